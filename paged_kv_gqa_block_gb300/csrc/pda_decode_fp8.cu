// pda_decode_fp8.cu -- instantiation and launch of the partition kernel for an fp8 e4m3 KV cache
// with one fp32 scale per token per KV head.
#include "pda_decode.cuh"
#include "pda_launch.cuh"

namespace pda {

int launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map, bool fused,
                      cudaStream_t stream) {
    // one-warp CTAs with a private ring of 4 KB stages (+128 B of scales).  QG <= 8: 3 stages and
    // 12 CTAs per SM (168 registers; 3 stages measured 2 % faster than 4 at the same occupancy,
    // and 13-15 CTAs per SM spill).  QG = 16: 4 stages, 8 CTAs per SM (the full register budget).
    if (fused) {
        if (a.QG <= 8) return launch_partition<PDA_KV_FP8_E4M3, 1, 3, 12, true>(a, kv_map, sc_map, stream);
        return launch_partition<PDA_KV_FP8_E4M3, 2, 4, 8, true>(a, kv_map, sc_map, stream);
    }
    if (a.QG <= 8) return launch_partition<PDA_KV_FP8_E4M3, 1, 3, 12, false>(a, kv_map, sc_map, stream);
    return launch_partition<PDA_KV_FP8_E4M3, 2, 4, 8, false>(a, kv_map, sc_map, stream);
}

}  // namespace pda
