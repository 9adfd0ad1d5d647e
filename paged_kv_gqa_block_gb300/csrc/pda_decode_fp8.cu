// pda_decode_fp8.cu -- instantiation and launch of the partition kernel for an fp8 e4m3 KV cache
// with one fp32 scale per token per KV head.
#include "pda_decode.cuh"
#include "pda_launch.cuh"

namespace pda {

int launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map, bool fused,
                      cudaStream_t stream) {
    // one-warp CTAs with a private ring of S = 4 stages of 4 KB (+128 B of scales); 12 CTAs per SM
    // for QG <= 8 (168 registers), 8 for QG = 16 (which needs the full register budget)
    if (fused) {
        if (a.QG <= 8) return launch_partition<PDA_KV_FP8_E4M3, 1, 4, 12, true>(a, kv_map, sc_map, stream);
        return launch_partition<PDA_KV_FP8_E4M3, 2, 4, 8, true>(a, kv_map, sc_map, stream);
    }
    if (a.QG <= 8) return launch_partition<PDA_KV_FP8_E4M3, 1, 4, 12, false>(a, kv_map, sc_map, stream);
    return launch_partition<PDA_KV_FP8_E4M3, 2, 4, 8, false>(a, kv_map, sc_map, stream);
}

}  // namespace pda
