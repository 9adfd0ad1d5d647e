// pda_decode_bf16.cu -- instantiation and launch of the partition kernel for a bf16 KV cache.
#include "pda_decode.cuh"
#include "pda_launch.cuh"

namespace pda {

int launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& kv_map, bool fused, cudaStream_t stream) {
    // one-warp CTAs with a private ring of S = 3 stages of 8 KB, 8 CTAs per SM (QG <= 8);
    // QG = 16: 4 stages, 6 CTAs per SM
    if (fused) {
        if (a.QG <= 8) return launch_partition<false, 1, 3, 8, true>(a, kv_map, kv_map, stream);
        return launch_partition<false, 2, 4, 1, true>(a, kv_map, kv_map, stream);
    }
    if (a.QG <= 8) return launch_partition<false, 1, 3, 8, false>(a, kv_map, kv_map, stream);
    return launch_partition<false, 2, 4, 1, false>(a, kv_map, kv_map, stream);
}

}  // namespace pda
