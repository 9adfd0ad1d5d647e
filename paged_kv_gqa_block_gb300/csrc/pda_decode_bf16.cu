// pda_decode_bf16.cu -- instantiation and launch of the partition kernel for a bf16 KV cache.
#include "pda_decode.cuh"
#include "pda_launch.cuh"

namespace pda {

int launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& kv_map, cudaStream_t stream) {
    // one-warp CTAs with a private ring of S = 4 stages of 8 KB
    if (a.QG <= 8) return launch_partition<false, 1, 4>(a, kv_map, kv_map, stream);
    return launch_partition<false, 2, 4>(a, kv_map, kv_map, stream);
}

}  // namespace pda
