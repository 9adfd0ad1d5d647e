// pda_decode_tq4.cu -- instantiation and launch of the partition kernel for a TQ4 cache (4-bit K
// codes into 16 centroids with a per-token norm, 4-bit V codes with a per-token scale and zero).
#include "pda_decode.cuh"
#include "pda_launch.cuh"

namespace pda {

int launch_decode_tq4(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map, cudaStream_t stream) {
    // one-warp CTAs with a private ring of S = 6 stages of 2 KB (+96 B of fields): the same
    // bytes in flight per warp as fp8's 4 stages would need twice the tiles; 12 CTAs per SM
    // for QG <= 8, 8 for QG = 16
    if (a.QG <= 8) return launch_partition<PDA_KV_TQ4, 1, 6, 12, false>(a, kv_map, sc_map, stream);
    return launch_partition<PDA_KV_TQ4, 2, 6, 8, false>(a, kv_map, sc_map, stream);
}

}  // namespace pda
