// pda_decode_bf16.cu -- instantiation and launch of the partition kernel for a bf16 KV cache.
#include "pda_decode.cuh"
#include "pda_launch.cuh"

namespace pda {

int launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& kv_map, bool fused, cudaStream_t stream) {
    // one-warp CTAs with a private ring of 8 KB stages.  QG <= 8: 3 stages and 8 CTAs per SM,
    // or, for a small batch of 256-token partitions (at most 2048 units: every warp then streams
    // one short partition and waits on its copies more than it computes), 4 stages and 6 CTAs
    // per SM.  QG = 16: 4 stages, 6 CTAs per SM.
    const bool short_units = a.W == kTokensPerTileGroup && (long long)a.B * a.Hk * a.P <= 2048;
    if (fused) {
        if (a.QG <= 8) return launch_partition<PDA_KV_BF16, 1, 3, 8, true>(a, kv_map, kv_map, stream);
        return launch_partition<PDA_KV_BF16, 2, 4, 1, true>(a, kv_map, kv_map, stream);
    }
    if (a.QG <= 8) {
        if (short_units) return launch_partition<PDA_KV_BF16, 1, 4, 6, false>(a, kv_map, kv_map, stream);
        return launch_partition<PDA_KV_BF16, 1, 3, 8, false>(a, kv_map, kv_map, stream);
    }
    return launch_partition<PDA_KV_BF16, 2, 4, 1, false>(a, kv_map, kv_map, stream);
}

}  // namespace pda
