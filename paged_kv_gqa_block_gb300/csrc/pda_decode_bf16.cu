// pda_decode_bf16.cu -- instantiation and launch of the partition kernel for a bf16 KV cache.
#include <mutex>

#include "pda_decode.cuh"
#include "pda_launch.cuh"
#include "pda_rows.cuh"

namespace pda {

int launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& kv_map, bool fused, cudaStream_t stream) {
    // one-warp CTAs with a private ring of 8 KB stages.  QG <= 8: 3 stages and 8 CTAs per SM,
    // or, for a small batch of 256-token partitions (at most 2048 units: every warp then streams
    // one short partition and waits on its copies more than it computes), 4 stages and 6 CTAs
    // per SM.  QG = 16: 4 stages, 6 CTAs per SM (the row-half kernel below is the faster layout
    // for QG = 16 when the step has enough units).
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

// Persistent grid of row-half CTAs for QG = 16: (SMs x resident CTAs per SM), each CTA one
// producer warp and two consumer warps of 8 query rows; units taken from a per-launch counter
// slot in the head-group order with groups of one head.
template <int S, int MINB>
static int launch_rows(const DecodeArgs& a, const CUtensorMap& kv_map, cudaStream_t stream) {
    auto kernel = pda_rows_kernel<S, MINB>;
    static int occ_cache[64] = {0};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PDA_ERR_CUDA;
    if (a.QG != 8 * kRowsConsumers) return PDA_ERR_INVALID_ARG;
    const int threads = 32 * (kRowsConsumers + 1), smem = rows_smem_bytes(S);
    int occ;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (occ_cache[dev] == 0) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
                return PDA_ERR_LAUNCH;
            int o = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, threads, smem) != cudaSuccess || o < 1)
                return PDA_ERR_LAUNCH;
            occ_cache[dev] = o;
        }
        occ = occ_cache[dev];
    }
    const int sms = device_sm_count();
    if (sms <= 0) return PDA_ERR_CUDA;
    int rc = PDA_OK;
    DecodeArgs ar = a;
    ar.HG = 1;   // the unit order of head groups of one head
    ar.sched = launch_counter_slot(&rc);
    if (rc != PDA_OK) return rc;
    const long long units = (long long)a.B * a.Hk * a.P;
    long long grid = (long long)sms * occ;
    if (grid > units) grid = units;
    if (grid < 1) return PDA_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, kv_map, ar) == cudaSuccess ? PDA_OK : PDA_ERR_LAUNCH;
}

int launch_decode_bf16_rows(const DecodeArgs& a, const CUtensorMap& kv_map, cudaStream_t stream) {
    // 6 stages of 8 KB and four CTAs per SM (167 registers, no spills): eight consumer warps per
    // SM against the head-warp kernel's six, the same 192 KB in flight
    return launch_rows<6, 4>(a, kv_map, stream);
}

}  // namespace pda
