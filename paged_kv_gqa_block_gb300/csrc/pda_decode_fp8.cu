// pda_decode_fp8.cu -- instantiation and launch of the partition kernels for an fp8 e4m3 KV cache
// with one fp32 scale per token per KV head: head warps (pda_decode.cuh) and head groups
// (pda_group.cuh).
#include <atomic>
#include <mutex>

#include "pda_decode.cuh"
#include "pda_group.cuh"
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

// Per-launch counters: kSchedSlots slots of kSchedInts counters ({next unit, producers done} for
// the head-group partition pass; {next unit, -, -, -, CTAs done} for its fused step; {arrived,
// left} for the grid barrier of the head-warp fused step), every slot zero between launches (each
// launch's last CTA returns its slot to zero).  Each launch takes the next slot in turn, so
// launches in flight at the same time (on other streams) use different slots as long as fewer than
// kSchedSlots of them overlap.  The array lives in every GPU that loads the library.
constexpr int kSchedSlots = 256, kSchedInts = 8;
static __device__ unsigned int g_group_sched[kSchedInts * kSchedSlots];

// Device address of this launch's slot (the array's address is looked up once per device).
unsigned int* launch_counter_slot(int* status) {
    static unsigned int* base[64] = {nullptr};
    static std::mutex mu;
    static std::atomic<unsigned long long> seq{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *status = PDA_ERR_CUDA;
        return nullptr;
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!base[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_group_sched) != cudaSuccess || !p) {
                *status = PDA_ERR_CUDA;
                return nullptr;
            }
            base[dev] = static_cast<unsigned int*>(p);
        }
    }
    *status = PDA_OK;
    return base[dev] + kSchedInts * (int)(seq.fetch_add(1) % kSchedSlots);
}

int group_heads(int Hk) {
    for (int d = kGroupMaxHeads; d > 1; --d)
        if (Hk % d == 0) return d;
    return 1;
}

// Persistent grid of head-group CTAs: (SMs x resident CTAs per SM), each CTA one producer warp
// and a.HG consumer warps.
template <int NT, int S, int NWARPS, int MINB, bool FUSED>
static int launch_groups(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map,
                         cudaStream_t stream) {
    auto kernel = pda_group_kernel<NT, S, NWARPS, MINB, FUSED>;
    static int occ_cache[64][kGroupMaxHeads + 1] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PDA_ERR_CUDA;
    const int threads = 32 * (a.HG + 1);   // producer, HG consumers
    const int smem = group_smem_bytes(a.HG, S);
    if (a.HG < 1 || threads > 32 * NWARPS) return PDA_ERR_INVALID_ARG;
    int occ;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (occ_cache[dev][a.HG] == 0) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     group_smem_bytes(kGroupMaxHeads, S)) != cudaSuccess)
                return PDA_ERR_LAUNCH;
            int o = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, threads, smem) != cudaSuccess || o < 1)
                return PDA_ERR_LAUNCH;
            occ_cache[dev][a.HG] = o;
        }
        occ = occ_cache[dev][a.HG];
    }
    const int sms = device_sm_count();
    if (sms <= 0) return PDA_ERR_CUDA;
    int rc = PDA_OK;
    DecodeArgs ag = a;
    ag.sched = launch_counter_slot(&rc);
    if (rc != PDA_OK) return rc;
    const long long units = (long long)a.B * (a.Hk / a.HG) * a.P;
    long long grid = (long long)sms * occ;
    if (grid > units) grid = units;
    if (grid < 1) return PDA_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (FUSED) {   // the fused step ends with a grid barrier: every CTA must be resident
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, kv_map, sc_map, ag) == cudaSuccess ? PDA_OK : PDA_ERR_LAUNCH;
}

int launch_decode_fp8_groups(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map,
                             bool fused, cudaStream_t stream) {
    // up to 4 heads a CTA: two CTAs of up to 5 warps per SM, each with 6
    // stages of up to 17 KB (two independent producers per SM, whose consumers reach their unit
    // boundaries at different times, measured faster than one CTA of 8 heads with 6 stages of 33 KB)
    if (fused) {
        if (a.QG <= 8) return launch_groups<1, 6, 5, 2, true>(a, kv_map, sc_map, stream);
        return launch_groups<2, 6, 5, 2, true>(a, kv_map, sc_map, stream);
    }
    if (a.QG <= 8) return launch_groups<1, 6, 5, 2, false>(a, kv_map, sc_map, stream);
    return launch_groups<2, 6, 5, 2, false>(a, kv_map, sc_map, stream);
}

}  // namespace pda
