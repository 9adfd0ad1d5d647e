// pda_launch.cuh -- grid sizing and launch of one instance of the partition kernel.
#pragma once

#include <mutex>

#include "pda.h"
#include "pda_decode.cuh"

namespace pda {

// Persistent grid of one-warp CTAs: (SMs x resident CTAs per SM), capped by the number of units.
template <int KV, int NT, int S, int MINB, bool FUSED>
int launch_partition(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map, cudaStream_t stream) {
    using Cfg = DecodeCfg<KV, S>;
    auto kernel = pda_partition_kernel<KV, NT, S, MINB, FUSED>;
    static int occ_cache[64] = {0};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PDA_ERR_CUDA;
    int occ;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (occ_cache[dev] == 0) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes) !=
                cudaSuccess)
                return PDA_ERR_LAUNCH;
            int o = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, Cfg::kThreads, Cfg::kSmemBytes) !=
                    cudaSuccess ||
                o < 1)
                return PDA_ERR_LAUNCH;
            occ_cache[dev] = o;
        }
        occ = occ_cache[dev];
    }
    const int sms = device_sm_count();
    if (sms <= 0) return PDA_ERR_CUDA;
    const long long units = (long long)a.B * a.Hk * a.P;
    long long grid = (long long)sms * occ;
    if (grid > units) grid = units;
    if (grid < 1) return PDA_OK;
    DecodeArgs af = a;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    // programmatic dependent launch: the prologue may overlap the tail of the previous grid; the
    // kernel waits for that grid before it reads any input
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (FUSED) {
        // the fused step ends with a grid barrier: a cooperative launch keeps every CTA resident
        // (the grid is at most the resident CTAs), and the barrier counts in this launch's slot
        int rc = PDA_OK;
        af.sched = launch_counter_slot(&rc);
        if (rc != PDA_OK) return rc;
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, kv_map, sc_map, af) == cudaSuccess ? PDA_OK : PDA_ERR_LAUNCH;
}

}  // namespace pda
