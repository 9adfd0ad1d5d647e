// pda_noalloc.cu -- a decode step (partition pass + reduce) for callers that cannot allocate
// device memory: the partials live in a fixed array inside this library instead of in a
// caller-provided workspace.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pda.h"

namespace pda {

// The partials of one step: partial_out, then exp_sums, then max_logits.  Every GPU that loads
// this library holds the array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PDA_NOALLOC_SCRATCH_BYTES];

// Device address of the array, looked up once per device.  In host code the array's name is only
// a host-side stand-in, so the kernels must be given this address instead.
static void* scratch_address_for_current_device(int* status) {
    static void* addr[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *status = PDA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            *status = PDA_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    *status = PDA_OK;
    return addr[dev];
}

static long long round_up_256(long long x) { return (x + 255) / 256 * 256; }

}  // namespace pda

extern "C" int pda_decode_step_noalloc(const pda_plan_t* plan, const void* query, const void* kv_cache,
                                       long long num_cache_blocks, const int* block_table, const int* context_lens,
                                       void* out, int out_dtype, int* err_word, void* stream) {
    if (!plan || pda_workspace_size(plan) < 0) return PDA_ERR_INVALID_ARG;
    if (plan->kv_dtype == PDA_KV_TQ4) return PDA_ERR_INVALID_ARG;   // TQ4 needs its centroids (pda_decode_tq4)
    if (plan->num_seqs == 0) return PDA_OK;
    const long long rows = (long long)plan->num_seqs * plan->num_kv_heads * plan->num_partitions *
                           plan->query_group_size;
    const long long partial_bytes = pda::round_up_256(rows * plan->head_dim * 4);
    const long long stat_bytes = pda::round_up_256(rows * 4);
    if (partial_bytes + 2 * stat_bytes > PDA_NOALLOC_SCRATCH_BYTES) return PDA_ERR_WORKSPACE_TOO_SMALL;
    int rc = PDA_OK;
    unsigned char* base = static_cast<unsigned char*>(pda::scratch_address_for_current_device(&rc));
    if (rc != PDA_OK) return rc;
    float* partial_out = reinterpret_cast<float*>(base);
    float* exp_sums = reinterpret_cast<float*>(base + partial_bytes);
    float* max_logits = reinterpret_cast<float*>(base + partial_bytes + stat_bytes);
    rc = pda_decode(plan, query, kv_cache, num_cache_blocks, block_table, context_lens, partial_out, exp_sums,
                    max_logits, err_word, stream);
    if (rc != PDA_OK) return rc;
    return pda_reduce(plan, context_lens, partial_out, exp_sums, max_logits, out, out_dtype, err_word, stream);
}
