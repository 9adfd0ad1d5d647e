// pda_api.cu -- host side of libpda: pda_plan, argument checks, tensor-map encoding, launches,
// and the reduce kernel that combines the partition partials.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pda.h"
#include "pda_internal.h"
#include "pda_ptx.cuh"
#include "pda_merge.cuh"

namespace pda {

constexpr int kMaxReduceWarps = 16;   // query rows of a unit (QG <= 16)

// ------------------------------------------------------------------------- reduce kernel
// One CTA per (sequence, KV head) unit, one warp per query row; the unit's partials stream through
// shared memory by bulk copies (merge_unit_smem, pda_merge.cuh).  Launched as a programmatic
// dependent of the partition pass: it waits for that grid before reading anything.
__global__ void __launch_bounds__(kMaxReduceWarps * 32, 1) pda_reduce_kernel(const ReduceArgs r) {
    extern __shared__ __align__(128) float reduce_smem[];
    __shared__ __align__(8) uint64_t bars[4];   // full[2], empty[2]
    // Everything this kernel reads, the context lengths included, is read after the wait: a kernel
    // that ran before the partition pass (an append, or an in-place ctx += 1) may still be in
    // flight when this grid is scheduled, and only the wait orders its writes before these reads.
    grid_dependency_wait();
    const int b = (int)(blockIdx.x / r.Hk), h = (int)(blockIdx.x - (unsigned)b * r.Hk);
    int ctx = r.context_lens[b];
    if (ctx < 0 || ctx > r.MB * r.BS) {
        if (h == 0 && threadIdx.x == 0 && r.err_word) atomicOr(r.err_word, PDA_ERRW_BAD_CONTEXT_LEN);
        ctx = 0;
    }
    const uint32_t bar0 = smem_addr(bars);
    if (threadIdx.x == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        mbar_init(bar0 + 16, (uint32_t)r.QG);
        mbar_init(bar0 + 24, (uint32_t)r.QG);
        fence_mbar_init();
    }
    __syncthreads();
    const MergeArgs m{r.partial_out, r.exp_sums, r.max_logits, r.out, r.Hk, r.QG, r.P, r.W, r.out_f32};
    bool timed_out = false;
    merge_unit_smem(m, b, h, ctx, reduce_smem, bar0, &timed_out);
    if (timed_out && (threadIdx.x & 31) == 0 && r.err_word) atomicOr(r.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
}

static int reduce_smem_bytes(int QG) { return 2 * kMergeChunk * QG * kHeadDim * 4; }

int launch_reduce(const ReduceArgs& r, cudaStream_t stream) {
    static bool attr_set[64] = {false};   // the shared-memory limit, set once per device
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PDA_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(pda_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     reduce_smem_bytes(kMaxReduceWarps)) != cudaSuccess)
                return PDA_ERR_LAUNCH;
            attr_set[dev] = true;
        }
    }
    const long long ctas = (long long)r.B * r.Hk;
    if (ctas > 0x7FFFFFFFll || r.QG > kMaxReduceWarps) return PDA_ERR_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(r.QG * 32);
    cfg.dynamicSmemBytes = reduce_smem_bytes(r.QG);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pda_reduce_kernel, r) == cudaSuccess ? PDA_OK : PDA_ERR_LAUNCH;
}

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

// ------------------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Bytes of K and V of one token of one KV head: 512 (bf16), 256 (fp8), 128 (TQ4 4-bit codes).
static long long token_head_bytes(int kv_dtype) {
    return kv_dtype == PDA_KV_BF16 ? 4ll * kHeadDim : kv_dtype == PDA_KV_FP8_E4M3 ? 2ll * kHeadDim : (long long)kHeadDim;
}

// K|V bytes of one 16-token tile of one KV head (or of heads_per_box consecutive heads).
// Dimensions (innermost first):
//   {128 bytes of a chunk, BS slots, chunks per token-head, Hk heads, NB blocks}
// with strides {-, Hk*token_head_bytes, 128, token_head_bytes, cache_block_bytes}.  The box
// {128, 16, chunks, heads_per_box, 1} lands as [head][chunk][token][128 B] in shared memory,
// 128-byte swizzle.
static bool encode_kv_map(CUtensorMap* m, const void* cache, const pda_plan_t* p, long long nb, int heads_per_box = 1) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t thb = (cuuint64_t)token_head_bytes(p->kv_dtype);
    const cuuint32_t chunks = (cuuint32_t)(thb / 128);
    cuuint64_t dims[5] = {128, (cuuint64_t)p->kv_block_size, chunks, (cuuint64_t)p->num_kv_heads, (cuuint64_t)nb};
    cuuint64_t strides[4] = {(cuuint64_t)p->num_kv_heads * thb, 128, thb, (cuuint64_t)p->cache_block_bytes};
    cuuint32_t box[5] = {128, (cuuint32_t)kTileTokens, chunks, (cuuint32_t)heads_per_box, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    // L2 fetches are widened to 256 bytes, or to 128 for TQ4 whose token-head rows are 128 bytes
    // (256 would also bring the next head's row, which another warp may read much later)
    const CUtensorMapL2promotion promo = thb >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(cache), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Metadata of one 16-token tile: {BS slots, F fields, Hk heads, NB blocks} starting at the metadata
// region; box {16, F, heads_per_box, 1} lands as [head][field][token].  fp8: F = 2 fp32 fields (K scale, V scale);
// TQ4: F = 3 fp16 fields (k_norm, v_scale, v_zero).
static bool encode_scale_map(CUtensorMap* m, const void* cache, const pda_plan_t* p, long long nb,
                             int heads_per_box = 1) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const bool tq = p->kv_dtype == PDA_KV_TQ4;
    const cuuint64_t fields = tq ? 3 : 2, esz = tq ? 2 : 4;
    const char* base = static_cast<const char*>(cache) + p->meta_offset_bytes;
    cuuint64_t dims[4] = {(cuuint64_t)p->kv_block_size, fields, (cuuint64_t)p->num_kv_heads, (cuuint64_t)nb};
    cuuint64_t strides[3] = {(cuuint64_t)p->kv_block_size * esz, (cuuint64_t)p->kv_block_size * esz * fields,
                             (cuuint64_t)p->cache_block_bytes};
    cuuint32_t box[4] = {(cuuint32_t)kTileTokens, (cuuint32_t)fields, (cuuint32_t)heads_per_box, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, tq ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<char*>(base),
              dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------- plan
static int compute_plan(const pda_plan_t* in, pda_plan_t* out) {
    *out = *in;
    if (in->num_seqs < 0 || in->num_kv_heads < 1 || in->max_blocks_per_seq < 1 || in->tile_groups_per_partition < 0 ||
        in->max_partitions < 0 || in->wait_timeout_ns < 0 || in->kernel_variant < PDA_VARIANT_AUTO ||
        in->kernel_variant > PDA_VARIANT_ROW_HALVES)
        return PDA_ERR_INVALID_ARG;
    if (in->query_group_size != 6 && in->query_group_size != 8 && in->query_group_size != 16)
        return PDA_ERR_UNSUPPORTED;
    if (in->kv_block_size != 16 && in->kv_block_size != 32) return PDA_ERR_UNSUPPORTED;
    if (in->head_dim != kHeadDim) return PDA_ERR_UNSUPPORTED;
    if (in->kv_dtype != PDA_KV_BF16 && in->kv_dtype != PDA_KV_FP8_E4M3 && in->kv_dtype != PDA_KV_TQ4)
        return PDA_ERR_UNSUPPORTED;
    if (in->kernel_variant == PDA_VARIANT_HEAD_GROUPS && in->kv_dtype != PDA_KV_FP8_E4M3) return PDA_ERR_UNSUPPORTED;
    if (in->kernel_variant == PDA_VARIANT_ROW_HALVES && (in->kv_dtype != PDA_KV_BF16 || in->query_group_size != 16))
        return PDA_ERR_UNSUPPORTED;
    if (!std::isfinite(in->softmax_scale)) return PDA_ERR_INVALID_ARG;
    const long long max_ctx = (long long)in->max_blocks_per_seq * in->kv_block_size;
    if (max_ctx > (1ll << 30)) return PDA_ERR_INVALID_ARG;   // context lengths are int32
    long long G = in->tile_groups_per_partition;
    if (G == 0)
        G = in->max_partitions <= 0 ? 1
                                    : (max_ctx + (long long)kTokensPerTileGroup * in->max_partitions - 1) /
                                          ((long long)kTokensPerTileGroup * in->max_partitions);
    if (G < 1) G = 1;
    if (G * kTokensPerTileGroup > (1ll << 30)) return PDA_ERR_INVALID_ARG;
    const long long W = G * kTokensPerTileGroup;
    const long long P = (max_ctx + W - 1) / W;
    // index ranges used by the kernels: units and tiles of a step in int64, grid and rows in int32
    const long long units = (long long)in->num_seqs * in->num_kv_heads * P;
    if ((long long)in->num_seqs * in->num_kv_heads > (1ll << 31) - 1 || units * in->query_group_size > (1ll << 40))
        return PDA_ERR_INVALID_ARG;
    const long long data = (long long)in->kv_block_size * in->num_kv_heads * token_head_bytes(in->kv_dtype);
    const long long meta = in->kv_dtype == PDA_KV_BF16     ? 0
                           : in->kv_dtype == PDA_KV_FP8_E4M3 ? (long long)in->num_kv_heads * 2 * in->kv_block_size * 4
                                                             : (long long)in->num_kv_heads * 3 * in->kv_block_size * 2;
    out->num_partitions = (int)P;
    out->partition_tokens = (int)W;
    out->resolved_tile_groups = (int)G;
    out->resolved_softmax_scale = in->softmax_scale > 0.f ? in->softmax_scale : 1.0f / std::sqrt((float)kHeadDim);
    out->cache_block_bytes = data + meta;
    out->meta_offset_bytes = data;
    out->workspace_bytes = units * in->query_group_size * (kHeadDim * 4 + 8);
    return PDA_OK;
}

static bool plan_matches(const pda_plan_t* p) {
    pda_plan_t chk;
    if (compute_plan(p, &chk) != PDA_OK) return false;
    return chk.num_partitions == p->num_partitions && chk.partition_tokens == p->partition_tokens &&
           chk.resolved_tile_groups == p->resolved_tile_groups &&
           chk.resolved_softmax_scale == p->resolved_softmax_scale && chk.cache_block_bytes == p->cache_block_bytes &&
           chk.meta_offset_bytes == p->meta_offset_bytes && chk.workspace_bytes == p->workspace_bytes;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pda

using namespace pda;

extern "C" {

int pda_plan(pda_plan_t* plan) {
    if (!plan) return PDA_ERR_INVALID_ARG;
    pda_plan_t out;
    const int rc = compute_plan(plan, &out);
    if (rc == PDA_OK) *plan = out;
    return rc;
}

}  // extern "C"

namespace pda {
// Head groups (fp8) when asked for, or, with PDA_VARIANT_AUTO, when the groups hold 4 heads and
// the plan has room for at least two (sequence, head group, partition) units per resident CTA
// (two per SM); otherwise head warps.
static bool use_head_groups(const pda_plan_t* plan) {
    if (plan->kernel_variant != PDA_VARIANT_AUTO) return plan->kernel_variant == PDA_VARIANT_HEAD_GROUPS;
    const int HG = group_heads(plan->num_kv_heads);
    if (HG < 4) return false;
    const long long units = (long long)plan->num_seqs * (plan->num_kv_heads / HG) * plan->num_partitions;
    return units >= 2ll * 2 * device_sm_count();
}

// Row halves (bf16, QG 16) when asked for, or, with PDA_VARIANT_AUTO, when the plan has room for
// at least two (sequence, KV head, partition) units per resident row-half CTA (four per SM).
static bool use_row_halves(const pda_plan_t* plan) {
    if (plan->kernel_variant != PDA_VARIANT_AUTO) return plan->kernel_variant == PDA_VARIANT_ROW_HALVES;
    if (plan->kv_dtype != PDA_KV_BF16 || plan->query_group_size != 16) return false;
    const long long units = (long long)plan->num_seqs * plan->num_kv_heads * plan->num_partitions;
    return units >= 2ll * 4 * device_sm_count();
}

// The partition pass; with `fused`, the same (cooperative) launch also combines the partials
// into `out` after a grid barrier (`counters` is reserved and left untouched).
static int decode_launch(const pda_plan_t* plan, const void* query, const void* kv_cache, long long num_cache_blocks,
                         const int* block_table, const int* context_lens, float* partial_out, float* exp_sums,
                         float* max_logits, int* err_word, void* stream, bool fused, int* counters, void* out,
                         int out_dtype, const float* centroids) {
    if (!plan || !plan_matches(plan)) return PDA_ERR_INVALID_ARG;
    // a TQ4 cache is read only with its centroids (pda_decode_tq4), and only by the two-launch path
    const bool tq = plan->kv_dtype == PDA_KV_TQ4;
    if (tq != (centroids != nullptr) || (tq && fused) || ((uintptr_t)centroids & 3u)) return PDA_ERR_INVALID_ARG;
    if (fused && out_dtype != PDA_OUT_BF16 && out_dtype != PDA_OUT_F32) return PDA_ERR_INVALID_ARG;
    if (plan->num_seqs == 0) return PDA_OK;
    if (!query || !kv_cache || !block_table || !context_lens || !partial_out || !exp_sums || !max_logits)
        return PDA_ERR_INVALID_ARG;
    if (fused && (!counters || !out || ((uintptr_t)counters & 3u) ||
                  ((uintptr_t)out & (out_dtype == PDA_OUT_F32 ? 15u : 7u))))
        return PDA_ERR_INVALID_ARG;
    if (num_cache_blocks < 1 || num_cache_blocks > (1ll << 31) - 1) return PDA_ERR_INVALID_ARG;
    if (!aligned16(query) || !aligned16(kv_cache) || !aligned16(partial_out)) return PDA_ERR_INVALID_ARG;
    if (((uintptr_t)exp_sums & 3u) || ((uintptr_t)max_logits & 3u) || ((uintptr_t)block_table & 3u) ||
        ((uintptr_t)context_lens & 3u) || ((uintptr_t)err_word & 3u))
        return PDA_ERR_INVALID_ARG;

    DecodeArgs a;
    a.query = static_cast<const uint16_t*>(query);
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.centroids = centroids;
    a.partial_out = partial_out;
    a.exp_sums = exp_sums;
    a.max_logits = max_logits;
    a.err_word = err_word;
    a.num_cache_blocks = num_cache_blocks;
    a.B = plan->num_seqs;
    a.Hk = plan->num_kv_heads;
    a.QG = plan->query_group_size;
    a.MB = plan->max_blocks_per_seq;
    a.BS = plan->kv_block_size;
    a.P = plan->num_partitions;
    a.W = plan->partition_tokens;
    a.bs_shift = plan->kv_block_size == 32 ? 5 : 4;
    a.qk_scale_log2 = plan->resolved_softmax_scale * 1.4426950408889634f;
    a.timeout_ns = plan->wait_timeout_ns > 0 ? (unsigned long long)plan->wait_timeout_ns : kDefaultTimeoutNs;
    a.counters = counters;
    a.out = out;
    a.out_f32 = out_dtype == PDA_OUT_F32;

    a.HG = 1;
    a.sched = nullptr;
    CUtensorMap kv_map, sc_map;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan->kv_dtype == PDA_KV_FP8_E4M3 && use_head_groups(plan)) {
        a.HG = group_heads(plan->num_kv_heads);
        if (!encode_kv_map(&kv_map, kv_cache, plan, num_cache_blocks, a.HG) ||
            !encode_scale_map(&sc_map, kv_cache, plan, num_cache_blocks, a.HG))
            return PDA_ERR_LAUNCH;
        return launch_decode_fp8_groups(a, kv_map, sc_map, fused, s);
    }
    if (!encode_kv_map(&kv_map, kv_cache, plan, num_cache_blocks)) return PDA_ERR_LAUNCH;
    if (plan->kv_dtype == PDA_KV_BF16 && !fused && use_row_halves(plan)) return launch_decode_bf16_rows(a, kv_map, s);
    if (plan->kv_dtype == PDA_KV_BF16) return launch_decode_bf16(a, kv_map, fused, s);
    if (!encode_scale_map(&sc_map, kv_cache, plan, num_cache_blocks)) return PDA_ERR_LAUNCH;
    if (tq) return launch_decode_tq4(a, kv_map, sc_map, s);
    return launch_decode_fp8(a, kv_map, sc_map, fused, s);
}
}  // namespace pda

extern "C" {

int pda_decode(const pda_plan_t* plan, const void* query, const void* kv_cache, long long num_cache_blocks,
               const int* block_table, const int* context_lens, float* partial_out, float* exp_sums,
               float* max_logits, int* err_word, void* stream) {
    return decode_launch(plan, query, kv_cache, num_cache_blocks, block_table, context_lens, partial_out, exp_sums,
                         max_logits, err_word, stream, false, nullptr, nullptr, PDA_OUT_BF16, nullptr);
}

int pda_decode_tq4(const pda_plan_t* plan, const void* query, const void* kv_cache, long long num_cache_blocks,
                   const float* centroids, const int* block_table, const int* context_lens, float* partial_out,
                   float* exp_sums, float* max_logits, int* err_word, void* stream) {
    if (!plan || plan->kv_dtype != PDA_KV_TQ4 || !centroids) return PDA_ERR_INVALID_ARG;
    return decode_launch(plan, query, kv_cache, num_cache_blocks, block_table, context_lens, partial_out, exp_sums,
                         max_logits, err_word, stream, false, nullptr, nullptr, PDA_OUT_BF16, centroids);
}

int pda_decode_fused(const pda_plan_t* plan, const void* query, const void* kv_cache, long long num_cache_blocks,
                     const int* block_table, const int* context_lens, float* partial_out, float* exp_sums,
                     float* max_logits, int* counters, void* out, int out_dtype, int* err_word, void* stream) {
    return decode_launch(plan, query, kv_cache, num_cache_blocks, block_table, context_lens, partial_out, exp_sums,
                         max_logits, err_word, stream, true, counters, out, out_dtype, nullptr);
}

int pda_reduce(const pda_plan_t* plan, const int* context_lens, const float* partial_out, const float* exp_sums,
               const float* max_logits, void* out, int out_dtype, int* err_word, void* stream) {
    if (!plan || !plan_matches(plan)) return PDA_ERR_INVALID_ARG;
    if (out_dtype != PDA_OUT_BF16 && out_dtype != PDA_OUT_F32) return PDA_ERR_INVALID_ARG;
    if (plan->num_seqs == 0) return PDA_OK;
    if (!context_lens || !partial_out || !exp_sums || !max_logits || !out) return PDA_ERR_INVALID_ARG;
    if (!aligned16(partial_out) || ((uintptr_t)out & (out_dtype == PDA_OUT_F32 ? 15u : 7u)) ||
        ((uintptr_t)exp_sums & 3u) || ((uintptr_t)max_logits & 3u) || ((uintptr_t)context_lens & 3u) ||
        ((uintptr_t)err_word & 3u))
        return PDA_ERR_INVALID_ARG;
    ReduceArgs r;
    r.context_lens = context_lens;
    r.partial_out = partial_out;
    r.exp_sums = exp_sums;
    r.max_logits = max_logits;
    r.out = out;
    r.err_word = err_word;
    r.B = plan->num_seqs;
    r.Hk = plan->num_kv_heads;
    r.QG = plan->query_group_size;
    r.MB = plan->max_blocks_per_seq;
    r.BS = plan->kv_block_size;
    r.P = plan->num_partitions;
    r.W = plan->partition_tokens;
    r.out_f32 = out_dtype == PDA_OUT_F32;
    return launch_reduce(r, static_cast<cudaStream_t>(stream));
}

const char* pda_status_string(int status) {
    switch (status) {
        case PDA_OK: return "PDA_OK";
        case PDA_ERR_INVALID_ARG: return "PDA_ERR_INVALID_ARG";
        case PDA_ERR_UNSUPPORTED: return "PDA_ERR_UNSUPPORTED";
        case PDA_ERR_WORKSPACE_TOO_SMALL: return "PDA_ERR_WORKSPACE_TOO_SMALL";
        case PDA_ERR_LAUNCH: return "PDA_ERR_LAUNCH";
        case PDA_ERR_NOT_IMPLEMENTED: return "PDA_ERR_NOT_IMPLEMENTED";
        case PDA_ERR_CUDA: return "PDA_ERR_CUDA";
        default: return "PDA_ERR_UNKNOWN";
    }
}

long long pda_workspace_size(const pda_plan_t* plan) {
    if (!plan || !plan_matches(plan)) return -1;
    return plan->workspace_bytes;
}

int pda_plan_struct_size(void) { return (int)sizeof(pda_plan_t); }

int pda_kernel_variant(const pda_plan_t* plan) {
    if (!plan || !plan_matches(plan)) return PDA_ERR_INVALID_ARG;
    const bool rows_possible = plan->kv_dtype == PDA_KV_BF16 && plan->query_group_size == 16;
    if (plan->kv_dtype != PDA_KV_FP8_E4M3 && !rows_possible) return PDA_VARIANT_HEAD_WARPS;
    if (plan->kernel_variant == PDA_VARIANT_AUTO && device_sm_count() <= 0) return PDA_ERR_CUDA;
    if (rows_possible) return use_row_halves(plan) ? PDA_VARIANT_ROW_HALVES : PDA_VARIANT_HEAD_WARPS;
    return use_head_groups(plan) ? PDA_VARIANT_HEAD_GROUPS : PDA_VARIANT_HEAD_WARPS;
}

}  // extern "C"
