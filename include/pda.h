/*
 * pda.h -- C ABI of libpda: single-token decode attention over a paged KV cache with GQA
 * grouping ("paged decode attention"), for NVIDIA GB300 (sm_103a).
 *
 * One decode step, for every sequence b and KV head h: the query_group_size (QG) query rows
 * of head group h (query heads h*QG .. h*QG+QG-1) attend over the sequence's context
 * (context_lens[b] tokens), gathered through the block table in kv_block_size-token blocks.
 * The context is split FA-2 style into partitions of G*256 tokens; pda_decode computes one
 * partial per non-empty partition (normalised output, running max, sum of exponentials) and
 * pda_reduce combines the partials into the softmax-weighted sum of V.
 *
 * Source of the method: the vLLM "tq_decode" page (build_tq_decode_module and the kernel body
 * tq_decode_kernel): argument list, grid (sequence, KV head, partition), block-table walk,
 * partition split with tile_groups_per_partition, mask, online softmax and partial epilogue.
 * The KV element formats here are bf16, fp8 e4m3 with one fp32 scale per token per KV head, and
 * the page's own 4-bit format (TQ4: K codes into 16 centroids times a per-token norm, V codes
 * with a per-token scale and zero point; pda_decode_tq4).
 *
 * Conventions for every call
 *   - Pointers named "device" are device pointers owned by the caller; the library allocates
 *     nothing, frees nothing and keeps no per-call state.  Process-wide state: a cache of the
 *     driver's tensor-map encoder and of per-device occupancy figures, and, in every GPU that
 *     loads the library, two static arrays: 256 slots of per-launch counters, used by the fp8
 *     head-group kernel and by the fused step's grid barrier (each such launch takes the next
 *     slot in turn; the launch's last CTA returns it to zero, so a captured launch can be
 *     replayed; two launches whose slots coincide, one taken 256 such launches after the other,
 *     must not overlap on the GPU, and a graph replay keeps the slot taken at capture), and the
 *     64 MiB array of pda_decode_step_noalloc.  The first such launch on a device looks up the
 *     slots' address; make it before any stream capture, and make no launch on a device after
 *     cudaDeviceReset in the same process.
 *   - Launches are asynchronous on the caller's stream (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).  Calls that share output or workspace buffers race
 *     if they overlap on the GPU.
 *   - Every call returns a pda_status.  Argument errors are reported before anything is
 *     launched.  Errors found in the data on the device (a context length or a block id out
 *     of range, a pipeline wait that timed out) never fault or trap: the kernel sets a bit
 *     in the optional device word *err_word (atomicOr) and carries on with the rule stated
 *     at pda_decode; the caller reads the word after synchronising.
 */
#ifndef PDA_H
#define PDA_H

#if defined(__GNUC__)
#define PDA_API __attribute__((visibility("default")))
#else
#define PDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pda_status {
    PDA_OK = 0,
    PDA_ERR_INVALID_ARG = -1,         /* null pointer, bad size, misaligned buffer, edited plan */
    PDA_ERR_UNSUPPORTED = -2,         /* QG not in {6,8,16}, BS not in {16,32}, head_dim != 128 */
    PDA_ERR_WORKSPACE_TOO_SMALL = -3, /* a size passed with a buffer is below the plan's need */
    PDA_ERR_LAUNCH = -4,              /* the CUDA launch (or tensor-map encode) failed */
    PDA_ERR_NOT_IMPLEMENTED = -5,
    PDA_ERR_CUDA = -6                 /* a CUDA runtime query failed (no device, ...) */
} pda_status;

enum { PDA_KV_BF16 = 0, PDA_KV_FP8_E4M3 = 1, PDA_KV_TQ4 = 2 };
enum { PDA_OUT_BF16 = 0, PDA_OUT_F32 = 1 };
enum { PDA_VARIANT_AUTO = 0, PDA_VARIANT_HEAD_WARPS = 1, PDA_VARIANT_HEAD_GROUPS = 2, PDA_VARIANT_ROW_HALVES = 3 };

/* Bits of the device error word. */
enum {
    PDA_ERRW_BAD_CONTEXT_LEN = 1,   /* context_lens[b] < 0 or > max_blocks_per_seq*kv_block_size */
    PDA_ERRW_BAD_BLOCK_ID = 2,      /* a block-table entry used by the context is outside [0, NB) */
    PDA_ERRW_PIPELINE_TIMEOUT = 4,  /* a bounded wait inside the kernel gave up */
    PDA_ERRW_BAD_POSITION = 8       /* pda_append_kv: a position >= max_blocks_per_seq*kv_block_size */
};

/*
 * Problem description.  The caller fills the input fields and calls pda_plan, which checks
 * them and fills the output fields.  The launch calls recompute the outputs from the inputs
 * and reject a plan whose outputs were edited (PDA_ERR_INVALID_ARG).
 * Field names follow build_tq_decode_module's arguments.
 */
typedef struct pda_plan_t {
    /* ---- inputs ---- */
    int num_seqs;                  /* B >= 0 (0 = nothing to do)                                  */
    int num_kv_heads;              /* Hk >= 1                                                      */
    int query_group_size;          /* QG = query heads / KV heads, one of 6, 8, 16                */
    int head_dim;                  /* D, must be 128                                              */
    int kv_block_size;             /* BS tokens per cache block, 16 or 32                         */
    int max_blocks_per_seq;        /* MB, row length of the block table, >= 1                     */
    int tile_groups_per_partition; /* G >= 1, or 0 = smallest G with num_partitions <= max_partitions */
    int max_partitions;            /* cap used when G == 0 (0 = no cap, i.e. G = 1)              */
    int kv_dtype;                  /* PDA_KV_BF16, PDA_KV_FP8_E4M3 or PDA_KV_TQ4                  */
    float softmax_scale;           /* <= 0 selects 1/sqrt(head_dim)                                */
    int wait_timeout_ns;           /* limit of each bounded wait inside pda_decode's kernel, in
                                      nanoseconds; 0 = 1 s.  A wait that gives up sets
                                      PDA_ERRW_PIPELINE_TIMEOUT.  Copies already in flight are
                                      always waited for (up to 1 s) before a warp leaves.  No
                                      counterpart on the pages; small values exist for testing
                                      the timeout path.                                          */
    int kernel_variant;            /* how pda_decode lays out the partition pass on the GPU (the
                                      results agree within the parity tolerances; each variant is
                                      deterministic on its own):
                                        PDA_VARIANT_AUTO (0): chosen at launch from the shape
                                          (head groups for fp8 and row halves for bf16 with
                                          query_group_size 16 when the plan has at least two
                                          units per resident CTA, else head warps),
                                        PDA_VARIANT_HEAD_WARPS (1): one warp per (sequence, KV head,
                                          partition) unit, any format,
                                        PDA_VARIANT_HEAD_GROUPS (2): one CTA per (sequence, group of
                                          up to 4 KV heads, partition) unit, fp8 e4m3 only,
                                        PDA_VARIANT_ROW_HALVES (3): one CTA per (sequence, KV head,
                                          partition) unit, its 16 query rows split between two
                                          warps, bf16 with query_group_size 16 only (the
                                          partials equal head warps' bit for bit).
                                      pda_decode_fused runs head groups where pda_decode would,
                                      else head warps.  No counterpart on the pages.              */
    /* ---- outputs of pda_plan ---- */
    int num_partitions;            /* P = ceil(MB*BS / W)                                          */
    int partition_tokens;          /* W = G * 256                                                 */
    int resolved_tile_groups;      /* G actually used                                              */
    float resolved_softmax_scale;
    long long cache_block_bytes;   /* bytes per cache block (data region + metadata region)       */
    long long meta_offset_bytes;   /* offset of the metadata region inside a block                */
    long long workspace_bytes;     /* bytes of partial_out + exp_sums + max_logits                 */
} pda_plan_t;

/*
 * pda_plan -- host only; launches nothing.
 * Checks the inputs (build_tq_decode_module's asserts: QG in {6,8,16}, BS in {16,32}, G >= 1)
 * and fills the outputs.  G == 0 follows the long-context launcher policy described with
 * tile_groups_per_partition on the same page: the smallest G with ceil(MB*BS / (G*256)) <=
 * max_partitions (the page's example: BS 32, cap 32 partitions -> G = 5, 32*5*256 = 40960
 * tokens).  Also rejects sizes whose index arithmetic would not fit the kernels' int32/int64
 * ranges (PDA_ERR_INVALID_ARG).
 *
 * Cache block layout (the page's stride block; formats of this library):
 *   data region   [BS slots][Hk heads][K: D elements | V: D elements], elements bf16, e4m3, or
 *                 TQ4 4-bit codes (two per byte, dimension 2j in the low nibble of byte j),
 *   meta region   at meta_offset_bytes: fp8: fp32 [Hk][2: K scale, V scale][BS];
 *                 TQ4: fp16 [Hk][3: k_norm, v_scale, v_zero][BS]; bf16: none.
 *   cache_block_bytes = BS*Hk*2*D*elem (+ Hk*2*BS*4 for fp8), or BS*Hk*D + Hk*3*BS*2 for TQ4.
 * Returns PDA_OK, PDA_ERR_INVALID_ARG or PDA_ERR_UNSUPPORTED.
 */
PDA_API int pda_plan(pda_plan_t* plan);

/*
 * pda_decode -- the partition pass (tq_decode_kernel: steps B to G).
 *   query          device, bf16 [B][Hk*QG][D] contiguous, 16-byte aligned.
 *                  query, block_table and context_lens may instead be pinned host memory that
 *                  the device can address (cudaHostAlloc, or cudaHostRegister, under unified
 *                  addressing): the kernels then read them across the host link, with no copy.
 *   kv_cache       device, bytes [num_cache_blocks][cache_block_bytes], 16-byte aligned.
 *   num_cache_blocks  NB >= 1, < 2^31; block ids outside [0, NB) are data errors.
 *   block_table    device, int32 [B][max_blocks_per_seq]; only entries t/BS for t < ctx are read.
 *   context_lens   device, int32 [B], each in [0, MB*BS].
 *   partial_out    device, fp32 [B][Hk][P][QG][D]   (normalised partial o_p)
 *   exp_sums       device, fp32 [B][Hk][P][QG]      (l_p = sum of exp(s - m_p) over the partition)
 *   max_logits     device, fp32 [B][Hk][P][QG]      (m_p = max of s = softmax_scale * q.k)
 *   err_word       device int or NULL.
 *   stream         cudaStream_t or NULL.
 * Only partitions p < ceil(ctx_b / W) are written; rows >= QG do not exist in the layout;
 * other partitions' slots are left untouched.
 * Data errors: a context length out of range is treated as 0 (nothing written for that
 * sequence) and sets PDA_ERRW_BAD_CONTEXT_LEN; a block id out of range is read as zeros
 * (the tensor copy's out-of-bounds fill) and sets PDA_ERRW_BAD_BLOCK_ID.
 * A TQ4 plan is rejected (PDA_ERR_INVALID_ARG): that format needs pda_decode_tq4.
 */
PDA_API int pda_decode(const pda_plan_t* plan, const void* query, const void* kv_cache, long long num_cache_blocks,
               const int* block_table, const int* context_lens, float* partial_out, float* exp_sums,
               float* max_logits, int* err_word, void* stream);

/*
 * pda_decode_tq4 -- the partition pass for a TQ4 cache (plan->kv_dtype == PDA_KV_TQ4): the
 * page's own format, decoded as its STEP F does (tq_decode_kernel):
 *   K[t][d] = centroids[code] * k_norm[t],   V[t][d] = code * v_scale[t] + v_zero[t]
 * with code the 4-bit code of dimension d of token t (K codes: bytes 0..63 of the token-head
 * row, V codes: bytes 64..127; dimension 2j in the low nibble of byte j) and the fp16 fields
 * of the metadata region.  The query is taken as given: on the page it arrives already rotated
 * into the basis the codes were made in (STEP B), so the rotation is the caller's.
 *   centroids      device, fp32 [16], finite (STEP A's codebook).
 * Every other argument, the partial layout and the error rules are those of pda_decode;
 * pda_reduce combines the partials.  A non-TQ4 plan is rejected (PDA_ERR_INVALID_ARG).
 */
PDA_API int pda_decode_tq4(const pda_plan_t* plan, const void* query, const void* kv_cache,
                           long long num_cache_blocks, const float* centroids, const int* block_table,
                           const int* context_lens, float* partial_out, float* exp_sums, float* max_logits,
                           int* err_word, void* stream);

/*
 * pda_reduce -- combines the partials of pda_decode (the reduce that follows the partition
 * pass; the page's per-partition exp_sums / max_logits outputs exist for it):
 *   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p (w_p / sum_q w_q) * o_p
 * over p < ceil(ctx_b / W).  One partition is copied bit for bit; ctx 0 gives 0.
 *   out            device, [B][Hk*QG][D], bf16 (PDA_OUT_BF16, round to nearest even) or fp32.
 *                  out and context_lens may be pinned host memory, as for pda_decode's inputs.
 * A context length out of range gives 0 and sets PDA_ERRW_BAD_CONTEXT_LEN.
 */
PDA_API int pda_reduce(const pda_plan_t* plan, const int* context_lens, const float* partial_out,
               const float* exp_sums, const float* max_logits, void* out, int out_dtype, int* err_word,
               void* stream);

/*
 * pda_append_kv -- the write side of the same cache: stores K and V of one new token for every
 * sequence b with positions[b] >= 0, at token index positions[b]: cache block
 * block_table[b][pos / BS], slot pos % BS (the paged slot formula of the KV insert on the
 * DeepSeek attention-front page: block = slot // block_size, offset = slot % block_size, and a
 * negative slot means no write).
 *   k_new, v_new  device, bf16 [B][Hk][D], 8-byte aligned
 *   kv_cache      device, the cache pda_decode reads (16-byte aligned)
 *   positions     device, int32 [B]
 * bf16 caches store the values as given.  fp8 caches store, per (token, KV head) and separately
 * for K and V, scale = absmax / 448 in fp32 (1 when the row is all zero) in the metadata region
 * and codes e4m3(x / scale), both divisions correctly rounded in fp32, the conversion rounding to
 * nearest even and saturating at +-448.  TQ4 caches are not supported (PDA_ERR_UNSUPPORTED): the
 * pages give no encoder for that format (its rotation and codebook are not on them).
 * Data errors (nothing is written for that sequence): a position >= MB*BS sets
 * PDA_ERRW_BAD_POSITION, a block id outside [0, NB) sets PDA_ERRW_BAD_BLOCK_ID.
 * Two sequences whose table entries name the same block and slot race.
 */
PDA_API int pda_append_kv(const pda_plan_t* plan, const void* k_new, const void* v_new, void* kv_cache,
                          long long num_cache_blocks, const int* block_table, const int* positions, int* err_word,
                          void* stream);

/*
 * pda_decode_fused -- one launch for the whole step: the partition pass of pda_decode, then, in
 * the same launch, the reduce of pda_reduce.  The launch is cooperative (every CTA resident): once
 * every CTA has written its partials they meet at a grid barrier (a bounded wait on a counter of
 * the library's per-launch slots; a wait that gives up sets PDA_ERRW_PIPELINE_TIMEOUT), and then
 * all of them merge the output rows, each row in partition order with pda_reduce's arithmetic, so
 * results are deterministic and equal pda_decode + pda_reduce's bit for bit.  On head-warp plans a
 * (sequence, KV head) whose context fits one partition is written to `out` by its partition's
 * epilogue (its partial is not stored).  The rows of a sequence with no tokens (context 0, or an
 * invalid length, which also sets PDA_ERRW_BAD_CONTEXT_LEN) are written as zeros, as pda_reduce
 * writes them.
 *   partial_out, exp_sums, max_logits   as for pda_decode (scratch here)
 *   counters   device int32 [B][Hk], zero: reserved (an earlier form of this step counted arrivals
 *              there); the call leaves them zero.
 *   out, out_dtype                      as for pda_reduce
 * query, block_table, context_lens and out may be pinned host memory, as for pda_decode.
 * Calls that share partials race if they overlap on the GPU; fewer than 256 launches of this
 * library's counter-slot kernels may be in flight on a device at once.
 * A TQ4 plan is rejected (PDA_ERR_INVALID_ARG): that format is read by pda_decode_tq4 only.
 * On GB300 this step measured slower than pda_decode followed by pda_reduce on every workload
 * timed (the reduce launch is already resident when the partition pass ends; the barrier and
 * the merge after it cost more); it exists for callers that want a single launch.
 */
PDA_API int pda_decode_fused(const pda_plan_t* plan, const void* query, const void* kv_cache,
                             long long num_cache_blocks, const int* block_table, const int* context_lens,
                             float* partial_out, float* exp_sums, float* max_logits, int* counters, void* out,
                             int out_dtype, int* err_word, void* stream);

/*
 * pda_decode_step_noalloc -- pda_decode followed by pda_reduce, for callers that cannot
 * allocate device memory when they run a step: for example a plugin inside an engine that owns
 * every byte of device memory, or code that must not call cudaMalloc because it can synchronise
 * the device.  Such callers can pass inputs and outputs but no partials workspace, so this entry
 * point keeps the partials in a fixed array inside the library.  The pages describe no such
 * entry point; it has no counterpart there.
 *   Arguments are those of pda_decode and pda_reduce without the three partial buffers:
 *   query, kv_cache, num_cache_blocks, block_table, context_lens as for pda_decode; out and
 *   out_dtype as for pda_reduce.
 * The array holds PDA_NOALLOC_SCRATCH_BYTES (64 MiB) on every GPU that loads the library, until
 * the process exits.  A plan whose partials (B*Hk*P*QG*(D*4 + 8) bytes, each part rounded up to
 * 256 bytes) do not fit returns PDA_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 * query, block_table, context_lens and out may be pinned host memory, as for pda_decode and
 * pda_reduce.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  The address is kept for
 * the life of the process: after cudaDeviceReset, or anything else that destroys the device's
 * primary context, do not call this entry point again in the same process.  The call allocates
 * nothing and frees nothing.
 * All calls share the one array and it keeps the last call's contents (nothing in it needs to
 * start at zero); calls that overlap on the GPU, on any streams, race.
 * A TQ4 plan is rejected (PDA_ERR_INVALID_ARG): that format is read by pda_decode_tq4 only.
 */
#define PDA_NOALLOC_SCRATCH_BYTES (64ll << 20)
PDA_API int pda_decode_step_noalloc(const pda_plan_t* plan, const void* query, const void* kv_cache,
                                    long long num_cache_blocks, const int* block_table, const int* context_lens,
                                    void* out, int out_dtype, int* err_word, void* stream);

/*
 * pda_kernel_variant -- host only; launches nothing.  The partition-pass layout pda_decode would
 * launch for this plan on the current device: PDA_VARIANT_HEAD_WARPS, PDA_VARIANT_HEAD_GROUPS or
 * PDA_VARIANT_ROW_HALVES (plan->kernel_variant resolved, PDA_VARIANT_AUTO included).  Returns PDA_ERR_INVALID_ARG for
 * a NULL or edited plan, PDA_ERR_CUDA when the device cannot be queried.  No counterpart on the
 * pages.
 */
PDA_API int pda_kernel_variant(const pda_plan_t* plan);

/* Human-readable name of a pda_status value (static string; never NULL). */
PDA_API const char* pda_status_string(int status);

/* plan->workspace_bytes after pda_plan (-1 for a NULL or unplanned plan). */
PDA_API long long pda_workspace_size(const pda_plan_t* plan);

/* sizeof(pda_plan_t), for bindings that mirror the structure. */
PDA_API int pda_plan_struct_size(void);

#ifdef __cplusplus
}
#endif
#endif /* PDA_H */
