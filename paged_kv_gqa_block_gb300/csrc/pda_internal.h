// pda_internal.h -- declarations shared by the translation units of libpda (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace pda {

constexpr int kHeadDim = 128;
constexpr int kTileTokens = 16;          // tokens per MMA tile (TILE_SIZE on the page)
constexpr int kTokensPerTileGroup = 256; // 16 tiles (KV_COMPUTE_BLOCK on the page)
constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;   // 1 s per bounded wait

// Arguments of the partition kernel (plain values, passed by value).
struct DecodeArgs {
    const uint16_t* query;     // bf16 [B][Hk*QG][D]
    const int* block_table;    // [B][MB]
    const int* context_lens;   // [B]
    const float* centroids;    // TQ4 only: [16]
    float* partial_out;        // [B][Hk][P][QG][D]
    float* exp_sums;           // [B][Hk][P][QG]
    float* max_logits;         // [B][Hk][P][QG]
    int* err_word;             // may be null
    long long num_cache_blocks;
    int B, Hk, QG, MB, BS, P, W;
    int bs_shift;              // log2(BS)
    int HG;                    // head-group kernel: KV heads per CTA (a divisor of Hk, <= 4)
    unsigned int* sched;       // this launch's slot of counters (head-group kernel; the fused step's
                               // grid barrier), zero at launch and left zero by its last CTA
    float qk_scale_log2;       // softmax_scale * log2(e)
    unsigned long long timeout_ns;
    // fused step only: the caller's reserved counters (untouched) and the final output
    int* counters;             // [B][Hk], zero
    void* out;                 // [B][Hk*QG][D] bf16 or fp32
    int out_f32;
};

struct ReduceArgs {
    const int* context_lens;
    const float* partial_out;
    const float* exp_sums;
    const float* max_logits;
    void* out;
    int* err_word;
    int B, Hk, QG, MB, BS, P, W;
    int out_f32;
};

// Launches the partition kernel for one KV format; returns a pda_status value.
int launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& kv_map, bool fused, cudaStream_t stream);
int launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map, bool fused,
                      cudaStream_t stream);
// The row-half kernel (bf16, QG 16): two consumer warps of 8 query rows per CTA.
int launch_decode_bf16_rows(const DecodeArgs& a, const CUtensorMap& kv_map, cudaStream_t stream);
// The head-group kernel (fp8): a.HG heads per CTA; the maps' boxes span a.HG heads.
// With `fused`, the same (cooperative) launch also combines the partials into `out` after a
// grid barrier.
int launch_decode_fp8_groups(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map,
                             bool fused, cudaStream_t stream);
// KV heads per CTA of the head-group kernel for Hk heads: the largest divisor of Hk not above 4.
int group_heads(int Hk);
int launch_decode_tq4(const DecodeArgs& a, const CUtensorMap& kv_map, const CUtensorMap& sc_map, cudaStream_t stream);
int launch_reduce(const ReduceArgs& r, cudaStream_t stream);

// The next slot of per-launch counters on the current device (zero; the launch's last CTA leaves
// it zero).  Sets *status to a pda_status value.
unsigned int* launch_counter_slot(int* status);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace pda
