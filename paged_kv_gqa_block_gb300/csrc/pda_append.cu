// pda_append.cu -- the write side of the paged cache: one new token per sequence.
//
// Token position pos of sequence b goes to cache block block_table[b][pos / BS], slot pos % BS
// (the paged slot formula block = slot // block_size, offset = slot % block_size of the KV insert
// on the DeepSeek attention-front page, where a negative slot means "no write").  bf16 caches take
// the values as given; fp8 caches take, per (token, KV head) and separately for K and V,
// scale = absmax / 448 (fp32, 1 for an all-zero row) and codes e4m3(x / scale) rounded to nearest
// even with saturation, the scale stored in the metadata region [kv_head][K, V][slot].
#include <cuda_runtime.h>

#include <cstdint>

#include "pda.h"
#include "pda_ptx.cuh"

namespace pda {

struct AppendArgs {
    const uint16_t* k_new;   // bf16 [B][Hk][D]
    const uint16_t* v_new;
    uint8_t* cache;
    const int* block_table;
    const int* positions;
    int* err_word;
    long long num_cache_blocks;
    long long cache_block_bytes, meta_offset_bytes;
    int B, Hk, MB, BS, fp8;
};


// One warp per (sequence, KV head); lane l handles head dims 4l .. 4l+3.
__global__ void __launch_bounds__(256) pda_append_kernel(const AppendArgs a) {
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (long long)a.B * a.Hk) return;
    const int b = (int)(wid / a.Hk), h = (int)(wid - (long long)b * a.Hk);
    const int pos = __ldg(a.positions + b);
    if (pos < 0) return;
    if (pos >= a.MB * a.BS) {
        if (h == 0 && lane == 0 && a.err_word) atomicOr(a.err_word, PDA_ERRW_BAD_POSITION);
        return;
    }
    const int blk = __ldg(a.block_table + (long long)b * a.MB + pos / a.BS);
    if (blk < 0 || (long long)blk >= a.num_cache_blocks) {
        if (h == 0 && lane == 0 && a.err_word) atomicOr(a.err_word, PDA_ERRW_BAD_BLOCK_ID);
        return;
    }
    const int slot = pos % a.BS;
    uint8_t* block = a.cache + (long long)blk * a.cache_block_bytes;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        const uint16_t* src = (which == 0 ? a.k_new : a.v_new) + ((long long)b * a.Hk + h) * 128 + 4 * lane;
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(src));
        if (!a.fp8) {
            uint8_t* row = block + ((long long)slot * a.Hk + h) * 512 + which * 256 + 8 * lane;
            *reinterpret_cast<uint2*>(row) = raw;
            continue;
        }
        const float x0 = __uint_as_float(raw.x << 16), x1 = __uint_as_float(raw.x & 0xFFFF0000u);
        const float x2 = __uint_as_float(raw.y << 16), x3 = __uint_as_float(raw.y & 0xFFFF0000u);
        float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale));
        const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(x2, scale), __fdiv_rn(x3, scale));
        uint8_t* row = block + ((long long)slot * a.Hk + h) * 256 + which * 128 + 4 * lane;
        *reinterpret_cast<uint32_t*>(row) = lo | (hi << 16);
        if (lane == 0)
            *reinterpret_cast<float*>(block + a.meta_offset_bytes + (((long long)h * 2 + which) * a.BS + slot) * 4) =
                scale;
    }
}

}  // namespace pda

extern "C" int pda_append_kv(const pda_plan_t* plan, const void* k_new, const void* v_new, void* kv_cache,
                             long long num_cache_blocks, const int* block_table, const int* positions, int* err_word,
                             void* stream) {
    if (!plan || pda_workspace_size(plan) < 0) return PDA_ERR_INVALID_ARG;
    if (plan->kv_dtype == PDA_KV_TQ4) return PDA_ERR_UNSUPPORTED;   // no encoder for that format
    if (plan->num_seqs == 0) return PDA_OK;
    if (!k_new || !v_new || !kv_cache || !block_table || !positions) return PDA_ERR_INVALID_ARG;
    if (num_cache_blocks < 1 || num_cache_blocks > (1ll << 31) - 1) return PDA_ERR_INVALID_ARG;
    if (((uintptr_t)k_new & 7u) || ((uintptr_t)v_new & 7u) || ((uintptr_t)kv_cache & 15u) ||
        ((uintptr_t)block_table & 3u) || ((uintptr_t)positions & 3u) || ((uintptr_t)err_word & 3u))
        return PDA_ERR_INVALID_ARG;
    pda::AppendArgs a;
    a.k_new = static_cast<const uint16_t*>(k_new);
    a.v_new = static_cast<const uint16_t*>(v_new);
    a.cache = static_cast<uint8_t*>(kv_cache);
    a.block_table = block_table;
    a.positions = positions;
    a.err_word = err_word;
    a.num_cache_blocks = num_cache_blocks;
    a.cache_block_bytes = plan->cache_block_bytes;
    a.meta_offset_bytes = plan->meta_offset_bytes;
    a.B = plan->num_seqs;
    a.Hk = plan->num_kv_heads;
    a.MB = plan->max_blocks_per_seq;
    a.BS = plan->kv_block_size;
    a.fp8 = plan->kv_dtype == PDA_KV_FP8_E4M3;
    const long long warps = (long long)a.B * a.Hk;
    const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
    pda::pda_append_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? PDA_OK : PDA_ERR_LAUNCH;
}
