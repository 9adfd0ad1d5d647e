// pda_decode.cuh -- the partition pass of paged-KV GQA decode attention for sm_103a.
//
// What one work unit computes (vLLM "tq_decode" page, tq_decode_kernel): for sequence b, KV
// head h and partition p, the QG query rows h*QG..h*QG+QG-1 attend over tokens
// [p*W, min((p+1)*W, ctx_b)) (STEP E); each 16-token tile finds its cache block through the
// block table, entry t/BS, slot t%BS (STEP F); scores are scaled and tokens >= ctx masked to
// -inf; an online softmax carries (max, sum, acc) across tiles; the epilogue writes the
// normalised partial, the running max and the running sum (STEP G).
//
// How it is laid out on GB300 (not the page's AMD design):
//   * One warp per CTA, many CTAs per SM, persistent grid.  Every warp owns whole units: the
//     tiles of the step are split evenly over all warps of the grid and a warp takes the units
//     whose first tile falls in its share, so empty partitions cost nothing and no warp ever
//     waits for another (no cross-warp merge, no barrier).
//   * The warp feeds itself: lane 0 keeps S 16-token tiles in flight with ONE 5-D TMA tensor
//     copy per tile (K and V of one KV head, 8 KB bf16 / 4 KB fp8, 128-byte swizzle) into a
//     private S-stage ring of mbarriers; for fp8 a 4-D TMA copy brings the tile's 16 K and 16
//     V scales.  Block-table entries are loaded 32 at a time one chunk ahead, and the next
//     unit's Q rows are loaded into registers while the current unit runs.
//   * Per tile: S^T = K Q^T and O^T += V^T P^T with warp-level mma.sync (m16n8k16, fp32
//     accumulate).  Tokens are the M dimension of the score MMA so QG = 8 fills it; P is moved
//     to the B-operand layout with movmatrix.
//   * bf16 KV: bf16 MMAs, P split into bf16 hi + lo parts (two PV MMAs) so P keeps ~16 bits.
//     fp8 KV: e4m3 -> f16 conversion (exact), Q scaled by a power of two into f16 range,
//     K scales applied to the fp32 scores, V scales folded into P relative to the tile's
//     largest V scale (the factor is carried in the running rescale).
//     TQ4 KV (the page's own 4-bit format, STEP F): K codes become f16 centroid pairs through a
//     256-entry table in shared memory (one byte = two dimensions), k_norm scales the fp32
//     scores; V codes enter the PV MMA as exact f16 integers (the code itself as a subnormal
//     bit pattern, code * 2^-24), v_scale is folded into P like fp8's V scale, and v_zero
//     contributes sum_t p_t v_zero_t to every dimension, kept per query row beside the
//     running sum.
//   * The epilogue stages the partial through the stage it has just consumed and writes it
//     with coalesced 16-byte stores.
//   * Every wait is bounded; a wait that gives up sets PDA_ERRW_PIPELINE_TIMEOUT, and the
//     warp waits (bounded) for its own copies in flight before it leaves.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "pda.h"
#include "pda_internal.h"
#include "pda_ptx.cuh"
#include "pda_merge.cuh"

namespace pda {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kFull = 0xFFFFFFFFu;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int KV, int S>
struct DecodeCfg {
    static constexpr bool kBf16 = KV == PDA_KV_BF16, kTq = KV == PDA_KV_TQ4;
    static constexpr int kThreads = 32;
    // K and V of 16 tokens of one KV head: 8 KB bf16, 4 KB fp8, 2 KB of TQ4 codes
    static constexpr int kTileBytes = kBf16 ? 8192 : kTq ? 2048 : 4096;
    static constexpr int kChunks = kTileBytes / 2048;       // 128-byte chunks per token-head
    // metadata copied per tile: fp8 16 K + 16 V scales (fp32); TQ4 16 x {k_norm, v_scale, v_zero} (fp16)
    static constexpr int kScaleTx = kBf16 ? 0 : kTq ? 96 : 128;
    static constexpr int kScaleBytes = kBf16 ? 0 : 128;     // per stage (16-byte aligned slots)
    static constexpr int kOffStages = 0;
    static constexpr int kOffScales = S * kTileBytes;
    static constexpr int kOffBar = align_up(kOffScales + S * kScaleBytes, 8);
    static constexpr int kSmemBytes = kOffBar + S * 8 + 1024;   // + base alignment slack
};

// ---------------------------------------------------------------------------------------------
// unit iteration (same order everywhere): sequences b ascending, then KV head h, then partition
// p; a unit's first tile index is its position in that order counted in 16-token tiles.
struct UnitIt {
    int b, h, p, ctx, nv;
    long long start;
};

__device__ __forceinline__ int sanitize_ctx(int c, int max_ctx) { return (c < 0 || c > max_ctx) ? 0 : c; }

__device__ __forceinline__ void it_settle(UnitIt& u, const DecodeArgs& a) {
    const int max_ctx = a.MB * a.BS;
    while (u.b < a.B) {
        u.ctx = sanitize_ctx(__ldg(a.context_lens + u.b), max_ctx);
        u.nv = (u.ctx + a.W - 1) / a.W;
        if (u.nv > 0) break;
        ++u.b;
        u.h = 0;
        u.p = 0;
    }
}
__device__ __forceinline__ int unit_tokens(const UnitIt& u, int W) {
    const int rem = u.ctx - u.p * W;
    return rem < W ? rem : W;
}
__device__ __forceinline__ int unit_tiles(const UnitIt& u, int W) { return (unit_tokens(u, W) + 15) >> 4; }
__device__ __forceinline__ void it_advance(UnitIt& u, const DecodeArgs& a) {
    u.start += unit_tiles(u, a.W);
    if (++u.p == u.nv) {
        u.p = 0;
        if (++u.h == a.Hk) {
            u.h = 0;
            ++u.b;
            it_settle(u, a);
        }
    }
}

// One warp: count the tiles and the units of the step and choose this warp's work.  With no
// more units than warps, warp k takes unit k alone (nothing is gained by pairing units: the
// longest warp would hold two).  Otherwise the tiles are split evenly over the warps and a warp
// takes the units whose first tile falls in its share.  Returns the warp's first unit
// (u.b == B when it has none) and the end of its tile range.  Sets the data-error bit for
// out-of-range context lengths (block 0 only).
__device__ inline void find_range(const DecodeArgs& a, UnitIt& u, long long& hi) {
    const int lane = threadIdx.x & 31;
    const int max_ctx = a.MB * a.BS;
    const int per = (a.B + 31) >> 5;
    const int b0 = min(a.B, lane * per), b1 = min(a.B, b0 + per);
    long long mine = 0, mine_u = 0;   // tiles and units of this lane's sequences
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
        const int raw = __ldg(a.context_lens + b);
        if (raw < 0 || raw > max_ctx) bad = true;
        const int c = sanitize_ctx(raw, max_ctx);
        mine += (long long)a.Hk * ((c + 15) >> 4);
        mine_u += (long long)a.Hk * ((c + a.W - 1) / a.W);
    }
    if (bad && blockIdx.x == 0 && a.err_word) atomicOr(a.err_word, PDA_ERRW_BAD_CONTEXT_LEN);
    long long incl = mine, incl_u = mine_u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(kFull, incl, o);
        const long long nu = __shfl_up_sync(kFull, incl_u, o);
        if (lane >= o) {
            incl += n;
            incl_u += nu;
        }
    }
    const long long total = __shfl_sync(kFull, incl, 31);
    const long long units = __shfl_sync(kFull, incl_u, 31);
    const long long excl = incl - mine, excl_u = incl_u - mine_u;
    int fb = a.B, fh = 0, fp = 0;
    long long fs = 0;
    int found = 0;
    if (units <= gridDim.x) {
        // unit k = blockIdx.x, found by the lane whose sequences hold it
        const long long k = blockIdx.x;
        hi = 0;
        if (mine_u > 0 && excl_u <= k && k < excl_u + mine_u) {
            long long pos = excl, pos_u = excl_u;
            for (int b = b0; b < b1; ++b) {
                const int c = sanitize_ctx(__ldg(a.context_lens + b), max_ctx);
                const long long th = (c + 15) >> 4;
                const long long nv = (c + a.W - 1) / a.W;
                if (k < pos_u + a.Hk * nv) {
                    const long long r = k - pos_u;
                    fb = b;
                    fh = (int)(r / nv);
                    fp = (int)(r - fh * nv);
                    fs = pos + fh * th + (long long)fp * (a.W >> 4);
                    found = 1;
                    break;
                }
                pos += a.Hk * th;
                pos_u += a.Hk * nv;
            }
        }
        const unsigned m = __ballot_sync(kFull, found);
        const int src = m ? __ffs(m) - 1 : 0;
        u.b = m ? __shfl_sync(kFull, fb, src) : a.B;
        u.h = __shfl_sync(kFull, fh, src);
        u.p = __shfl_sync(kFull, fp, src);
        u.start = __shfl_sync(kFull, fs, src);
        u.ctx = 0;
        u.nv = 0;
        if (u.b < a.B) {
            it_settle(u, a);
            hi = u.start + unit_tiles(u, a.W);
        }
        return;
    }
    const long long lo = (long long)blockIdx.x * total / gridDim.x;
    hi = ((long long)blockIdx.x + 1) * total / gridDim.x;
    // the lane whose sequences contain tile `lo` finds the first unit starting at or after it
    if (mine > 0 && excl <= lo && lo < excl + mine) {
        long long pos = excl;
        for (int b = b0; b < b1; ++b) {
            const int c = sanitize_ctx(__ldg(a.context_lens + b), max_ctx);
            const long long th = (c + 15) >> 4;           // tiles of one KV head of this sequence
            const long long tb = (long long)a.Hk * th;
            if (lo < pos + tb) {
                const long long off = lo - pos;
                int h = (int)(off / th);
                const long long r = off - h * th;
                const long long tp = a.W >> 4;                // tiles of a full partition
                int p = (int)((r + tp - 1) / tp);
                const int nv = (c + a.W - 1) / a.W;
                if (p >= nv) {
                    p = 0;
                    ++h;
                }
                if (h < a.Hk) {
                    fb = b; fh = h; fp = p;
                    fs = pos + h * th + p * tp;
                } else {            // the next sequence's first unit (empty sequences are skipped below)
                    fb = b + 1; fh = 0; fp = 0;
                    fs = pos + tb;
                }
                found = 1;
                break;
            }
            pos += tb;
        }
    }
    const unsigned m = __ballot_sync(kFull, found);
    const int src = m ? __ffs(m) - 1 : 0;
    u.b = m ? __shfl_sync(kFull, fb, src) : a.B;
    u.h = __shfl_sync(kFull, fh, src);
    u.p = __shfl_sync(kFull, fp, src);
    u.start = __shfl_sync(kFull, fs, src);
    u.ctx = 0;
    u.nv = 0;
    it_settle(u, a);
}

// ---------------------------------------------------------------------------------------------
// EAGER: the eager softmax update even where kLazy would apply (the QG = 16 row-half kernel,
// whose 8-row blocks must give the bits of this kernel's two n-tiles).
template <int KV, int NT, int S, bool FUSED, bool EAGER = false>
struct Decode {
    using Cfg = DecodeCfg<KV, S>;
    static constexpr bool FP8 = KV == PDA_KV_FP8_E4M3;
    static constexpr bool TQ = KV == PDA_KV_TQ4;
    static constexpr bool F16 = KV != PDA_KV_BF16;   // f16 MMAs, Q scaled into f16, V scale folded into P

    // ------------------------------------------------------------------ tile feeding
    // The issue side walks (unit, 32-entry chunk) pairs; the entries of the next chunk are
    // loaded when the current chunk becomes current, one full chunk of issue time ahead.
    struct Feed {
        UnitIt u;      // unit of the current chunk
        int e0;        // first block-table entry of the current chunk (relative to the unit)
        int ent;       // this lane's entry of the current chunk
        int t;         // next tile of the unit to issue
        int nt;        // tiles of the unit
        bool valid;
        bool pf;       // the next chunk has been looked up and its entries requested
        UnitIt nu;     // next chunk
        int ne0, nent;
        bool nvalid;
        uint64_t policy;   // L2 policy of the tile copies (read once: evict first)
    };

    static __device__ __forceinline__ int n_entries(const DecodeArgs& a, const UnitIt& u) {
        return (unit_tokens(u, a.W) + a.BS - 1) >> a.bs_shift;
    }
    static __device__ __forceinline__ int load_entry(const DecodeArgs& a, const UnitIt& u, int e0, int lane) {
        const int idx = e0 + lane;
        if (idx >= n_entries(a, u)) return 0;
        return __ldg(a.block_table + (long long)u.b * a.MB + ((u.p * a.W) >> a.bs_shift) + idx);
    }
    static __device__ void prefetch_next(const DecodeArgs& a, long long hi, Feed& f, int lane) {
        f.nu = f.u;
        if (f.e0 + 32 < n_entries(a, f.u)) {
            f.ne0 = f.e0 + 32;
            f.nvalid = true;
        } else {
            it_advance(f.nu, a);
            f.ne0 = 0;
            f.nvalid = f.nu.b < a.B && f.nu.start < hi;
        }
        f.nent = f.nvalid ? load_entry(a, f.nu, f.ne0, lane) : 0;
        f.pf = true;
    }
    static __device__ __forceinline__ void feed_init(const DecodeArgs& a, long long hi, const UnitIt& first, Feed& f,
                                                     int lane) {
        f.u = first;
        f.e0 = 0;
        f.t = 0;
        f.valid = first.b < a.B && first.start < hi;
        f.nt = f.valid ? unit_tiles(first, a.W) : 0;
        f.ent = f.valid ? load_entry(a, f.u, 0, lane) : 0;
        f.pf = false;
        f.nvalid = false;
        f.policy = l2_policy_evict_first();
    }
    // Issues the next tile into `stage` (whole warp; lane 0 issues).  Returns false when the
    // warp's range has no more tiles.
    static __device__ __forceinline__ bool feed_one(const DecodeArgs& a, long long hi, const CUtensorMap* kv_map,
                                                    const CUtensorMap* sc_map, uint32_t sbase, uint32_t bar, int stage,
                                                    Feed& f, int lane) {
        if (!f.valid) return false;
        const int ts = a.bs_shift - 4;   // log2(16-token tiles per block-table entry)
        const int phys = __shfl_sync(kFull, f.ent, (f.t >> ts) - f.e0);
        if (lane == 0) {
            const int slot0 = (f.t & ((1 << ts) - 1)) * kTileTokens;
            mbar_arrive_expect_tx(bar, Cfg::kTileBytes + Cfg::kScaleTx);
            tma_load_5d(sbase + Cfg::kOffStages + stage * Cfg::kTileBytes, kv_map, bar, 0, slot0, 0, f.u.h, phys,
                        f.policy);
            if constexpr (F16)
                tma_load_4d(sbase + Cfg::kOffScales + stage * Cfg::kScaleBytes, sc_map, bar, slot0, 0, f.u.h, phys,
                            f.policy);
            if ((phys < 0 || (long long)phys >= a.num_cache_blocks) && a.err_word)
                atomicOr(a.err_word, PDA_ERRW_BAD_BLOCK_ID);
        }
        ++f.t;
        if (f.t == f.nt || (f.t >> ts) - f.e0 >= 32) {     // move to the next chunk
            if (!f.pf) prefetch_next(a, hi, f, lane);
            const bool same_unit = f.t < f.nt;
            f.u = f.nu;
            f.e0 = f.ne0;
            f.ent = f.nent;
            f.valid = f.nvalid;
            if (!same_unit) {
                f.t = 0;
                f.nt = unit_tiles(f.u, a.W);
            }
            f.pf = false;
            if (f.valid) prefetch_next(a, hi, f, lane);   // one chunk ahead
        }
        return true;
    }

    // ------------------------------------------------------------------ Q of a unit
    // Raw words of the unit's Q rows as this lane needs them (rows >= QG read as zero).
    //   bf16: w[n][2kk + j] = Q[8n + gid][16kk + 8j + 2tig .. +1]  (the mma B fragments)
    //   fp8, TQ4: w[n][c]   = Q[8n + gid][32tig + 2c .. +1]         (converted at unit start)
    static __device__ __forceinline__ void load_q(const DecodeArgs& a, const UnitIt& u, uint32_t (&w)[NT][16],
                                                  int lane) {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int r = n * 8 + gid;
            if (r < a.QG) {
                const uint32_t* row = reinterpret_cast<const uint32_t*>(
                    a.query + ((long long)u.b * a.Hk * a.QG + (long long)u.h * a.QG + r) * kHeadDim);
                if constexpr (F16) {
                    const uint4* p4 = reinterpret_cast<const uint4*>(row + tig * 16);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v = __ldg(p4 + c);
                        w[n][4 * c] = v.x;
                        w[n][4 * c + 1] = v.y;
                        w[n][4 * c + 2] = v.z;
                        w[n][4 * c + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        w[n][2 * kk] = __ldg(row + kk * 8 + tig);
                        w[n][2 * kk + 1] = __ldg(row + kk * 8 + 4 + tig);
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < 16; ++c) w[n][c] = 0u;
            }
        }
    }

    // ------------------------------------------------------------------ online softmax
    // The eager update (no kLazy): with scaled V (VS) the V weights are first divided by the step's
    // largest one, F, and the accumulators rebased on it (ratio); then, n-tile by n-tile, each
    // query row reduces the step's maximum across the lanes, rescales its state to the new
    // maximum and adds the step.
    template <int NTL>
    static __device__ __forceinline__ float eager_v_rebase(float (&w0)[NTL], float (&w1)[NTL], float& F) {
        float fv = 0.f;
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) fv = fmaxf(fv, fmaxf(fabsf(w0[tl]), fabsf(w1[tl])));
        fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 4));
        fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 8));
        fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 16));
        if (!(fv > 0.f)) fv = 1.f;
        const float rF = rcp_approx(fv);   // acc and F move together: only their product matters
        // acc holds true_acc / F: rebase it on this step's factor (exactly 1 when F is unchanged,
        // which F * rcp(F) need not be)
        const float ratio = fv == F ? 1.f : F * rF;
        F = fv;
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            w0[tl] *= rF;
            w1[tl] *= rF;
        }
        return ratio;
    }
    template <int NTL, bool VS, bool ZS>
    static __device__ __forceinline__ void eager_rows(int n, float (&s)[NTL][NT][4], const float (&w0)[NTL],
                                                      const float (&w1)[NTL], const float (&z0)[NTL],
                                                      const float (&z1)[NTL], float (&acc)[NT][8][4],
                                                      float (&m2)[NT][2], float (&ls)[NT][2], float (&zs)[NT][2],
                                                      float ratio) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(s[0][n][j], s[0][n][j + 2]);
#pragma unroll
            for (int tl = 1; tl < NTL; ++tl) mx = fmaxf(mx, fmaxf(s[tl][n][j], s[tl][n][j + 2]));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float mnew = fmaxf(m2[n][j], mx);
            const float alpha = ex2(m2[n][j] - mnew);
            m2[n][j] = mnew;
            float sum = 0.f, zsum = 0.f;
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) {
                const float p0 = ex2(s[tl][n][j] - mnew), p1 = ex2(s[tl][n][j + 2] - mnew);
                sum += p0 + p1;
                if constexpr (ZS) zsum = fmaf(p0, z0[tl], fmaf(p1, z1[tl], zsum));
                s[tl][n][j] = VS ? p0 * w0[tl] : p0;
                s[tl][n][j + 2] = VS ? p1 * w1[tl] : p1;
            }
            ls[n][j] = ls[n][j] * alpha + sum;
            if constexpr (ZS) zs[n][j] = zs[n][j] * alpha + zsum;
            const float ar = alpha * ratio;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                acc[n][m][j] *= ar;
                acc[n][m][j + 2] *= ar;
            }
        }
    }

    // One step's update of the running softmax state, given the step's scores s (log2 units,
    // -inf where masked).  The reference point m2 of each query row, and with scaled V (VS) the
    // factor F that the V weights w are divided by, move lazily: only when a score exceeds m2 by
    // more than kLazyLog2, or a V weight leaves (F/64, 64F].  Most steps then skip the cross-lane
    // reductions and the rescale of the accumulators; P = 2^(s - m2) stays below 2^kLazyLog2 and
    // P w / F below 2^14 (f16 range).  mt keeps this lane's true running maximum (reduced once, in
    // the epilogue).  On return s holds P, times w/F with scaled V; ls (and zs, the zero-point
    // sum, with ZS) include the step.
    //
    // Without kLazy every step rebases, row by row (m2 is then the running maximum and F the
    // step's largest V weight).  That order is kept where the lazy form measured slower: the fp8
    // kernel, whose 168-register budget (12 CTAs per SM) it strains, and QG = 16 (two n-tiles).
    static constexpr float kLazyLog2 = 8.f;
    static constexpr bool kLazy = NT == 1 && !FP8 && !EAGER;
    template <int NTL, bool VS, bool ZS>
    static __device__ __forceinline__ void softmax_step(float (&s)[NTL][NT][4], float (&w0)[NTL], float (&w1)[NTL],
                                                        const float (&z0)[NTL], const float (&z1)[NTL],
                                                        float (&acc)[NT][8][4], float (&m2)[NT][2],
                                                        float (&mt)[NT][2], float (&ls)[NT][2], float (&zs)[NT][2],
                                                        float& F, float& rF) {
        float mx[NT][2];
        bool up = false;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float x = fmaxf(s[0][n][j], s[0][n][j + 2]);
#pragma unroll
                for (int tl = 1; tl < NTL; ++tl) x = fmaxf(x, fmaxf(s[tl][n][j], s[tl][n][j + 2]));
                mx[n][j] = x;
                mt[n][j] = fmaxf(mt[n][j], x);
                up |= x > m2[n][j] + kLazyLog2;
            }
        float fl = 0.f;
        if constexpr (VS) {
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) fl = fmaxf(fl, fmaxf(fabsf(w0[tl]), fabsf(w1[tl])));
            up |= fl > F * 64.f;
        }
        bool need = __any_sync(kFull, up);
        if constexpr (VS) need = need || __all_sync(kFull, fl < F * 0.015625f);
        if (need) {   // warp-uniform: move the reference points to this step's maxima
            float ratio = 1.f;
            if constexpr (VS) {
                float fv = fl;
                fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 4));
                fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 8));
                fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 16));
                if (!(fv > 0.f)) fv = 1.f;
                const float r = rcp_approx(fv);
                ratio = fv == F ? 1.f : F * r;   // acc holds true_acc / F: rebase it on the new factor
                F = fv;
                rF = r;
            }
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float x = mx[n][j];
                    x = fmaxf(x, __shfl_xor_sync(kFull, x, 4));
                    x = fmaxf(x, __shfl_xor_sync(kFull, x, 8));
                    x = fmaxf(x, __shfl_xor_sync(kFull, x, 16));
                    const float mnew = fmaxf(m2[n][j], x);
                    const float alpha = mnew == -INFINITY ? 1.f : ex2(m2[n][j] - mnew);
                    m2[n][j] = mnew;
                    ls[n][j] *= alpha;
                    if constexpr (ZS) zs[n][j] *= alpha;
                    const float ar = alpha * ratio;
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        acc[n][m][j] *= ar;
                        acc[n][m][j + 2] *= ar;
                    }
                }
        }
        if constexpr (VS) {
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) {
                w0[tl] *= rF;
                w1[tl] *= rF;
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float sum = 0.f, zsum = 0.f;
#pragma unroll
                for (int tl = 0; tl < NTL; ++tl) {
                    const float p0 = ex2(s[tl][n][j] - m2[n][j]), p1 = ex2(s[tl][n][j + 2] - m2[n][j]);
                    sum += p0 + p1;
                    if constexpr (ZS) zsum = fmaf(p0, z0[tl], fmaf(p1, z1[tl], zsum));
                    s[tl][n][j] = VS ? p0 * w0[tl] : p0;
                    s[tl][n][j + 2] = VS ? p1 * w1[tl] : p1;
                }
                ls[n][j] += sum;
                if constexpr (ZS) zs[n][j] += zsum;
            }
    }

    // ------------------------------------------------------------------ tile math
    // One step processes NTL (1 or 2) consecutive 16-token tiles of a unit with a single online-
    // softmax update; two tiles give the warp two independent score-MMA chains and halve the
    // max reductions and accumulator rescales per token.
    //
    // bf16 stage layout: chunk c (K0 = d 0..63, K1, V0, V1) x 16 tokens x 128 bytes, 16-byte
    // units swizzled by (token & 7).
    template <int NTL>
    static __device__ __forceinline__ void step_bf16(const uint32_t (&st)[NTL], const int (&valid)[NTL], float scale2,
                                                     const uint32_t (&qf)[NT][8][2], float (&acc)[NT][8][4],
                                                     float (&m2)[NT][2], float (&mt)[NT][2], float (&ls)[NT][2],
                                                     int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        constexpr int CH = NTL == 1 ? 2 : 1;   // independent MMA chains per tile
        float s[NTL][NT][4];
        {
            float sx[NTL][CH][NT][4];
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl)
#pragma unroll
                for (int ch = 0; ch < CH; ++ch)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int c = 0; c < 4; ++c) sx[tl][ch][n][c] = 0.f;
            const int ktok = lane & 15, khalf = lane >> 4;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int u = ((kk & 3) << 1) | khalf;
                const uint32_t off = (kk >> 2) * 2048 + ktok * 128 + ((u ^ (ktok & 7)) << 4);
#pragma unroll
                for (int tl = 0; tl < NTL; ++tl) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(st[tl] + off, a0, a1, a2, a3);
#pragma unroll
                    for (int n = 0; n < NT; ++n) mma_bf16(sx[tl][kk % CH][n], a0, a1, a2, a3, qf[n][kk][0], qf[n][kk][1]);
                }
            }
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int c = 0; c < 4; ++c) s[tl][n][c] = CH == 2 ? sx[tl][0][n][c] + sx[tl][CH - 1][n][c] : sx[tl][0][n][c];
        }
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            const bool v0 = gid < valid[tl], v1 = gid + 8 < valid[tl];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                s[tl][n][0] = v0 ? s[tl][n][0] * scale2 : -INFINITY;
                s[tl][n][1] = v0 ? s[tl][n][1] * scale2 : -INFINITY;
                s[tl][n][2] = v1 ? s[tl][n][2] * scale2 : -INFINITY;
                s[tl][n][3] = v1 ? s[tl][n][3] * scale2 : -INFINITY;
            }
        }
        float w[NTL], zz[NTL], zsd[NT][2];
        if constexpr (kLazy) {
            float Fd = 1.f, rFd = 1.f;
            softmax_step<NTL, false, false>(s, w, w, zz, zz, acc, m2, mt, ls, zsd, Fd, rFd);
        }
        uint32_t bh[NTL][NT][2], bl[NTL][NT][2];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            if constexpr (!kLazy) eager_rows<NTL, false, false>(n, s, w, w, zz, zz, acc, m2, ls, zsd, 1.f);
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) {
                const uint32_t h01 = pack_bf16(s[tl][n][0], s[tl][n][1]);
                const uint32_t h23 = pack_bf16(s[tl][n][2], s[tl][n][3]);
                const uint32_t l01 = pack_bf16(s[tl][n][0] - bf16_lo(h01), s[tl][n][1] - bf16_hi(h01));
                const uint32_t l23 = pack_bf16(s[tl][n][2] - bf16_lo(h23), s[tl][n][3] - bf16_hi(h23));
                bh[tl][n][0] = movmatrix_trans(h01);
                bh[tl][n][1] = movmatrix_trans(h23);
                bl[tl][n][0] = movmatrix_trans(l01);
                bl[tl][n][1] = movmatrix_trans(l23);
            }
        }
        // Only a step's last tile can be partial (the one before it is followed by another); its
        // V rows past the context may hold anything (NaN included) and are zeroed, 0 * NaN = NaN.
        if (valid[NTL - 1] < kTileTokens)
            pv_bf16<NTL, true>(st, valid, bh, bl, acc, lane);
        else
            pv_bf16<NTL, false>(st, valid, bh, bl, acc, lane);
    }
    template <int NTL, bool MASKED>
    static __device__ __forceinline__ void pv_bf16(const uint32_t (&st)[NTL], const int (&valid)[NTL],
                                                   const uint32_t (&bh)[NTL][NT][2], const uint32_t (&bl)[NTL][NT][2],
                                                   float (&acc)[NT][8][4], int lane) {
        const int tig = lane & 3;
        uint32_t mlo = kFull, mhi = kFull;   // the last tile's token mask, 16 bits per token
        if constexpr (MASKED) {
            const int v = valid[NTL - 1];
            mlo = (2 * tig < v ? 0x0000FFFFu : 0u) | (2 * tig + 1 < v ? 0xFFFF0000u : 0u);
            mhi = (2 * tig + 8 < v ? 0x0000FFFFu : 0u) | (2 * tig + 9 < v ? 0xFFFF0000u : 0u);
        }
        const int vtok = (lane & 7) + ((lane >> 4) << 3), vhalf = (lane >> 3) & 1;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int u = ((m & 3) << 1) | vhalf;
            const uint32_t off = (2 + (m >> 2)) * 2048 + vtok * 128 + ((u ^ (vtok & 7)) << 4);
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(st[tl] + off, a0, a1, a2, a3);
                if (MASKED && tl == NTL - 1) {
                    a0 &= mlo;
                    a1 &= mlo;
                    a2 &= mhi;
                    a3 &= mhi;
                }
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    mma_bf16(acc[n][m], a0, a1, a2, a3, bh[tl][n][0], bh[tl][n][1]);
                    mma_bf16(acc[n][m], a0, a1, a2, a3, bl[tl][n][0], bl[tl][n][1]);
                }
            }
        }
    }

    // fp8 stage layout: chunk 0 = K (16 tokens x 128 bytes), chunk 1 = V, swizzled as above;
    // scale stage: 16 fp32 K scales then 16 V scales.
    template <int NTL>
    static __device__ __forceinline__ void step_fp8(const uint32_t (&st)[NTL], const float* const (&scl)[NTL],
                                                    const int (&valid)[NTL], float cq, const uint32_t (&qf)[NT][8][2],
                                                    float (&acc)[NT][8][4], float (&m2)[NT][2], float (&mt)[NT][2],
                                                    float (&ls)[NT][2], float& F, float& rF, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        constexpr int CH = NTL == 1 ? 2 : 1;
        float s[NTL][NT][4];
        {
            // K rows gid and gid+8, bytes d = 32*tig .. 32*tig+31
            uint32_t k0[NTL][8], k1[NTL][8];
            const int u0 = ((2 * tig) ^ (gid & 7)) << 4, u1 = ((2 * tig + 1) ^ (gid & 7)) << 4;
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) {
                const uint32_t r0 = st[tl] + gid * 128, r1 = st[tl] + (gid + 8) * 128;
                lds128(r0 + u0, k0[tl][0], k0[tl][1], k0[tl][2], k0[tl][3]);
                lds128(r0 + u1, k0[tl][4], k0[tl][5], k0[tl][6], k0[tl][7]);
                lds128(r1 + u0, k1[tl][0], k1[tl][1], k1[tl][2], k1[tl][3]);
                lds128(r1 + u1, k1[tl][4], k1[tl][5], k1[tl][6], k1[tl][7]);
            }
            float sx[NTL][CH][NT][4];
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl)
#pragma unroll
                for (int ch = 0; ch < CH; ++ch)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int c = 0; c < 4; ++c) sx[tl][ch][n][c] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
#pragma unroll
                for (int tl = 0; tl < NTL; ++tl) {
                    uint32_t a0, a1, a2, a3;
                    e4m3x4_to_f16x2x2(k0[tl][kk], a0, a2);
                    e4m3x4_to_f16x2x2(k1[tl][kk], a1, a3);
#pragma unroll
                    for (int n = 0; n < NT; ++n) mma_f16(sx[tl][kk % CH][n], a0, a1, a2, a3, qf[n][kk][0], qf[n][kk][1]);
                }
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int c = 0; c < 4; ++c) s[tl][n][c] = CH == 2 ? sx[tl][0][n][c] + sx[tl][CH - 1][n][c] : sx[tl][0][n][c];
        }
        // scales; the V scales are folded into P relative to the factor F
        float w0[NTL], w1[NTL];
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            const bool v0 = gid < valid[tl], v1 = gid + 8 < valid[tl];
            const float f0 = cq * scl[tl][gid], f1 = cq * scl[tl][gid + 8];
            w0[tl] = v0 ? scl[tl][16 + gid] : 0.f;
            w1[tl] = v1 ? scl[tl][24 + gid] : 0.f;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                s[tl][n][0] = v0 ? s[tl][n][0] * f0 : -INFINITY;
                s[tl][n][1] = v0 ? s[tl][n][1] * f0 : -INFINITY;
                s[tl][n][2] = v1 ? s[tl][n][2] * f1 : -INFINITY;
                s[tl][n][3] = v1 ? s[tl][n][3] * f1 : -INFINITY;
            }
        }
        float zz[NTL], zsd[NT][2], ratio = 1.f;
        if constexpr (kLazy)
            softmax_step<NTL, true, false>(s, w0, w1, zz, zz, acc, m2, mt, ls, zsd, F, rF);
        else
            ratio = eager_v_rebase<NTL>(w0, w1, F);
        uint32_t b[NTL][NT][2];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            if constexpr (!kLazy) eager_rows<NTL, true, false>(n, s, w0, w1, zz, zz, acc, m2, ls, zsd, ratio);
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) {
                b[tl][n][0] = movmatrix_trans(pack_f16(s[tl][n][0], s[tl][n][1]));
                b[tl][n][1] = movmatrix_trans(pack_f16(s[tl][n][2], s[tl][n][3]));
            }
        }
        // V: rows 2tig, 2tig+1, 2tig+8, 2tig+9; 16-byte unit gid (d = 16*gid .. 16*gid+15)
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            uint32_t vx[4], vy[4], vx2[4], vy2[4];
            const uint32_t vb = st[tl] + 2048;
            const int x = 2 * tig, y = 2 * tig + 1, x2 = 2 * tig + 8, y2 = 2 * tig + 9;
            lds128(vb + x * 128 + ((gid ^ (x & 7)) << 4), vx[0], vx[1], vx[2], vx[3]);
            lds128(vb + y * 128 + ((gid ^ (y & 7)) << 4), vy[0], vy[1], vy[2], vy[3]);
            lds128(vb + x2 * 128 + ((gid ^ (x2 & 7)) << 4), vx2[0], vx2[1], vx2[2], vx2[3]);
            lds128(vb + y2 * 128 + ((gid ^ (y2 & 7)) << 4), vy2[0], vy2[1], vy2[2], vy2[3]);
            if (valid[tl] < kTileTokens) {   // rows past the context may hold NaN codes
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (x >= valid[tl]) vx[j] = 0u;
                    if (y >= valid[tl]) vy[j] = 0u;
                    if (x2 >= valid[tl]) vx2[j] = 0u;
                    if (y2 >= valid[tl]) vy2[j] = 0u;
                }
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                // M row gid <-> d = 16*gid + 2m, M row gid+8 <-> d = 16*gid + 2m + 1
                const int j = m >> 1;
                const uint32_t sel = (m & 1) ? 0x7362u : 0x5140u;
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(__byte_perm(vx[j], vy[j], sel), a0, a1);
                e4m3x4_to_f16x2x2(__byte_perm(vx2[j], vy2[j], sel), a2, a3);
#pragma unroll
                for (int n = 0; n < NT; ++n) mma_f16(acc[n][m], a0, a1, a2, a3, b[tl][n][0], b[tl][n][1]);
            }
        }
    }

    // TQ4 stage layout: per token one 128-byte row, K codes in 16-byte units 0..3 (byte i of the
    // row holds dimensions 2i and 2i + 1, low nibble first), V codes in units 4..7, swizzled as
    // above; metadata stage: 16 k_norm, 16 v_scale, 16 v_zero (fp16).  `lut` maps a code byte to
    // the f16 pair (centroid[low nibble], centroid[high nibble]), both scaled by 2^e (cq holds 2^-e).
    template <int NTL>
    static __device__ __forceinline__ void step_tq(const uint32_t (&st)[NTL], const __half* const (&scl)[NTL],
                                                   const int (&valid)[NTL], float cq, const uint32_t* lut,
                                                   const uint32_t (&qf)[NT][8][2], float (&acc)[NT][8][4],
                                                   float (&m2)[NT][2], float (&mt)[NT][2], float (&ls)[NT][2],
                                                   float (&zs)[NT][2], float& F, float& rF, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        constexpr int CH = NTL == 1 ? 2 : 1;
        float s[NTL][NT][4];
        {
            // K codes of rows gid and gid+8, bytes 16*tig .. 16*tig+15 (dimensions 32*tig .. 32*tig+31)
            uint32_t k0[NTL][4], k1[NTL][4];
            const uint32_t u = (uint32_t)((tig ^ (gid & 7)) << 4);
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) {
                lds128(st[tl] + gid * 128 + u, k0[tl][0], k0[tl][1], k0[tl][2], k0[tl][3]);
                lds128(st[tl] + (gid + 8) * 128 + u, k1[tl][0], k1[tl][1], k1[tl][2], k1[tl][3]);
            }
            float sx[NTL][CH][NT][4];
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl)
#pragma unroll
                for (int ch = 0; ch < CH; ++ch)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int c = 0; c < 4; ++c) sx[tl][ch][n][c] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
#pragma unroll
                for (int tl = 0; tl < NTL; ++tl) {
                    // code bytes 2kk (dimensions 32tig + 4kk, +1) and 2kk + 1 (+2, +3) of each row
                    const int sh = (kk & 1) * 16;
                    const uint32_t w0 = k0[tl][kk >> 1], w1 = k1[tl][kk >> 1];
                    const uint32_t a0 = lut[(w0 >> sh) & 0xFFu], a2 = lut[(w0 >> (sh + 8)) & 0xFFu];
                    const uint32_t a1 = lut[(w1 >> sh) & 0xFFu], a3 = lut[(w1 >> (sh + 8)) & 0xFFu];
#pragma unroll
                    for (int n = 0; n < NT; ++n) mma_f16(sx[tl][kk % CH][n], a0, a1, a2, a3, qf[n][kk][0], qf[n][kk][1]);
                }
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int c = 0; c < 4; ++c) s[tl][n][c] = CH == 2 ? sx[tl][0][n][c] + sx[tl][CH - 1][n][c] : sx[tl][0][n][c];
        }
        // k_norm scales the scores; v_scale is folded into P relative to the factor F; v_zero
        // enters the per-row zero-point sum.  Tokens past the context contribute nothing (their
        // fields may hold anything, NaN included).
        float w0[NTL], w1[NTL], z0[NTL], z1[NTL];
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            const bool v0 = gid < valid[tl], v1 = gid + 8 < valid[tl];
            const float f0 = cq * __half2float(scl[tl][gid]), f1 = cq * __half2float(scl[tl][gid + 8]);
            w0[tl] = v0 ? __half2float(scl[tl][16 + gid]) : 0.f;
            w1[tl] = v1 ? __half2float(scl[tl][24 + gid]) : 0.f;
            z0[tl] = v0 ? __half2float(scl[tl][32 + gid]) : 0.f;
            z1[tl] = v1 ? __half2float(scl[tl][40 + gid]) : 0.f;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                s[tl][n][0] = v0 ? s[tl][n][0] * f0 : -INFINITY;
                s[tl][n][1] = v0 ? s[tl][n][1] * f0 : -INFINITY;
                s[tl][n][2] = v1 ? s[tl][n][2] * f1 : -INFINITY;
                s[tl][n][3] = v1 ? s[tl][n][3] * f1 : -INFINITY;
            }
        }
        float ratio = 1.f;
        if constexpr (kLazy)
            softmax_step<NTL, true, true>(s, w0, w1, z0, z1, acc, m2, mt, ls, zs, F, rF);
        else
            ratio = eager_v_rebase<NTL>(w0, w1, F);
        uint32_t b[NTL][NT][2];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            if constexpr (!kLazy) eager_rows<NTL, true, true>(n, s, w0, w1, z0, z1, acc, m2, ls, zs, ratio);
#pragma unroll
            for (int tl = 0; tl < NTL; ++tl) {
                b[tl][n][0] = movmatrix_trans(pack_f16(s[tl][n][0], s[tl][n][1]));
                b[tl][n][1] = movmatrix_trans(pack_f16(s[tl][n][2], s[tl][n][3]));
            }
        }
        // V codes by ldmatrix.trans: matrix (token half th, V code unit k = 16-byte unit 4 + k of the
        // row) is 8 tokens x 8 code pairs; lane (gid, tig) receives, for tokens 8th + 2tig and
        // 8th + 2tig + 1 (low and high half), the code pair at bytes 16k + 2gid, 16k + 2gid + 1, i.e.
        // dimensions 32k + 4gid + e, e = 0..3 in bits 4e .. 4e+3 of each half.  M rows of chunk m:
        // gid <-> d = 32(m >> 1) + 4gid + 2(m & 1), gid+8 <-> d + 1.  A code enters the MMA as an
        // f16 subnormal, exactly: the low nibble of a byte as c * 2^-24, the high nibble, unshifted,
        // as 16c * 2^-24 (the epilogue scales rows gid by 2^24 and rows gid+8 by 2^20).
        const int lmat = lane >> 3, vtok = 8 * (lmat & 1) + (lane & 7);
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            uint32_t z[2][4];   // [kp][th + 2 * (k & 1)] for k = 2kp + (k & 1)
#pragma unroll
            for (int kp = 0; kp < 2; ++kp) {
                const int u = 4 + 2 * kp + (lmat >> 1);
                ldsm_x4_trans(st[tl] + vtok * 128 + ((u ^ (vtok & 7)) << 4), z[kp][0], z[kp][1], z[kp][2], z[kp][3]);
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int k = m >> 1;
                const uint32_t x0 = z[k >> 1][2 * (k & 1)], x1 = z[k >> 1][2 * (k & 1) + 1];   // token halves
                const uint32_t y0 = (m & 1) ? (x0 >> 8) : x0, y1 = (m & 1) ? (x1 >> 8) : x1;
                const uint32_t a0 = y0 & 0x000F000Fu, a1 = y0 & 0x00F000F0u;
                const uint32_t a2 = y1 & 0x000F000Fu, a3 = y1 & 0x00F000F0u;
#pragma unroll
                for (int n = 0; n < NT; ++n) mma_f16(acc[n][m], a0, a1, a2, a3, b[tl][n][0], b[tl][n][1]);
            }
        }
    }

    // ------------------------------------------------------------------ fused step: output
    static __device__ __forceinline__ void store_out(const DecodeArgs& a, long long orow, int lane, float4 v) {
        if (a.out_f32) {
            *reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow * kHeadDim + (lane << 2)) = v;
        } else {
            uint2 u;
            u.x = pack_bf16(v.x, v.y);
            u.y = pack_bf16(v.z, v.w);
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow * kHeadDim + (lane << 2)) = u;
        }
    }
    // The fused step's reduce, after the partition pass of every CTA: a grid barrier (the launch is
    // cooperative, so every CTA is resident and the bounded wait ends), then the CTAs (one warp
    // each) take the output rows round robin and merge each with merge_row, the arithmetic of the
    // reduce kernel (same bits as pda_decode + pda_reduce).  A row of a single-partition unit was
    // written by that unit's epilogue; a row of a sequence without tokens is written as zeros.
    // The launch's counter slot {arrived, left} is zero at launch; its last CTA to leave resets it.
    static __device__ __noinline__ void finish_fused(const DecodeArgs& a, int lane, bool ok) {
        unsigned int* const bar = a.sched;
        const bool alone = gridDim.x == 1;   // one CTA: it waits for no one and counts nothing
        if (!alone) __threadfence();         // this CTA's partials and statistics, before it is counted
        __syncwarp();
        int arrived = alone ? 1 : 0;
        if (lane == 0 && !alone) {
            atomicAdd(bar, 1u);
            const uint64_t t0 = global_timer_ns();
            unsigned int backoff = 32;
            while ((arrived = ld_acquire_gpu(reinterpret_cast<const int*>(bar))) < (int)gridDim.x) {
                if (global_timer_ns() - t0 > a.timeout_ns) break;
                __nanosleep(backoff);
                backoff = min(backoff * 2, 256u);
            }
        }
        arrived = __shfl_sync(kFull, arrived, 0);
        if (arrived < (int)gridDim.x) {
            ok = false;
        } else {
            const MergeArgs mg{a.partial_out, a.exp_sums, a.max_logits, a.out, a.Hk, a.QG, a.P, a.W, a.out_f32};
            const int max_ctx = a.MB * a.BS;
            const long long rows = (long long)a.B * a.Hk * a.QG, rps = (long long)a.Hk * a.QG;
            int cb = -1, c = 0;   // the last sequence whose context length was read, and that length
            for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
                const int b = (int)(row / rps);
                const int rem = (int)(row - (long long)b * rps);
                const int h = rem / a.QG, q = rem - h * a.QG;
                if (b != cb) {
                    cb = b;
                    c = sanitize_ctx(__ldcg(a.context_lens + b), max_ctx);
                }
                if ((c + a.W - 1) / a.W == 1) continue;   // written by the unit's epilogue
                merge_row(mg, b, h, q, c);
            }
        }
        if (lane == 0) {
            if (!ok && a.err_word) atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
            if (!alone) {
                __threadfence();
                if (atomicAdd(bar + 1, 1u) == gridDim.x - 1) {   // every CTA has left the barrier
                    bar[0] = 0u;
                    bar[1] = 0u;
                }
            }
        }
        __syncwarp();
    }

    // ------------------------------------------------------------------ the warp
    static __device__ void run(const DecodeArgs& a, const CUtensorMap* kv_map, const CUtensorMap* sc_map,
                               uint8_t* smem, uint32_t* tq_lut) {
        const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
        const uint32_t sbase = smem_addr(smem);
        const uint32_t bar0 = sbase + Cfg::kOffBar;
        if (lane == 0) {
            for (int s = 0; s < S; ++s) mbar_init(bar0 + 8 * s, 1);
            fence_mbar_init();
            prefetch_tensormap(kv_map);
            if (F16) prefetch_tensormap(sc_map);
        }
        __syncwarp();
        allow_dependent_launch();   // the reduce may be scheduled as soon as CTAs of this grid retire
        grid_dependency_wait();     // inputs may come from the previous grid on the stream

        UnitIt cu;
        long long hi;
        find_range(a, cu, hi);
        if (!(cu.b < a.B && cu.start < hi)) {
            if constexpr (FUSED) finish_fused(a, lane, true);
            return;
        }

        // Q rows and the first block-table entries are requested before anything waits
        uint32_t qn[NT][16];
        load_q(a, cu, qn, lane);
        float cent = 0.f;
        if constexpr (TQ) cent = __ldg(a.centroids + (lane & 15));
        Feed f;
        feed_init(a, hi, cu, f, lane);
        // fill the ring, then look up the next chunk
        long long issued = 0;
        for (int s = 0; s < S; ++s)
            if (feed_one(a, hi, kv_map, sc_map, sbase, bar0 + 8 * s, s, f, lane)) ++issued;
        if (f.valid && !f.pf) prefetch_next(a, hi, f, lane);

        // TQ4: the 16 centroids, scaled by a power of two into f16 range (each keeps 11 significant
        // bits), as a table of f16 pairs indexed by one byte of codes (low nibble -> low half)
        const uint32_t* lut = tq_lut;
        float cscale = 1.f;
        if constexpr (TQ) {
            float amax = fabsf(cent);
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
            int e = 0;
            if (amax > 0.f) e = 14 - ((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127);
            e = max(-100, min(100, e));
            cscale = __uint_as_float((uint32_t)(127 - e) << 23);
            const uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn(cent * __uint_as_float((uint32_t)(e + 127) << 23)));
            uint32_t* lut_w = tq_lut;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int x = 8 * lane + i;   // code byte: low nibble 8*(lane&1) + i, high nibble lane/2
                const uint32_t lo = __shfl_sync(kFull, h, x & 15), hi16 = __shfl_sync(kFull, h, x >> 4);
                lut_w[x] = lo | (hi16 << 16);
            }
            __syncwarp();
        }

        int cs = 0;                          // next stage to consume and its barrier phase
        uint32_t cph = 0;
        bool ok = true;
        // Q fragments of the current unit.  The f16 kernels with QG <= 8 rebuild them only when the
        // unit's (sequence, head) differs from the previous unit's (consecutive partitions of one
        // head share their Q rows; the conversion to f16 costs ~0.6 us of a warp per unit).  The
        // others rebuild them every unit: keeping them across the epilogue costs registers (QG = 16
        // measured 5 % slower), and for bf16 they are plain register moves.
        constexpr bool kKeepQ = F16 && NT == 1;
        uint32_t qf[NT][8][2];
        float cq = a.qk_scale_log2;
        bool new_q = true;
        while (ok) {
            // ---- unit start: Q fragments, next unit's Q in flight
            if (!new_q) {
            } else if constexpr (!F16) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        qf[n][kk][0] = qn[n][2 * kk];
                        qf[n][kk][1] = qn[n][2 * kk + 1];
                    }
            } else {
                float amax = 0.f;
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(qn[n][c])), fabsf(bf16_hi(qn[n][c]))));
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
                // a power of two that brings the largest |q| into [2^14, 2^15): f16 keeps every bf16 bit
                int e = 0;
                if (amax > 0.f) e = 14 - ((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127);
                e = max(-100, min(100, e));
                const float pw = __uint_as_float((uint32_t)(e + 127) << 23);
                cq = a.qk_scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23) * cscale;
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t x = qn[n][2 * kk], y = qn[n][2 * kk + 1];
                        qf[n][kk][0] = pack_f16(bf16_lo(x) * pw, bf16_hi(x) * pw);
                        qf[n][kk][1] = pack_f16(bf16_lo(y) * pw, bf16_hi(y) * pw);
                    }
            }
            UnitIt nx = cu;
            it_advance(nx, a);
            const bool has_next = nx.b < a.B && nx.start < hi;
            const bool other_rows = nx.b != cu.b || nx.h != cu.h;
            if (has_next && other_rows) load_q(a, nx, qn, lane);   // else: same rows
            new_q = !kKeepQ || (has_next && other_rows);

            float acc[NT][8][4];
            float m2[NT][2], mt[NT][2], ls[NT][2], zs[NT][2];
            float F = 1.f, rF = 1.f;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
#pragma unroll
                for (int m = 0; m < 8; ++m) acc[n][m][0] = acc[n][m][1] = acc[n][m][2] = acc[n][m][3] = 0.f;
                m2[n][0] = m2[n][1] = -INFINITY;
                mt[n][0] = mt[n][1] = -INFINITY;
                ls[n][0] = ls[n][1] = 0.f;
                zs[n][0] = zs[n][1] = 0.f;
            }
            const int nt = unit_tiles(cu, a.W);
            const int tok_base = cu.p * a.W;
            int stage = 0;
            for (int t = 0; t < nt;) {
                const bool two = t + 1 < nt;
                const int s0 = cs;
                const uint32_t ph0 = cph;
                const int s1 = s0 + 1 == S ? 0 : s0 + 1;
                const uint32_t ph1 = s0 + 1 == S ? cph ^ 1u : cph;
                if (!mbar_wait(bar0 + 8 * s0, ph0, a.timeout_ns) || (two && !mbar_wait(bar0 + 8 * s1, ph1, a.timeout_ns))) {
                    ok = false;
                    break;
                }
                const int v0 = cu.ctx - (tok_base + t * kTileTokens);
                if (two) {
                    const uint32_t st[2] = {sbase + Cfg::kOffStages + s0 * Cfg::kTileBytes,
                                            sbase + Cfg::kOffStages + s1 * Cfg::kTileBytes};
                    const int vv[2] = {v0, v0 - kTileTokens};
                    if constexpr (TQ) {
                        const __half* const sc[2] = {
                            reinterpret_cast<const __half*>(smem + Cfg::kOffScales + s0 * Cfg::kScaleBytes),
                            reinterpret_cast<const __half*>(smem + Cfg::kOffScales + s1 * Cfg::kScaleBytes)};
                        step_tq<2>(st, sc, vv, cq, lut, qf, acc, m2, mt, ls, zs, F, rF, lane);
                    } else if constexpr (FP8) {
                        const float* const sc[2] = {
                            reinterpret_cast<const float*>(smem + Cfg::kOffScales + s0 * Cfg::kScaleBytes),
                            reinterpret_cast<const float*>(smem + Cfg::kOffScales + s1 * Cfg::kScaleBytes)};
                        step_fp8<2>(st, sc, vv, cq, qf, acc, m2, mt, ls, F, rF, lane);
                    } else {
                        step_bf16<2>(st, vv, a.qk_scale_log2, qf, acc, m2, mt, ls, lane);
                    }
                } else {
                    const uint32_t st[1] = {sbase + Cfg::kOffStages + s0 * Cfg::kTileBytes};
                    const int vv[1] = {v0};
                    if constexpr (TQ) {
                        const __half* const sc[1] = {
                            reinterpret_cast<const __half*>(smem + Cfg::kOffScales + s0 * Cfg::kScaleBytes)};
                        step_tq<1>(st, sc, vv, cq, lut, qf, acc, m2, mt, ls, zs, F, rF, lane);
                    } else if constexpr (FP8) {
                        const float* const sc[1] = {
                            reinterpret_cast<const float*>(smem + Cfg::kOffScales + s0 * Cfg::kScaleBytes)};
                        step_fp8<1>(st, sc, vv, cq, qf, acc, m2, mt, ls, F, rF, lane);
                    } else {
                        step_bf16<1>(st, vv, a.qk_scale_log2, qf, acc, m2, mt, ls, lane);
                    }
                }
                __syncwarp();
                const int used = two ? 2 : 1;
                t += used;
                stage = two ? s1 : s0;
                // refill the stages just consumed, in tile order; the unit's last stage is kept for
                // the epilogue and refilled after it
                if (t < nt) {
                    if (feed_one(a, hi, kv_map, sc_map, sbase, bar0 + 8 * s0, s0, f, lane)) ++issued;
                    if (two && feed_one(a, hi, kv_map, sc_map, sbase, bar0 + 8 * s1, s1, f, lane)) ++issued;
                } else if (two) {
                    if (feed_one(a, hi, kv_map, sc_map, sbase, bar0 + 8 * s0, s0, f, lane)) ++issued;
                }
                cs = two ? (s1 + 1 == S ? 0 : s1 + 1) : s1;
                cph = two ? (s1 + 1 == S ? ph1 ^ 1u : ph1) : ph1;
            }
            if (!ok) break;

            // ---- epilogue: the last stage is free; stage the normalised partial through it
            // o = acc * F / l (F: the V-scale factor; TQ4 codes carry another 2^24, or 2^20 for the
            // high nibbles), plus, for TQ4, the zero-point sum z / l.  acc, l and z all count from
            // the reference point m2; the stored statistics count from the true maximum M:
            // m_p = M, l_p = l * 2^(m2 - M).
            float inv[NT][2], zq[NT][2];
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float l = ls[n][j];
                    l += __shfl_xor_sync(kFull, l, 4);
                    l += __shfl_xor_sync(kFull, l, 8);
                    l += __shfl_xor_sync(kFull, l, 16);
                    if constexpr (kLazy) {
                        float M = mt[n][j];
                        M = fmaxf(M, __shfl_xor_sync(kFull, M, 4));
                        M = fmaxf(M, __shfl_xor_sync(kFull, M, 8));
                        M = fmaxf(M, __shfl_xor_sync(kFull, M, 16));
                        ls[n][j] = M == -INFINITY ? l : l * ex2(m2[n][j] - M);
                        mt[n][j] = M;
                    } else {
                        ls[n][j] = l;
                        mt[n][j] = m2[n][j];
                    }
                    const float il = l > 0.f ? 1.f / l : 0.f;
                    inv[n][j] = il * (FP8 ? F : TQ ? F * 16777216.f : 1.f);
                    zq[n][j] = 0.f;
                    if constexpr (TQ) {
                        float z = zs[n][j];
                        z += __shfl_xor_sync(kFull, z, 4);
                        z += __shfl_xor_sync(kFull, z, 8);
                        z += __shfl_xor_sync(kFull, z, 16);
                        zq[n][j] = z * il;
                    }
                }
            float* stg = reinterpret_cast<float*>(smem + Cfg::kOffStages + stage * Cfg::kTileBytes);
            const long long row0 = ((long long)(cu.b * a.Hk + cu.h) * a.P + cu.p) * a.QG;
            // one stage holds 16 (bf16), 8 (fp8) or 4 (TQ4) rows of the partial: a pass stages that many
            // rows, at most the unit's 8*NT
            constexpr int kStageRows = Cfg::kTileBytes / (kHeadDim * 4);
            constexpr int kPassRows = kStageRows < NT * 8 ? kStageRows : NT * 8;
#pragma unroll
            for (int r0 = 0; r0 < NT * 8; r0 += kPassRows) {
                // write [row][d] floats of rows r0 .. r0 + kPassRows - 1 (local row ql = q - r0), 16-byte
                // chunk c of local row ql stored at c ^ (ql & 6)
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if (n * 8 + 8 <= r0 || n * 8 >= r0 + kPassRows) continue;
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        if constexpr (F16) {
                            // elements c and c + 2 are dimensions d and d + 1 of one row: one 8-byte store
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int ql = n * 8 + 2 * tig + j - r0;
                                if (ql < 0 || ql >= kPassRows) continue;   // a pass of 4 rows holds half an n-tile
                                const int d = TQ ? (32 * (m >> 1) + 4 * gid + 2 * (m & 1)) : (16 * gid + 2 * m);
                                float2 v;
                                if constexpr (TQ) {
                                    v.x = fmaf(acc[n][m][j], inv[n][j], zq[n][j]);
                                    v.y = fmaf(acc[n][m][j + 2], inv[n][j] * 0.0625f, zq[n][j]);
                                } else {
                                    v.x = acc[n][m][j] * inv[n][j];
                                    v.y = acc[n][m][j + 2] * inv[n][j];
                                }
                                *reinterpret_cast<float2*>(stg + ql * kHeadDim + ((((d >> 2) ^ (ql & 6))) << 2) + (d & 3)) = v;
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const int ql = n * 8 + 2 * tig + (c & 1) - r0;
                                if (ql < 0 || ql >= kPassRows) continue;
                                const int d = 16 * m + gid + 8 * (c >> 1);
                                stg[ql * kHeadDim + ((((d >> 2) ^ (ql & 6))) << 2) + (d & 3)] = acc[n][m][c] * inv[n][c & 1];
                            }
                        }
                    }
                }
                __syncwarp();
                const int rows = min(kPassRows, a.QG - r0);
                if (FUSED && cu.nv == 1) {   // the partial is the output (the reduce would copy it)
                    const long long orow = (long long)cu.b * a.Hk * a.QG + (long long)cu.h * a.QG + r0;
                    for (int q = 0; q < rows; ++q) {
                        const float4 v = *reinterpret_cast<const float4*>(stg + q * kHeadDim + ((lane ^ (q & 6)) << 2));
                        store_out(a, orow + q, lane, v);
                    }
                } else {
                    for (int q = 0; q < rows; ++q) {
                        const float4 v = *reinterpret_cast<const float4*>(stg + q * kHeadDim + ((lane ^ (q & 6)) << 2));
                        *reinterpret_cast<float4*>(a.partial_out + (row0 + r0 + q) * kHeadDim + (lane << 2)) = v;
                    }
                }
                __syncwarp();
            }
            if (gid == 0 && !(FUSED && cu.nv == 1)) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int q = n * 8 + 2 * tig + j;
                        if (q < a.QG) {
                            a.exp_sums[row0 + q] = ls[n][j];
                            a.max_logits[row0 + q] = mt[n][j] * kLn2;
                        }
                    }
            }
            // the staging stage goes back to the feed (its generic writes precede the copy)
            fence_proxy_async_shared();
            if (feed_one(a, hi, kv_map, sc_map, sbase, bar0 + 8 * stage, stage, f, lane)) ++issued;
            if (!has_next) break;
            cu = nx;
        }
        if (!ok) {
            if (lane == 0) {
                if (a.err_word) atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
                // wait (bounded, by the default limit whatever the plan asked for) for the last copy
                // issued into every stage: no copy may land in this CTA's memory after it leaves
                for (int s = 0; s < S; ++s) {
                    if (issued <= s) continue;
                    const long long j = s + ((issued - 1 - s) / S) * S;
                    (void)mbar_wait(bar0 + 8 * s, (uint32_t)((j / S) & 1), kDefaultTimeoutNs);
                }
            }
            __syncwarp();
        }
        if constexpr (FUSED) finish_fused(a, lane, ok);
    }
};

// MINB: CTAs per SM the register allocation must allow (more resident warps hide the latency of
// each warp's serial chain of loads, MMAs and shuffles).
template <int KV, int NT, int S, int MINB, bool FUSED>
__global__ void __launch_bounds__(32, MINB) pda_partition_kernel(const __grid_constant__ CUtensorMap kv_map,
                                                          const __grid_constant__ CUtensorMap sc_map,
                                                          const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // TQ4 centroid table: static, so that its lookups address it with an immediate offset
    __shared__ uint32_t tq_lut[KV == PDA_KV_TQ4 ? 256 : 1];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Decode<KV, NT, S, FUSED>::run(a, &kv_map, &sc_map, smem, tq_lut);
}

}  // namespace pda
