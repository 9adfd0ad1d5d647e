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
//   * Persistent, tile-balanced grid: every CTA takes the units whose first tile falls in its
//     equal share of all tiles of the step, so empty partitions cost nothing and long and
//     short contexts spread evenly over the SMs.
//   * One producer warp per CTA: it walks the block table (entries loaded 32 at a time, one
//     chunk ahead) and issues ONE 5-D TMA tensor copy per 16-token tile (K and V of one KV
//     head, 8 KB bf16 / 4 KB fp8, 128-byte swizzle) into an S-stage ring guarded by
//     mbarriers; for fp8 a second 4-D TMA copy brings the tile's 16 K and 16 V scales.
//   * NW consumer warps split the tiles of a unit; per tile: S^T = K Q^T and O^T += V^T P^T
//     with warp-level mma.sync (m16n8k16, fp32 accumulate).  Tokens are the M dimension of
//     the score MMA so QG = 8 fills it; P is moved to the B-operand layout with movmatrix.
//   * bf16 KV: bf16 MMAs, P split into bf16 hi + lo parts (two PV MMAs) so P keeps ~16 bits.
//     fp8 KV: e4m3 -> f16 conversion (exact), Q scaled by a power of two into f16 range,
//     K scales applied to the fp32 scores, V scales folded into P relative to the tile's
//     largest V scale (the factor is carried in the running rescale).
//   * Warps merge their (max, sum, acc) through shared memory at the end of a unit and
//     write the partial with coalesced 16-byte stores.
//   * Every wait is bounded; a wait that gives up sets PDA_ERRW_PIPELINE_TIMEOUT and the
//     CTA leaves collectively (bar.red.or) after draining its own copies in flight.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "pda.h"
#include "pda_internal.h"
#include "pda_ptx.cuh"

namespace pda {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kFull = 0xFFFFFFFFu;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

struct UnitInfo {
    int b, h, p, nt, ctx, pad0, pad1, pad2;
};

struct Misc {
    long long warp_sums[16];
    long long start_tile, hi_tile;
    int b, h, p, pad;
};

template <bool FP8, int NT, int NW, int S>
struct DecodeCfg {
    static constexpr int kThreads = (NW + 1) * 32;
    static constexpr int kTileBytes = FP8 ? 4096 : 8192;   // K and V of 16 tokens of one KV head
    static constexpr int kChunks = FP8 ? 2 : 4;             // 128-byte chunks per token-head
    static constexpr int kScaleBytes = FP8 ? 128 : 0;       // 16 K scales + 16 V scales
    static constexpr int kQRows = NT * 8;
    static constexpr int kQBytes = kQRows * 256;
    static constexpr int kMStride = 132;                    // floats per row of the merge buffer
    static constexpr int kMergeFloats = kQRows * kMStride + 2 * kQRows;
    static constexpr int kOffStages = 0;
    static constexpr int kOffScales = kOffStages + S * kTileBytes;
    static constexpr int kOffQ = align_up(kOffScales + S * kScaleBytes, 128);
    static constexpr int kOffMerge = kOffQ + 2 * kQBytes;
    static constexpr int kOffInfo = align_up(kOffMerge + NW * kMergeFloats * 4, 16);
    static constexpr int kOffBar = kOffInfo + 2 * (int)sizeof(UnitInfo);
    static constexpr int kNumBars = 2 * S + 4;
    static constexpr int kOffMisc = align_up(kOffBar + kNumBars * 8, 16);
    static constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc) + 1024;   // + base alignment slack
};

// ---------------------------------------------------------------------------------------------
// unit iteration (same order in every CTA and role): sequences b ascending, then KV head h,
// then partition p; a unit's first tile index is its position in that order counted in tiles.
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

// All threads: count the tiles of the step, split them evenly over the grid and find the first
// unit of this CTA.  Sets the data-error bit for out-of-range context lengths (CTA 0 only).
__device__ inline void find_range(const DecodeArgs& a, Misc* misc) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int max_ctx = a.MB * a.BS;
    const int per = (a.B + nthr - 1) / nthr;
    const int b0 = min(a.B, tid * per), b1 = min(a.B, b0 + per);
    long long mine = 0;
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
        const int raw = __ldg(a.context_lens + b);
        if (raw < 0 || raw > max_ctx) bad = true;
        mine += (long long)a.Hk * ((sanitize_ctx(raw, max_ctx) + 15) >> 4);
    }
    if (bad && blockIdx.x == 0 && a.err_word) atomicOr(a.err_word, PDA_ERRW_BAD_CONTEXT_LEN);
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) misc->warp_sums[warp] = incl;
    if (tid == 0) {
        misc->b = a.B;   // "no unit" unless a thread below finds one
        misc->h = 0;
        misc->p = 0;
        misc->start_tile = 0;
    }
    __syncthreads();
    long long before = 0, total = 0;
    const int nwarps = nthr >> 5;
    for (int w = 0; w < nwarps; ++w) {
        const long long s = misc->warp_sums[w];
        if (w < warp) before += s;
        total += s;
    }
    const long long excl = before + incl - mine;
    const long long lo = (long long)blockIdx.x * total / gridDim.x;
    const long long hi = ((long long)blockIdx.x + 1) * total / gridDim.x;
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
                int p = (int)((r + tp - 1) / tp);             // first unit starting at or after lo
                const int nv = (c + a.W - 1) / a.W;
                if (p >= nv) {
                    p = 0;
                    ++h;
                }
                if (h < a.Hk) {
                    misc->b = b;
                    misc->h = h;
                    misc->p = p;
                    misc->start_tile = pos + h * th + p * tp;
                } else {            // the next sequence's first unit (empty sequences are skipped later)
                    misc->b = b + 1;
                    misc->h = 0;
                    misc->p = 0;
                    misc->start_tile = pos + tb;
                }
                break;
            }
            pos += tb;
        }
    }
    if (tid == 0) misc->hi_tile = hi;
    __syncthreads();
}

__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------------------------------------
template <bool FP8, int NT, int NW, int S>
struct Decode {
    using Cfg = DecodeCfg<FP8, NT, NW, S>;

    // barrier addresses
    struct Bars {
        uint32_t base;
        __device__ uint32_t full(int s) const { return base + 8u * s; }
        __device__ uint32_t empty(int s) const { return base + 8u * (S + s); }
        __device__ uint32_t qfull(int i) const { return base + 8u * (2 * S + i); }
        __device__ uint32_t qempty(int i) const { return base + 8u * (2 * S + 2 + i); }
    };

    // ------------------------------------------------------------------ producer (one warp)
    static __device__ int load_entry(const DecodeArgs& a, const UnitIt& u, int e0, int lane) {
        const int nent = (unit_tokens(u, a.W) + a.BS - 1) / a.BS;
        const int idx = e0 + lane;
        if (idx >= nent) return 0;
        return __ldg(a.block_table + (long long)u.b * a.MB + (u.p * a.W) / a.BS + idx);
    }
    static __device__ void next_chunk(const DecodeArgs& a, long long hi, const UnitIt& u, int e0, UnitIt& nu,
                                      int& ne0, bool& nvalid) {
        const int nent = (unit_tokens(u, a.W) + a.BS - 1) / a.BS;
        nu = u;
        if (e0 + 32 < nent) {
            ne0 = e0 + 32;
            nvalid = true;
        } else {
            it_advance(nu, a);
            ne0 = 0;
            nvalid = nu.b < a.B && nu.start < hi;
        }
    }

    static __device__ void producer(const DecodeArgs& a, const CUtensorMap* kv_map, const CUtensorMap* sc_map,
                                    uint8_t* smem, Bars bars, Misc* misc, UnitInfo* info) {
        const int lane = threadIdx.x & 31;
        const uint32_t sbase = smem_addr(smem);
        const long long hi = misc->hi_tile;
        UnitIt u;
        u.b = misc->b;
        u.h = misc->h;
        u.p = misc->p;
        u.start = misc->start_tile;
        u.ctx = 0;
        u.nv = 0;
        it_settle(u, a);

        long long tile_i = 0;
        int ucount = 0;
        bool ok = true;
        bool cvalid = u.b < a.B && u.start < hi;
        int ce0 = 0;
        int cent = cvalid ? load_entry(a, u, 0, lane) : 0;
        UnitIt nu = u;
        int ne0 = 0, nent = 0;
        bool nvalid = false;
        if (cvalid) {
            next_chunk(a, hi, u, 0, nu, ne0, nvalid);
            if (nvalid) nent = load_entry(a, nu, ne0, lane);
        }
        const int tpe = a.BS >> 4;   // 16-token tiles per block-table entry (1 or 2)
        while (cvalid && ok) {
            if (ce0 == 0) {          // unit header: its description and its Q rows
                if (lane == 0) {
                    const int slot = ucount & 1;
                    if (ucount >= 2) ok = mbar_wait(bars.qempty(slot), ((ucount >> 1) - 1) & 1, a.timeout_ns);
                    if (ok) {
                        UnitInfo ui;
                        ui.b = u.b;
                        ui.h = u.h;
                        ui.p = u.p;
                        ui.nt = unit_tiles(u, a.W);
                        ui.ctx = u.ctx;
                        ui.pad0 = ui.pad1 = ui.pad2 = 0;
                        info[slot] = ui;
                        const uint32_t qbytes = (uint32_t)a.QG * 256u;
                        mbar_arrive_expect_tx(bars.qfull(slot), qbytes);
                        const uint16_t* src = a.query + ((long long)u.b * a.Hk * a.QG + (long long)u.h * a.QG) * kHeadDim;
                        bulk_load(sbase + Cfg::kOffQ + slot * Cfg::kQBytes, src, qbytes, bars.qfull(slot));
                    }
                }
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok) break;
                ++ucount;
            }
            const int nt = unit_tiles(u, a.W);
            const int t_begin = ce0 * tpe;
            const int t_end = min(nt, (ce0 + 32) * tpe);
            for (int t = t_begin; t < t_end; ++t) {
                const int phys = __shfl_sync(kFull, cent, t / tpe - ce0);
                if (lane == 0) {
                    const int stage = (int)(tile_i % S);
                    const long long round = tile_i / S;
                    if (tile_i >= S) ok = mbar_wait(bars.empty(stage), (uint32_t)((round - 1) & 1), a.timeout_ns);
                    if (ok) {
                        const int slot0 = (t & (tpe - 1)) * kTileTokens;
                        mbar_arrive_expect_tx(bars.full(stage), Cfg::kTileBytes + Cfg::kScaleBytes);
                        tma_load_5d(sbase + Cfg::kOffStages + stage * Cfg::kTileBytes, kv_map, bars.full(stage), 0,
                                    slot0, 0, u.h, phys);
                        if constexpr (FP8)
                            tma_load_4d(sbase + Cfg::kOffScales + stage * Cfg::kScaleBytes, sc_map, bars.full(stage),
                                        slot0, 0, u.h, phys);
                        if ((phys < 0 || (long long)phys >= a.num_cache_blocks) && a.err_word)
                            atomicOr(a.err_word, PDA_ERRW_BAD_BLOCK_ID);
                    }
                }
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok) break;
                ++tile_i;
            }
            u = nu;
            ce0 = ne0;
            cvalid = nvalid;
            cent = nent;
            if (cvalid && ok) {
                next_chunk(a, hi, u, ce0, nu, ne0, nvalid);
                nent = nvalid ? load_entry(a, nu, ne0, lane) : 0;
            }
        }
        if (lane == 0) {
            if (ok) {            // end marker: a header with nt = -1 and no bytes
                const int slot = ucount & 1;
                if (ucount >= 2) ok = mbar_wait(bars.qempty(slot), ((ucount >> 1) - 1) & 1, a.timeout_ns);
                if (ok) {
                    info[slot].nt = -1;
                    mbar_arrive(bars.qfull(slot));
                }
            }
            if (!ok) {
                if (a.err_word) atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
                // drain: wait (bounded) for the last copy issued into every stage and Q slot
                for (int s = 0; s < S; ++s) {
                    if (tile_i <= s) continue;
                    const long long j = s + ((tile_i - 1 - s) / S) * S;   // last issued tile that used stage s
                    (void)mbar_wait(bars.full(s), (uint32_t)((j / S) & 1), a.timeout_ns);
                }
                for (int k = ucount - 1; k >= 0 && k >= ucount - 2; --k)
                    (void)mbar_wait(bars.qfull(k & 1), (uint32_t)((k >> 1) & 1), a.timeout_ns);
            }
        }
        __syncwarp();
    }

    // ------------------------------------------------------------------ consumer tile math
    // bf16 K/V.  Stage layout: chunk c (K0 = d 0..63, K1, V0, V1) x 16 tokens x 128 bytes,
    // 16-byte units swizzled by (token & 7).
    static __device__ __forceinline__ void tile_bf16(uint32_t st, int valid, float scale2, const uint32_t (&qf)[NT][8][2],
                                                     float (&acc)[NT][8][4], float (&m2)[NT][2], float (&ls)[NT][2],
                                                     int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        float s[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
        const int ktok = lane & 15, khalf = lane >> 4;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int u = ((kk & 3) << 1) | khalf;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(st + (kk >> 2) * 2048 + ktok * 128 + ((u ^ (ktok & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
            for (int n = 0; n < NT; ++n) mma_bf16(s[n], a0, a1, a2, a3, qf[n][kk][0], qf[n][kk][1]);
        }
        const bool v0 = gid < valid, v1 = gid + 8 < valid;
        uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            s[n][0] = v0 ? s[n][0] * scale2 : -INFINITY;
            s[n][1] = v0 ? s[n][1] * scale2 : -INFINITY;
            s[n][2] = v1 ? s[n][2] * scale2 : -INFINITY;
            s[n][3] = v1 ? s[n][3] * scale2 : -INFINITY;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = fmaxf(s[n][j], s[n][j + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
                const float mnew = fmaxf(m2[n][j], mx);
                const float alpha = ex2(m2[n][j] - mnew);
                m2[n][j] = mnew;
                const float p0 = ex2(s[n][j] - mnew), p1 = ex2(s[n][j + 2] - mnew);
                s[n][j] = p0;
                s[n][j + 2] = p1;
                ls[n][j] = ls[n][j] * alpha + (p0 + p1);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    acc[n][m][j] *= alpha;
                    acc[n][m][j + 2] *= alpha;
                }
            }
            const uint32_t h01 = pack_bf16(s[n][0], s[n][1]);
            const uint32_t h23 = pack_bf16(s[n][2], s[n][3]);
            const uint32_t l01 = pack_bf16(s[n][0] - bf16_lo(h01), s[n][1] - bf16_hi(h01));
            const uint32_t l23 = pack_bf16(s[n][2] - bf16_lo(h23), s[n][3] - bf16_hi(h23));
            bh[n][0] = movmatrix_trans(h01);
            bh[n][1] = movmatrix_trans(h23);
            bl[n][0] = movmatrix_trans(l01);
            bl[n][1] = movmatrix_trans(l23);
        }
        // V rows past the context may hold anything (NaN included): zero them, 0 * NaN = NaN.
        uint32_t mlo = kFull, mhi = kFull;
        if (valid < kTileTokens) {
            mlo = (2 * tig < valid ? 0x0000FFFFu : 0u) | (2 * tig + 1 < valid ? 0xFFFF0000u : 0u);
            mhi = (2 * tig + 8 < valid ? 0x0000FFFFu : 0u) | (2 * tig + 9 < valid ? 0xFFFF0000u : 0u);
        }
        const int vtok = (lane & 7) + ((lane >> 4) << 3), vhalf = (lane >> 3) & 1;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int u = ((m & 3) << 1) | vhalf;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(st + (2 + (m >> 2)) * 2048 + vtok * 128 + ((u ^ (vtok & 7)) << 4), a0, a1, a2, a3);
            a0 &= mlo;
            a1 &= mlo;
            a2 &= mhi;
            a3 &= mhi;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                mma_bf16(acc[n][m], a0, a1, a2, a3, bh[n][0], bh[n][1]);
                mma_bf16(acc[n][m], a0, a1, a2, a3, bl[n][0], bl[n][1]);
            }
        }
    }

    // fp8 K/V.  Stage layout: chunk 0 = K (16 tokens x 128 bytes), chunk 1 = V, swizzled as
    // above; scale stage: 16 fp32 K scales then 16 V scales.
    static __device__ __forceinline__ void tile_fp8(uint32_t st, const float* scl, int valid, float cq,
                                                    const uint32_t (&qf)[NT][8][2], float (&acc)[NT][8][4],
                                                    float (&m2)[NT][2], float (&ls)[NT][2], float& F, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        uint32_t k0[8], k1[8];
        {
            const uint32_t r0 = st + gid * 128, r1 = st + (gid + 8) * 128;
            const int u0 = ((2 * tig) ^ (gid & 7)) << 4, u1 = ((2 * tig + 1) ^ (gid & 7)) << 4;
            lds128(r0 + u0, k0[0], k0[1], k0[2], k0[3]);
            lds128(r0 + u1, k0[4], k0[5], k0[6], k0[7]);
            lds128(r1 + u0, k1[0], k1[1], k1[2], k1[3]);
            lds128(r1 + u1, k1[4], k1[5], k1[6], k1[7]);
        }
        float s[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_f16x2x2(k0[kk], a0, a2);
            e4m3x4_to_f16x2x2(k1[kk], a1, a3);
#pragma unroll
            for (int n = 0; n < NT; ++n) mma_f16(s[n], a0, a1, a2, a3, qf[n][kk][0], qf[n][kk][1]);
        }
        const bool v0 = gid < valid, v1 = gid + 8 < valid;
        const float f0 = cq * scl[gid], f1 = cq * scl[gid + 8];
        const float vs0 = v0 ? scl[16 + gid] : 0.f, vs1 = v1 ? scl[24 + gid] : 0.f;
        float fv = fmaxf(fabsf(vs0), fabsf(vs1));
        fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 4));
        fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 8));
        fv = fmaxf(fv, __shfl_xor_sync(kFull, fv, 16));
        if (!(fv > 0.f)) fv = 1.f;
        const float rF = 1.f / fv;
        const float ratio = F * rF;   // acc holds true_acc / F; rebase it on this tile's factor
        F = fv;
        const float w0 = vs0 * rF, w1 = vs1 * rF;
        uint32_t b[NT][2];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            s[n][0] = v0 ? s[n][0] * f0 : -INFINITY;
            s[n][1] = v0 ? s[n][1] * f0 : -INFINITY;
            s[n][2] = v1 ? s[n][2] * f1 : -INFINITY;
            s[n][3] = v1 ? s[n][3] * f1 : -INFINITY;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = fmaxf(s[n][j], s[n][j + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
                const float mnew = fmaxf(m2[n][j], mx);
                const float alpha = ex2(m2[n][j] - mnew);
                m2[n][j] = mnew;
                const float p0 = ex2(s[n][j] - mnew), p1 = ex2(s[n][j + 2] - mnew);
                ls[n][j] = ls[n][j] * alpha + (p0 + p1);
                s[n][j] = p0 * w0;
                s[n][j + 2] = p1 * w1;
                const float ar = alpha * ratio;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    acc[n][m][j] *= ar;
                    acc[n][m][j + 2] *= ar;
                }
            }
            b[n][0] = movmatrix_trans(pack_f16(s[n][0], s[n][1]));
            b[n][1] = movmatrix_trans(pack_f16(s[n][2], s[n][3]));
        }
        // V: rows 2tig, 2tig+1, 2tig+8, 2tig+9; 16-byte unit gid (d = 16*gid .. 16*gid+15)
        uint32_t vx[4], vy[4], vx2[4], vy2[4];
        {
            const uint32_t vb = st + 2048;
            const int x = 2 * tig, y = 2 * tig + 1, x2 = 2 * tig + 8, y2 = 2 * tig + 9;
            lds128(vb + x * 128 + ((gid ^ (x & 7)) << 4), vx[0], vx[1], vx[2], vx[3]);
            lds128(vb + y * 128 + ((gid ^ (y & 7)) << 4), vy[0], vy[1], vy[2], vy[3]);
            lds128(vb + x2 * 128 + ((gid ^ (x2 & 7)) << 4), vx2[0], vx2[1], vx2[2], vx2[3]);
            lds128(vb + y2 * 128 + ((gid ^ (y2 & 7)) << 4), vy2[0], vy2[1], vy2[2], vy2[3]);
            if (valid < kTileTokens) {   // rows past the context may hold NaN codes
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (x >= valid) vx[j] = 0u;
                    if (y >= valid) vy[j] = 0u;
                    if (x2 >= valid) vx2[j] = 0u;
                    if (y2 >= valid) vy2[j] = 0u;
                }
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
            for (int n = 0; n < NT; ++n) mma_f16(acc[n][m], a0, a1, a2, a3, b[n][0], b[n][1]);
        }
    }

    // ------------------------------------------------------------------ consumers
    static __device__ void consumer(const DecodeArgs& a, uint8_t* smem, Bars bars, UnitInfo* info, int warp) {
        const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
        const uint32_t sbase = smem_addr(smem);
        float* merge = reinterpret_cast<float*>(smem + Cfg::kOffMerge);
        float* mw = merge + warp * Cfg::kMergeFloats;
        constexpr int kCons = NW * 32;
        int ucount = 0;
        long long tile_base = 0;
        while (true) {
            const int slot = ucount & 1;
            bool failed = !mbar_wait(bars.qfull(slot), (ucount >> 1) & 1, a.timeout_ns);
            UnitInfo ui{};
            if (!failed) ui = info[slot];
            // every consumer warp leaves together (end marker or a failed wait anywhere)
            if (bar_red_or(1, kCons, failed || ui.nt < 0)) {
                if (failed && lane == 0 && a.err_word) atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
                break;
            }
            // ---- Q fragments (B operand of the score MMA)
            uint32_t qf[NT][8][2];
            float cq = a.qk_scale_log2;
            const uint32_t qb = sbase + Cfg::kOffQ + slot * Cfg::kQBytes;
            if constexpr (!FP8) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int kk = 0; kk < 8; kk += 2) {
                        const int row = n * 8 + (lane & 7);
                        const int d0 = kk * 16 + (lane >> 3) * 8;
                        ldsm_x4(qb + row * 256 + d0 * 2, qf[n][kk][0], qf[n][kk][1], qf[n][kk + 1][0], qf[n][kk + 1][1]);
                    }
            } else {
                uint32_t w[NT][16];
                float amax = 0.f;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint32_t rb = qb + (n * 8 + gid) * 256 + tig * 64;
#pragma unroll
                    for (int c = 0; c < 4; ++c) lds128(rb + c * 16, w[n][4 * c], w[n][4 * c + 1], w[n][4 * c + 2], w[n][4 * c + 3]);
#pragma unroll
                    for (int c = 0; c < 16; ++c) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[n][c])), fabsf(bf16_hi(w[n][c]))));
                }
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
                // power of two that brings the largest |q| into [2^14, 2^15): f16 keeps every bf16 bit
                int e = 0;
                if (amax > 0.f) e = 14 - ((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127);
                e = max(-100, min(100, e));
                const float pw = __uint_as_float((uint32_t)(e + 127) << 23);
                cq = a.qk_scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t x = w[n][2 * kk], y = w[n][2 * kk + 1];
                        qf[n][kk][0] = pack_f16(bf16_lo(x) * pw, bf16_hi(x) * pw);
                        qf[n][kk][1] = pack_f16(bf16_lo(y) * pw, bf16_hi(y) * pw);
                    }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.qempty(slot));

            float acc[NT][8][4];
            float m2[NT][2], ls[NT][2];
            float F = 1.f;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
#pragma unroll
                for (int m = 0; m < 8; ++m) acc[n][m][0] = acc[n][m][1] = acc[n][m][2] = acc[n][m][3] = 0.f;
                m2[n][0] = m2[n][1] = -INFINITY;
                ls[n][0] = ls[n][1] = 0.f;
            }
            const int tok_base = ui.p * a.W;
            for (int t = warp; t < ui.nt; t += NW) {
                const long long i = tile_base + t;
                const int stage = (int)(i % S);
                if (!mbar_wait(bars.full(stage), (uint32_t)((i / S) & 1), a.timeout_ns)) {
                    failed = true;
                    break;
                }
                const int valid = ui.ctx - (tok_base + t * kTileTokens);
                const uint32_t st = sbase + Cfg::kOffStages + stage * Cfg::kTileBytes;
                if constexpr (FP8) {
                    const float* scl = reinterpret_cast<const float*>(smem + Cfg::kOffScales + stage * Cfg::kScaleBytes);
                    tile_fp8(st, scl, valid, cq, qf, acc, m2, ls, F, lane);
                } else {
                    tile_bf16(st, valid, a.qk_scale_log2, qf, acc, m2, ls, lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.empty(stage));
            }
            tile_base += ui.nt;

            // ---- per-warp state -> merge buffer
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float l = ls[n][j];
                    l += __shfl_xor_sync(kFull, l, 4);
                    l += __shfl_xor_sync(kFull, l, 8);
                    l += __shfl_xor_sync(kFull, l, 16);
                    ls[n][j] = l;
                }
            const float fmul = FP8 ? F : 1.f;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int q = n * 8 + 2 * tig + (c & 1);
                        const int d = FP8 ? (16 * gid + 2 * m + (c >> 1)) : (16 * m + gid + 8 * (c >> 1));
                        mw[q * Cfg::kMStride + d] = acc[n][m][c] * fmul;
                    }
            if (gid == 0) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int q = n * 8 + 2 * tig + j;
                        mw[Cfg::kQRows * Cfg::kMStride + q] = m2[n][j];
                        mw[Cfg::kQRows * Cfg::kMStride + Cfg::kQRows + q] = ls[n][j];
                    }
            }
            if (bar_red_or(1, kCons, failed)) {
                if (failed && lane == 0 && a.err_word) atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
                break;
            }
            // ---- combine the NW warps and store the partial
            const int ctid = threadIdx.x;   // consumers are threads 0 .. kCons-1
            const long long row0 = ((long long)(ui.b * a.Hk + ui.h) * a.P + ui.p) * a.QG;
            for (int e = ctid; e < a.QG * 32; e += kCons) {
                const int q = e >> 5, d4 = (e & 31) << 2;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < NW; ++w) M = fmaxf(M, merge[w * Cfg::kMergeFloats + Cfg::kQRows * Cfg::kMStride + q]);
                float L = 0.f;
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < NW; ++w) {
                        const float* mwv = merge + w * Cfg::kMergeFloats;
                        const float f = ex2(mwv[Cfg::kQRows * Cfg::kMStride + q] - M);
                        L += f * mwv[Cfg::kQRows * Cfg::kMStride + Cfg::kQRows + q];
                        const float4 v = *reinterpret_cast<const float4*>(mwv + q * Cfg::kMStride + d4);
                        o.x += f * v.x;
                        o.y += f * v.y;
                        o.z += f * v.z;
                        o.w += f * v.w;
                    }
                }
                const float inv = L > 0.f ? 1.f / L : 0.f;
                o.x *= inv;
                o.y *= inv;
                o.z *= inv;
                o.w *= inv;
                *reinterpret_cast<float4*>(a.partial_out + (row0 + q) * kHeadDim + d4) = o;
                if (d4 == 0) {
                    a.exp_sums[row0 + q] = L;
                    a.max_logits[row0 + q] = M * kLn2;
                }
            }
            ++ucount;
        }
    }
};

template <bool FP8, int NT, int NW, int S>
__global__ void __launch_bounds__((NW + 1) * 32, 1)
    pda_partition_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap sc_map,
                         const DecodeArgs a) {
    using D = Decode<FP8, NT, NW, S>;
    using Cfg = typename D::Cfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc* misc = reinterpret_cast<Misc*>(smem + Cfg::kOffMisc);
    UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + Cfg::kOffInfo);
    typename D::Bars bars{smem_addr(smem + Cfg::kOffBar)};
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bars.full(s), 1);
            mbar_init(bars.empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars.qfull(i), 1);
            mbar_init(bars.qempty(i), NW);
        }
        fence_mbar_init();
        prefetch_tensormap(&kv_map);
        if (FP8) prefetch_tensormap(&sc_map);
    }
    // Q rows QG..7 (QG = 6) are never copied: they must read as zero.
    for (int i = a.QG * 256 + tid * 16; i < Cfg::kQBytes; i += blockDim.x * 16) {
        *reinterpret_cast<uint4*>(smem + Cfg::kOffQ + i) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + Cfg::kOffQ + Cfg::kQBytes + i) = make_uint4(0, 0, 0, 0);
    }
    find_range(a, misc);   // ends with __syncthreads()

    if (warp == NW)
        D::producer(a, &kv_map, &sc_map, smem, bars, misc, info);
    else
        D::consumer(a, smem, bars, info, warp);
}

}  // namespace pda
