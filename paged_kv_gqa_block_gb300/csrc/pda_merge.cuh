// pda_merge.cuh -- the combination of one query row's partition partials into its output row,
// shared by the reduce kernel and the fused steps, so all give the same bits.
//
// For sequence b, KV head h and query row q with nv = ceil(ctx / W) partitions:
//   M = max_p m_p,  w_p = l_p * e^(m_p - M),  out = sum_p (w_p / sum_p w_p) * o_p   (p < nv)
// (the partials' epilogue is STEP G of the vLLM "tq_decode" page; the combination is the split
// reduce its per-partition max_logits and exp_sums exist for).  No partitions (ctx = 0) gives a
// zero row.
#pragma once

#include <cstdint>

#include "pda_internal.h"
#include "pda_ptx.cuh"

namespace pda {

struct MergeArgs {
    const float* partial_out;   // [B][Hk][P][QG][D]
    const float* exp_sums;      // [B][Hk][P][QG]
    const float* max_logits;    // [B][Hk][P][QG]
    void* out;                  // [B][Hk*QG][D], bf16 or fp32
    int Hk, QG, P, W;
    int out_f32;
};

constexpr int kMergeRegParts = 2;   // partitions whose (m, l) a lane holds (up to 64); beyond that they are reloaded
constexpr int kMergeBatch = 16;     // partial loads in flight per lane

__device__ __forceinline__ void merge_load_batch(const float* op, int pstride, int p0, int plast,
                                                 float4 (&o)[kMergeBatch]) {
    const float4* o4 = reinterpret_cast<const float4*>(op);
    const int s4 = pstride >> 2;   // float4s between partitions (QG * D / 4)
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)   // clamped index: every load is in bounds, extras are discarded
        o[j] = __ldcg(o4 + (long long)min(p0 + j, plast) * s4);
}

// One warp.  Lane j holds (m_p, l_p) of partitions p = j, j+32, ...; warp reductions give M and
// sum_p w_p; every lane then accumulates four output elements over p in partition order, sixteen
// partial loads in flight.  The (m, l) of the first 64 partitions and the first sixteen partials
// are requested in one round (indices clamped to the row's partitions; values past nv are
// discarded by selects, never multiplied in), so a row of up to sixteen partitions costs one
// round trip to L2.  With one partition w_0 / w_0 == 1 exactly, so the partial is copied bit for
// bit.  The partials are read through L2 (ld.global.cg): they may have been written by other SMs
// during the same launch.  merge_unit_smem below gives the same bits from a shared-memory copy.
__device__ inline void merge_row(const MergeArgs& r, int b, int h, int q, int ctx) {
    const int lane = threadIdx.x & 31, d4 = lane << 2;
    const long long unit = (long long)b * r.Hk + h;
    const long long base = unit * r.P * r.QG + q;   // index of (unit, p = 0, q)
    const float* op = r.partial_out + base * kHeadDim + d4;
    const int pstride = r.QG * kHeadDim;
    const int nv = (ctx + r.W - 1) / r.W;

    float mr[kMergeRegParts], lr[kMergeRegParts];
#pragma unroll
    for (int k = 0; k < kMergeRegParts; ++k) {
        const long long i = base + (long long)max(0, min(lane + 32 * k, nv - 1)) * r.QG;
        mr[k] = __ldcg(r.max_logits + i);
        lr[k] = __ldcg(r.exp_sums + i);
    }
    float4 o[kMergeBatch];
    if (nv > 0) merge_load_batch(op, pstride, 0, nv - 1, o);
#pragma unroll
    for (int k = 0; k < kMergeRegParts; ++k) {
        const bool ok = lane + 32 * k < nv;
        mr[k] = ok ? mr[k] : -INFINITY;
        lr[k] = ok ? lr[k] : 0.f;
    }

    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMergeRegParts; ++k) M = fmaxf(M, mr[k]);
    for (int p = lane + 32 * kMergeRegParts; p < nv; p += 32)
        M = fmaxf(M, __ldcg(r.max_logits + base + (long long)p * r.QG));
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o_));
    float wsum = 0.f;
#pragma unroll
    for (int k = 0; k < kMergeRegParts; ++k) {
        lr[k] = partition_weight(lr[k], mr[k], M);   // w_p (0 for p >= nv)
        wsum = __fadd_rn(wsum, lr[k]);
    }
    for (int p = lane + 32 * kMergeRegParts; p < nv; p += 32) {
        const long long i = base + (long long)p * r.QG;
        wsum = __fadd_rn(wsum, partition_weight(__ldcg(r.exp_sums + i), __ldcg(r.max_logits + i), M));
    }
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) wsum = __fadd_rn(wsum, __shfl_xor_sync(0xFFFFFFFFu, wsum, o_));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < nv; c0 += 32) {
        const int k = c0 >> 5;
        float coef;
        if (k < kMergeRegParts) {
            float w = lr[0];
#pragma unroll
            for (int kk = 1; kk < kMergeRegParts; ++kk)
                if (kk == k) w = lr[kk];
            coef = __fdiv_rn(w, wsum);
        } else {
            const int p = c0 + lane;
            coef = 0.f;
            if (p < nv) {
                const long long i = base + (long long)p * r.QG;
                coef = __fdiv_rn(partition_weight(__ldcg(r.exp_sums + i), __ldcg(r.max_logits + i), M), wsum);
            }
        }
        const int cn = min(32, nv - c0);
        for (int j0 = 0; j0 < cn; j0 += kMergeBatch) {
            if (c0 + j0 > 0) merge_load_batch(op, pstride, c0 + j0, nv - 1, o);
#pragma unroll
            for (int j = 0; j < kMergeBatch; ++j) {
                const float cf = __shfl_sync(0xFFFFFFFFu, coef, (j0 + j) & 31);
                if (j0 + j < cn) {
                    acc.x = fmaf(cf, o[j].x, acc.x);
                    acc.y = fmaf(cf, o[j].y, acc.y);
                    acc.z = fmaf(cf, o[j].z, acc.z);
                    acc.w = fmaf(cf, o[j].w, acc.w);
                }
            }
        }
    }
    const long long orow = unit * r.QG + q;
    if (r.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(r.out) + orow * kHeadDim + d4) = acc;
    } else {
        uint2 v;
        v.x = pack_bf16(acc.x, acc.y);
        v.y = pack_bf16(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(r.out) + orow * kHeadDim + d4) = v;
    }
}

// The merge of a whole (sequence, KV head) unit, for the reduce kernel: one CTA, warp q merges
// query row q.  The unit's partials of partitions p < nv are one contiguous range
// ([p][q][D] within the unit), streamed into a ring of two shared-memory buffers of kMergeChunk
// partitions each by bulk copies (thread 0 issues; the copies need no registers, so a long row's
// partials are all in flight at once instead of sixteen loads per lane); the (m_p, l_p) are
// loaded per row as in merge_row, and the arithmetic, order included, is merge_row's, so the
// result has the same bits.  `buf` holds 2 * kMergeChunk * QG * D floats (16-byte aligned),
// `bars` four mbarriers.  Every wait is bounded; one that gives up sets `*timed_out`.
constexpr int kMergeChunk = 8;   // partitions per shared-memory buffer

__device__ inline void merge_unit_smem(const MergeArgs& r, int b, int h, int ctx, float* buf, uint32_t bars,
                                       bool* timed_out) {
    const int lane = threadIdx.x & 31, q = threadIdx.x >> 5, d4 = lane << 2;
    const long long unit = (long long)b * r.Hk + h;
    const long long base = unit * r.P * r.QG + q;   // index of (unit, p = 0, q)
    const int nv = (ctx + r.W - 1) / r.W;
    const int nch = (nv + kMergeChunk - 1) / kMergeChunk;
    const uint32_t full0 = bars, empty0 = bars + 16;
    const uint32_t chunk_floats = (uint32_t)kMergeChunk * r.QG * kHeadDim;
    const float* src = r.partial_out + unit * r.P * r.QG * kHeadDim;
    auto issue = [&](int k) {   // thread 0: chunk k into buffer k & 1
        const int cnt = min(kMergeChunk, nv - k * kMergeChunk);
        const uint32_t bytes = (uint32_t)cnt * r.QG * kHeadDim * 4;
        const uint32_t bar = full0 + 8 * (k & 1);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(smem_addr(buf + (k & 1) * chunk_floats), src + (long long)k * chunk_floats, bytes, bar);
    };
    int issued = 0;   // thread 0: chunks issued
    if (threadIdx.x == 0) {
        for (; issued < 2 && issued < nch; ++issued) issue(issued);
    }

    // M and sum_p w_p of this row, exactly as merge_row
    float mr[kMergeRegParts], lr[kMergeRegParts];
#pragma unroll
    for (int k = 0; k < kMergeRegParts; ++k) {
        const long long i = base + (long long)max(0, min(lane + 32 * k, nv - 1)) * r.QG;
        const bool ok = lane + 32 * k < nv;
        const float m = __ldcg(r.max_logits + i), l = __ldcg(r.exp_sums + i);
        mr[k] = ok ? m : -INFINITY;
        lr[k] = ok ? l : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMergeRegParts; ++k) M = fmaxf(M, mr[k]);
    for (int p = lane + 32 * kMergeRegParts; p < nv; p += 32)
        M = fmaxf(M, __ldcg(r.max_logits + base + (long long)p * r.QG));
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o_));
    float wsum = 0.f;
#pragma unroll
    for (int k = 0; k < kMergeRegParts; ++k) {
        lr[k] = partition_weight(lr[k], mr[k], M);
        wsum = __fadd_rn(wsum, lr[k]);
    }
    for (int p = lane + 32 * kMergeRegParts; p < nv; p += 32) {
        const long long i = base + (long long)p * r.QG;
        wsum = __fadd_rn(wsum, partition_weight(__ldcg(r.exp_sums + i), __ldcg(r.max_logits + i), M));
    }
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) wsum = __fadd_rn(wsum, __shfl_xor_sync(0xFFFFFFFFu, wsum, o_));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float coef = 0.f;
    bool ok = true;
    for (int k = 0; k < nch; ++k) {
        if (!mbar_wait(full0 + 8 * (k & 1), (uint32_t)((k >> 1) & 1), kDefaultTimeoutNs)) {
            ok = false;
            break;
        }
        const float* cb = buf + (k & 1) * chunk_floats;
        const int cnt = min(kMergeChunk, nv - k * kMergeChunk);
        for (int j = 0; j < cnt; ++j) {
            const int p = k * kMergeChunk + j;
            if ((p & 31) == 0) {   // the coefficients of partitions p .. p+31, one per lane
                const int kk = p >> 5;
                if (kk < kMergeRegParts) {
                    float w = lr[0];
#pragma unroll
                    for (int k2 = 1; k2 < kMergeRegParts; ++k2)
                        if (k2 == kk) w = lr[k2];
                    coef = __fdiv_rn(w, wsum);
                } else {
                    const int pl = p + lane;
                    coef = 0.f;
                    if (pl < nv) {
                        const long long i = base + (long long)pl * r.QG;
                        coef = __fdiv_rn(partition_weight(__ldcg(r.exp_sums + i), __ldcg(r.max_logits + i), M), wsum);
                    }
                }
            }
            const float cf = __shfl_sync(0xFFFFFFFFu, coef, p & 31);
            const float4 o = *reinterpret_cast<const float4*>(cb + ((long long)j * r.QG + q) * kHeadDim + d4);
            acc.x = fmaf(cf, o.x, acc.x);
            acc.y = fmaf(cf, o.y, acc.y);
            acc.z = fmaf(cf, o.z, acc.z);
            acc.w = fmaf(cf, o.w, acc.w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * (k & 1));
        if (threadIdx.x == 0 && k + 2 < nch) {   // refill this buffer once every row is done with it
            if (!mbar_wait(empty0 + 8 * (k & 1), (uint32_t)((k >> 1) & 1), kDefaultTimeoutNs)) {
                ok = false;
            } else {
                issue(k + 2);
                ++issued;
            }
        }
        if (!ok) break;
    }
    if (threadIdx.x == 0) {   // no copy may land in this CTA's memory after it leaves
        for (int k = max(0, issued - 2); k < issued; ++k)
            (void)mbar_wait(full0 + 8 * (k & 1), (uint32_t)((k >> 1) & 1), kDefaultTimeoutNs);
    }
    if (!ok) {
        *timed_out = true;
        return;
    }
    const long long orow = unit * r.QG + q;
    if (r.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(r.out) + orow * kHeadDim + d4) = acc;
    } else {
        uint2 v;
        v.x = pack_bf16(acc.x, acc.y);
        v.y = pack_bf16(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(r.out) + orow * kHeadDim + d4) = v;
    }
}

}  // namespace pda
