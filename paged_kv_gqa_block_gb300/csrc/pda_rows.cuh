// pda_rows.cuh -- the partition pass for QG = 16 over a bf16 KV cache with the sixteen query rows
// of a unit split between two warps of one CTA.
//
// What is computed is the partition pass of the vLLM "tq_decode" page (tq_decode_kernel, steps B
// to G), as in pda_decode.cuh: for sequence b, KV head h and partition p, the QG query rows of
// head h attend over tokens [p*W, min((p+1)*W, ctx_b)); the epilogue writes the normalised
// partial, the running max and the running sum.
//
// How the work is laid out (a GB300 design, not the page's):
//   * With sixteen rows a one-warp unit carries two 8-row MMA blocks through every tile, and at
//     the registers that needs only six such warps fit an SM: each warp's long dependent chain
//     is hidden by few others.  Here a CTA is one producer warp and two consumer warps; consumer
//     c runs query rows 8c .. 8c+7 of the unit with the one-block math, and both read every tile
//     of the ring the producer keeps full (one TMA copy per 16-token tile, 8 KB).
//   * The per-row arithmetic is the head-warp kernel's two-block form, block by block (the eager
//     update: Decode<bf16, 1, S, false, true>), so the partials equal that kernel's bit for bit
//     and the fused step (head warps) still gives pda_decode + pda_reduce's bits.
//   * Units (sequence, KV head, partition) come longest first from the launch's counter slot,
//     by the head-group kernel's order with groups of one head (pda_group.cuh); the producer
//     passes each unit to the consumers through a ring of descriptors in shared memory, one unit
//     ahead.
//   * The epilogue stores the partial straight from the accumulators (the tile stages are shared
//     by both consumers, so neither can stage its rows in one while the other may still read it).
//   * Every wait is bounded; a wait that gives up sets PDA_ERRW_PIPELINE_TIMEOUT.  The producer,
//     the only warp that issues copies, waits (bounded) for every copy it issued before it leaves.
#pragma once

#include "pda_group.cuh"

namespace pda {

constexpr int kRowsConsumers = 2;   // consumer warps per CTA, 8 query rows each
constexpr int kRowsTileBytes = 8192;   // K|V of 16 tokens of one KV head, bf16

__host__ __device__ constexpr int rows_smem_bytes(int S) {
    // stages + stage barriers + unit-descriptor barriers and descriptors (4 in flight) + bucket
    // table and its scratch + alignment slack
    return S * kRowsTileBytes + 2 * S * 8 + 4 * 32 + 8 * (kGroupBuckets + 2) + 1024;
}

template <int S>
struct RowsDecode {
    using D = Decode<PDA_KV_BF16, 1, S, false, true>;   // one 8-row block, eager update
    static constexpr int R = 4;                           // unit descriptors in flight

    struct Smem {
        uint32_t base;            // shared address of the stages
        uint32_t full0, empty0;   // stage barriers: data landed / both consumers done with it
        uint32_t ufull0, uempty0; // unit-descriptor barriers
        int4* udesc;              // R descriptors {b, h, p, ctx}; b < 0: no more units
        const int* above;         // partial-unit bucket table
    };

    // ------------------------------------------------------------------ producer warp
    static __device__ void publish(const Smem& m, long long i, const GroupUnit& u, int lane, bool& ok,
                                   unsigned long long timeout) {
        const int slot = (int)(i % R);
        const long long n = i / R;
        if (n > 0 && !mbar_wait(m.uempty0 + 8 * slot, (uint32_t)((n - 1) & 1), timeout)) {
            ok = false;
            return;
        }
        if (lane == 0) {
            m.udesc[slot] = make_int4(u.valid ? u.b : -1, u.g, u.p, u.ctx);
            mbar_arrive(m.ufull0 + 8 * slot);   // release: the descriptor is visible to its readers
        }
        __syncwarp();
    }

    static __device__ void produce(const DecodeArgs& a, const CUtensorMap* kv_map, const Smem& m) {
        const int lane = threadIdx.x & 31;
        const uint64_t policy = l2_policy_evict_first();
        const int ts = a.bs_shift - 4;   // log2(16-token tiles per block-table entry)
        GroupSched s;
        group_sched_init(a, s, m.above, blockIdx.x == 0);
        long long issued = 0;
        bool ok = true;
        // this lane's block-table entry e of unit x (0 past the unit's entries)
        auto load_entry = [&](const GroupUnit& x, int e) -> int {
            const int tokens = min(a.W, x.ctx - x.p * a.W);
            const int n_ent = (tokens + a.BS - 1) >> a.bs_shift;
            if (e >= n_ent) return 0;
            return __ldg(a.block_table + (long long)x.b * a.MB + ((x.p * a.W) >> a.bs_shift) + e);
        };
        GroupUnit u = group_unit(a, s, group_take(a));
        int ent = u.valid ? load_entry(u, lane) : 0;
        publish(m, 0, u, lane, ok, a.timeout_ns);
        for (long long i = 0; u.valid && ok; ++i) {
            // the consumers learn unit i + 1 while they start unit i (for its Q rows)
            const GroupUnit nx = group_unit(a, s, group_take(a));
            const int nent = nx.valid ? load_entry(nx, lane) : 0;   // in flight while this unit issues
            publish(m, i + 1, nx, lane, ok, a.timeout_ns);
            if (!ok) break;
            const int tokens = min(a.W, u.ctx - u.p * a.W);
            const int nt = (tokens + 15) >> 4;
            for (int t = 0; t < nt; ++t) {
                const int e = t >> ts;
                if (e > 0 && (e & 31) == 0 && (t & ((1 << ts) - 1)) == 0)
                    ent = load_entry(u, e + lane);   // the next 32 entries (units of more than 32)
                const int phys = __shfl_sync(kFull, ent, e & 31);
                const int st = (int)(issued % S);
                const long long n = issued / S;
                if (n > 0 && !mbar_wait(m.empty0 + 8 * st, (uint32_t)((n - 1) & 1), a.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int slot0 = (t & ((1 << ts) - 1)) * kTileTokens;
                    const uint32_t bar = m.full0 + 8 * st;
                    mbar_arrive_expect_tx(bar, kRowsTileBytes);
                    tma_load_5d(m.base + st * kRowsTileBytes, kv_map, bar, 0, slot0, 0, u.g, phys, policy);
                    if ((phys < 0 || (long long)phys >= a.num_cache_blocks) && a.err_word)
                        atomicOr(a.err_word, PDA_ERRW_BAD_BLOCK_ID);
                }
                __syncwarp();
                ++issued;
            }
            u = nx;
            ent = nent;
        }
        if (lane == 0) {
            if (!ok && a.err_word) atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
            // this CTA takes no more units; the launch's last CTA to get here returns the counter
            // pair to zero
            __threadfence();
            if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
                a.sched[0] = 0u;
                a.sched[1] = 0u;
            }
            // no copy may land in this CTA's memory after it leaves: wait (bounded, by the default
            // limit whatever the plan asked for) for the last copy issued into every stage
            for (int st = 0; st < S; ++st) {
                if (issued <= st) continue;
                const long long j = st + ((issued - 1 - st) / S) * S;
                (void)mbar_wait(m.full0 + 8 * st, (uint32_t)((j / S) & 1), kDefaultTimeoutNs);
            }
        }
        __syncwarp();
    }

    // ------------------------------------------------------------------ consumer warp (rows 8c .. 8c+7)
    // Unit i as the producer published it (u.valid false: no unit i, or the wait gave up and ok is false).
    static __device__ GroupUnit read_unit(const Smem& m, long long i, int lane, bool& ok, unsigned long long timeout) {
        GroupUnit u;
        u.valid = false;
        u.b = u.g = u.p = u.ctx = 0;
        const int slot = (int)(i % R);
        if (!mbar_wait(m.ufull0 + 8 * slot, (uint32_t)((i / R) & 1), timeout)) {
            ok = false;
            return u;
        }
        const int4 d = m.udesc[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(m.uempty0 + 8 * slot);
        u.valid = d.x >= 0;
        u.b = d.x;
        u.g = d.y;
        u.p = d.z;
        u.ctx = d.w;
        return u;
    }

    // Query rows 8c + gid of unit u's KV head, as the bf16 B-operand fragments of the score MMA
    // (lane (gid, tig) holds words tig and tig + 4 of each 8-word chunk of its row).
    static __device__ __forceinline__ void load_rows(const DecodeArgs& a, const GroupUnit& u, int c, uint32_t (&w)[16],
                                                     int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(
            a.query + ((long long)u.b * a.Hk * a.QG + (long long)u.g * a.QG + 8 * c + gid) * kHeadDim);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            w[2 * kk] = __ldg(row + kk * 8 + tig);
            w[2 * kk + 1] = __ldg(row + kk * 8 + 4 + tig);
        }
    }

    static __device__ void consume(const DecodeArgs& a, int c, const Smem& m) {
        const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
        bool ok = true;
        GroupUnit u = read_unit(m, 0, lane, ok, a.timeout_ns);
        uint32_t qn[16];
        if (u.valid) load_rows(a, u, c, qn, lane);
        int cs = 0;
        uint32_t cph = 0;
        for (long long i = 0; u.valid && ok; ++i) {
            uint32_t qf[1][8][2];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                qf[0][kk][0] = qn[2 * kk];
                qf[0][kk][1] = qn[2 * kk + 1];
            }
            // ---- the next unit's Q rows are requested while this unit runs
            const GroupUnit nx = read_unit(m, i + 1, lane, ok, a.timeout_ns);
            if (!ok) break;
            if (nx.valid) load_rows(a, nx, c, qn, lane);

            float acc[1][8][4], m2[1][2], mt[1][2], ls[1][2];
#pragma unroll
            for (int mm = 0; mm < 8; ++mm) acc[0][mm][0] = acc[0][mm][1] = acc[0][mm][2] = acc[0][mm][3] = 0.f;
            m2[0][0] = m2[0][1] = -INFINITY;
            mt[0][0] = mt[0][1] = -INFINITY;
            ls[0][0] = ls[0][1] = 0.f;
            const int tokens = min(a.W, u.ctx - u.p * a.W);
            const int nt = (tokens + 15) >> 4;
            const int tok_base = u.p * a.W;
            for (int t = 0; t < nt;) {
                const bool two = t + 1 < nt;
                const int s0 = cs;
                const uint32_t ph0 = cph;
                const int s1 = s0 + 1 == S ? 0 : s0 + 1;
                const uint32_t ph1 = s0 + 1 == S ? cph ^ 1u : cph;
                if (!mbar_wait(m.full0 + 8 * s0, ph0, a.timeout_ns) ||
                    (two && !mbar_wait(m.full0 + 8 * s1, ph1, a.timeout_ns))) {
                    ok = false;
                    break;
                }
                const int v0 = u.ctx - (tok_base + t * kTileTokens);
                if (two) {
                    const uint32_t st[2] = {m.base + s0 * kRowsTileBytes, m.base + s1 * kRowsTileBytes};
                    const int vv[2] = {v0, v0 - kTileTokens};
                    D::template step_bf16<2>(st, vv, a.qk_scale_log2, qf, acc, m2, mt, ls, lane);
                } else {
                    const uint32_t st[1] = {m.base + s0 * kRowsTileBytes};
                    const int vv[1] = {v0};
                    D::template step_bf16<1>(st, vv, a.qk_scale_log2, qf, acc, m2, mt, ls, lane);
                }
                t += two ? 2 : 1;
                // the stages go back to the producer once every lane's reads of them are done
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(m.empty0 + 8 * s0);
                    if (two) mbar_arrive(m.empty0 + 8 * s1);
                }
                cs = two ? (s1 + 1 == S ? 0 : s1 + 1) : s1;
                cph = two ? (s1 + 1 == S ? ph1 ^ 1u : ph1) : ph1;
            }
            if (!ok) break;

            // ---- epilogue (the eager update: m2 is the running maximum): o = acc / l, m_p = m2,
            // l_p = l, in the head-warp kernel's arithmetic; lane (gid, tig) holds dimension
            // 16*mm + gid + 8*(k >> 1) of rows 2*tig + (k & 1) of this consumer's block
            float inv[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float l = ls[0][j];
                l += __shfl_xor_sync(kFull, l, 4);
                l += __shfl_xor_sync(kFull, l, 8);
                l += __shfl_xor_sync(kFull, l, 16);
                ls[0][j] = l;
                inv[j] = l > 0.f ? 1.f / l : 0.f;
            }
            const long long row0 = ((long long)(u.b * a.Hk + u.g) * a.P + u.p) * a.QG + 8 * c;
#pragma unroll
            for (int mm = 0; mm < 8; ++mm)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int q = 2 * tig + (k & 1), d = 16 * mm + gid + 8 * (k >> 1);
                    a.partial_out[(row0 + q) * kHeadDim + d] = acc[0][mm][k] * inv[k & 1];
                }
            if (gid == 0) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    a.exp_sums[row0 + 2 * tig + j] = ls[0][j];
                    a.max_logits[row0 + 2 * tig + j] = m2[0][j] * kLn2;
                }
            }
            u = nx;
        }
        if (lane == 0 && !ok && a.err_word) atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
        __syncwarp();
    }

    static __device__ void run(const DecodeArgs& a, const CUtensorMap* kv_map, uint8_t* smem) {
        const int warp = threadIdx.x >> 5;
        Smem m;
        m.base = smem_addr(smem);
        const uint32_t off_bar = (uint32_t)(S * kRowsTileBytes);
        m.full0 = m.base + off_bar;
        m.empty0 = m.full0 + 8 * S;
        m.ufull0 = m.empty0 + 8 * S;
        m.uempty0 = m.ufull0 + 8 * R;
        m.udesc = reinterpret_cast<int4*>(smem + off_bar + 16 * S + 16 * R);
        int* above = reinterpret_cast<int*>(smem + off_bar + 16 * S + 16 * R + 16 * R);
        int* hist = above + (kGroupBuckets + 2);
        m.above = above;
        if (threadIdx.x == 0) {
            for (int st = 0; st < S; ++st) {
                mbar_init(m.full0 + 8 * st, 1);
                mbar_init(m.empty0 + 8 * st, (uint32_t)kRowsConsumers);
            }
            for (int r = 0; r < R; ++r) {
                mbar_init(m.ufull0 + 8 * r, 1);
                mbar_init(m.uempty0 + 8 * r, (uint32_t)kRowsConsumers);
            }
            fence_mbar_init();
            prefetch_tensormap(kv_map);
        }
        allow_dependent_launch();   // the reduce may be scheduled as soon as CTAs of this grid retire
        grid_dependency_wait();     // inputs may come from the previous grid on the stream
        group_buckets_init(a, above, hist);
        __syncthreads();            // the barriers and the bucket table are ready
        if (warp == 0)
            produce(a, kv_map, m);
        else if (warp <= kRowsConsumers)
            consume(a, warp - 1, m);
    }
};

// MINB: CTAs per SM the register allocation must allow.
template <int S, int MINB>
__global__ void __launch_bounds__((kRowsConsumers + 1) * 32, MINB) pda_rows_kernel(const __grid_constant__ CUtensorMap kv_map,
                                                                                   const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    RowsDecode<S>::run(a, &kv_map, smem);
}

}  // namespace pda
