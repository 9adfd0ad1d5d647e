// pda_group.cuh -- the partition pass with head-group CTAs, for an fp8 e4m3 KV cache.
//
// What is computed is the partition pass of the vLLM "tq_decode" page (tq_decode_kernel, steps B
// to G), exactly as in pda_decode.cuh: for sequence b, KV head h and partition p, the QG query
// rows of head h attend over tokens [p*W, min((p+1)*W, ctx_b)); the epilogue writes the normalised
// partial, the running max and the running sum.
//
// How the work is laid out (a GB300 design, not the page's):
//   * A block of the paged cache holds all KV heads of its 16 or 32 tokens contiguously
//     ([slot][head][K|V]), so one TMA box {128 B, 16 tokens, K|V, HG heads} brings a 16-token tile
//     of HG heads (32 KB for 8 heads) and one more box brings their 2*16*HG fp32 scales: two copy
//     instructions per HG head-tiles instead of two per head-tile.
//   * A CTA is one producer warp and HG consumer warps, one per head of the group.  The producer
//     walks the block table and keeps an S-stage ring of such tiles in flight; consumer c reads
//     head c's 4 KB slice of every stage and runs the same per-tile math as the head-warp kernel
//     (scores, mask, online softmax, PV), then releases the stage.  A consumer never issues a copy.
//   * Work unit = (sequence, head group, partition), every head of the group on the same tokens.
//     Two CTAs per SM (persistent).  Units are taken longest first: all full partitions, then the
//     partial last partitions in decreasing order of their tile count.  A CTA's producer takes the
//     next unit from a counter shared by the launch's CTAs (atomicAdd), so a CTA that streams
//     faster takes more units; the launch's last CTA returns the counter to zero.  The producer
//     passes each unit to its consumers through a small ring of descriptors in shared memory,
//     one unit ahead, so that each consumer loads the next unit's Q rows while it runs the
//     current one.
//   * The epilogue stores the partial straight from the MMA accumulators: lane (gid, tig) holds
//     dimensions 16*gid .. 16*gid+15 of query rows 2*tig and 2*tig+1, 64 contiguous bytes each.
//   * Every wait is bounded; a wait that gives up sets PDA_ERRW_PIPELINE_TIMEOUT.  The producer,
//     the only warp that issues copies, waits (bounded) for every copy it issued before it leaves.
#pragma once

#include "pda_decode.cuh"
#include "pda_merge.cuh"

namespace pda {

constexpr int kGroupMaxHeads = 4;

__host__ __device__ constexpr int group_stage_bytes(int HG) { return HG * 4096; }   // K|V of HG heads, 16 tokens
__host__ __device__ constexpr int group_scale_bytes(int HG) { return HG * 128; }    // 16 K + 16 V fp32 scales per head
// Partial units are ordered by their tile count, in buckets 1..kGroupBuckets (a partial partition
// longer than that many tiles falls in the top bucket).
constexpr int kGroupBuckets = 256;
__host__ __device__ constexpr int group_smem_bytes(int HG, int S) {
    // stages + scales + stage barriers + unit-descriptor barriers and descriptors (4 in flight) +
    // bucket table and its scratch + alignment slack
    return S * (group_stage_bytes(HG) + group_scale_bytes(HG)) + 2 * S * 8 + 4 * 32 + 8 * (kGroupBuckets + 2) + 1024;
}

// One unit of the head-group pass.
struct GroupUnit {
    int b, g, p, ctx;
    bool valid;
};

// The launch's unit order, in three classes:
//   L: every unit of the long sequences (at least kGroupLongPartitions partitions), in (sequence,
//      head group, partition) order;
//   F: the full partitions of the other sequences, in the same order;
//   P: the partial last partitions of the other sequences, by decreasing tile count (bucket), then
//      sequence, then head group.
// Longest first keeps the end of the launch to the smallest units, and the long sequences, whose
// partials take the longest to combine, are complete well before the end.
// GroupSched is the order as one warp derives it from the context lengths: lane l looks after
// sequences [b0, b1); NL, NF and NP count the units of each class (x NG head groups); `above` is the
// CTA's table of class-P sequences per tile-count bucket: above[t] = number of such sequences
// whose partial partition falls in a bucket above t (built once per CTA).
constexpr int kGroupLongPartitions = 8;

struct GroupSched {
    int b0, b1;
    long long excl_l, mine_l;   // class-L units (per head group) of the sequences before / inside this lane's range
    long long excl_f, mine_f;   // class-F units (per head group), likewise
    long long NL, NF, NP;
    long long nonempty;         // sequences with at least one token
    int NG, TWc;                // head groups, top bucket
    const int* above;
};

// Partitions of a sequence of c tokens; whether it is long (class L).
__device__ __forceinline__ int group_nv(int c, int W) { return (c + W - 1) / W; }
__device__ __forceinline__ bool group_long(int c, int W) { return group_nv(c, W) >= kGroupLongPartitions; }

// Class-P bucket of a sequence of c tokens (0: no class-P unit).
__device__ __forceinline__ int group_bucket(int c, int W, int TWc) {
    const int rem = c % W;
    return (rem == 0 || group_long(c, W)) ? 0 : min((rem + 15) >> 4, TWc);
}

// The bucket table (whole CTA, after the grid-dependency wait; a __syncthreads must follow):
// above[t] for t = 0..TWc, above[TWc + 1] = 0.  hist is scratch of TWc + 2 ints.
__device__ inline void group_buckets_init(const DecodeArgs& a, int* above, int* hist) {
    const int TWc = min(a.W >> 4, kGroupBuckets), max_ctx = a.MB * a.BS;
    for (int t = threadIdx.x; t <= TWc + 1; t += blockDim.x) hist[t] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        const int t = group_bucket(sanitize_ctx(__ldg(a.context_lens + b), max_ctx), a.W, TWc);
        if (t) atomicAdd(hist + t, 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {   // above[t] = sum of hist over buckets t+1 .. TWc (a reverse scan, 8 buckets a lane)
        const int lane = threadIdx.x;
        const int per = (TWc + 1 + 31) >> 5, t0 = lane * per;
        int mine = 0;
        for (int t = t0; t < t0 + per && t <= TWc; ++t) mine += hist[t];
        int incl = mine;   // sum over lanes >= this one
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_down_sync(kFull, incl, o);
            if (lane + o < 32) incl += n;
        }
        int run = incl - mine;   // buckets of the lanes above
        for (int t = min(t0 + per, TWc + 1) - 1; t >= t0; --t) {
            above[t] = run;
            run += hist[t];
        }
        if (lane == 0) above[TWc + 1] = 0;
    }
}

__device__ __forceinline__ long long warp_excl_scan(long long x, long long& total) {
    const int lane = threadIdx.x & 31;
    long long incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    total = __shfl_sync(kFull, incl, 31);
    return incl - x;
}

// Sets the data-error bit for out-of-range context lengths when `report`.
__device__ inline void group_sched_init(const DecodeArgs& a, GroupSched& s, const int* above, bool report) {
    const int lane = threadIdx.x & 31;
    const int max_ctx = a.MB * a.BS;
    const int per = (a.B + 31) >> 5;
    s.b0 = min(a.B, lane * per);
    s.b1 = min(a.B, s.b0 + per);
    s.NG = a.Hk / a.HG;
    s.TWc = min(a.W >> 4, kGroupBuckets);
    s.above = above;
    long long nl = 0, nf = 0, np = 0, ne = 0;
    bool bad = false;
    for (int b = s.b0; b < s.b1; ++b) {
        const int raw = __ldg(a.context_lens + b);
        if (raw < 0 || raw > max_ctx) bad = true;
        const int c = sanitize_ctx(raw, max_ctx);
        ne += c > 0;
        if (group_long(c, a.W)) {
            nl += group_nv(c, a.W);
        } else {
            nf += c / a.W;
            np += (c % a.W) != 0;
        }
    }
    if (report && bad && a.err_word) atomicOr(a.err_word, PDA_ERRW_BAD_CONTEXT_LEN);
    long long tl, tf, tp, te;
    s.excl_l = warp_excl_scan(nl, tl);
    s.excl_f = warp_excl_scan(nf, tf);
    (void)warp_excl_scan(np, tp);
    (void)warp_excl_scan(ne, te);
    s.mine_l = nl;
    s.mine_f = nf;
    s.NL = tl * s.NG;
    s.NF = tf * s.NG;
    s.NP = tp * s.NG;
    s.nonempty = te;
}

// Unit k of the launch's order (whole warp; the result is warp-uniform).
__device__ inline GroupUnit group_unit(const DecodeArgs& a, const GroupSched& s, long long k) {
    const int max_ctx = a.MB * a.BS;
    GroupUnit u;
    u.valid = false;
    u.b = u.g = u.p = u.ctx = 0;
    if (k < 0 || k >= s.NL + s.NF + s.NP) return u;
    int fb = -1, fg = 0, fp = 0, fc = 0;
    if (k < s.NL + s.NF) {
        // classes L and F: (sequence, head group, partition) order over the class's sequences
        const bool L = k < s.NL;
        const long long kk = L ? k : k - s.NL;
        const long long lo = (L ? s.excl_l : s.excl_f) * s.NG, mine = L ? s.mine_l : s.mine_f;
        if (mine > 0 && lo <= kk && kk < lo + mine * s.NG) {
            long long pos = lo;
            for (int b = s.b0; b < s.b1; ++b) {
                const int c = sanitize_ctx(__ldg(a.context_lens + b), max_ctx);
                if (group_long(c, a.W) != L) continue;
                const int nu = L ? group_nv(c, a.W) : c / a.W;   // units of one head group
                const long long n = (long long)nu * s.NG;
                if (kk < pos + n) {
                    const int r = (int)(kk - pos);
                    fb = b;
                    fg = r / nu;
                    fp = r - fg * nu;
                    fc = c;
                    break;
                }
                pos += n;
            }
        }
    } else {
        // class P by decreasing tile count (bucket), then sequence, then head group: the bucket
        // from the CTA's table (the largest t with above[t] <= i), the sequence by one scan
        const long long j = k - s.NL - s.NF;
        const int i = (int)(j / s.NG);
        int lo = 1, hi = s.TWc;   // above[] is non-increasing in t; above[TWc] = 0 <= i
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s.above[mid] <= i) hi = mid;
            else lo = mid + 1;
        }
        const int t = lo, r = i - s.above[t];
        int mine = 0;
        for (int b = s.b0; b < s.b1; ++b)
            mine += group_bucket(sanitize_ctx(__ldg(a.context_lens + b), max_ctx), a.W, s.TWc) == t;
        long long tot;
        const int excl = (int)warp_excl_scan(mine, tot);
        if (mine > 0 && excl <= r && r < excl + mine) {
            int cnt = excl;
            for (int b = s.b0; b < s.b1; ++b) {
                const int c = sanitize_ctx(__ldg(a.context_lens + b), max_ctx);
                if (group_bucket(c, a.W, s.TWc) == t) {
                    if (cnt == r) {
                        fb = b;
                        fg = (int)(j - (long long)i * s.NG);
                        fp = c / a.W;
                        fc = c;
                        break;
                    }
                    ++cnt;
                }
            }
        }
    }
    const unsigned m = __ballot_sync(kFull, fb >= 0);
    if (!m) return u;
    const int src = __ffs(m) - 1;
    u.b = __shfl_sync(kFull, fb, src);
    u.g = __shfl_sync(kFull, fg, src);
    u.p = __shfl_sync(kFull, fp, src);
    u.ctx = __shfl_sync(kFull, fc, src);
    u.valid = true;
    return u;
}

// The next unit of the launch's order for this CTA (whole warp; lane 0 takes it).
__device__ __forceinline__ long long group_take(const DecodeArgs& a) {
    unsigned int k = 0;
    if ((threadIdx.x & 31) == 0) k = atomicAdd(a.sched, 1u);
    return (long long)__shfl_sync(kFull, k, 0);
}

template <int NT, int S, bool FUSED>
struct GroupDecode {
    using D = Decode<PDA_KV_FP8_E4M3, NT, 3, false>;
    static constexpr int R = 4;   // unit descriptors in flight from the producer to the consumers

    struct Smem {
        uint32_t base;            // shared address of the stages
        const uint8_t* ptr;       // the same, generic
        uint32_t off_scales;      // stage scales
        uint32_t full0, empty0;   // stage barriers: data landed / every consumer done with it
        uint32_t ufull0, uempty0; // unit-descriptor barriers
        int4* udesc;              // R descriptors {b, g, p, ctx}; b < 0: no more units
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

    static __device__ void produce(const DecodeArgs& a, const CUtensorMap* kv_map, const CUtensorMap* sc_map,
                                   const Smem& m) {
        const int lane = threadIdx.x & 31;
        const int HG = a.HG;
        const uint32_t stage_bytes = group_stage_bytes(HG), scale_bytes = group_scale_bytes(HG);
        const uint32_t tx = stage_bytes + scale_bytes;
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
                    mbar_arrive_expect_tx(bar, tx);
                    tma_load_5d(m.base + st * stage_bytes, kv_map, bar, 0, slot0, 0, u.g * HG, phys, policy);
                    tma_load_4d(m.base + m.off_scales + st * scale_bytes, sc_map, bar, slot0, 0, u.g * HG, phys,
                                policy);
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
            // this CTA takes no more units (its last take, or a wait that gave up, came first);
            // the launch's last CTA to get here returns the counter pair to zero (the fused step
            // returns its counters to zero at its end instead)
            if constexpr (!FUSED) {
                __threadfence();
                if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
                    a.sched[0] = 0u;
                    a.sched[1] = 0u;
                }
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

    // ------------------------------------------------------------------ consumer warp (head c of the group)
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

    static __device__ void consume(const DecodeArgs& a, int c, const Smem& m) {
        const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
        const int HG = a.HG;
        const uint32_t stage_bytes = group_stage_bytes(HG), scale_bytes = group_scale_bytes(HG);
        bool ok = true;
        GroupUnit u = read_unit(m, 0, lane, ok, a.timeout_ns);
        uint32_t qn[NT][16];
        if (u.valid) {
            UnitIt ui{u.b, u.g * HG + c, u.p, u.ctx, 0, 0};
            D::load_q(a, ui, qn, lane);
        }
        int cs = 0;
        uint32_t cph = 0;
        for (long long i = 0; u.valid && ok; ++i) {
            const int h = u.g * HG + c;
            // ---- Q fragments: every bf16 bit of Q kept in f16 by a power-of-two scale
            uint32_t qf[NT][8][2];
            float cq;
            {
                float amax = 0.f;
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(qn[n][k])), fabsf(bf16_hi(qn[n][k]))));
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
                int e = 0;
                if (amax > 0.f) e = 14 - ((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127);
                e = max(-100, min(100, e));
                const float pw = __uint_as_float((uint32_t)(e + 127) << 23);
                cq = a.qk_scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t x = qn[n][2 * kk], y = qn[n][2 * kk + 1];
                        qf[n][kk][0] = pack_f16(bf16_lo(x) * pw, bf16_hi(x) * pw);
                        qf[n][kk][1] = pack_f16(bf16_lo(y) * pw, bf16_hi(y) * pw);
                    }
            }
            // ---- the next unit's Q rows are requested while this unit runs
            const GroupUnit nx = read_unit(m, i + 1, lane, ok, a.timeout_ns);
            if (!ok) break;
            if (nx.valid) {
                UnitIt ui{nx.b, nx.g * HG + c, nx.p, nx.ctx, 0, 0};
                D::load_q(a, ui, qn, lane);
            }

            float acc[NT][8][4];
            float m2[NT][2], mt[NT][2], ls[NT][2];
            float F = 1.f, rF = 1.f;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
#pragma unroll
                for (int mm = 0; mm < 8; ++mm) acc[n][mm][0] = acc[n][mm][1] = acc[n][mm][2] = acc[n][mm][3] = 0.f;
                m2[n][0] = m2[n][1] = -INFINITY;
                mt[n][0] = mt[n][1] = -INFINITY;
                ls[n][0] = ls[n][1] = 0.f;
            }
            const int tokens = min(a.W, u.ctx - u.p * a.W);
            const int nt = (tokens + 15) >> 4;
            const int tok_base = u.p * a.W;
            int last = 0;   // the stage of the unit's last tile: released after the epilogue has used it
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
                    const uint32_t st[2] = {m.base + s0 * stage_bytes + c * 4096, m.base + s1 * stage_bytes + c * 4096};
                    const float* const sc[2] = {
                        reinterpret_cast<const float*>(m.ptr + m.off_scales + s0 * scale_bytes + c * 128),
                        reinterpret_cast<const float*>(m.ptr + m.off_scales + s1 * scale_bytes + c * 128)};
                    const int vv[2] = {v0, v0 - kTileTokens};
                    D::template step_fp8<2>(st, sc, vv, cq, qf, acc, m2, mt, ls, F, rF, lane);
                } else {
                    const uint32_t st[1] = {m.base + s0 * stage_bytes + c * 4096};
                    const float* const sc[1] = {
                        reinterpret_cast<const float*>(m.ptr + m.off_scales + s0 * scale_bytes + c * 128)};
                    const int vv[1] = {v0};
                    D::template step_fp8<1>(st, sc, vv, cq, qf, acc, m2, mt, ls, F, rF, lane);
                }
                t += two ? 2 : 1;
                // the stages go back to the producer once every lane's reads of them are done; the
                // unit's last stage is kept for the epilogue's staging
                __syncwarp();
                last = two ? s1 : s0;
                if (lane == 0) {
                    if (two) mbar_arrive(m.empty0 + 8 * s0);
                    if (t < nt) mbar_arrive(m.empty0 + 8 * last);
                }
                cs = two ? (s1 + 1 == S ? 0 : s1 + 1) : s1;
                cph = two ? (s1 + 1 == S ? ph1 ^ 1u : ph1) : ph1;
            }
            if (!ok) break;

            // ---- epilogue: o = acc * F / l (m_p = running max, l_p = running sum; the eager update
            // keeps the reference point at the true maximum)
            float inv[NT][2];
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float l = ls[n][j];
                    l += __shfl_xor_sync(kFull, l, 4);
                    l += __shfl_xor_sync(kFull, l, 8);
                    l += __shfl_xor_sync(kFull, l, 16);
                    ls[n][j] = l;
                    inv[n][j] = (l > 0.f ? 1.f / l : 0.f) * F;
                }
            const long long row0 = ((long long)(u.b * a.Hk + h) * a.P + u.p) * a.QG;
            if constexpr (NT == 1) {
                // the partial, QG rows of 512 bytes, is staged in this consumer's 4 KB slice of the
                // unit's last stage and written by one bulk copy; lane (gid, tig) holds dimensions
                // 16*gid .. 16*gid+15 of rows 2*tig and 2*tig+1
                float* stg = reinterpret_cast<float*>(const_cast<uint8_t*>(m.ptr) + last * stage_bytes + c * 4096);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int q = 2 * tig + j;
                    if (q >= a.QG) continue;
#pragma unroll
                    for (int mm = 0; mm < 8; mm += 2) {
                        float4 v;
                        v.x = acc[0][mm][j] * inv[0][j];
                        v.y = acc[0][mm][j + 2] * inv[0][j];
                        v.z = acc[0][mm + 1][j] * inv[0][j];
                        v.w = acc[0][mm + 1][j + 2] * inv[0][j];
                        *reinterpret_cast<float4*>(stg + q * kHeadDim + 16 * gid + 2 * mm) = v;
                    }
                }
                fence_proxy_async_shared();   // each lane's staging writes, before the bulk copy reads them
                __syncwarp();
                if (lane == 0) {
                    bulk_store(a.partial_out + row0 * kHeadDim, smem_addr(stg), (uint32_t)(a.QG * kHeadDim * 4));
                    bulk_commit();
                    bulk_wait_read_all();
                    mbar_arrive(m.empty0 + 8 * last);
                }
            } else {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int q = n * 8 + 2 * tig + j;
                        if (q >= a.QG) continue;
                        float* dst = a.partial_out + (row0 + q) * kHeadDim + 16 * gid;
#pragma unroll
                        for (int mm = 0; mm < 8; mm += 2) {
                            float4 v;
                            v.x = acc[n][mm][j] * inv[n][j];
                            v.y = acc[n][mm][j + 2] * inv[n][j];
                            v.z = acc[n][mm + 1][j] * inv[n][j];
                            v.w = acc[n][mm + 1][j + 2] * inv[n][j];
                            *reinterpret_cast<float4*>(dst + 2 * mm) = v;
                        }
                    }
                __syncwarp();
                if (lane == 0) mbar_arrive(m.empty0 + 8 * last);
            }
            if (gid == 0) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int q = n * 8 + 2 * tig + j;
                        if (q < a.QG) {
                            a.exp_sums[row0 + q] = ls[n][j];
                            a.max_logits[row0 + q] = m2[n][j] * kLn2;
                        }
                    }
            }
            u = nx;
        }
        if (lane == 0) {
            if (!ok && a.err_word) atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
            bulk_wait_all();   // the partials are written before the CTA retires
        }
        __syncwarp();
    }

    // ------------------------------------------------------------------ fused step
    // After every CTA's partition pass (a grid barrier: the launch is cooperative, so every CTA is
    // resident and the bounded wait ends), every warp of the launch merges its share of the output
    // rows, dealt round robin, with merge_row (the reduce kernel's arithmetic: the same bits as
    // pda_decode + pda_reduce).  Rows of sequences without tokens are written as zeros.  The
    // launch's counter slot holds {next unit, -, -, -, CTAs done, CTAs arrived}.
    static __device__ __noinline__ void merge_all(const DecodeArgs& a) {
        const int max_ctx = a.MB * a.BS, nwarps = blockDim.x >> 5;
        const long long rows = (long long)a.B * a.Hk * a.QG, rps = (long long)a.Hk * a.QG;
        const MergeArgs mg{a.partial_out, a.exp_sums, a.max_logits, a.out, a.Hk, a.QG, a.P, a.W, a.out_f32};
        int cb = -1, c = 0;   // the last sequence whose context length was read, and that length
        for (long long row = (long long)blockIdx.x * nwarps + (threadIdx.x >> 5); row < rows;
             row += (long long)gridDim.x * nwarps) {
            const int b = (int)(row / rps);
            const int rem = (int)(row - (long long)b * rps);
            const int h = rem / a.QG, q = rem - h * a.QG;
            if (b != cb) {
                cb = b;
                c = sanitize_ctx(__ldcg(a.context_lens + b), max_ctx);
            }
            merge_row(mg, b, h, q, c);
        }
    }
    static __device__ void run(const DecodeArgs& a, const CUtensorMap* kv_map, const CUtensorMap* sc_map,
                               uint8_t* smem) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int HG = a.HG;
        Smem m;
        m.base = smem_addr(smem);
        m.ptr = smem;
        m.off_scales = (uint32_t)(S * group_stage_bytes(HG));
        const uint32_t off_bar = m.off_scales + (uint32_t)(S * group_scale_bytes(HG));
        m.full0 = m.base + off_bar;
        m.empty0 = m.full0 + 8 * S;
        m.ufull0 = m.empty0 + 8 * S;
        m.uempty0 = m.ufull0 + 8 * R;
        m.udesc = reinterpret_cast<int4*>(smem + off_bar + 16 * S + 16 * R);
        int* above = reinterpret_cast<int*>(smem + off_bar + 16 * S + 16 * R + 16 * R);
        int* hist = above + (kGroupBuckets + 2);
        m.above = above;
        if (warp == 0 && lane == 0) {
            for (int st = 0; st < S; ++st) {
                mbar_init(m.full0 + 8 * st, 1);
                mbar_init(m.empty0 + 8 * st, (uint32_t)HG);
            }
            for (int r = 0; r < R; ++r) {
                mbar_init(m.ufull0 + 8 * r, 1);
                mbar_init(m.uempty0 + 8 * r, (uint32_t)HG);
            }
            fence_mbar_init();
            prefetch_tensormap(kv_map);
            prefetch_tensormap(sc_map);
        }
        allow_dependent_launch();   // the reduce may be scheduled as soon as CTAs of this grid retire
        grid_dependency_wait();     // inputs may come from the previous grid on the stream
        group_buckets_init(a, above, hist);
        __syncthreads();            // the barriers and the bucket table are ready
        if constexpr (!FUSED) {
            if (warp == 0)
                produce(a, kv_map, sc_map, m);
            else if (warp <= HG)
                consume(a, warp - 1, m);
        } else {
            if (warp == 0)
                produce(a, kv_map, sc_map, m);
            else if (warp <= HG)
                consume(a, warp - 1, m);
            // the CTA's partials are written (each consumer waited for its bulk copies): order them,
            // and the statistics, before the CTA is counted
            if (warp >= 1 && warp <= HG && lane == 0) fence_proxy_async_global();
            __threadfence();
            __syncthreads();
            __shared__ int arrived_all;
            const bool alone = gridDim.x == 1;   // one CTA: it waits for no one
            if (threadIdx.x == 0 && alone) arrived_all = 1;
            if (threadIdx.x == 0 && !alone) {
                atomicAdd(a.sched + 5, 1u);
                const uint64_t t0 = global_timer_ns();
                unsigned int backoff = 32;
                int arrived = 0;
                while ((arrived = ld_acquire_gpu(reinterpret_cast<const int*>(a.sched + 5))) < (int)gridDim.x) {
                    if (global_timer_ns() - t0 > a.timeout_ns) break;
                    __nanosleep(backoff);
                    backoff = min(backoff * 2, 256u);
                }
                arrived_all = arrived >= (int)gridDim.x;
            }
            __syncthreads();
            if (arrived_all)
                merge_all(a);
            else if (threadIdx.x == 0 && a.err_word)
                atomicOr(a.err_word, PDA_ERRW_PIPELINE_TIMEOUT);
            // the launch's last CTA returns the slot to zero
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                if (atomicAdd(a.sched + 4, 1u) == gridDim.x - 1) {   // (also resets the unit counter)
                    a.sched[0] = a.sched[1] = a.sched[2] = a.sched[3] = a.sched[5] = 0u;
                    __threadfence();
                    a.sched[4] = 0u;
                }
            }
        }
    }
};

// NWARPS: warps per CTA the register allocation is sized for (producer + up to NWARPS - 1
// consumers); MINB: CTAs per SM it must allow.
template <int NT, int S, int NWARPS, int MINB, bool FUSED>
__global__ void __launch_bounds__(NWARPS * 32, MINB) pda_group_kernel(const __grid_constant__ CUtensorMap kv_map,
                                                                     const __grid_constant__ CUtensorMap sc_map,
                                                                     const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GroupDecode<NT, S, FUSED>::run(a, &kv_map, &sc_map, smem);
}

}  // namespace pda
