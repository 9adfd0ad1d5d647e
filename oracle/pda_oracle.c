/*
 * pda_oracle.c -- fp64 CPU oracle for single-token paged-KV GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this file:
 * only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg use it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes is the plain definition of softmax attention (the split over context
 * partitions and the online softmax of the GPU path reach the same value up to rounding):
 *
 *   for every sequence b, KV head h and query row r < QG (query head h*QG + r):
 *     q        = Q[b][h*QG + r][:]                                        (bf16 -> double)
 *     for t < ctx_b:  blk = block_table[b][t / BS],  slot = t % BS          (the block walk)
 *                     k_t, v_t = decode(cache[blk] data region, slot, h)
 *                     s_t = softmax_scale * sum_d q_d k_{t,d}
 *     m   = max_t s_t
 *     out = sum_t exp(s_t - m) v_t / sum_t exp(s_t - m)      (ctx_b == 0  ->  out = 0)
 *
 * plus, for every partition p with p*W < ctx_b (W = partition extent in tokens), the
 * partial over tokens [p*W, min((p+1)*W, ctx_b)):
 *     m_p = max s_t,   l_p = sum exp(s_t - m_p),   o_p = sum exp(s_t - m_p) v_t / l_p.
 *
 * Sources (the vLLM "tq_decode" page, build_tq_decode_module and tq_decode_kernel):
 *   - grid unit (sequence, KV head, partition) and the partition base p*W: kernel "IDs" and
 *     STEP E;  empty partitions run no iterations (STEP E/F trip-count clamp);
 *   - block-table walk, entry t/BS, slot t%BS, one entry reused for the two 16-token tiles
 *     of a 32-token block: build_tq_decode_module docstring (kv_block_size) and STEP F;
 *   - cache block = data region [slot][kv_head][K bytes | V bytes] then a structure-of-
 *     arrays metadata region [kv_head][field][slot]: the stride block of the module builder;
 *   - scale then mask (tokens >= seq_len get -inf), online softmax: STEP F;
 *   - partial epilogue (normalised partial, running max, running sum; sum<=0 treated as 1):
 *     STEP G;   default softmax_scale = 1/sqrt(head_size): module builder.
 * The KV element formats are bf16, or OCP FP8 E4M3 ("e4m3fn") with one fp32 scale per
 * token per KV head for K and for V, kept in the metadata region as [kv_head][K,V][slot], or
 * the page's own 4-bit format ("TQ4"), decoded as its STEP F does it:
 *   - a token-head row is 64 bytes of K codes then 64 bytes of V codes; dimension d is the
 *     low nibble of byte d/2 when d is even, the high nibble when d is odd (the page reads
 *     32-bit words and takes nibble n of word w, low bits first, as dimension 8w + n);
 *   - K element = centroid[code] * k_norm, V element = code * v_scale + v_zero, with k_norm,
 *     v_scale and v_zero fp16 fields of the metadata region [kv_head][field][slot] and the
 *     16 fp32 centroids a separate input (STEP A loads them);
 *   - the page rounds each decoded element to bf16 before its MFMAs; the oracle keeps the
 *     exact products (the rounding is the kernel's business, as for P);
 *   - Q is taken as given: the page's Q arrives already rotated (STEP B), so the rotation is
 *     not part of this computation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Mirrors the field order of the Python ctypes structure in oracle/__init__.py. */
typedef struct {
    int64_t num_seqs;          /* B                                   */
    int64_t num_kv_heads;      /* Hk                                  */
    int64_t query_group_size;  /* QG; query heads = Hk * QG           */
    int64_t head_dim;          /* D                                   */
    int64_t kv_block_size;     /* BS tokens per cache block           */
    int64_t max_blocks_per_seq;/* MB, row length of the block table   */
    int64_t kv_dtype;          /* 0 = bf16, 1 = fp8 e4m3 + fp32 scale, 2 = TQ4 */
    int64_t partition_tokens;  /* W = G * 256                         */
    int64_t num_partitions;    /* P                                   */
    int64_t num_cache_blocks;  /* NB, blocks in the pool              */
    int64_t cache_block_bytes; /* bytes per cache block               */
    int64_t meta_offset_bytes; /* start of the metadata region        */
    double softmax_scale;
    const float* centroids;    /* TQ4 only: the 16 centroids          */
} oracle_problem;

enum { KV_BF16 = 0, KV_FP8_E4M3 = 1, KV_TQ4 = 2 };
enum { TQ4_K_NORM = 0, TQ4_V_SCALE = 1, TQ4_V_ZERO = 2, TQ4_FIELDS = 3 };

enum { ORACLE_OK = 0, ORACLE_BAD_CTX = -1, ORACLE_BAD_BLOCK = -2, ORACLE_NOMEM = -3, ORACLE_UNSUPPORTED = -4 };

/* bf16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 * Exponent field 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no infinity. */
double oracle_e4m3_to_double(uint8_t x) {
    int sign = (x >> 7) & 1;
    int e = (x >> 3) & 0xF;
    int m = x & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits with bias 15, 10 mantissa bits; exponent field 0
 * encodes subnormals m/1024 * 2^-14, field 31 encodes infinity (m = 0) or NaN. */
double oracle_f16_to_double(uint16_t x) {
    int sign = (x >> 15) & 1;
    int e = (x >> 10) & 0x1F;
    int m = x & 0x3FF;
    double v;
    if (e == 0x1F) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m / 1024.0, -14);
    else v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -v : v;
}

static float load_f32_le(const uint8_t* p) {
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t load_u16_le(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Decodes K (which == 0) or V (which == 1) of token slot `slot`, KV head h, cache block blk. */
static void decode_row(const oracle_problem* pr, const uint8_t* cache, int64_t blk, int64_t slot,
                       int64_t h, int which, double* dst) {
    const int64_t D = pr->head_dim, BS = pr->kv_block_size;
    const uint8_t* block = cache + blk * pr->cache_block_bytes;
    if (pr->kv_dtype == KV_TQ4) {
        /* K codes then V codes, D/2 bytes each, per token-head */
        const int64_t token_head_bytes = D;
        const uint8_t* row = block + (slot * pr->num_kv_heads + h) * token_head_bytes + (int64_t)which * (D / 2);
        const uint8_t* meta = block + pr->meta_offset_bytes + h * TQ4_FIELDS * BS * 2;
        if (which == 0) {
            const double k_norm = oracle_f16_to_double(load_u16_le(meta + (TQ4_K_NORM * BS + slot) * 2));
            for (int64_t d = 0; d < D; ++d) {
                const int code = (row[d / 2] >> ((d % 2) * 4)) & 0xF;
                dst[d] = (double)pr->centroids[code] * k_norm;
            }
        } else {
            const double v_scale = oracle_f16_to_double(load_u16_le(meta + (TQ4_V_SCALE * BS + slot) * 2));
            const double v_zero = oracle_f16_to_double(load_u16_le(meta + (TQ4_V_ZERO * BS + slot) * 2));
            for (int64_t d = 0; d < D; ++d) {
                const int code = (row[d / 2] >> ((d % 2) * 4)) & 0xF;
                dst[d] = (double)code * v_scale + v_zero;
            }
        }
        return;
    }
    const int64_t elem = pr->kv_dtype == KV_BF16 ? 2 : 1;
    const int64_t token_head_bytes = 2 * D * elem;           /* K bytes then V bytes */
    const uint8_t* row = block + slot * pr->num_kv_heads * token_head_bytes + h * token_head_bytes +
                         (int64_t)which * D * elem;
    if (pr->kv_dtype == KV_BF16) {
        for (int64_t d = 0; d < D; ++d) dst[d] = bf16_bits_to_double(load_u16_le(row + 2 * d));
    } else {
        /* metadata region: [kv_head][field: 0 = K scale, 1 = V scale][slot] fp32 */
        const uint8_t* sp = block + pr->meta_offset_bytes +
                            ((h * 2 + which) * pr->kv_block_size + slot) * 4;
        double scale = (double)load_f32_le(sp);
        for (int64_t d = 0; d < D; ++d) dst[d] = oracle_e4m3_to_double(row[d]) * scale;
    }
}

/*
 * Computes the listed (sequence, KV head) units.  unit = b * Hk + h.
 *   query        bf16 bits [B][Hk*QG][D]
 *   cache        bytes     [NB][cache_block_bytes]
 *   block_table  int32     [B][MB]
 *   context_lens int32     [B]
 *   out          double    [B][Hk*QG][D]         rows of the listed units are written
 *   part_o       double    [B][Hk][P][QG][D]     may be NULL; partitions >= ceil(ctx/W) untouched
 *   part_m/l     double    [B][Hk][P][QG]        may be NULL
 * Returns ORACLE_OK, or a negative code for a context length outside [0, MB*BS] or a block
 * id outside [0, NB) (the oracle does not define results for such inputs).
 */
int oracle_decode_units(const oracle_problem* pr, const uint16_t* query, const uint8_t* cache,
                        const int32_t* block_table, const int32_t* context_lens,
                        const int64_t* units, int64_t n_units, double* out, double* part_o,
                        double* part_m, double* part_l) {
    const int64_t Hk = pr->num_kv_heads, QG = pr->query_group_size, D = pr->head_dim;
    const int64_t BS = pr->kv_block_size, MB = pr->max_blocks_per_seq;
    const int64_t W = pr->partition_tokens, P = pr->num_partitions;
    const int64_t Hq = Hk * QG;

    for (int64_t ui = 0; ui < n_units; ++ui) {
        const int64_t b = units[ui] / Hk, h = units[ui] % Hk;
        const int64_t ctx = context_lens[b];
        if (ctx < 0 || ctx > MB * BS) return ORACLE_BAD_CTX;

        double* K = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * (size_t)D);
        double* V = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * (size_t)D);
        double* s = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
        double* q = (double*)malloc(sizeof(double) * (size_t)D);
        if (!K || !V || !s || !q) {
            free(K); free(V); free(s); free(q);
            return ORACLE_NOMEM;
        }

        /* gather every token of the context through the block table */
        for (int64_t t = 0; t < ctx; ++t) {
            const int64_t blk = block_table[b * MB + t / BS];
            const int64_t slot = t % BS;
            if (blk < 0 || blk >= pr->num_cache_blocks) {
                free(K); free(V); free(s); free(q);
                return ORACLE_BAD_BLOCK;
            }
            decode_row(pr, cache, blk, slot, h, 0, K + t * D);
            decode_row(pr, cache, blk, slot, h, 1, V + t * D);
        }

        for (int64_t r = 0; r < QG; ++r) {
            const int64_t qh = h * QG + r;
            for (int64_t d = 0; d < D; ++d) q[d] = bf16_bits_to_double(query[(b * Hq + qh) * D + d]);

            for (int64_t t = 0; t < ctx; ++t) {
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d) dot += q[d] * K[t * D + d];
                s[t] = pr->softmax_scale * dot;
            }

            /* the whole-context softmax */
            double* o = out + (b * Hq + qh) * D;
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            if (ctx > 0) {
                double m = -INFINITY;
                for (int64_t t = 0; t < ctx; ++t) m = fmax(m, s[t]);
                double l = 0.0;
                for (int64_t t = 0; t < ctx; ++t) {
                    const double e = exp(s[t] - m);
                    l += e;
                    for (int64_t d = 0; d < D; ++d) o[d] += e * V[t * D + d];
                }
                for (int64_t d = 0; d < D; ++d) o[d] /= l;
            }

            /* per-partition partials over [p*W, min((p+1)*W, ctx)) */
            if (part_o || part_m || part_l) {
                for (int64_t p = 0; p < P && p * W < ctx; ++p) {
                    const int64_t lo = p * W, hi = (p + 1) * W < ctx ? (p + 1) * W : ctx;
                    const int64_t idx = ((b * Hk + h) * P + p) * QG + r;
                    double mp = -INFINITY;
                    for (int64_t t = lo; t < hi; ++t) mp = fmax(mp, s[t]);
                    double lp = 0.0;
                    double* op = part_o ? part_o + idx * D : NULL;
                    if (op)
                        for (int64_t d = 0; d < D; ++d) op[d] = 0.0;
                    for (int64_t t = lo; t < hi; ++t) {
                        const double e = exp(s[t] - mp);
                        lp += e;
                        if (op)
                            for (int64_t d = 0; d < D; ++d) op[d] += e * V[t * D + d];
                    }
                    if (op)
                        for (int64_t d = 0; d < D; ++d) op[d] /= lp;
                    if (part_m) part_m[idx] = mp;
                    if (part_l) part_l[idx] = lp;
                }
            }
        }
        free(K); free(V); free(s); free(q);
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------------------------
 * The write side of the same cache: appending one token per sequence.
 *
 * OCP FP8 E4M3 encoding by brute force over the format's finite values: the code of |x| is the
 * finite non-negative code nearest to |x| (ties to the code with an even mantissa, i.e. round to
 * nearest even), values above the largest finite value (448) saturate to it, and the sign of x
 * is copied into the sign bit.  NaN input gives the NaN code.
 */
uint8_t oracle_e4m3_encode(float x) {
    if (x != x) return 0x7F;
    const double ax = fabs((double)x);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {               /* 0x7F is NaN */
        const double v = oracle_e4m3_to_double((uint8_t)c);
        const double d = fabs(v - ax);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(best | (signbit(x) ? 0x80 : 0));
}

/*
 * Writes K and V of one new token for every sequence b with positions[b] >= 0, at token index
 * positions[b]: cache block block_table[b][pos / BS], slot pos % BS (the paged slot formula
 * block = slot // block_size, offset = slot % block_size of the KV insert on the DeepSeek
 * attention-front page; a negative slot means "no write" there too).
 * bf16: the values are stored as given.  fp8: per (token, KV head) and separately for K and V,
 * scale = absmax / 448 in fp32 (1 when the row is all zero), code = e4m3(x / scale) with x / scale
 * rounded to fp32, and the scale is stored in the metadata region [kv_head][K,V][slot].
 *   k_new, v_new  bf16 bits [B][Hk][D];  positions int32 [B].
 * Returns ORACLE_OK, ORACLE_BAD_CTX for a position >= MB*BS, ORACLE_BAD_BLOCK for a block id
 * outside the pool (nothing is written for that sequence in either case), ORACLE_UNSUPPORTED for
 * a TQ4 cache (the pages give no encoder for that format: its rotation and codebook are not on
 * them).
 */
int oracle_append_kv(const oracle_problem* pr, const uint16_t* k_new, const uint16_t* v_new, uint8_t* cache,
                     const int32_t* block_table, const int32_t* positions) {
    const int64_t Hk = pr->num_kv_heads, D = pr->head_dim, BS = pr->kv_block_size, MB = pr->max_blocks_per_seq;
    int rc = ORACLE_OK;
    if (pr->kv_dtype == KV_TQ4) return ORACLE_UNSUPPORTED;
    for (int64_t b = 0; b < pr->num_seqs; ++b) {
        const int64_t pos = positions[b];
        if (pos < 0) continue;
        if (pos >= MB * BS) { rc = ORACLE_BAD_CTX; continue; }
        const int64_t blk = block_table[b * MB + pos / BS], slot = pos % BS;
        if (blk < 0 || blk >= pr->num_cache_blocks) { rc = ORACLE_BAD_BLOCK; continue; }
        uint8_t* block = cache + blk * pr->cache_block_bytes;
        for (int64_t h = 0; h < Hk; ++h) {
            for (int which = 0; which < 2; ++which) {
                const uint16_t* src = (which == 0 ? k_new : v_new) + (b * Hk + h) * D;
                if (pr->kv_dtype == KV_BF16) {
                    uint8_t* row = block + (slot * Hk + h) * 2 * D * 2 + (int64_t)which * D * 2;
                    for (int64_t d = 0; d < D; ++d) {
                        row[2 * d] = (uint8_t)(src[d] & 0xFF);
                        row[2 * d + 1] = (uint8_t)(src[d] >> 8);
                    }
                } else {
                    uint8_t* row = block + (slot * Hk + h) * 2 * D + (int64_t)which * D;
                    float amax = 0.0f;
                    for (int64_t d = 0; d < D; ++d) {
                        const float v = (float)bf16_bits_to_double(src[d]);
                        amax = fmaxf(amax, fabsf(v));
                    }
                    const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
                    for (int64_t d = 0; d < D; ++d) {
                        const float v = (float)bf16_bits_to_double(src[d]);
                        const float y = v / scale;
                        row[d] = oracle_e4m3_encode(y);
                    }
                    uint8_t* sp = block + pr->meta_offset_bytes + ((h * 2 + which) * BS + slot) * 4;
                    uint32_t u;
                    memcpy(&u, &scale, 4);
                    sp[0] = (uint8_t)u; sp[1] = (uint8_t)(u >> 8); sp[2] = (uint8_t)(u >> 16); sp[3] = (uint8_t)(u >> 24);
                }
            }
        }
    }
    return rc;
}
