"""Seeded synthetic inputs for single-token paged-KV GQA decode attention.

This module draws values, rounds them to the storage formats (bf16, OCP FP8 E4M3 with one
fp32 scale per token per KV head, scale = absmax / 448, or the 4-bit "TQ4" codes of the
"tq_decode" page) and writes them into the paged cache layout.  It holds none of the attention
arithmetic and imports neither the CUDA binding nor the oracle; both sides of every parity test
take their inputs from here.

Draw order for one workload (one ``numpy.random.PCG64`` stream seeded with ``seed``):
  1. context lengths, 2. block table, 3. Q, 4. the per-head K bias (if any),
  5. for each sequence in order: its K values, then its V values.
Values are N(0, 1) float32 unless stated.  Bytes the attention must never read (slots past a
sequence's context in its last block, blocks no table references, the scales of those slots)
are filled with 0xFF: NaN in bf16, fp8 e4m3 and fp32 alike ("poison").

Cache block layout (the stride block of build_tq_decode_module on the vLLM "tq_decode" page,
with the element formats of this library):
  data region  [BS slots][Hk kv heads][K: D elements | V: D elements]
  meta region  [Hk][2 fields: K scale, V scale][BS] fp32        (fp8; absent for bf16)
               [Hk][3 fields: k_norm, v_scale, v_zero][BS] fp16 (TQ4)
TQ4 elements are 4-bit codes, two per byte, the even dimension in the low nibble.

The pages give neither the TQ4 codebook nor the quantiser that fills such a cache (the page's
Q and K live in a rotated basis whose rotation is not given either).  The stand-ins here: the
16 centroids are Gaussian quantiles at (j + 1/2)/16 scaled by 1/sqrt(D) (the spread of one
coordinate of a random unit vector in D dimensions); K and Q are drawn directly in the rotated
basis (a rotation of i.i.d. N(0, 1) values is i.i.d. N(0, 1)); a K row stores k_norm = |k| and,
per dimension, the centroid nearest to k_d / k_norm; a V row stores v_zero = min v,
v_scale = (max v - min v) / 15 and codes round((v - v_zero) / v_scale) clipped to [0, 15].
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_TQ4 = 2
E4M3_MAX = 448.0
TQ4_FIELDS = 3      # k_norm, v_scale, v_zero (fp16)


@dataclass(frozen=True)
class Workload:
    name: str
    num_seqs: int
    num_kv_heads: int
    query_group_size: int
    kv_block_size: int
    max_blocks_per_seq: int
    num_cache_blocks: int
    ctx: tuple                      # ("fixed", n) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi) | ("list", tuple)
    seed: int
    kv_dtype: int = KV_BF16
    tile_groups_per_partition: int = 1   # 0 = choose from max_partitions
    max_partitions: int = 0
    head_dim: int = 128
    k_bias_std: float = 0.0
    softmax_scale: float = 0.0      # <= 0: 1/sqrt(head_dim)

    @property
    def num_q_heads(self) -> int:
        return self.num_kv_heads * self.query_group_size

    @property
    def token_head_bytes(self) -> int:
        """K and V bytes of one token of one KV head."""
        return {KV_BF16: 4, KV_FP8_E4M3: 2, KV_TQ4: 1}[self.kv_dtype] * self.head_dim

    @property
    def data_region_bytes(self) -> int:
        return self.kv_block_size * self.num_kv_heads * self.token_head_bytes

    @property
    def meta_region_bytes(self) -> int:
        if self.kv_dtype == KV_FP8_E4M3:
            return self.num_kv_heads * 2 * self.kv_block_size * 4
        if self.kv_dtype == KV_TQ4:
            return self.num_kv_heads * TQ4_FIELDS * self.kv_block_size * 2
        return 0

    @property
    def cache_block_bytes(self) -> int:
        return self.data_region_bytes + self.meta_region_bytes

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The decode workloads: sizes, distributions and seeds (1000 + index).
WORKLOADS = {
    w.name: w for w in [
        Workload("b1_hk1_qg8_bs16_ctx256", 1, 1, 8, 16, 16, 64, ("fixed", 256), seed=1001),
        Workload("b8_hk8_qg8_bs16_ctx1-4096", 8, 8, 8, 16, 256, 8 * 256, ("uniform", 1, 4096), seed=1002),
        Workload("b32_hk4_qg16_bs32_ctx2048-8192_kbias", 32, 4, 16, 32, 256, 32 * 256,
                 ("uniform", 2048, 8192), seed=1003, k_bias_std=2.0),
        Workload("b4_hk8_qg8_bs32_ctx32768_g5p32", 4, 8, 8, 32, 1280, 4 * 1280, ("fixed", 32768), seed=1004,
                 tile_groups_per_partition=0, max_partitions=32),
        Workload("b64_hk8_qg6_bs16_fp8_lognormal2048", 64, 8, 6, 16, 1024, 64 * 1024,
                 ("lognormal", 2048, 1.0, 16, 16384), seed=1005, kv_dtype=KV_FP8_E4M3),
        # the same step with the page's own 4-bit TQ4 cache
        Workload("b64_hk8_qg6_bs16_tq4_lognormal2048", 64, 8, 6, 16, 1024, 64 * 1024,
                 ("lognormal", 2048, 1.0, 16, 16384), seed=1006, kv_dtype=KV_TQ4),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclass
class Inputs:
    workload: Workload
    query: np.ndarray          # uint16 bf16 bits [B][Hq][D]
    cache: np.ndarray          # uint8 [NB * cache_block_bytes]
    block_table: np.ndarray    # int32 [B][MB]
    context_lens: np.ndarray   # int32 [B]
    extra: dict = field(default_factory=dict)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits (round to nearest even), as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantize_e4m3_rows(x: np.ndarray):
    """Per row over the last axis: scale = absmax/448 (fp32; 1 when the row is all zero),
    codes = e4m3(x / scale) rounded to nearest even.  Returns (uint8 codes, float32 scales)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    scale[amax == 0] = 1.0
    y = x / scale[..., None]
    codes = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scale


def tq4_codebook(head_dim: int = 128) -> np.ndarray:
    """The 16 TQ4 centroids of this generator: N(0, 1/D) quantiles at (j + 1/2) / 16 (float32)."""
    p = (torch.arange(16, dtype=torch.float64) + 0.5) / 16.0
    return (torch.special.ndtri(p) / np.sqrt(head_dim)).numpy().astype(np.float32)


def round_f16(x: np.ndarray) -> np.ndarray:
    """float32 -> fp16 bits (round to nearest even), as uint16."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def quantize_tq4_k(K: np.ndarray, centroids: np.ndarray):
    """K rows [..][D] -> (codes uint8 [..][D], k_norm fp16 bits [..]): k_norm = |k| in fp16 and the
    nearest centroid to k_d / k_norm per dimension."""
    K = np.asarray(K, dtype=np.float32)
    norm_bits = round_f16(np.sqrt((K.astype(np.float64) ** 2).sum(axis=-1)))
    norm = norm_bits.view(np.float16).astype(np.float32)
    unit = K / np.where(norm > 0, norm, 1.0)[..., None]
    c = np.asarray(centroids, dtype=np.float32)
    assert np.all(np.diff(c) > 0), "centroids must be increasing"
    mid = (c[1:] + c[:-1]) / 2                      # nearest centroid, ties to the lower one
    codes = np.searchsorted(mid, unit, side="left").astype(np.uint8)
    return codes, norm_bits


def quantize_tq4_v(V: np.ndarray):
    """V rows [..][D] -> (codes uint8 [..][D], v_scale fp16 bits, v_zero fp16 bits)."""
    V = np.asarray(V, dtype=np.float32)
    zero_bits = round_f16(V.min(axis=-1))
    scale_bits = round_f16((V.max(axis=-1) - V.min(axis=-1)) / np.float32(15.0))
    z = zero_bits.view(np.float16).astype(np.float32)[..., None]
    sc = scale_bits.view(np.float16).astype(np.float32)[..., None]
    codes = np.clip(np.rint((V - z) / np.where(sc > 0, sc, 1.0)), 0, 15).astype(np.uint8)
    return codes, scale_bits, zero_bits


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """4-bit codes [..][D] -> bytes [..][D/2], dimension 2j in the low nibble of byte j."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def cache_views(w: Workload, cache: np.ndarray):
    """Writable strided views: data [NB][BS][Hk][2][D] (uint16 for bf16, uint8 for fp8; packed
    codes [NB][BS][Hk][2][D/2] for TQ4) and meta [NB][Hk][2][BS] float32 (fp8) or
    [NB][Hk][3][BS] fp16 bits (TQ4)."""
    from numpy.lib.stride_tricks import as_strided
    NB, BS, Hk, D = w.num_cache_blocks, w.kv_block_size, w.num_kv_heads, w.head_dim
    cbb = w.cache_block_bytes
    if w.kv_dtype == KV_BF16:
        data = cache.view(np.uint16).reshape(NB, BS, Hk, 2, D)
        return data, None
    if w.kv_dtype == KV_TQ4:
        data = as_strided(cache, shape=(NB, BS, Hk, 2, D // 2), strides=(cbb, Hk * D, D, D // 2, 1), writeable=True)
        meta_base = cache[w.data_region_bytes:].view(np.uint16)
        meta = as_strided(meta_base, shape=(NB, Hk, TQ4_FIELDS, BS), strides=(cbb, TQ4_FIELDS * BS * 2, BS * 2, 2),
                          writeable=True)
        return data, meta
    data = as_strided(cache, shape=(NB, BS, Hk, 2, D), strides=(cbb, Hk * 2 * D, 2 * D, D, 1), writeable=True)
    meta_base = cache[w.data_region_bytes:].view(np.float32)
    meta = as_strided(meta_base, shape=(NB, Hk, 2, BS), strides=(cbb, 2 * BS * 4, BS * 4, 4), writeable=True)
    return data, meta


def draw_context_lens(w: Workload, rng: np.random.Generator) -> np.ndarray:
    kind = w.ctx[0]
    B = w.num_seqs
    if kind == "fixed":
        c = np.full(B, w.ctx[1])
    elif kind == "uniform":
        c = rng.integers(w.ctx[1], w.ctx[2] + 1, size=B)
    elif kind == "lognormal":
        _, median, sigma, lo, hi = w.ctx
        c = np.clip(np.rint(np.exp(rng.normal(np.log(median), sigma, size=B))), lo, hi)
    elif kind == "list":
        c = np.asarray(w.ctx[1])
        assert c.size == B
    else:
        raise ValueError(kind)
    return c.astype(np.int32)


def draw_block_table(w: Workload, rng: np.random.Generator) -> np.ndarray:
    """Blocks drawn without replacement from the pool (a random permutation)."""
    n = w.num_seqs * w.max_blocks_per_seq
    assert w.num_cache_blocks >= n, "pool smaller than the tables"
    return rng.permutation(w.num_cache_blocks)[:n].astype(np.int32).reshape(w.num_seqs, w.max_blocks_per_seq)


def write_tokens(w: Workload, cache: np.ndarray, table_row: np.ndarray, K: np.ndarray, V: np.ndarray,
                 centroids: np.ndarray | None = None):
    """Writes float32 K, V of shape [n][Hk][D] as tokens 0..n-1 of one sequence (TQ4: quantised
    with the given centroids)."""
    n = K.shape[0]
    if n == 0:
        return
    t = np.arange(n)
    blk = table_row[t // w.kv_block_size]
    slot = t % w.kv_block_size
    data, meta = cache_views(w, cache)
    if w.kv_dtype == KV_TQ4:
        kc, kn = quantize_tq4_k(K, centroids)
        vc, vs, vz = quantize_tq4_v(V)
        write_tq4_codes(w, cache, table_row, pack_nibbles(kc), pack_nibbles(vc), kn, vs, vz)
    elif w.kv_dtype == KV_BF16:
        data[blk, slot, :, 0, :] = round_bf16(K)
        data[blk, slot, :, 1, :] = round_bf16(V)
    else:
        kc, ks = quantize_e4m3_rows(K)
        vc, vs = quantize_e4m3_rows(V)
        data[blk, slot, :, 0, :] = kc
        data[blk, slot, :, 1, :] = vc
        meta[blk, :, 0, slot] = ks
        meta[blk, :, 1, slot] = vs


def write_tq4_codes(w: Workload, cache: np.ndarray, table_row: np.ndarray, k_bytes, v_bytes, k_norm, v_scale, v_zero):
    """Writes packed TQ4 codes [n][Hk][D/2] and fp16 field bits [n][Hk] as tokens 0..n-1."""
    n = k_bytes.shape[0]
    if n == 0:
        return
    t = np.arange(n)
    blk = table_row[t // w.kv_block_size]
    slot = t % w.kv_block_size
    data, meta = cache_views(w, cache)
    data[blk, slot, :, 0, :] = k_bytes
    data[blk, slot, :, 1, :] = v_bytes
    meta[blk, :, 0, slot] = k_norm
    meta[blk, :, 1, slot] = v_scale
    meta[blk, :, 2, slot] = v_zero


def empty_cache(w: Workload, poison: bool = True) -> np.ndarray:
    return np.full(w.num_cache_blocks * w.cache_block_bytes, 0xFF if poison else 0, dtype=np.uint8)


def generate(w: Workload, poison: bool = True) -> Inputs:
    rng = np.random.Generator(np.random.PCG64(w.seed))
    B, Hk, D = w.num_seqs, w.num_kv_heads, w.head_dim
    ctx = draw_context_lens(w, rng)
    assert (ctx <= w.max_blocks_per_seq * w.kv_block_size).all()
    table = draw_block_table(w, rng)
    q = rng.standard_normal((B, w.num_q_heads, D), dtype=np.float32)
    bias = None
    if w.k_bias_std:
        bias = (rng.standard_normal((Hk, D), dtype=np.float32) * np.float32(w.k_bias_std)).astype(np.float32)
    cache = empty_cache(w, poison)
    cent = tq4_codebook(D) if w.kv_dtype == KV_TQ4 else None
    for b in range(B):
        n = int(ctx[b])
        K = rng.standard_normal((n, Hk, D), dtype=np.float32)
        if bias is not None:
            K += bias[None]
        V = rng.standard_normal((n, Hk, D), dtype=np.float32)
        write_tokens(w, cache, table[b], K, V, cent)
    extra = {"k_bias": bias}
    if cent is not None:
        extra["centroids"] = cent
    return Inputs(w, round_bf16(q), cache, table, ctx, extra)


def small(name="small", num_seqs=2, num_kv_heads=2, query_group_size=8, kv_block_size=16, ctx=(40, 17),
          kv_dtype=KV_BF16, tile_groups_per_partition=1, max_partitions=0, seed=7, extra_blocks=3,
          max_blocks_per_seq=None, k_bias_std=0.0) -> Workload:
    """A small workload for tests: explicit context lengths, a pool a few blocks larger than the
    tables so that unreferenced (poisoned) blocks exist."""
    ctx = tuple(int(c) for c in ctx)
    assert len(ctx) == num_seqs
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, -(-max(ctx) // kv_block_size))
    nb = num_seqs * max_blocks_per_seq + extra_blocks
    return Workload(name, num_seqs, num_kv_heads, query_group_size, kv_block_size, max_blocks_per_seq, nb,
                    ("list", ctx), seed=seed, kv_dtype=kv_dtype, tile_groups_per_partition=tile_groups_per_partition,
                    max_partitions=max_partitions, k_bias_std=k_bias_std)
