"""Test-side helpers: map a generated workload onto the oracle's problem description and run
independent brute-force checks.  Only the test suite and the bench's CPU leg use this."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_gqa_block_gb300 import workloads as wl


def resolve_G(w: wl.Workload) -> int:
    return oracle.plan(w.max_blocks_per_seq, w.kv_block_size, w.tile_groups_per_partition, w.max_partitions)["G"]


def problem(w: wl.Workload, G: int | None = None) -> oracle.Problem:
    return oracle.Problem(w.num_seqs, w.num_kv_heads, w.query_group_size, w.kv_block_size,
                          w.max_blocks_per_seq, w.num_cache_blocks, kv_dtype=w.kv_dtype, head_dim=w.head_dim,
                          tile_groups_per_partition=resolve_G(w) if G is None else G,
                          softmax_scale=w.softmax_scale)


def run_oracle(inp: wl.Inputs, partials=False, G=None, units=None, lib=None, threads=None):
    return oracle.decode(problem(inp.workload, G), inp.query, inp.cache, inp.block_table, inp.context_lens,
                         units=units, partials=partials, lib=lib, threads=threads,
                         centroids=inp.extra.get("centroids"))


def build_from_values(w: wl.Workload, q: np.ndarray, K_list, V_list, table: np.ndarray, poison=True) -> wl.Inputs:
    """Inputs from explicit float32 values (for probes); ctx_b = len(K_list[b])."""
    cache = wl.empty_cache(w, poison)
    cent = wl.tq4_codebook(w.head_dim) if w.kv_dtype == wl.KV_TQ4 else None
    for b in range(w.num_seqs):
        wl.write_tokens(w, cache, table[b], K_list[b], V_list[b], cent)
    ctx = np.array([k.shape[0] for k in K_list], dtype=np.int32)
    return wl.Inputs(w, wl.round_bf16(q), cache, table.astype(np.int32), ctx,
                     {} if cent is None else {"centroids": cent})


def tq4_values(codes: np.ndarray, centroids=None, k_norm_bits=None, v_scale_bits=None, v_zero_bits=None):
    """Float64 values of unpacked TQ4 codes [..][D] (independent of any reader): K with centroids
    and k_norm, or V with v_scale and v_zero (fp16 bits, one per row)."""
    f16 = lambda b: np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)[..., None]
    if centroids is not None:
        return np.asarray(centroids, dtype=np.float32).astype(np.float64)[codes] * f16(k_norm_bits)
    return codes.astype(np.float64) * f16(v_scale_bits) + f16(v_zero_bits)


def stored_values(w: wl.Workload, K: np.ndarray):
    """What the cache holds for float32 rows K [n][Hk][D], as float64 (independent of any reader)."""
    if w.kv_dtype == wl.KV_BF16:
        return wl.bf16_bits_to_f32(wl.round_bf16(K)).astype(np.float64)
    codes, scale = wl.quantize_e4m3_rows(K)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return dec * scale.astype(np.float64)[..., None]


def sdpa_reference(w: wl.Workload, q_bits: np.ndarray, Kst, Vst, lo=0, hi=None) -> np.ndarray:
    """torch scaled_dot_product_attention in float64 over tokens [lo, hi) of each sequence, on
    values gathered directly (no cache, no block table).  Returns [B][Hq][D] (NaN where empty)."""
    B, Hk, QG, D = w.num_seqs, w.num_kv_heads, w.query_group_size, w.head_dim
    scale = w.softmax_scale if w.softmax_scale > 0 else 1.0 / np.sqrt(D)
    q = wl.bf16_bits_to_f32(q_bits).astype(np.float64)
    out = np.full((B, Hk * QG, D), np.nan)
    for b in range(B):
        k = Kst[b][lo:hi]
        v = Vst[b][lo:hi]
        if k.shape[0] == 0:
            continue
        qt = torch.from_numpy(q[b]).reshape(1, Hk * QG, 1, D)
        kt = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 0, 2))).reshape(1, Hk, -1, D)
        vt = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 0, 2))).reshape(1, Hk, -1, D)
        # query head h*QG + r reads KV head h
        kt = kt.repeat_interleave(QG, dim=1)
        vt = vt.repeat_interleave(QG, dim=1)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        out[b] = o.reshape(Hk * QG, D).numpy()
    return out
