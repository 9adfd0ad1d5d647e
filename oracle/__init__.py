"""fp64 CPU oracle for single-token paged-KV GQA decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The product path (the
CUDA library and its Python binding) never imports, loads or calls it, and the two share no
code: this package computes the cache layout, the partition plan and the attention from their
definitions on its own.

Contents
  * ``build()``            compiles ``pda_oracle.c`` (plain C, fp64, no fast-math) with gcc.
  * ``Problem``            the sizes of one decode step.
  * ``cache_layout()``     cache block layout of the vLLM "tq_decode" page (stride block of
                           build_tq_decode_module), with the bf16 / fp8+fp32-scale element formats.
  * ``plan()``             partition arithmetic: W = G*256 tokens (build_tq_decode_module,
                           tile_groups_per_partition), P = ceil(MB*BS / W), and the launcher's
                           cap policy G = ceil(MB*BS / (256*cap)) from the same docstring.
  * ``decode()``           the attention itself (see ``pda_oracle.c`` for the definition and the
                           passages it follows), optionally with per-partition partials.
  * ``e4m3_to_float64()``  the OCP FP8 E4M3 decode written from the format definition.
  * ``e4m3_encode()``      its encode: nearest finite code by brute force, ties to even, saturating.
  * ``f16_to_float64()``   the IEEE binary16 decode (the TQ4 format's metadata fields).
  * ``append_kv()``        the write side: one new token per sequence into the paged cache.

Parity of every function here is pinned by ``tests/test_oracle_pins.py`` against closed forms,
invariants, brute force, library routines and the page's worked sizing example.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_TQ4 = 2          # the page's 4-bit format: K codes into 16 centroids times k_norm, V codes affine
TQ4_FIELDS = 3      # fp16 metadata fields per (kv_head, slot): k_norm, v_scale, v_zero
TOKENS_PER_TILE_GROUP = 256   # KV_COMPUTE_BLOCK: 16 tiles of 16 tokens


def build(force: bool = False) -> str:
    """Compiles the oracle into ``oracle/_liboracle.so`` (IEEE fp64, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "num_seqs", "num_kv_heads", "query_group_size", "head_dim", "kv_block_size",
        "max_blocks_per_seq", "kv_dtype", "partition_tokens", "num_partitions",
        "num_cache_blocks", "cache_block_bytes", "meta_offset_bytes")] + [("softmax_scale", ctypes.c_double),
                                                                         ("centroids", ctypes.c_void_p)]


def load_library(path: str):
    """Loads an oracle shared library (the built one, or a test's deliberately broken copy)."""
    lib = ctypes.CDLL(path)
    lib.oracle_decode_units.restype = ctypes.c_int
    lib.oracle_decode_units.argtypes = [ctypes.POINTER(_Problem)] + [ctypes.c_void_p] * 5 + [
        ctypes.c_int64] + [ctypes.c_void_p] * 4
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_f16_to_double.restype = ctypes.c_double
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_append_kv.restype = ctypes.c_int
    lib.oracle_append_kv.argtypes = [ctypes.POINTER(_Problem)] + [ctypes.c_void_p] * 5
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


@dataclass(frozen=True)
class Problem:
    num_seqs: int
    num_kv_heads: int
    query_group_size: int
    kv_block_size: int
    max_blocks_per_seq: int
    num_cache_blocks: int
    kv_dtype: int = KV_BF16
    head_dim: int = 128
    tile_groups_per_partition: int = 1
    softmax_scale: float | None = None

    @property
    def scale(self) -> float:
        # default 1/sqrt(head_size): build_tq_decode_module
        return 1.0 / math.sqrt(self.head_dim) if not self.softmax_scale or self.softmax_scale <= 0 \
            else float(self.softmax_scale)


def cache_layout(num_kv_heads: int, kv_block_size: int, head_dim: int, kv_dtype: int) -> dict:
    """Byte layout of one cache block.

    Data region ``[slot][kv_head][K | V]`` (the page's data stride per slot is
    num_kv_heads * bytes-per-slot-per-head), followed by the metadata region
    ``[kv_head][field][slot]``: fp32 {K scale, V scale} for fp8, fp16 {k_norm, v_scale, v_zero}
    for TQ4 (head_dim/2 bytes of 4-bit codes each for K and V), absent for bf16.
    """
    if kv_dtype == KV_TQ4:
        token_head_bytes = head_dim                      # 2 * head_dim codes of 4 bits
        meta = num_kv_heads * TQ4_FIELDS * kv_block_size * 2
    else:
        token_head_bytes = 2 * head_dim * (2 if kv_dtype == KV_BF16 else 1)
        meta = 0 if kv_dtype == KV_BF16 else num_kv_heads * 2 * kv_block_size * 4
    data = kv_block_size * num_kv_heads * token_head_bytes
    return {"token_head_bytes": token_head_bytes, "data_region_bytes": data,
            "meta_offset_bytes": data, "meta_region_bytes": meta,
            "cache_block_bytes": data + meta}


def plan(max_blocks_per_seq: int, kv_block_size: int, tile_groups_per_partition: int = 1,
         max_partitions: int = 0) -> dict:
    """Partition arithmetic of build_tq_decode_module and its launcher policy.

    G = tile_groups_per_partition, or (G == 0) the smallest G with P <= max_partitions;
    W = G * 256 tokens; P = ceil(max_context / W) with max_context = MB * BS.
    """
    max_ctx = max_blocks_per_seq * kv_block_size
    G = tile_groups_per_partition
    if G == 0:
        G = 1 if max_partitions <= 0 else max(1, -(-max_ctx // (TOKENS_PER_TILE_GROUP * max_partitions)))
    W = G * TOKENS_PER_TILE_GROUP
    P = -(-max_ctx // W)
    return {"G": G, "W": W, "P": P, "max_context": max_ctx, "coverage": P * W}


def e4m3_to_float64(codes, lib=None) -> np.ndarray:
    lib = lib or _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_to_double(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def decode(problem: Problem, query: np.ndarray, cache: np.ndarray, block_table: np.ndarray,
           context_lens: np.ndarray, units=None, partials: bool = False, threads: int | None = None,
           lib=None, centroids=None):
    """Runs the oracle.

    query: uint16 bf16 bits [B][Hk*QG][D]; cache: uint8 [NB * cache_block_bytes];
    block_table: int32 [B][MB]; context_lens: int32 [B].
    ``units``: iterable of b*Hk + h to compute (default: all).  Returns a dict with ``out``
    float64 [B][Hq][D] (NaN for rows not computed) and, if ``partials``, ``part_o`` [B][Hk][P][QG][D],
    ``part_m``, ``part_l`` [B][Hk][P][QG] (NaN where the partition is empty or not computed),
    plus ``threads`` (the worker threads actually used).  ``lib`` overrides the library.
    ``centroids``: the 16 float32 centroids of a TQ4 cache (required for that format only).
    """
    lib = lib or _load()
    pr = problem
    lay = cache_layout(pr.num_kv_heads, pr.kv_block_size, pr.head_dim, pr.kv_dtype)
    pl = plan(pr.max_blocks_per_seq, pr.kv_block_size, pr.tile_groups_per_partition)
    B, Hk, QG, D, P = pr.num_seqs, pr.num_kv_heads, pr.query_group_size, pr.head_dim, pl["P"]

    query = np.ascontiguousarray(query, dtype=np.uint16)
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    assert query.size == B * Hk * QG * D
    assert cache.size == pr.num_cache_blocks * lay["cache_block_bytes"]
    assert block_table.size == B * pr.max_blocks_per_seq and context_lens.size == B

    cent = None
    if pr.kv_dtype == KV_TQ4:
        cent = np.ascontiguousarray(centroids, dtype=np.float32)
        assert cent.shape == (16,), "a TQ4 cache needs its 16 centroids"
    cp = _Problem(B, Hk, QG, D, pr.kv_block_size, pr.max_blocks_per_seq, pr.kv_dtype, pl["W"], P,
                  pr.num_cache_blocks, lay["cache_block_bytes"], lay["meta_offset_bytes"], pr.scale,
                  None if cent is None else cent.ctypes.data)

    out = np.full((B, Hk * QG, D), np.nan)
    po = pm = plv = None
    if partials:
        po = np.full((B, Hk, P, QG, D), np.nan)
        pm = np.full((B, Hk, P, QG), np.nan)
        plv = np.full((B, Hk, P, QG), np.nan)
    ulist = np.arange(B * Hk, dtype=np.int64) if units is None else np.asarray(list(units), dtype=np.int64)
    if ulist.size == 0:
        return {"out": out, "part_o": po, "part_m": pm, "part_l": plv, "threads": 0}

    nthreads = max(1, min(threads or os.cpu_count() or 1, ulist.size))
    chunks = [c for c in np.array_split(ulist, nthreads) if c.size]

    def ptr(a):
        return None if a is None else a.ctypes.data

    def run(chunk):
        chunk = np.ascontiguousarray(chunk)
        return lib.oracle_decode_units(ctypes.byref(cp), ptr(query), ptr(cache), ptr(block_table),
                                       ptr(context_lens), chunk.ctypes.data, chunk.size, ptr(out),
                                       ptr(po), ptr(pm), ptr(plv))

    if len(chunks) == 1:
        rcs = [run(chunks[0])]
    else:
        with ThreadPoolExecutor(max_workers=len(chunks)) as ex:   # ctypes releases the GIL
            rcs = list(ex.map(run, chunks))
    for rc in rcs:
        if rc != 0:
            raise ValueError({-1: "context length outside [0, MB*BS]", -2: "block id outside the pool",
                              -3: "out of memory"}.get(rc, f"oracle error {rc}"))
    return {"out": out, "part_o": po, "part_m": pm, "part_l": plv, "threads": len(chunks)}


def f16_to_float64(bits, lib=None) -> np.ndarray:
    lib = lib or _load()
    c = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.oracle_f16_to_double(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(values, lib=None) -> np.ndarray:
    lib = lib or _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.oracle_e4m3_encode(float(x)) for x in v.ravel()], dtype=np.uint8).reshape(v.shape)


def append_kv(problem: Problem, cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray, block_table: np.ndarray,
              positions: np.ndarray, lib=None) -> np.ndarray:
    """Returns a copy of ``cache`` with one token per sequence appended (see pda_oracle.c).
    k_new, v_new: uint16 bf16 bits [B][Hk][D]; positions: int32 [B] (negative: no write)."""
    lib = lib or _load()
    pr = problem
    lay = cache_layout(pr.num_kv_heads, pr.kv_block_size, pr.head_dim, pr.kv_dtype)
    pl = plan(pr.max_blocks_per_seq, pr.kv_block_size, pr.tile_groups_per_partition)
    cp = _Problem(pr.num_seqs, pr.num_kv_heads, 8, pr.head_dim, pr.kv_block_size, pr.max_blocks_per_seq, pr.kv_dtype,
                  pl["W"], pl["P"], pr.num_cache_blocks, lay["cache_block_bytes"], lay["meta_offset_bytes"], pr.scale)
    out = np.array(cache, dtype=np.uint8, copy=True)
    kn = np.ascontiguousarray(k_new, dtype=np.uint16)
    vn = np.ascontiguousarray(v_new, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    rc = lib.oracle_append_kv(ctypes.byref(cp), kn.ctypes.data, vn.ctypes.data, out.ctypes.data, bt.ctypes.data,
                              pos.ctypes.data)
    if rc != 0:
        raise ValueError({-1: "position outside [0, MB*BS)", -2: "block id outside the pool",
                          -4: "no encoder for this cache format"}.get(rc, f"oracle error {rc}"))
    return out
