"""paged_kv_gqa_block_gb300: single-token paged-KV GQA decode attention for GB300 (sm_103a).

Thin binding over the C ABI of ``libpda.so`` (declared in ``include/pda.h``): it checks and
marshals torch tensors into device pointers and calls the library.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and a
missing library raises.  PyTorch provides device memory and streams only.

    p   = plan(num_seqs=..., num_kv_heads=..., query_group_size=8, kv_block_size=16,
               max_blocks_per_seq=..., tile_groups_per_partition=1)
    ws  = workspace(p, device)                    # partial_out, exp_sums, max_logits
    decode(p, query, kv_cache, num_cache_blocks, block_table, context_lens, **ws)
    reduce(p, context_lens, out=out, **ws)        # or decode_step(...) for both
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpda.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_TQ4 = 2
OUT_BF16 = 0
OUT_F32 = 1
ERRW_BAD_CONTEXT_LEN = 1
ERRW_BAD_BLOCK_ID = 2
ERRW_PIPELINE_TIMEOUT = 4
ERRW_BAD_POSITION = 8
HEAD_DIM = 128
VARIANT_AUTO = 0
VARIANT_HEAD_WARPS = 1
VARIANT_HEAD_GROUPS = 2
VARIANT_ROW_HALVES = 3

STATUS = {0: "PDA_OK", -1: "PDA_ERR_INVALID_ARG", -2: "PDA_ERR_UNSUPPORTED", -3: "PDA_ERR_WORKSPACE_TOO_SMALL",
          -4: "PDA_ERR_LAUNCH", -5: "PDA_ERR_NOT_IMPLEMENTED", -6: "PDA_ERR_CUDA"}


class PdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Plan(ctypes.Structure):
    """Mirror of pda_plan_t."""
    _fields_ = [
        ("num_seqs", ctypes.c_int), ("num_kv_heads", ctypes.c_int), ("query_group_size", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("kv_block_size", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
        ("tile_groups_per_partition", ctypes.c_int), ("max_partitions", ctypes.c_int), ("kv_dtype", ctypes.c_int),
        ("softmax_scale", ctypes.c_float), ("wait_timeout_ns", ctypes.c_int), ("kernel_variant", ctypes.c_int),
        ("num_partitions", ctypes.c_int), ("partition_tokens", ctypes.c_int), ("resolved_tile_groups", ctypes.c_int),
        ("resolved_softmax_scale", ctypes.c_float),
        ("cache_block_bytes", ctypes.c_longlong), ("meta_offset_bytes", ctypes.c_longlong),
        ("workspace_bytes", ctypes.c_longlong),
    ]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None
_lock = threading.Lock()
_VP = ctypes.c_void_p


def lib():
    """The loaded libpda.so.  Raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.POINTER(Plan)
            L.pda_plan.argtypes = [P]
            L.pda_plan.restype = ctypes.c_int
            L.pda_decode.argtypes = [P, _VP, _VP, ctypes.c_longlong, _VP, _VP, _VP, _VP, _VP, _VP, _VP]
            L.pda_decode.restype = ctypes.c_int
            L.pda_decode_tq4.argtypes = [P, _VP, _VP, ctypes.c_longlong, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]
            L.pda_decode_tq4.restype = ctypes.c_int
            L.pda_reduce.argtypes = [P, _VP, _VP, _VP, _VP, _VP, ctypes.c_int, _VP, _VP]
            L.pda_reduce.restype = ctypes.c_int
            L.pda_status_string.argtypes = [ctypes.c_int]
            L.pda_status_string.restype = ctypes.c_char_p
            L.pda_workspace_size.argtypes = [P]
            L.pda_workspace_size.restype = ctypes.c_longlong
            L.pda_append_kv.argtypes = [P, _VP, _VP, _VP, ctypes.c_longlong, _VP, _VP, _VP, _VP]
            L.pda_append_kv.restype = ctypes.c_int
            L.pda_decode_fused.argtypes = [P, _VP, _VP, ctypes.c_longlong, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                           ctypes.c_int, _VP, _VP]
            L.pda_decode_fused.restype = ctypes.c_int
            L.pda_decode_step_noalloc.argtypes = [P, _VP, _VP, ctypes.c_longlong, _VP, _VP, _VP, ctypes.c_int, _VP,
                                                  _VP]
            L.pda_decode_step_noalloc.restype = ctypes.c_int
            L.pda_kernel_variant.argtypes = [P]
            L.pda_kernel_variant.restype = ctypes.c_int
            L.pda_plan_struct_size.argtypes = []
            L.pda_plan_struct_size.restype = ctypes.c_int
            if L.pda_plan_struct_size() != ctypes.sizeof(Plan):
                raise RuntimeError("pda_plan_t layout mismatch between include/pda.h and the binding")
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pda_status_string(status).decode()


def plan(num_seqs: int, num_kv_heads: int, query_group_size: int, kv_block_size: int, max_blocks_per_seq: int,
         tile_groups_per_partition: int = 1, max_partitions: int = 0, kv_dtype: int = KV_BF16,
         softmax_scale: float = 0.0, head_dim: int = HEAD_DIM, wait_timeout_ns: int = 0,
         kernel_variant: int = 0) -> Plan:
    p = Plan(num_seqs, num_kv_heads, query_group_size, head_dim, kv_block_size, max_blocks_per_seq,
             tile_groups_per_partition, max_partitions, kv_dtype, softmax_scale, wait_timeout_ns, kernel_variant)
    rc = lib().pda_plan(ctypes.byref(p))
    if rc != 0:
        raise PdaError(rc, "pda_plan")
    return p


def kernel_variant(p: Plan) -> int:
    """pda_kernel_variant: the partition-pass layout pda_decode launches for this plan on the
    current device (VARIANT_HEAD_WARPS, VARIANT_HEAD_GROUPS or VARIANT_ROW_HALVES)."""
    rc = lib().pda_kernel_variant(ctypes.byref(p))
    if rc < 0:
        raise PdaError(rc, "pda_kernel_variant")
    return rc


def partial_shapes(p: Plan):
    B, Hk, P, QG = p.num_seqs, p.num_kv_heads, p.num_partitions, p.query_group_size
    return (B, Hk, P, QG, p.head_dim), (B, Hk, P, QG)


def workspace(p: Plan, device, fill: float | None = None) -> dict:
    """partial_out / exp_sums / max_logits for one step (allocated by torch)."""
    so, ss = partial_shapes(p)
    mk = (lambda s: torch.empty(s, dtype=torch.float32, device=device)) if fill is None else \
        (lambda s: torch.full(s, fill, dtype=torch.float32, device=device))
    return {"partial_out": mk(so), "exp_sums": mk(ss), "max_logits": mk(ss)}


def _need(t: torch.Tensor, name: str, dtype, numel: int, host_ok: bool = False):
    """Pointer of a contiguous tensor of at least `numel` bytes.  With host_ok, pinned host memory
    is accepted too: the kernels then read or write it across the host link (unified addressing
    gives pinned memory one address on both sides)."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (host_ok and t.device.type == "cpu" and t.is_pinned())):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() * t.element_size() < numel:
        raise ValueError(f"{name} is too small ({t.numel() * t.element_size()} < {numel} bytes)")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream if isinstance(s, torch.cuda.Stream) else int(s))


def decode(p: Plan, query, kv_cache, num_cache_blocks: int, block_table, context_lens, partial_out, exp_sums,
           max_logits, err_word=None, stream=None) -> None:
    """pda_decode: the partition pass (see include/pda.h)."""
    B, Hk, QG, D, P = p.num_seqs, p.num_kv_heads, p.query_group_size, p.head_dim, p.num_partitions
    args = (
        _need(query, "query", (torch.bfloat16, torch.int16, torch.uint16), B * Hk * QG * D * 2, host_ok=True),
        _need(kv_cache, "kv_cache", None, num_cache_blocks * p.cache_block_bytes),
        ctypes.c_longlong(num_cache_blocks),
        _need(block_table, "block_table", torch.int32, B * p.max_blocks_per_seq * 4, host_ok=True),
        _need(context_lens, "context_lens", torch.int32, B * 4, host_ok=True),
        _need(partial_out, "partial_out", torch.float32, B * Hk * P * QG * D * 4),
        _need(exp_sums, "exp_sums", torch.float32, B * Hk * P * QG * 4),
        _need(max_logits, "max_logits", torch.float32, B * Hk * P * QG * 4),
        None if err_word is None else _need(err_word, "err_word", torch.int32, 4),
        _stream(stream),
    )
    rc = lib().pda_decode(ctypes.byref(p), *args)
    if rc != 0:
        raise PdaError(rc, "pda_decode")


def decode_tq4(p: Plan, query, kv_cache, num_cache_blocks: int, centroids, block_table, context_lens, partial_out,
               exp_sums, max_logits, err_word=None, stream=None) -> None:
    """pda_decode_tq4: the partition pass over a TQ4 cache (see include/pda.h); centroids: fp32 [16]."""
    B, Hk, QG, D, P = p.num_seqs, p.num_kv_heads, p.query_group_size, p.head_dim, p.num_partitions
    args = (
        _need(query, "query", (torch.bfloat16, torch.int16, torch.uint16), B * Hk * QG * D * 2, host_ok=True),
        _need(kv_cache, "kv_cache", None, num_cache_blocks * p.cache_block_bytes),
        ctypes.c_longlong(num_cache_blocks),
        _need(centroids, "centroids", torch.float32, 16 * 4),
        _need(block_table, "block_table", torch.int32, B * p.max_blocks_per_seq * 4, host_ok=True),
        _need(context_lens, "context_lens", torch.int32, B * 4, host_ok=True),
        _need(partial_out, "partial_out", torch.float32, B * Hk * P * QG * D * 4),
        _need(exp_sums, "exp_sums", torch.float32, B * Hk * P * QG * 4),
        _need(max_logits, "max_logits", torch.float32, B * Hk * P * QG * 4),
        None if err_word is None else _need(err_word, "err_word", torch.int32, 4),
        _stream(stream),
    )
    rc = lib().pda_decode_tq4(ctypes.byref(p), *args)
    if rc != 0:
        raise PdaError(rc, "pda_decode_tq4")


def reduce(p: Plan, context_lens, partial_out, exp_sums, max_logits, out, err_word=None, stream=None) -> None:
    """pda_reduce: combines the partials into out [B][Hk*QG][D] (bf16 or fp32 by out's dtype)."""
    B, Hk, QG, D, P = p.num_seqs, p.num_kv_heads, p.query_group_size, p.head_dim, p.num_partitions
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    args = (
        _need(context_lens, "context_lens", torch.int32, B * 4, host_ok=True),
        _need(partial_out, "partial_out", torch.float32, B * Hk * P * QG * D * 4),
        _need(exp_sums, "exp_sums", torch.float32, B * Hk * P * QG * 4),
        _need(max_logits, "max_logits", torch.float32, B * Hk * P * QG * 4),
        _need(out, "out", (torch.float32, torch.bfloat16), B * Hk * QG * D * out.element_size(), host_ok=True),
        ctypes.c_int(out_dtype),
        None if err_word is None else _need(err_word, "err_word", torch.int32, 4),
        _stream(stream),
    )
    rc = lib().pda_reduce(ctypes.byref(p), *args)
    if rc != 0:
        raise PdaError(rc, "pda_reduce")


def append_kv(p: Plan, k_new, v_new, kv_cache, num_cache_blocks: int, block_table, positions, err_word=None,
              stream=None) -> None:
    """pda_append_kv: writes one new token per sequence into the paged cache (see include/pda.h).
    k_new, v_new: bf16 [B][Hk][D]; positions: int32 [B] (negative: no write)."""
    B, Hk, D = p.num_seqs, p.num_kv_heads, p.head_dim
    args = (
        _need(k_new, "k_new", (torch.bfloat16, torch.int16, torch.uint16), B * Hk * D * 2),
        _need(v_new, "v_new", (torch.bfloat16, torch.int16, torch.uint16), B * Hk * D * 2),
        _need(kv_cache, "kv_cache", None, num_cache_blocks * p.cache_block_bytes),
        ctypes.c_longlong(num_cache_blocks),
        _need(block_table, "block_table", torch.int32, B * p.max_blocks_per_seq * 4),
        _need(positions, "positions", torch.int32, B * 4),
        None if err_word is None else _need(err_word, "err_word", torch.int32, 4),
        _stream(stream),
    )
    rc = lib().pda_append_kv(ctypes.byref(p), *args)
    if rc != 0:
        raise PdaError(rc, "pda_append_kv")


def counters(p: Plan, device):
    """The fused step's reserved counters argument, int32 [B][Hk], zeroed (the step leaves them zero)."""
    return torch.zeros((p.num_seqs, p.num_kv_heads), dtype=torch.int32, device=device)


def decode_fused(p: Plan, query, kv_cache, num_cache_blocks: int, block_table, context_lens, partial_out, exp_sums,
                 max_logits, counters, out, err_word=None, stream=None) -> None:
    """pda_decode_fused: the partition pass and the reduce in one launch (see include/pda.h)."""
    B, Hk, QG, D, P = p.num_seqs, p.num_kv_heads, p.query_group_size, p.head_dim, p.num_partitions
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    args = (
        _need(query, "query", (torch.bfloat16, torch.int16, torch.uint16), B * Hk * QG * D * 2, host_ok=True),
        _need(kv_cache, "kv_cache", None, num_cache_blocks * p.cache_block_bytes),
        ctypes.c_longlong(num_cache_blocks),
        _need(block_table, "block_table", torch.int32, B * p.max_blocks_per_seq * 4, host_ok=True),
        _need(context_lens, "context_lens", torch.int32, B * 4, host_ok=True),
        _need(partial_out, "partial_out", torch.float32, B * Hk * P * QG * D * 4),
        _need(exp_sums, "exp_sums", torch.float32, B * Hk * P * QG * 4),
        _need(max_logits, "max_logits", torch.float32, B * Hk * P * QG * 4),
        _need(counters, "counters", torch.int32, B * Hk * 4),
        _need(out, "out", (torch.float32, torch.bfloat16), B * Hk * QG * D * out.element_size(), host_ok=True),
        ctypes.c_int(out_dtype),
        None if err_word is None else _need(err_word, "err_word", torch.int32, 4),
        _stream(stream),
    )
    rc = lib().pda_decode_fused(ctypes.byref(p), *args)
    if rc != 0:
        raise PdaError(rc, "pda_decode_fused")


def decode_step(p: Plan, query, kv_cache, num_cache_blocks: int, block_table, context_lens, ws: dict | None = None,
                out=None, out_dtype=torch.bfloat16, err_word=None, stream=None, centroids=None):
    """pda_decode (pda_decode_tq4 for a TQ4 plan, with its centroids) then pda_reduce on one stream;
    returns out [B][Hk*QG][D]."""
    if ws is None:
        ws = workspace(p, query.device)
    if out is None:
        out = torch.empty((p.num_seqs, p.num_kv_heads * p.query_group_size, p.head_dim), dtype=out_dtype,
                          device=query.device)
    if p.kv_dtype == KV_TQ4:
        decode_tq4(p, query, kv_cache, num_cache_blocks, centroids, block_table, context_lens, ws["partial_out"],
                   ws["exp_sums"], ws["max_logits"], err_word=err_word, stream=stream)
    else:
        decode(p, query, kv_cache, num_cache_blocks, block_table, context_lens, ws["partial_out"], ws["exp_sums"],
               ws["max_logits"], err_word=err_word, stream=stream)
    reduce(p, context_lens, ws["partial_out"], ws["exp_sums"], ws["max_logits"], out, err_word=err_word,
           stream=stream)
    return out


NOALLOC_SCRATCH_BYTES = 64 << 20


def decode_step_noalloc(p: Plan, query, kv_cache, num_cache_blocks: int, block_table, context_lens, out,
                        err_word=None, stream=None) -> None:
    """pda_decode_step_noalloc: a whole step with the partials kept inside the library, for callers
    that cannot allocate a workspace (see include/pda.h).  out [B][Hk*QG][D], bf16 or fp32."""
    B, Hk, QG, D = p.num_seqs, p.num_kv_heads, p.query_group_size, p.head_dim
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    args = (
        _need(query, "query", (torch.bfloat16, torch.int16, torch.uint16), B * Hk * QG * D * 2, host_ok=True),
        _need(kv_cache, "kv_cache", None, num_cache_blocks * p.cache_block_bytes),
        ctypes.c_longlong(num_cache_blocks),
        _need(block_table, "block_table", torch.int32, B * p.max_blocks_per_seq * 4, host_ok=True),
        _need(context_lens, "context_lens", torch.int32, B * 4, host_ok=True),
        _need(out, "out", (torch.float32, torch.bfloat16), B * Hk * QG * D * out.element_size(), host_ok=True),
        ctypes.c_int(out_dtype),
        None if err_word is None else _need(err_word, "err_word", torch.int32, 4),
        _stream(stream),
    )
    rc = lib().pda_decode_step_noalloc(ctypes.byref(p), *args)
    if rc != 0:
        raise PdaError(rc, "pda_decode_step_noalloc")
