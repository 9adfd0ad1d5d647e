"""The C-ABI library on the host (no GPU): it loads, exports every symbol the header declares,
its plan arithmetic agrees with the oracle's, and argument errors come back as statuses."""
import ctypes
import os
import re

import pytest

import oracle
from paged_kv_gqa_block_gb300 import _build
from paged_kv_gqa_block_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pda():
    _build.build()
    import paged_kv_gqa_block_gb300 as pda
    pda.lib()
    return pda


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            names |= set(re.findall(r"^PDA_API\s+[\w\s\*]+?\b(pda_\w+)\s*\(", open(os.path.join(inc, f)).read(), re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    assert {"pda_plan", "pda_decode", "pda_reduce", "pda_status_string", "pda_workspace_size"} <= set(declared_symbols())


def test_library_exports_every_declared_symbol(pda):
    L = pda.lib()
    for name in declared_symbols():
        assert hasattr(L, name), name
    assert L.pda_plan_struct_size() == ctypes.sizeof(pda.Plan)


def test_status_strings(pda):
    for code, name in pda.STATUS.items():
        assert pda.status_string(code) == name
    assert pda.status_string(12345) == "PDA_ERR_UNKNOWN"


@pytest.mark.parametrize("name", wl.WORKLOAD_ORDER)
def test_plan_agrees_with_oracle(pda, name):
    w = wl.WORKLOADS[name]
    p = pda.plan(w.num_seqs, w.num_kv_heads, w.query_group_size, w.kv_block_size, w.max_blocks_per_seq,
                 w.tile_groups_per_partition, w.max_partitions, w.kv_dtype)
    o = oracle.plan(w.max_blocks_per_seq, w.kv_block_size, w.tile_groups_per_partition, w.max_partitions)
    lay = oracle.cache_layout(w.num_kv_heads, w.kv_block_size, 128, w.kv_dtype)
    assert (p.resolved_tile_groups, p.num_partitions, p.partition_tokens) == (o["G"], o["P"], o["W"])
    assert p.cache_block_bytes == lay["cache_block_bytes"] == w.cache_block_bytes
    assert p.meta_offset_bytes == lay["meta_offset_bytes"]
    assert p.workspace_bytes == w.num_seqs * w.num_kv_heads * o["P"] * w.query_group_size * (128 * 4 + 8)
    assert abs(p.resolved_softmax_scale - 128 ** -0.5) < 1e-8
    assert pda.lib().pda_workspace_size(ctypes.byref(p)) == p.workspace_bytes


def test_plan_worked_example(pda):
    p = pda.plan(4, 8, 8, 32, 1280, tile_groups_per_partition=0, max_partitions=32)
    assert (p.resolved_tile_groups, p.num_partitions, p.partition_tokens) == (5, 32, 1280)
    assert p.num_partitions * p.partition_tokens == 40960


@pytest.mark.parametrize("kw,code", [
    (dict(query_group_size=7), -2), (dict(query_group_size=4), -2), (dict(kv_block_size=8), -2),
    (dict(kv_block_size=64), -2), (dict(head_dim=64), -2), (dict(kv_dtype=3), -2), (dict(kv_dtype=-1), -2),
    (dict(num_kv_heads=0), -1), (dict(max_blocks_per_seq=0), -1), (dict(tile_groups_per_partition=-1), -1),
    (dict(num_seqs=-1), -1), (dict(max_partitions=-2), -1), (dict(softmax_scale=float("nan")), -1),
    (dict(wait_timeout_ns=-1), -1), (dict(kernel_variant=-1), -1), (dict(kernel_variant=4), -1),
    (dict(kernel_variant=2), -2), (dict(kernel_variant=2, kv_dtype=2), -2),
    (dict(kernel_variant=3), -2), (dict(kernel_variant=3, query_group_size=16, kv_dtype=1), -2),
    (dict(kernel_variant=3, query_group_size=16, kv_dtype=2), -2),
])
def test_plan_rejects(pda, kw, code):
    args = dict(num_seqs=2, num_kv_heads=2, query_group_size=8, kv_block_size=16, max_blocks_per_seq=4)
    args.update(kw)
    with pytest.raises(pda.PdaError) as e:
        pda.plan(**args)
    assert e.value.status == code


def test_launch_argument_errors_without_a_gpu(pda):
    L = pda.lib()
    p = pda.plan(2, 2, 8, 16, 4)
    good = ctypes.c_void_p(1 << 20)
    args = [good, good, ctypes.c_longlong(8), good, good, good, good, good, None, None]
    assert L.pda_decode(None, *args) == -1
    edited = pda.Plan.from_buffer_copy(p)
    edited.num_partitions += 1
    assert L.pda_decode(ctypes.byref(edited), *args) == -1
    bad = list(args)
    bad[0] = None
    assert L.pda_decode(ctypes.byref(p), *bad) == -1             # null query
    bad = list(args)
    bad[1] = ctypes.c_void_p((1 << 20) + 4)
    assert L.pda_decode(ctypes.byref(p), *bad) == -1             # kv cache not 16-byte aligned
    bad = list(args)
    bad[2] = ctypes.c_longlong(0)
    assert L.pda_decode(ctypes.byref(p), *bad) == -1             # empty pool
    assert L.pda_reduce(ctypes.byref(p), good, good, good, good, good, 7, None, None) == -1   # bad out dtype
    assert L.pda_reduce(ctypes.byref(p), good, None, good, good, good, 0, None, None) == -1
    empty = pda.plan(0, 2, 8, 16, 4)                            # nothing to do: no launch, no CUDA call
    assert L.pda_decode(ctypes.byref(empty), *args) == 0
    assert L.pda_reduce(ctypes.byref(empty), good, good, good, good, good, 0, None, None) == 0
    assert L.pda_workspace_size(None) == -1


def test_tq4_entry_point_rules_without_a_gpu(pda):
    """A TQ4 cache is read only through pda_decode_tq4, with its centroids; the other entry points
    turn a TQ4 plan away before launching anything."""
    L = pda.lib()
    tq = pda.plan(2, 2, 8, 16, 4, kv_dtype=pda.KV_TQ4)
    assert tq.cache_block_bytes == 16 * 2 * 128 + 2 * 3 * 16 * 2 and tq.meta_offset_bytes == 16 * 2 * 128
    bf = pda.plan(2, 2, 8, 16, 4)
    good = ctypes.c_void_p(1 << 20)
    dec = [good, good, ctypes.c_longlong(8), good, good, good, good, good, None, None]
    assert L.pda_decode(ctypes.byref(tq), *dec) == -1                           # needs the centroids
    tq4 = [good, good, ctypes.c_longlong(8), good, good, good, good, good, good, None, None]
    assert L.pda_decode_tq4(ctypes.byref(bf), *tq4) == -1                       # not a TQ4 plan
    no_cent = list(tq4)
    no_cent[3] = None
    assert L.pda_decode_tq4(ctypes.byref(tq), *no_cent) == -1
    odd = list(tq4)
    odd[3] = ctypes.c_void_p((1 << 20) + 2)
    assert L.pda_decode_tq4(ctypes.byref(tq), *odd) == -1                       # centroids not 4-byte aligned
    fused = [good, good, ctypes.c_longlong(8), good, good, good, good, good, good, good, ctypes.c_int(0), None, None]
    assert L.pda_decode_fused(ctypes.byref(tq), *fused) == -1
    assert L.pda_decode_step_noalloc(ctypes.byref(tq), good, good, ctypes.c_longlong(8), good, good, good,
                                     ctypes.c_int(0), None, None) == -1
    assert L.pda_append_kv(ctypes.byref(tq), good, good, good, ctypes.c_longlong(8), good, good, None, None) == -2
    empty = pda.plan(0, 2, 8, 16, 4, kv_dtype=pda.KV_TQ4)
    assert L.pda_decode_tq4(ctypes.byref(empty), *tq4) == 0


def test_head_group_variant_is_accepted_for_fp8(pda):
    for v in (0, 1, 2):
        p = pda.plan(2, 8, 6, 16, 4, kv_dtype=pda.KV_FP8_E4M3, kernel_variant=v)
        assert p.kernel_variant == v


def test_row_half_variant_is_accepted_for_bf16_with_sixteen_rows(pda):
    for v, want in ((1, pda.VARIANT_HEAD_WARPS), (3, pda.VARIANT_ROW_HALVES)):
        p = pda.plan(2, 4, 16, 32, 4, kv_dtype=pda.KV_BF16, kernel_variant=v)
        assert p.kernel_variant == v
        assert pda.kernel_variant(p) == want


def test_kernel_variant_of_a_plan(pda):
    L = pda.lib()
    assert L.pda_kernel_variant(None) == -1
    p = pda.plan(2, 8, 6, 16, 4, kv_dtype=pda.KV_BF16)
    assert pda.kernel_variant(p) == pda.VARIANT_HEAD_WARPS            # head groups are fp8 only
    for v, want in ((1, pda.VARIANT_HEAD_WARPS), (2, pda.VARIANT_HEAD_GROUPS)):
        p = pda.plan(2, 8, 6, 16, 4, kv_dtype=pda.KV_FP8_E4M3, kernel_variant=v)
        assert pda.kernel_variant(p) == want
    edited = pda.Plan.from_buffer_copy(p)
    edited.num_partitions += 1
    assert L.pda_kernel_variant(ctypes.byref(edited)) == -1
