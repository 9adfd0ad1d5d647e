"""The allocation-free decode step, for callers that cannot allocate device memory while they run
(an engine that owns all device memory, or code that must not let cudaMalloc synchronise the
device).  It keeps the partials in a fixed array inside the library; this checks, through the C
ABI, that two calls in a row give what the workspace-based entry points give and what the fp64
oracle gives, that a smaller plan after a larger one reads none of the larger one's leftovers,
that pinned host buffers work as for the other entry points, and that a plan whose partials do
not fit the array is turned away.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh
from tests.gpu_helpers import bf16_half_ulp, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pda():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_block_gb300 as pda
    return pda


def plan_of(pda, w):
    return pda.plan(w.num_seqs, w.num_kv_heads, w.query_group_size, w.kv_block_size, w.max_blocks_per_seq,
                    w.tile_groups_per_partition, w.max_partitions, w.kv_dtype)


def tol_of(w):
    return 2e-3 if w.kv_dtype == wl.KV_BF16 else 1e-2


@pytest.mark.parametrize("name,kwargs", [
    ("b8_hk8_qg8_bs16_ctx1-4096", {}),
    # fp8 with 64-partition rows: 16 sequences x 8 heads x 64 partitions x 6 rows x 520 bytes = 26 MB
    ("mid_fp8", dict(num_seqs=16, num_kv_heads=8, query_group_size=6, kv_block_size=16,
                     ctx=(16384, 1, 900, 4000, 255, 256, 257, 12000, 3000, 7, 16000, 2048, 100, 5000, 640, 9000),
                     kv_dtype=wl.KV_FP8_E4M3, seed=95)),
    ("small_fp8", dict(num_seqs=3, num_kv_heads=2, query_group_size=6, kv_block_size=16, ctx=(300, 1, 1100),
                       kv_dtype=wl.KV_FP8_E4M3, seed=91)),
])
def test_two_calls_match_the_workspace_entry_points_and_the_oracle(oracle_mod, pda, name, kwargs):
    w = wl.WORKLOADS[name] if not kwargs else wl.small(name=name, **kwargs)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_of(pda, w)
    shape = (w.num_seqs, w.num_q_heads, 128)
    ref = torch.empty(shape, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pda.decode_step(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"], out=ref,
                    err_word=err)
    oracle_out = oh.run_oracle(inp)["out"]
    tol = tol_of(w)
    for _ in range(2):
        got = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        pda.decode_step_noalloc(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                                got, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        g = got.cpu().numpy().astype(np.float64)
        diff = float(np.abs(g - ref.cpu().numpy()).max())
        assert np.isfinite(diff) and diff <= tol, diff
        assert np.abs(g - oracle_out).max() <= tol
    got16 = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    pda.decode_step_noalloc(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"], got16)
    torch.cuda.synchronize()
    g16 = got16.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(g16 - oracle_out) <= tol + bf16_half_ulp(oracle_out))


def test_smaller_plan_after_a_larger_one(oracle_mod, pda):
    # the array keeps the last call's partials; a later, smaller step must read only its own
    big = wl.small(name="big", num_seqs=6, num_kv_heads=4, query_group_size=16, kv_block_size=16,
                   ctx=(4000, 3000, 2000, 4096, 100, 3500), seed=92)
    small = wl.small(name="small", num_seqs=2, num_kv_heads=2, query_group_size=8, kv_block_size=32, ctx=(700, 33),
                     seed=93)
    for w in (big, small, big):
        inp = wl.generate(w)
        d = to_device(inp)
        p = plan_of(pda, w)
        got = torch.full((w.num_seqs, w.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pda.decode_step_noalloc(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                                got, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert np.abs(got.cpu().numpy() - oh.run_oracle(inp)["out"]).max() <= tol_of(w), w.name


def test_pinned_host_inputs_and_output(oracle_mod, pda):
    w = wl.small(num_seqs=3, num_kv_heads=2, query_group_size=8, kv_block_size=16, ctx=(500, 20, 257),
                 kv_dtype=wl.KV_FP8_E4M3, seed=94)
    inp = wl.generate(w)
    p = plan_of(pda, w)
    cache = torch.from_numpy(inp.cache).cuda()
    q = torch.from_numpy(inp.query.view(np.int16)).view(torch.bfloat16).pin_memory()
    bt = torch.from_numpy(inp.block_table).pin_memory()
    ctx = torch.from_numpy(inp.context_lens).pin_memory()
    out = torch.full((w.num_seqs, w.num_q_heads, 128), float("nan"), dtype=torch.float32).pin_memory()
    pda.decode_step_noalloc(p, q, cache, w.num_cache_blocks, bt, ctx, out)
    torch.cuda.synchronize()
    assert np.abs(out.numpy() - oh.run_oracle(inp)["out"]).max() <= tol_of(w)


def test_plan_larger_than_the_array_is_refused(pda):
    # 64 sequences x 8 heads x 64 partitions x 16 rows x 520 bytes = 272 MB of partials > 64 MiB
    p = pda.plan(64, 8, 16, 16, 1024)
    assert p.workspace_bytes > pda.NOALLOC_SCRATCH_BYTES
    L = pda.lib()
    dummy = ctypes.c_void_p(1 << 20)
    rc = L.pda_decode_step_noalloc(ctypes.byref(p), dummy, dummy, ctypes.c_longlong(1), dummy, dummy, dummy,
                                   ctypes.c_int(0), None, None)
    assert rc == -3 and pda.status_string(rc) == "PDA_ERR_WORKSPACE_TOO_SMALL"
