"""The allocation-free decode step, for callers that cannot allocate device memory while they run
(an engine that owns all device memory, or code that must not let cudaMalloc synchronise the
device).  It keeps the partials in a fixed array inside the library; this checks, through the C
ABI, that two calls in a row give what the workspace-based entry points give, and that a plan
whose partials do not fit the array is turned away.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_gqa_block_gb300 import workloads as wl
from tests.gpu_helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pda():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_block_gb300 as pda
    return pda


@pytest.mark.parametrize("name,kwargs", [
    ("b8_hk8_qg8_bs16_ctx1-4096", {}),
    ("small_fp8", dict(num_seqs=3, num_kv_heads=2, query_group_size=6, kv_block_size=16, ctx=(300, 1, 1100),
                       kv_dtype=wl.KV_FP8_E4M3, seed=91)),
])
def test_two_calls_match_the_workspace_entry_points(pda, name, kwargs):
    w = wl.WORKLOADS[name] if not kwargs else wl.small(name=name, **kwargs)
    inp = wl.generate(w)
    d = to_device(inp)
    p = pda.plan(w.num_seqs, w.num_kv_heads, w.query_group_size, w.kv_block_size, w.max_blocks_per_seq,
                 w.tile_groups_per_partition, w.max_partitions, w.kv_dtype)
    shape = (w.num_seqs, w.num_q_heads, 128)
    ref = torch.empty(shape, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pda.decode_step(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"], out=ref,
                    err_word=err)
    tol = 2e-3 if w.kv_dtype == wl.KV_BF16 else 1e-2
    for _ in range(2):
        got = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        pda.decode_step_noalloc(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                                got, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        diff = (got - ref).abs().max().item()
        assert np.isfinite(diff) and diff <= tol, diff
    got16 = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    pda.decode_step_noalloc(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"], got16)
    torch.cuda.synchronize()
    assert (got16.float() - ref).abs().max().item() <= tol + 2.0 ** -7 * ref.abs().max().item()


def test_plan_larger_than_the_array_is_refused(pda):
    # 64 sequences x 8 heads x 64 partitions x 16 rows x 520 bytes = 272 MB of partials > 64 MiB
    p = pda.plan(64, 8, 16, 16, 1024)
    assert p.workspace_bytes > pda.NOALLOC_SCRATCH_BYTES
    L = pda.lib()
    dummy = ctypes.c_void_p(1 << 20)
    rc = L.pda_decode_step_noalloc(ctypes.byref(p), dummy, dummy, ctypes.c_longlong(1), dummy, dummy, dummy,
                                   ctypes.c_int(0), None, None)
    assert rc == -3 and pda.status_string(rc) == "PDA_ERR_WORKSPACE_TOO_SMALL"
