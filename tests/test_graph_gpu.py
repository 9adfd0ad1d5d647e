"""The decode step (partition pass + reduce, both launched with programmatic dependent launch)
captured in a CUDA graph: replays equal direct launches, and context lengths changed in device
memory between replays are honoured (the grid depends only on the plan)."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh
from tests.gpu_helpers import KV_VARIANTS, plan_for, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pda():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_block_gb300 as pda
    return pda


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_captured_step_replays_and_follows_context_lengths(oracle_mod, pda, kv, variant):
    ctx = (700, 33, 256, 1500)
    w = wl.small(num_seqs=4, num_kv_heads=4, ctx=ctx, kv_dtype=kv, seed=80, max_blocks_per_seq=100)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w, variant=variant)
    ws = pda.workspace(p, "cuda")
    out = torch.empty((w.num_seqs, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    cent = d.get("centroids")
    with torch.cuda.stream(s):     # one direct call first: per-device set-up happens outside capture
        pda.decode_step(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"], ws=ws,
                        out=out, centroids=cent)
    torch.cuda.synchronize()
    direct = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pda.decode_step(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"], ws=ws,
                        out=out, centroids=cent)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, direct)
    # shorter contexts, written in place: the replay reads them from device memory
    new_ctx = np.array([300, 1, 0, 1499], np.int32)
    d["context_lens"].copy_(torch.from_numpy(new_ctx))
    g.replay()
    torch.cuda.synchronize()
    ref = oh.run_oracle(wl.Inputs(w, inp.query, inp.cache, inp.block_table, new_ctx, inp.extra))["out"]
    tol = 2e-3 if kv == wl.KV_BF16 else 1e-2
    assert np.abs(out.cpu().numpy() - ref).max() <= tol
