"""The fused step (partition pass and reduce in one launch) against the oracle and against the
two-launch path, through the C ABI."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh
from tests.gpu_helpers import bf16_half_ulp, plan_for, to_device

pytestmark = pytest.mark.gpu

TOL = {wl.KV_BF16: 2e-3, wl.KV_FP8_E4M3: 1e-2}


@pytest.fixture(scope="module")
def pda():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_block_gb300 as pda
    return pda


def run_both(pda, inp, G=None, repeats=2, variant=0):
    w = inp.workload
    p = plan_for(w, G, variant)
    d = to_device(inp)
    shape = (w.num_seqs, w.num_q_heads, 128)
    two = torch.empty(shape, dtype=torch.float32, device="cuda")
    pda.decode_step(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"], out=two)
    ws = pda.workspace(p, "cuda")
    cnt = pda.counters(p, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(repeats):
        for dt in (torch.float32, torch.bfloat16):
            o = torch.full(shape, float("nan"), dtype=dt, device="cuda")
            pda.decode_fused(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                             ws["partial_out"], ws["exp_sums"], ws["max_logits"], cnt, o, err_word=err)
            outs.append(o)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert int(cnt.abs().sum().item()) == 0, "counters must be left at zero"
    return two.cpu().numpy().astype(np.float64), [o.float().cpu().numpy().astype(np.float64) for o in outs]


CASES = [
    (wl.KV_BF16, 8, 16, 1, 2, (1, 15, 256, 257, 700, 4000)),
    (wl.KV_BF16, 16, 32, 2, 2, (33, 600, 2049)),
    (wl.KV_BF16, 6, 32, 5, 3, (1281, 40, 3000)),
    (wl.KV_FP8_E4M3, 6, 16, 1, 2, (1, 300, 1100, 5000)),
    (wl.KV_FP8_E4M3, 16, 16, 1, 2, (16, 900)),
    # empty sequences among others (their rows are zeroed, as the reduce does), and 79 partitions
    # in one sequence (the in-kernel merge's path for more than 64)
    (wl.KV_BF16, 8, 32, 1, 2, (20000, 0, 300, 0)),
    (wl.KV_FP8_E4M3, 6, 32, 1, 1, (0, 18000, 5)),
    (wl.KV_BF16, 8, 16, 1, 2, (0, 0, 0)),
]


CASES += [
    # the fused head-group step: groups of 4 (one and two per sequence), 2 and 3 heads, 79 partitions
    (wl.KV_FP8_E4M3, 6, 16, 1, 8, (1, 17, 300, 2048, 5000, 0, 4097)),
    (wl.KV_FP8_E4M3, 8, 32, 1, 4, (20000, 1, 0, 255)),
    (wl.KV_FP8_E4M3, 16, 16, 2, 2, (513, 2000, 1)),
    (wl.KV_FP8_E4M3, 6, 32, 5, 6, (1281, 40, 3000, 0)),
]
FUSED_CASES = [(*c, v) for c in CASES for v in ((1, 2) if c[0] == wl.KV_FP8_E4M3 else (0,))]


@pytest.mark.parametrize("kv,QG,BS,G,Hk,ctx,variant", FUSED_CASES)
def test_fused_matches_oracle_and_the_two_launch_path(oracle_mod, pda, kv, QG, BS, G, Hk, ctx, variant):
    w = wl.small(num_seqs=len(ctx), num_kv_heads=Hk, query_group_size=QG, kv_block_size=BS, ctx=ctx, kv_dtype=kv,
                 tile_groups_per_partition=G, seed=200 + QG + BS + G, extra_blocks=5)
    inp = wl.generate(w)
    two, fused = run_both(pda, inp, variant=variant)
    ref = oh.run_oracle(inp, G=G)["out"]
    tol = TOL[kv]
    for k, o in enumerate(fused):
        if k % 2 == 0:   # fp32 outputs: same combination, same order as the two-launch path
            assert np.array_equal(o, two), "fused and two-launch results differ"
            assert np.abs(o - ref).max() <= tol
        else:            # bf16 outputs
            assert np.all(np.abs(o - ref) <= tol + bf16_half_ulp(ref))


@pytest.mark.parametrize("kv,variant", [(wl.KV_BF16, 0), (wl.KV_FP8_E4M3, 1), (wl.KV_FP8_E4M3, 2)])
def test_fused_bad_context_length_sets_the_bit_and_zeroes_that_sequence(oracle_mod, pda, kv, variant):
    w = wl.small(num_seqs=3, num_kv_heads=4, ctx=(300, 20, 33), kv_dtype=kv, seed=38)
    inp = wl.generate(w)
    ref = oh.run_oracle(inp)["out"]
    ctx = inp.context_lens.copy()
    ctx[1] = -5
    d = to_device(wl.Inputs(w, inp.query, inp.cache, inp.block_table, ctx))
    p = plan_for(w, variant=variant)
    ws = pda.workspace(p, "cuda")
    cnt = pda.counters(p, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full((w.num_seqs, w.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    pda.decode_fused(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                     ws["partial_out"], ws["exp_sums"], ws["max_logits"], cnt, o, err_word=err)
    torch.cuda.synchronize()
    out = o.cpu().numpy().astype(np.float64)
    assert int(err.item()) & 1
    assert np.all(out[1] == 0)
    for b in (0, 2):
        assert np.abs(out[b] - ref[b]).max() <= TOL[kv]
    assert int(cnt.abs().sum().item()) == 0


@pytest.mark.parametrize("name,variant", [("b8_hk8_qg8_bs16_ctx1-4096", 0), ("b64_hk8_qg6_bs16_fp8_lognormal2048", 1),
                                          ("b64_hk8_qg6_bs16_fp8_lognormal2048", 2)])
def test_fused_full_size_equals_two_launch(pda, name, variant):
    inp = wl.generate(wl.WORKLOADS[name])
    two, fused = run_both(pda, inp, repeats=2, variant=variant)
    for o in fused[::2]:
        assert np.array_equal(o, two)


@pytest.mark.parametrize("kv,variant", [(wl.KV_BF16, 0), (wl.KV_FP8_E4M3, 1), (wl.KV_FP8_E4M3, 2)])
def test_fused_counters_return_to_zero_across_many_launches(oracle_mod, pda, kv, variant):
    # the fused step takes a counter slot per launch (256 of them: the head-group scheduler's, or
    # the head-warp step's grid barrier) and leaves its slot and the caller's counters at zero:
    # 600 launches in a row give the first launch's bits (a slot left non-zero would let a later
    # launch merge before its partials exist)
    w = wl.small(num_seqs=5, num_kv_heads=8, query_group_size=6, kv_block_size=16, ctx=(3000, 17, 0, 1200, 256),
                 kv_dtype=kv, seed=97)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w, variant=variant)
    ws = pda.workspace(p, "cuda")
    cnt = pda.counters(p, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = (w.num_seqs, w.num_q_heads, 128)
    first = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    last = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    for i in range(600):
        o = first if i == 0 else last
        pda.decode_fused(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                         ws["partial_out"], ws["exp_sums"], ws["max_logits"], cnt, o, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(cnt.abs().sum().item()) == 0
    assert torch.equal(first, last)
    assert np.abs(first.cpu().numpy() - oh.run_oracle(inp)["out"]).max() <= TOL[kv]


@pytest.mark.parametrize("kv,variant", [(wl.KV_BF16, 0), (wl.KV_FP8_E4M3, 1), (wl.KV_FP8_E4M3, 2)])
def test_fused_step_replays_in_a_cuda_graph(oracle_mod, pda, kv, variant):
    # a captured fused step keeps the counter slot it took at capture: every replay finds it zero
    # again (the launch's last CTA resets it) and reads the context lengths as they are then
    w = wl.small(num_seqs=4, num_kv_heads=4, ctx=(700, 33, 256, 1500), kv_dtype=kv, seed=81, max_blocks_per_seq=100)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w, variant=variant)
    ws = pda.workspace(p, "cuda")
    cnt = pda.counters(p, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((w.num_seqs, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def step():
        pda.decode_fused(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                         ws["partial_out"], ws["exp_sums"], ws["max_logits"], cnt, out, err_word=err)
    with torch.cuda.stream(s):     # one direct call first: per-device set-up happens outside capture
        step()
    torch.cuda.synchronize()
    direct = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, direct)
    new_ctx = np.array([300, 1, 0, 1499], np.int32)
    d["context_lens"].copy_(torch.from_numpy(new_ctx))
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(cnt.abs().sum().item()) == 0
    ref = oh.run_oracle(wl.Inputs(w, inp.query, inp.cache, inp.block_table, new_ctx, inp.extra))["out"]
    assert np.abs(out.cpu().numpy() - ref).max() <= TOL[kv]


@pytest.mark.parametrize("kv,variant", [(wl.KV_BF16, 0), (wl.KV_FP8_E4M3, 1), (wl.KV_FP8_E4M3, 2)])
def test_fused_repeat_runs_are_bitwise_identical(pda, kv, variant):
    # the fused step's merges run in whichever warp takes them, but always in partition order
    w = wl.small(num_seqs=4, num_kv_heads=4, ctx=(1000, 3, 513, 2000), seed=36, kv_dtype=kv)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w, variant=variant)
    ws = pda.workspace(p, "cuda")
    cnt = pda.counters(p, "cuda")
    outs, parts = [], []
    for _ in range(3):
        o = torch.empty((w.num_seqs, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
        pda.decode_fused(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                         ws["partial_out"], ws["exp_sums"], ws["max_logits"], cnt, o)
        torch.cuda.synchronize()
        outs.append(o.cpu().numpy())
        parts.append([ws[k].cpu().numpy().copy() for k in ("partial_out", "exp_sums", "max_logits")])
    for o, pr in zip(outs[1:], parts[1:]):
        assert np.array_equal(o.view(np.int32), outs[0].view(np.int32))
        # the partials of multi-partition units (single-partition units write the output directly)
        for a, b in zip(pr, parts[0]):
            assert np.array_equal(a.view(np.int32), b.view(np.int32))
