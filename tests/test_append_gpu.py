"""The append kernel (write side of the paged cache) against the oracle: bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh
from tests.gpu_helpers import plan_for, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pda():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_block_gb300 as pda
    return pda


def new_tokens(w, rng, scale=1.0):
    k = wl.round_bf16((rng.standard_normal((w.num_seqs, w.num_kv_heads, 128)) * scale).astype(np.float32))
    v = wl.round_bf16((rng.standard_normal((w.num_seqs, w.num_kv_heads, 128)) * scale).astype(np.float32))
    return k, v


@pytest.mark.parametrize("kv,BS,Hk", [(wl.KV_BF16, 16, 2), (wl.KV_BF16, 32, 3), (wl.KV_FP8_E4M3, 16, 2),
                                      (wl.KV_FP8_E4M3, 32, 8)])
def test_append_matches_oracle_bytes(oracle_mod, pda, kv, BS, Hk):
    ctx = (0, 5, 31, 32, 100)
    w = wl.small(num_seqs=len(ctx), num_kv_heads=Hk, kv_block_size=BS, ctx=ctx, kv_dtype=kv, seed=60 + BS + Hk,
                 max_blocks_per_seq=8)
    inp = wl.generate(w)
    rng = np.random.default_rng(3)
    for scale in (1.0, 300.0, 1e-3):        # scales that exercise saturation-free rounding, large and tiny rows
        k, v = new_tokens(w, rng, scale)
        k[1, 0] = 0                         # an all-zero row: scale 1, codes 0
        pos = np.array(ctx, np.int32)
        pos[2] = -1                          # skipped
        d = to_device(inp)
        p = plan_for(w)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kt = torch.from_numpy(k.view(np.int16)).cuda()
        vt = torch.from_numpy(v.view(np.int16)).cuda()
        pda.append_kv(p, kt, vt, d["cache"], w.num_cache_blocks, d["block_table"], torch.from_numpy(pos).cuda(),
                      err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref = oracle.append_kv(oh.problem(w), inp.cache, k, v, inp.block_table, pos)
        got = d["cache"].cpu().numpy()
        assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"


def test_append_then_decode_sees_the_new_token(oracle_mod, pda):
    w = wl.small(num_seqs=2, num_kv_heads=2, kv_block_size=16, ctx=(40, 16), kv_dtype=wl.KV_FP8_E4M3, seed=70,
                 max_blocks_per_seq=4)
    inp = wl.generate(w)
    rng = np.random.default_rng(4)
    k, v = new_tokens(w, rng)
    d = to_device(inp)
    p = plan_for(w)
    pda.append_kv(p, torch.from_numpy(k.view(np.int16)).cuda(), torch.from_numpy(v.view(np.int16)).cuda(),
                  d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"])
    ctx1 = d["context_lens"] + 1
    out = pda.decode_step(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], ctx1,
                          out_dtype=torch.float32)
    torch.cuda.synchronize()
    cache1 = oracle.append_kv(oh.problem(w), inp.cache, k, v, inp.block_table, inp.context_lens)
    ref = oh.run_oracle(wl.Inputs(w, inp.query, cache1, inp.block_table, inp.context_lens + 1))["out"]
    assert np.abs(out.cpu().numpy() - ref).max() <= 1e-2


def test_append_data_errors(pda):
    w = wl.small(num_seqs=2, num_kv_heads=1, ctx=(3, 3), seed=71, max_blocks_per_seq=2)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w)
    z = torch.zeros((2, 1, 128), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.tensor([w.max_blocks_per_seq * w.kv_block_size, 0], dtype=torch.int32, device="cuda")
    bt = d["block_table"].clone()
    bt[1, 0] = w.num_cache_blocks + 3
    before = d["cache"].clone()
    pda.append_kv(p, z, z, d["cache"], w.num_cache_blocks, bt, pos, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pda.ERRW_BAD_POSITION and int(err.item()) & pda.ERRW_BAD_BLOCK_ID
    assert torch.equal(before, d["cache"])


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_FP8_E4M3])
def test_in_stream_context_update_is_ordered_before_decode_and_reduce(oracle_mod, pda, kv):
    # A serving loop on one stream: append the new token at position ctx, add 1 to the device
    # context lengths in place, then the partition pass and the reduce, with no host sync in
    # between.  Both kernels must see the lengths the in-place update wrote (the reduce reads them
    # only after its grid-dependency wait).  Three steps in a row, each against the oracle.
    ctx0 = (255, 256, 511, 17)
    w = wl.small(num_seqs=len(ctx0), num_kv_heads=2, query_group_size=8, kv_block_size=16, ctx=ctx0, kv_dtype=kv,
                 seed=73, max_blocks_per_seq=40)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w)
    rng = np.random.default_rng(5)
    cache = inp.cache.copy()
    ctx = inp.context_lens.copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(3):
        k, v = new_tokens(w, rng)
        pda.append_kv(p, torch.from_numpy(k.view(np.int16)).cuda(), torch.from_numpy(v.view(np.int16)).cuda(),
                      d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"], err_word=err)
        d["context_lens"].add_(1)
        out = pda.decode_step(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                              out_dtype=torch.float32, err_word=err)
        got = out.cpu().numpy()          # the one host synchronisation of the step
        cache = oracle.append_kv(oh.problem(w), cache, k, v, inp.block_table, ctx)
        ctx = ctx + 1
        ref = oh.run_oracle(wl.Inputs(w, inp.query, cache, inp.block_table, ctx))["out"]
        assert int(err.item()) == 0
        tol = 2e-3 if kv == wl.KV_BF16 else 1e-2
        assert np.abs(got - ref).max() <= tol, f"step {step}"
