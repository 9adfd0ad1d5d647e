"""Pins of the fp64 oracle against things other than itself (no GPU).

Each check ties the oracle to a library routine, a closed form, an invariant of softmax
attention, brute force on tiny inputs, or a value the pages print.  A plausible slip in the
oracle (a wrong slot or block index, a swapped K/V, a dropped scale, a sign error, a wrong
GQA mapping, a wrong e4m3 bias, a partition range that runs past the context) fails at
least one of them; test_oracle_mutations.py plants such slips and checks that they do.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp8 e4m3 decode
def test_e4m3_all_codes_match_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_float64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_e4m3_format_points(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "e4m3_format_points.json")))
    for code, val in g["points"]:
        got = oracle.e4m3_to_float64([int(code, 16)])[0]
        if val == "nan":
            assert np.isnan(got), code
        else:
            assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)


# ---------------------------------------------------------------- plan arithmetic
def test_plan_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "plan_worked_example.json")))
    p = oracle.plan(g["max_blocks_per_seq"], g["kv_block_size"], 0, g["max_partitions"])
    for k, v in g["expected"].items():
        assert p[k] == v, (k, p[k], v)
    assert p["coverage"] == g["worst_case_context_tokens"]


@pytest.mark.parametrize("name,G,P", [
    ("b1_hk1_qg8_bs16_ctx256", 1, 1),
    ("b8_hk8_qg8_bs16_ctx1-4096", 1, 16),
    ("b32_hk4_qg16_bs32_ctx2048-8192_kbias", 1, 32),
    ("b4_hk8_qg8_bs32_ctx32768_g5p32", 5, 32),
    ("b64_hk8_qg6_bs16_fp8_lognormal2048", 1, 64),
])
def test_plan_for_workloads(name, G, P):
    w = wl.WORKLOADS[name]
    p = oracle.plan(w.max_blocks_per_seq, w.kv_block_size, w.tile_groups_per_partition, w.max_partitions)
    assert (p["G"], p["P"]) == (G, P)


def test_plan_layout_by_hand():
    # bf16, BS=16, Hk=8: data 16*8*2*128*2 = 65536 B, no metadata.
    a = oracle.cache_layout(8, 16, 128, oracle.KV_BF16)
    assert a["cache_block_bytes"] == 65536 and a["meta_region_bytes"] == 0 and a["token_head_bytes"] == 512
    # fp8, BS=16, Hk=8: data 16*8*256 = 32768 B, then 8 heads * 2 fields * 16 slots * 4 B = 1024 B.
    b = oracle.cache_layout(8, 16, 128, oracle.KV_FP8_E4M3)
    assert b["meta_offset_bytes"] == 32768 and b["cache_block_bytes"] == 33792


# ---------------------------------------------------------------- brute force vs SDPA
CASES = [
    dict(kv_dtype=wl.KV_BF16, query_group_size=8, kv_block_size=16, ctx=(40, 17)),
    dict(kv_dtype=wl.KV_BF16, query_group_size=6, kv_block_size=32, ctx=(1, 33)),
    dict(kv_dtype=wl.KV_BF16, query_group_size=16, kv_block_size=16, ctx=(16, 15)),
    dict(kv_dtype=wl.KV_FP8_E4M3, query_group_size=6, kv_block_size=16, ctx=(31, 2)),
    dict(kv_dtype=wl.KV_FP8_E4M3, query_group_size=8, kv_block_size=32, ctx=(64, 9)),
]


def _random_case(case, seed=3, bias=None):
    w = wl.small(num_kv_heads=2, seed=seed, **case)
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((w.num_seqs, w.num_q_heads, w.head_dim), dtype=np.float32)
    K = [rng.standard_normal((c, w.num_kv_heads, w.head_dim), dtype=np.float32) for c in case["ctx"]]
    V = [rng.standard_normal((c, w.num_kv_heads, w.head_dim), dtype=np.float32) for c in case["ctx"]]
    table = wl.draw_block_table(w, rng)
    return w, q, K, V, table


@pytest.mark.parametrize("case", CASES)
def test_bruteforce_matches_sdpa(oracle_mod, case):
    w, q, K, V, table = _random_case(case)
    inp = oh.build_from_values(w, q, K, V, table)
    got = oh.run_oracle(inp)["out"]
    ref = oh.sdpa_reference(w, inp.query, [oh.stored_values(w, k) for k in K], [oh.stored_values(w, v) for v in V])
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("G", [1, 2])
def test_partials_match_sdpa_on_their_ranges(oracle_mod, G):
    case = dict(kv_dtype=wl.KV_BF16, query_group_size=8, kv_block_size=16, ctx=(700, 256))
    w, q, K, V, table = _random_case(case, seed=11)
    inp = oh.build_from_values(w, q, K, V, table)
    res = oh.run_oracle(inp, partials=True, G=G)
    W = 256 * G
    Ks = [oh.stored_values(w, k) for k in K]
    Vs = [oh.stored_values(w, v) for v in V]
    P = res["part_o"].shape[2]
    check_partials_by_brute_force(w, inp, res, Ks, Vs, W)


def check_partials_by_brute_force(w, inp, res, Ks, Vs, W):
    """o_p against SDPA on the partition's range; m_p and l_p against logits from numpy."""
    P = res["part_o"].shape[2]
    q = wl.bf16_bits_to_f32(inp.query).astype(np.float64)
    scale = 1.0 / np.sqrt(w.head_dim)
    QG = w.query_group_size
    for p in range(P):
        ref = oh.sdpa_reference(w, inp.query, Ks, Vs, lo=p * W, hi=(p + 1) * W)
        for b in range(w.num_seqs):
            got = res["part_o"][b, :, p].reshape(w.num_q_heads, w.head_dim)
            if p * W < inp.context_lens[b]:
                np.testing.assert_allclose(got, ref[b], rtol=0, atol=1e-12)
                for h in range(w.num_kv_heads):
                    s = scale * q[b, h * QG:(h + 1) * QG] @ Ks[b][p * W:(p + 1) * W, h].T     # [QG][n]
                    m = s.max(axis=1)
                    l = np.exp(s - m[:, None]).sum(axis=1)
                    np.testing.assert_allclose(res["part_m"][b, h, p], m, rtol=0, atol=1e-12)
                    np.testing.assert_allclose(res["part_l"][b, h, p], l, rtol=1e-12, atol=0)
            else:       # empty partitions are left untouched
                assert np.isnan(got).all() and np.isnan(res["part_m"][b, :, p]).all()


@pytest.mark.parametrize("G", [1, 2, 5])
def test_split_partials_combine_to_unsplit(oracle_mod, G):
    """Combining the partition partials (l_p e^{m_p - M} weights) gives the unsplit result."""
    w = wl.small(num_seqs=3, num_kv_heads=2, ctx=(1300, 256, 257), seed=5)
    inp = wl.generate(w)
    res = oh.run_oracle(inp, partials=True, G=G)
    W = 256 * G
    for b in range(w.num_seqs):
        nv = -(-int(inp.context_lens[b]) // W)
        m = res["part_m"][b, :, :nv]
        l = res["part_l"][b, :, :nv]
        o = res["part_o"][b, :, :nv]
        M = m.max(axis=1, keepdims=True)
        wgt = l * np.exp(m - M)
        comb = (wgt[..., None] * o).sum(axis=1) / wgt.sum(axis=1)[..., None]
        np.testing.assert_allclose(comb.reshape(w.num_q_heads, w.head_dim), res["out"][b], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- probes with closed forms
def _probe_workload(ctx=(37,), kv_dtype=wl.KV_BF16, QG=8, BS=16):
    return wl.small(num_seqs=len(ctx), num_kv_heads=2, query_group_size=QG, kv_block_size=BS, ctx=ctx,
                    kv_dtype=kv_dtype, seed=9)


@pytest.mark.parametrize("kv_dtype", [wl.KV_BF16, wl.KV_FP8_E4M3])
def test_one_hot_selects_one_v_row(oracle_mod, kv_dtype):
    w = _probe_workload(ctx=(37,), kv_dtype=kv_dtype)
    rng = np.random.default_rng(1)
    u = rng.standard_normal((w.num_kv_heads, w.head_dim)).astype(np.float32)
    q = np.repeat(u, w.query_group_size, axis=0)[None]              # every query row of head h equals u_h
    for j in (0, 15, 16, 36):
        K = np.zeros((37, w.num_kv_heads, w.head_dim), np.float32)
        K[j] = 40.0 * u / np.linalg.norm(u, axis=1, keepdims=True)   # s_j - s_t ~ 40 for t != j
        V = rng.standard_normal((37, w.num_kv_heads, w.head_dim)).astype(np.float32)
        inp = oh.build_from_values(w, q, [K], [V], wl.draw_block_table(w, rng))
        out = oh.run_oracle(inp)["out"][0].reshape(w.num_kv_heads, w.query_group_size, w.head_dim)
        vj = oh.stored_values(w, V)[j]
        for h in range(w.num_kv_heads):
            np.testing.assert_allclose(out[h], np.broadcast_to(vj[h], out[h].shape), rtol=0, atol=1e-12)


@pytest.mark.parametrize("kv_dtype", [wl.KV_BF16, wl.KV_FP8_E4M3])
def test_constant_v_returns_v(oracle_mod, kv_dtype):
    w = _probe_workload(ctx=(300,), kv_dtype=kv_dtype)
    rng = np.random.default_rng(2)
    K = rng.standard_normal((300, w.num_kv_heads, w.head_dim)).astype(np.float32)
    V = np.full((300, w.num_kv_heads, w.head_dim), 0.5, np.float32)
    q = rng.standard_normal((1, w.num_q_heads, w.head_dim)).astype(np.float32)
    inp = oh.build_from_values(w, q, [K], [V], wl.draw_block_table(w, rng))
    out = oh.run_oracle(inp)["out"]
    stored = oh.stored_values(w, V)            # 0.5 for bf16; 448 * fp32(0.5/448) for fp8
    c = stored.flat[0]
    assert np.all(stored == c)
    if kv_dtype == wl.KV_BF16:
        assert np.all(out == c)                # dyadic constant: every step is exact
    else:
        np.testing.assert_allclose(out, c, rtol=1e-13, atol=0)   # 300 fp64 roundings


def test_one_token_context_returns_its_v_row(oracle_mod):
    w = _probe_workload(ctx=(1,))
    rng = np.random.default_rng(3)
    K = rng.standard_normal((1, w.num_kv_heads, w.head_dim)).astype(np.float32)
    V = rng.standard_normal((1, w.num_kv_heads, w.head_dim)).astype(np.float32)
    q = rng.standard_normal((1, w.num_q_heads, w.head_dim)).astype(np.float32)
    inp = oh.build_from_values(w, q, [K], [V], wl.draw_block_table(w, rng))
    out = oh.run_oracle(inp)["out"][0].reshape(w.num_kv_heads, w.query_group_size, w.head_dim)
    v0 = oh.stored_values(w, V)[0]
    assert np.array_equal(out, np.broadcast_to(v0[:, None, :], out.shape))


def test_zero_keys_give_the_mean_of_v_and_exact_counts(oracle_mod):
    ctx = 600
    w = _probe_workload(ctx=(ctx,))
    rng = np.random.default_rng(4)
    K = np.zeros((ctx, w.num_kv_heads, w.head_dim), np.float32)
    V = rng.standard_normal((ctx, w.num_kv_heads, w.head_dim)).astype(np.float32)
    q = rng.standard_normal((1, w.num_q_heads, w.head_dim)).astype(np.float32)
    inp = oh.build_from_values(w, q, [K], [V], wl.draw_block_table(w, rng))
    res = oh.run_oracle(inp, partials=True, G=1)
    mean = oh.stored_values(w, V).mean(axis=0)                     # [Hk][D]
    out = res["out"][0].reshape(w.num_kv_heads, w.query_group_size, w.head_dim)
    np.testing.assert_allclose(out, np.broadcast_to(mean[:, None, :], out.shape), rtol=0, atol=1e-12)
    # m_p = 0 and l_p = number of tokens in the partition, exactly
    counts = [256, 256, 88]
    for p, c in enumerate(counts):
        assert np.all(res["part_m"][0, :, p] == 0.0)
        assert np.all(res["part_l"][0, :, p] == float(c))


def test_block_relocation_is_bitwise_invariant(oracle_mod):
    w = wl.small(num_seqs=2, num_kv_heads=2, ctx=(100, 77), seed=12, extra_blocks=9)
    inp = wl.generate(w)
    base = oh.run_oracle(inp)["out"]
    rng = np.random.default_rng(0)
    perm = rng.permutation(w.num_cache_blocks)                     # block i moves to perm[i]
    blocks = inp.cache.reshape(w.num_cache_blocks, w.cache_block_bytes)
    moved = np.empty_like(blocks)
    moved[perm] = blocks
    inp2 = wl.Inputs(w, inp.query, moved.reshape(-1), perm[inp.block_table].astype(np.int32), inp.context_lens)
    assert np.array_equal(oh.run_oracle(inp2)["out"], base)


def test_adding_one_vector_to_every_key_of_a_head_changes_nothing(oracle_mod):
    """Keys on a 1/16 grid in [-2, 2] and an integer bias in [-8, 8] are exact in bf16 both
    before and after the shift, so the logits of each query row move by the constant
    scale * q.b and the softmax is unchanged."""
    w = _probe_workload(ctx=(90,))
    rng = np.random.default_rng(6)
    K = (rng.integers(-32, 33, size=(90, w.num_kv_heads, w.head_dim)) / 16.0).astype(np.float32)
    bias = rng.integers(-8, 9, size=(w.num_kv_heads, w.head_dim)).astype(np.float32)
    V = rng.standard_normal((90, w.num_kv_heads, w.head_dim)).astype(np.float32)
    q = (rng.integers(-16, 17, size=(1, w.num_q_heads, w.head_dim)) / 64.0).astype(np.float32)
    table = wl.draw_block_table(w, rng)
    a = oh.run_oracle(oh.build_from_values(w, q, [K], [V], table))["out"]
    assert np.array_equal(wl.bf16_bits_to_f32(wl.round_bf16(K + bias)), K + bias)
    b = oh.run_oracle(oh.build_from_values(w, q, [K + bias], [V], table))["out"]
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_empty_context_gives_zero_and_no_partials(oracle_mod):
    w = wl.small(num_seqs=2, num_kv_heads=1, ctx=(0, 5), seed=13)
    inp = wl.generate(w)
    res = oh.run_oracle(inp, partials=True)
    assert np.all(res["out"][0] == 0.0)
    assert np.isnan(res["part_m"][0]).all() and np.isnan(res["part_o"][0]).all()


def test_invalid_inputs_are_rejected(oracle_mod):
    w = wl.small(num_seqs=1, num_kv_heads=1, ctx=(20,), seed=14)
    inp = wl.generate(w)
    bad = wl.Inputs(w, inp.query, inp.cache, inp.block_table, np.array([10_000], np.int32))
    with pytest.raises(ValueError):
        oh.run_oracle(bad)
    bt = inp.block_table.copy()
    bt[0, 0] = w.num_cache_blocks
    with pytest.raises(ValueError):
        oh.run_oracle(wl.Inputs(w, inp.query, inp.cache, bt, inp.context_lens))
