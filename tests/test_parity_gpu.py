"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerances (the problem's own bar): max-abs 2e-3 on the fp32 output for a bf16 KV cache and
1e-2 for fp8 e4m3 and for the 4-bit TQ4 cache (the bar stated for a quantised cache); the bf16
output may differ by that plus half a bf16 ulp of the oracle value.
Partition partials: o_p within the same tolerance, m_p within lt*max(1,|m|) and l_p within a
relative lt*max(1,|m|), with lt = 1e-4 (fp32 logits): a logit off by a relative lt moves every
term e^(s - m) of l_p by about lt*|s|, so both bounds grow with the logits' magnitude.  TQ4
takes lt = 2e-3: its centroids enter the score MMA as f16 (unit roundoff 2^-11), so a logit can
be off by up to softmax_scale * k_norm * sum_d |q_d c_d| * 2^-11, about 3.5e-3 on random inputs
if every rounding pointed the same way and ~3e-4 typically (with logits up to 25, f16
centroids alone move l_p by 3.5e-4*|m|).  Block-table walking and partition bookkeeping are checked bit for
bit: which partials are written (sentinel NaN payload elsewhere), the zero-key count probe
(m_p = 0 and l_p = token count exactly), the one-hot probe (the output equals one stored V row
exactly), block relocation and the G independence of short contexts.
"""
import numpy as np
import pytest
import torch

from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh
from tests.gpu_helpers import KV_VARIANTS, bf16_half_ulp, is_sentinel, run_gpu, to_device

pytestmark = pytest.mark.gpu

TOL = {wl.KV_BF16: 2e-3, wl.KV_FP8_E4M3: 1e-2, wl.KV_TQ4: 1e-2}
LOGIT_TOL = {wl.KV_BF16: 1e-4, wl.KV_FP8_E4M3: 1e-4, wl.KV_TQ4: 2e-3}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def check_against_oracle(inp, res, ref, units=None):
    """Every (sequence, KV head) unit in `units` (default: all): the fp32 and bf16 outputs, and,
    when the oracle computed them, every partition's partials and which partitions were written."""
    w = inp.workload
    tol, lt = TOL[w.kv_dtype], LOGIT_TOL[w.kv_dtype]
    B, Hk, QG, D = w.num_seqs, w.num_kv_heads, w.query_group_size, w.head_dim
    W, P = res["plan"].partition_tokens, res["plan"].num_partitions
    assert res["err"] == 0
    ul = np.arange(B * Hk) if units is None else np.asarray(units, dtype=np.int64)
    bs, hs = np.divmod(ul, Hk)

    def first_bad(ok, what):
        bad = np.flatnonzero(~ok)
        assert bad.size == 0, f"unit {int(ul[bad[0]])} (b={int(bs[bad[0]])}, h={int(hs[bad[0]])}): {what}"

    g = res["out"].reshape(B, Hk, QG, D)[bs, hs]
    o = ref["out"].reshape(B, Hk, QG, D)[bs, hs]
    first_bad(np.isfinite(g).all(axis=(1, 2)), "non-finite output")
    first_bad(np.abs(g - o).max(axis=(1, 2)) <= tol, f"out max-abs above {tol}")
    gb = res["out_bf16"].reshape(B, Hk, QG, D)[bs, hs]
    first_bad(np.all(np.abs(gb - o) <= tol + bf16_half_ulp(o), axis=(1, 2)), "bf16 out")
    if ref.get("part_o") is None:
        return
    nv = -(-inp.context_lens.astype(np.int64)[bs] // W)
    written = np.arange(P)[None, :] < nv[:, None]                                   # [U][P]
    go, gm, gl = res["part_o"][bs, hs], res["part_m"][bs, hs], res["part_l"][bs, hs]
    ro, rm, rl = ref["part_o"][bs, hs], ref["part_m"][bs, hs], ref["part_l"][bs, hs]
    sent_o = is_sentinel(go).all(axis=(2, 3))
    sent_s = is_sentinel(gm).all(axis=2) & is_sentinel(gl).all(axis=2)
    first_bad(np.all(~written | (~is_sentinel(go).any(axis=(2, 3)) & ~is_sentinel(gm).any(axis=2)), axis=1),
              "a partition below ceil(ctx/W) was not written")
    first_bad(np.all(written | (sent_o & sent_s), axis=1), "a partition at or above ceil(ctx/W) was written")
    with np.errstate(invalid="ignore"):
        eo = np.where(written[:, :, None, None], np.abs(go - ro), 0.0)
        first_bad(np.all(eo <= tol, axis=(1, 2, 3)), f"o_p max-abs above {tol}")
        mag = np.maximum(1.0, np.abs(rm))
        em = np.where(written[:, :, None], np.abs(gm - rm) <= lt * mag, True)
        first_bad(np.all(em, axis=(1, 2)), "m_p")
        # l_p: relative lt where |m_p| <= 1; beyond that a logit off by a relative lt moves every
        # term e^(s - m) of l_p by about lt*|s|, so the bound grows with |m_p|
        el = np.where(written[:, :, None], np.abs(gl - rl) <= lt * mag * rl, True)
        first_bad(np.all(el, axis=(1, 2)), "l_p")
        tight = written[:, :, None] & (np.abs(rm) <= 1.0)
        first_bad(np.all(np.where(tight, np.abs(gl - rl) <= lt * rl, True), axis=(1, 2)), "l_p (|m_p| <= 1)")


SWEEP = [
    # (kv dtype, QG, BS, G, Hk, context lengths); fp8 shapes run on both fp8 kernels
    (wl.KV_BF16, 8, 16, 1, 2, (1, 15, 16, 17, 255, 256, 257, 700)),
    (wl.KV_BF16, 6, 32, 1, 3, (2, 31, 33, 513, 1000)),
    (wl.KV_BF16, 16, 16, 2, 2, (1, 511, 512, 513, 1600)),
    (wl.KV_BF16, 8, 32, 5, 2, (1279, 1280, 1281, 3000)),
    (wl.KV_BF16, 16, 32, 1, 1, (64, 4097)),
    (wl.KV_FP8_E4M3, 6, 16, 1, 2, (1, 17, 300, 1100)),
    (wl.KV_FP8_E4M3, 8, 32, 2, 3, (5, 600, 1500)),
    (wl.KV_FP8_E4M3, 16, 16, 1, 2, (16, 257, 900)),
    (wl.KV_TQ4, 6, 16, 1, 2, (1, 17, 300, 1100)),
    (wl.KV_TQ4, 8, 32, 2, 3, (5, 600, 1500)),
    (wl.KV_TQ4, 16, 16, 1, 2, (16, 257, 900)),
    (wl.KV_TQ4, 8, 16, 5, 1, (1279, 1280, 1281, 2000)),
]


SWEEP += [
    # head groups of 8 (one group, and four), 4, 6 and 5 heads
    (wl.KV_FP8_E4M3, 6, 16, 1, 8, (1, 17, 255, 256, 257, 1100, 4000)),
    (wl.KV_FP8_E4M3, 8, 32, 5, 8, (1279, 1281, 40, 6000)),
    (wl.KV_FP8_E4M3, 6, 16, 1, 32, (700, 33)),
    (wl.KV_FP8_E4M3, 16, 16, 2, 4, (513, 2000, 1)),
    (wl.KV_FP8_E4M3, 8, 32, 1, 12, (300, 901)),
    (wl.KV_FP8_E4M3, 6, 16, 1, 5, (64, 777)),
]
def _variants(kv, QG):
    # fp8 on both of its kernels; bf16 with sixteen rows on head warps (automatic) and row halves
    if kv == wl.KV_FP8_E4M3:
        return (1, 2)
    return (0, 3) if kv == wl.KV_BF16 and QG == 16 else (0,)


SWEEP_CASES = [(*c, v) for c in SWEEP for v in _variants(c[0], c[1])]


@pytest.mark.parametrize("kv,QG,BS,G,Hk,ctx,variant", SWEEP_CASES)
def test_sweep_matches_oracle(oracle_mod, kv, QG, BS, G, Hk, ctx, variant):
    w = wl.small(num_seqs=len(ctx), num_kv_heads=Hk, query_group_size=QG, kv_block_size=BS, ctx=ctx, kv_dtype=kv,
                 tile_groups_per_partition=G, seed=100 + QG + BS + G + Hk, extra_blocks=5)
    inp = wl.generate(w)
    res = run_gpu(inp, variant=variant)
    ref = oh.run_oracle(inp, partials=True, G=G)
    check_against_oracle(inp, res, ref)


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_more_units_than_warps(oracle_mod, kv, variant):
    # 2600 to 3000 (sequence, KV head, partition) units: more than the persistent grid has warps,
    # so warps take tile-balanced runs of several units (fewer units give one unit per warp)
    rng = np.random.default_rng(9)
    ctx = tuple(int(c) for c in rng.integers(257, 1025, size=120))
    w = wl.small(num_seqs=120, num_kv_heads=8, query_group_size=6, kv_block_size=16, ctx=ctx, kv_dtype=kv, seed=41)
    inp = wl.generate(w)
    assert sum(8 * -(-c // 256) for c in ctx) > 2432
    check_against_oracle(inp, run_gpu(inp, variant=variant), oh.run_oracle(inp, partials=True))


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_large_batch_of_short_contexts(oracle_mod, kv, variant):
    # 1500 sequences: every lane of the work scan walks 47 of them; contexts 0-300 tokens (one or
    # two partitions, some empty), sampled units checked against the oracle with their partials
    rng = np.random.default_rng(13)
    ctx = tuple(int(c) for c in rng.integers(0, 301, size=1500))
    w = wl.small(num_seqs=1500, num_kv_heads=2, query_group_size=8, kv_block_size=16, ctx=ctx, kv_dtype=kv, seed=43,
                 max_blocks_per_seq=19)
    inp = wl.generate(w)
    res = run_gpu(inp, variant=variant)
    units = np.sort(rng.choice(1500 * 2, size=200, replace=False))
    check_against_oracle(inp, res, oh.run_oracle(inp, partials=True, units=units), units=units)
    empty = [b for b, c in enumerate(ctx) if c == 0]
    assert empty and np.all(res["out"][empty] == 0)


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_many_kv_heads(oracle_mod, kv, variant):
    # 32 KV heads of QG 6 (192 query heads): the head dimension of the tensor maps and the
    # per-head metadata offsets at a large head count; 1056 units (tile-balanced on the 912-warp
    # bf16 grid, one unit per warp on the 1824-warp fp8 and TQ4 grids)
    ctx = (4000, 1, 1300, 700, 256, 1500)
    w = wl.small(num_seqs=6, num_kv_heads=32, query_group_size=6, kv_block_size=16, ctx=ctx, kv_dtype=kv, seed=44)
    inp = wl.generate(w)
    res = run_gpu(inp, variant=variant)
    units = np.sort(np.random.default_rng(3).choice(6 * 32, size=48, replace=False))
    check_against_oracle(inp, res, oh.run_oracle(inp, partials=True, units=units), units=units)


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_one_unit_per_warp(oracle_mod, kv, variant):
    # room for 16 x 8 x 16 = 2048 partitions (more than the grid's warps) but short contexts
    # give at most 16 x 8 x 3 = 384 non-empty ones: each warp takes one whole unit
    rng = np.random.default_rng(11)
    ctx = tuple(int(c) for c in rng.integers(1, 769, size=16))
    w = wl.small(num_seqs=16, num_kv_heads=8, query_group_size=8, kv_block_size=16, ctx=ctx, kv_dtype=kv, seed=42,
                 max_blocks_per_seq=256)
    inp = wl.generate(w)
    res = run_gpu(inp, variant=variant)
    assert res["plan"].num_partitions == 16
    check_against_oracle(inp, res, oh.run_oracle(inp, partials=True))


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_more_than_64_partitions_and_empty_sequences(oracle_mod, kv, variant):
    # the longest sequence has 79 partitions of 256 tokens: the reduce holds (m_p, l_p) of 64
    # partitions per row in registers and reloads the rest; empty sequences sit in between
    ctx = (20000, 0, 16385, 300, 0, 1)
    w = wl.small(num_seqs=6, num_kv_heads=2, query_group_size=8, kv_block_size=32, ctx=ctx, kv_dtype=kv, seed=71)
    inp = wl.generate(w)
    res = run_gpu(inp, variant=variant)
    assert res["plan"].num_partitions == 79
    check_against_oracle(inp, res, oh.run_oracle(inp, partials=True))
    assert np.all(res["out"][[1, 4]] == 0) and np.all(res["out_bf16"][[1, 4]] == 0)


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_every_context_empty(oracle_mod, kv, variant):
    w = wl.small(num_seqs=3, num_kv_heads=2, ctx=(0, 0, 0), kv_dtype=kv, seed=72, max_blocks_per_seq=4)
    inp = wl.generate(w)
    res = run_gpu(inp, variant=variant)
    assert res["err"] == 0
    assert np.all(res["out"] == 0) and np.all(res["out_bf16"] == 0)
    for key in ("part_o", "part_m", "part_l"):
        assert is_sentinel(res[key]).all(), f"{key} was written"


def test_key_bias_workload_small(oracle_mod):
    w = wl.small(num_seqs=3, num_kv_heads=2, query_group_size=16, kv_block_size=32, ctx=(2048, 2100, 3000),
                 seed=5, k_bias_std=2.0)
    inp = wl.generate(w)
    check_against_oracle(inp, run_gpu(inp), oh.run_oracle(inp, partials=True))


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_zero_keys_count_probe_is_exact(oracle_mod, kv, variant):
    ctx = (600, 256, 1)
    w = wl.small(num_seqs=3, num_kv_heads=2, ctx=ctx, kv_dtype=kv, seed=31)
    rng = np.random.default_rng(0)
    K = [np.zeros((c, 2, 128), np.float32) for c in ctx]
    V = [rng.standard_normal((c, 2, 128)).astype(np.float32) for c in ctx]
    q = rng.standard_normal((3, w.num_q_heads, 128)).astype(np.float32)
    inp = oh.build_from_values(w, q, K, V, wl.draw_block_table(w, rng))
    res = run_gpu(inp, variant=variant)
    assert res["err"] == 0
    for b, c in enumerate(ctx):
        nv = -(-c // 256)
        for p in range(res["plan"].num_partitions):
            if p < nv:
                assert np.all(res["part_m"][b, :, p] == 0.0)
                assert np.all(res["part_l"][b, :, p] == float(min(256, c - 256 * p)))
            else:
                assert is_sentinel(res["part_m"][b, :, p]).all()


def stored_v_rows_f32(w, V):
    """The fp32 value of every stored V element [n][Hk][D], as the kernels produce it for a
    weight of exactly 1: bf16 values as they are; e4m3 codes times their fp32 scale, rounded
    once to fp32; TQ4 code * v_scale + v_zero, rounded once to fp32."""
    if w.kv_dtype == wl.KV_TQ4:
        codes, vs, vz = wl.quantize_tq4_v(V)
        return oh.tq4_values(codes, v_scale_bits=vs, v_zero_bits=vz).astype(np.float32).astype(np.float64)
    return oh.stored_values(w, V).astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
@pytest.mark.parametrize("BS,ctx,js", [(16, 37, (0, 15, 16, 36)), (16, 700, (0, 255, 256, 511, 699)),
                                       (32, 700, (31, 32, 300, 699))])
def test_one_hot_probe_returns_the_stored_row_exactly(oracle_mod, kv, variant, BS, ctx, js):
    # One key j points along the query (a logit gap above 140, so every other weight is exactly
    # 0 in fp32 and p_j = 1); the output is then the stored V row j itself, bit for bit, which
    # pins the block-table walk (entry t/BS, slot t%BS) of every format.  Every V row has the same
    # extremes (element 0 is 1, element 1 is -1, the rest lie between), so the quantised formats
    # store every row with the same scale (fp8) or the same scale and zero (TQ4), and the weight of
    # row j relative to the step's largest V weight is exactly 1.
    w = wl.small(num_seqs=1, num_kv_heads=2, kv_block_size=BS, ctx=(ctx,), seed=32, kv_dtype=kv)
    rng = np.random.default_rng(1)
    u = rng.standard_normal((2, 128)).astype(np.float32)
    q = np.repeat(u, 8, axis=0)[None]
    for j in js:
        K = np.zeros((ctx, 2, 128), np.float32)
        K[j] = 150.0 * u / np.linalg.norm(u, axis=1, keepdims=True)
        V = rng.uniform(-0.9, 0.9, (ctx, 2, 128)).astype(np.float32)
        V[:, :, 0], V[:, :, 1] = 1.0, -1.0
        inp = oh.build_from_values(w, q, [K], [V], wl.draw_block_table(w, rng))
        vj = stored_v_rows_f32(w, V)[j]
        ref = oh.run_oracle(inp)["out"][0].reshape(2, 8, 128)
        assert np.allclose(ref, vj[:, None, :], rtol=0, atol=1e-6)     # the probe is what it claims
        res = run_gpu(inp, variant=variant)
        assert res["err"] == 0
        out = res["out"][0].reshape(2, 8, 128)
        for h in range(2):
            assert np.array_equal(out[h], np.broadcast_to(vj[h], (8, 128))), f"j={j} h={h}"


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
@pytest.mark.parametrize("QG", [8, 16])
def test_running_maximum_and_v_scale_swings(oracle_mod, kv, variant, QG):
    # Key magnitudes that grow 160-fold across every 256-token partition move the running
    # maximum by several times 2^8 within a partition; the next sequence has them shrink instead
    # (the maximum is set by the first tiles); V rows jump between magnitude 1 and 2^-8 every
    # three tiles, so a step's V scales leave any window of 64x around the previous ones, up and
    # down.
    ctx = (1000, 700, 300, 40)
    w = wl.small(num_seqs=4, num_kv_heads=2, query_group_size=QG, kv_block_size=16, ctx=ctx, kv_dtype=kv,
                 tile_groups_per_partition=1, seed=61, extra_blocks=5)
    rng = np.random.default_rng(61)
    q = rng.standard_normal((4, w.num_q_heads, 128)).astype(np.float32)
    K, V = [], []
    for b, c in enumerate(ctx):
        gk = 0.05 * 160.0 ** ((np.arange(c) % 256) / 255.0)
        if b % 2:
            gk = gk[::-1]
        gv = np.where((np.arange(c) // 48) % 2 == 0, 1.0, 2.0 ** -8)
        K.append((rng.standard_normal((c, 2, 128)) * gk[:, None, None]).astype(np.float32))
        V.append((rng.standard_normal((c, 2, 128)) * gv[:, None, None]).astype(np.float32))
    inp = oh.build_from_values(w, q, K, V, wl.draw_block_table(w, rng))
    res = run_gpu(inp, variant=variant)
    assert res["plan"].partition_tokens == 256
    check_against_oracle(inp, res, oh.run_oracle(inp, partials=True))


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
@pytest.mark.parametrize("BS", [16, 32])
def test_block_relocation_is_bitwise_invariant(kv, variant, BS):
    # moving every block of the pool (data and metadata) and rewriting the tables to match changes
    # no bit of the output or of any partial: the arithmetic follows the logical token order only
    w = wl.small(num_seqs=2, num_kv_heads=2, kv_block_size=BS, ctx=(900, 77), seed=33, extra_blocks=11, kv_dtype=kv)
    inp = wl.generate(w)
    a = run_gpu(inp, variant=variant)
    perm = np.random.default_rng(0).permutation(w.num_cache_blocks)
    blocks = inp.cache.reshape(w.num_cache_blocks, w.cache_block_bytes)
    moved = np.empty_like(blocks)
    moved[perm] = blocks
    b = run_gpu(wl.Inputs(w, inp.query, moved.reshape(-1), perm[inp.block_table].astype(np.int32), inp.context_lens,
                          inp.extra), variant=variant)
    assert a["err"] == 0 and b["err"] == 0
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["out_bf16"], b["out_bf16"])
    for k in ("part_o", "part_m", "part_l"):
        assert np.array_equal(a[k].view(np.int32), b[k].view(np.int32)), k


def test_short_contexts_do_not_depend_on_G():
    w = wl.small(num_seqs=3, num_kv_heads=2, ctx=(1, 100, 256), seed=34, max_blocks_per_seq=64)
    inp = wl.generate(w)
    r1, r2, r5 = run_gpu(inp, G=1), run_gpu(inp, G=2), run_gpu(inp, G=5)
    assert r1["plan"].num_partitions != r2["plan"].num_partitions
    assert np.array_equal(r1["out"], r2["out"]) and np.array_equal(r1["out"], r5["out"])


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_repeat_runs_are_bitwise_identical(kv, variant):
    # the work assignment is a function of the inputs only, and every sum has a fixed order
    w = wl.small(num_seqs=4, num_kv_heads=2, ctx=(1000, 3, 513, 2000), seed=35, kv_dtype=kv)
    inp = wl.generate(w)
    d = to_device(inp)
    a, b = run_gpu(inp, d=d, variant=variant), run_gpu(inp, d=d, variant=variant)
    assert np.array_equal(a["out"], b["out"])
    for k in ("part_o", "part_m", "part_l"):     # compare bits: unwritten slots hold the NaN sentinel
        assert np.array_equal(a[k].view(np.int32), b[k].view(np.int32))


def test_bad_context_length_sets_error_bit_and_zeroes_that_sequence(oracle_mod):
    w = wl.small(num_seqs=3, num_kv_heads=2, ctx=(40, 20, 33), seed=36)
    inp = wl.generate(w)
    ref = oh.run_oracle(inp)
    ctx = inp.context_lens.copy()
    ctx[1] = w.max_blocks_per_seq * w.kv_block_size + 1
    res = run_gpu(wl.Inputs(w, inp.query, inp.cache, inp.block_table, ctx))
    assert res["err"] & 1
    assert np.all(res["out"][1] == 0)
    for b in (0, 2):
        assert np.abs(res["out"][b] - ref["out"][b]).max() <= 2e-3


def test_bad_block_id_sets_error_bit_without_faulting():
    w = wl.small(num_seqs=2, num_kv_heads=2, ctx=(40, 20), seed=37)
    inp = wl.generate(w)
    bt = inp.block_table.copy()
    bt[0, 1] = w.num_cache_blocks + 5
    bt[1, 0] = -3
    res = run_gpu(wl.Inputs(w, inp.query, inp.cache, bt, inp.context_lens))
    assert res["err"] & 2
    assert np.isfinite(res["out"]).all()
    torch.cuda.synchronize()


# ---------------------------------------------------------------- full-size workloads
FULL_CASES = [(n, 0) for n in wl.WORKLOAD_ORDER] + [
    (n, v) for n in wl.WORKLOAD_ORDER for v in _variants(wl.WORKLOADS[n].kv_dtype, wl.WORKLOADS[n].query_group_size)
    if v != 0]


@pytest.mark.parametrize("name,variant", FULL_CASES)
def test_full_size_workload_every_unit(oracle_mod, name, variant):
    # every (sequence, KV head) unit of the configuration, with every partition's partials, in
    # the launch configuration the bench times (variant 0), and for fp8 on each kernel
    w = wl.WORKLOADS[name]
    inp = wl.generate(w)
    res = run_gpu(inp, variant=variant)
    assert res["err"] == 0
    assert np.isfinite(res["out"]).all()
    check_against_oracle(inp, res, oh.run_oracle(inp, partials=True))


ROW_HALF_CASES = [
    ("b32_hk4_qg16_bs32_ctx2048-8192_kbias", None),
    # long and short sequences, an empty one, one of a single partial tile, BS 16 and 32, G 1 and 2
    (None, dict(num_seqs=6, num_kv_heads=2, query_group_size=16, kv_block_size=16, ctx=(5000, 1, 0, 700, 257, 4097),
                seed=131)),
    (None, dict(num_seqs=3, num_kv_heads=3, query_group_size=16, kv_block_size=32, ctx=(2049, 64, 9000),
                tile_groups_per_partition=2, seed=132)),
]


@pytest.mark.parametrize("name,kw", ROW_HALF_CASES)
def test_row_halves_equal_head_warps_bit_for_bit(oracle_mod, name, kw):
    # The row-half kernel runs each 8-row block with the head-warp kernel's arithmetic: the same
    # partials (and so the same outputs), bit for bit, written to the same partitions.
    w = wl.WORKLOADS[name] if name else wl.small(kv_dtype=wl.KV_BF16, extra_blocks=3, **kw)
    inp = wl.generate(w)
    d = to_device(inp)
    head, rows = run_gpu(inp, d=d, variant=1), run_gpu(inp, d=d, variant=3)
    assert head["err"] == 0 and rows["err"] == 0
    for k in ("part_o", "part_m", "part_l"):
        assert np.array_equal(head[k].view(np.int32), rows[k].view(np.int32)), k
    assert np.array_equal(head["out"], rows["out"])
    check_against_oracle(inp, rows, oh.run_oracle(inp, partials=True))


def test_row_half_counters_return_to_zero_across_many_launches(oracle_mod):
    # the row-half kernel takes units from the library's counter slots too: 300 launches in a row
    # (every slot reused) give the first launch's bits
    import paged_kv_gqa_block_gb300 as pda
    from tests.gpu_helpers import plan_for, sentinel_ws
    w = wl.small(num_seqs=4, num_kv_heads=4, query_group_size=16, kv_block_size=16, ctx=(3000, 17, 600, 2048),
                 kv_dtype=wl.KV_BF16, seed=133)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w, variant=3)
    ws = sentinel_ws(p)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for i in range(300):
        pda.decode(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                   ws["partial_out"], ws["exp_sums"], ws["max_logits"], err_word=err)
        if i in (0, 299):
            o = torch.empty((w.num_seqs, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
            pda.reduce(p, d["context_lens"], ws["partial_out"], ws["exp_sums"], ws["max_logits"], o, err_word=err)
            outs.append(o.cpu().numpy())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(outs[0].view(np.int32), outs[1].view(np.int32))
    assert np.abs(outs[0] - oh.run_oracle(inp)["out"]).max() <= TOL[wl.KV_BF16]


def test_head_group_counters_return_to_zero_across_many_launches(oracle_mod):
    # The head-group kernel takes units from a counter pair that its last CTA returns to zero; the
    # library cycles through 256 such pairs.  600 launches in a row (every pair reused twice) must
    # all give the same bits as the first, which matches the oracle.
    import paged_kv_gqa_block_gb300 as pda
    from tests.gpu_helpers import plan_for, sentinel_ws
    w = wl.small(num_seqs=6, num_kv_heads=8, query_group_size=6, kv_block_size=16,
                 ctx=(300, 5000, 17, 2048, 1000, 256), kv_dtype=wl.KV_FP8_E4M3, seed=96)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w, variant=2)
    ws = sentinel_ws(p)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for i in range(600):
        pda.decode(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                   ws["partial_out"], ws["exp_sums"], ws["max_logits"], err_word=err)
        if i in (0, 599):
            o = torch.empty((w.num_seqs, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
            pda.reduce(p, d["context_lens"], ws["partial_out"], ws["exp_sums"], ws["max_logits"], o, err_word=err)
            outs.append(o.cpu().numpy())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(outs[0].view(np.int32), outs[1].view(np.int32))
    assert np.abs(outs[0] - oh.run_oracle(inp)["out"]).max() <= TOL[wl.KV_FP8_E4M3]


def test_automatic_variant_on_the_full_size_workloads():
    # the fp8 configuration (64 sequences, 8 heads: head groups of 4, 256 units of room per group)
    # runs on head groups, the bf16 QG 16 configuration (4 096 units) on row halves; the others
    # run on head warps
    import paged_kv_gqa_block_gb300 as pda
    from tests.gpu_helpers import plan_for
    for name in wl.WORKLOAD_ORDER:
        w = wl.WORKLOADS[name]
        want = (pda.VARIANT_HEAD_GROUPS if w.kv_dtype == wl.KV_FP8_E4M3 else
                pda.VARIANT_ROW_HALVES if w.kv_dtype == wl.KV_BF16 and w.query_group_size == 16 else
                pda.VARIANT_HEAD_WARPS)
        assert pda.kernel_variant(plan_for(w)) == want, name
