"""Pins of the oracle's TQ4 decode (the 4-bit format of the vLLM "tq_decode" page) against
things other than itself (no GPU).

The format, as the page's STEP F reads it: per token and KV head, 64 bytes of K codes then 64
bytes of V codes, dimension d in nibble d % 2 (low first) of byte d / 2; K = centroid[code] *
k_norm, V = code * v_scale + v_zero, the three fp16 fields in the metadata region
[kv_head][field][slot].  The probes below write cache bytes by hand (not through the
generator's packer) and compare with closed forms, so a slip in the nibble order, the byte
position of a dimension, the centroid index, the field order or the fp16 decode fails one of
them; the planted-mistake test at the end checks that it does.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh

D = 128
# increasing, distinct and not symmetric, so that code j and code 15 - j differ
CENTROIDS = np.array([-0.30, -0.21, -0.15, -0.11, -0.08, -0.05, -0.03, -0.01,
                      0.02, 0.04, 0.07, 0.10, 0.14, 0.19, 0.26, 0.35], dtype=np.float32)


def f16_bits(x: float) -> int:
    return int(np.array(x, dtype=np.float16).view(np.uint16))


def _workload(ctx, QG=8, BS=16, Hk=2, seed=21):
    return wl.small(num_seqs=len(ctx), num_kv_heads=Hk, query_group_size=QG, kv_block_size=BS, ctx=ctx,
                    kv_dtype=wl.KV_TQ4, seed=seed)


class HandCache:
    """A TQ4 cache written byte by hand from the layout's definition."""

    def __init__(self, w):
        self.w = w
        self.cache = wl.empty_cache(w, poison=True)
        rng = np.random.default_rng(w.seed)
        self.table = wl.draw_block_table(w, rng)

    def _block_slot(self, b, t):
        return int(self.table[b, t // self.w.kv_block_size]), t % self.w.kv_block_size

    def put_row(self, b, t, h, which, row_bytes):
        blk, slot = self._block_slot(b, t)
        w = self.w
        off = blk * w.cache_block_bytes + (slot * w.num_kv_heads + h) * D + which * (D // 2)
        self.cache[off:off + D // 2] = np.asarray(row_bytes, dtype=np.uint8)

    def put_field(self, b, t, h, field, value):
        blk, slot = self._block_slot(b, t)
        w = self.w
        off = blk * w.cache_block_bytes + w.data_region_bytes + ((h * 3 + field) * w.kv_block_size + slot) * 2
        bits = f16_bits(value)
        self.cache[off] = bits & 0xFF
        self.cache[off + 1] = bits >> 8

    def inputs(self, q, ctx):
        return wl.Inputs(self.w, wl.round_bf16(q), self.cache, self.table,
                         np.asarray(ctx, dtype=np.int32), {"centroids": CENTROIDS})


# ---------------------------------------------------------------- fp16 fields
def test_f16_all_codes_match_numpy(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.f16_to_float64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_layout_by_hand():
    # BS 16, Hk 8: 16 slots * 8 heads * (64 + 64) code bytes, then 8 heads * 3 fields * 16 slots * 2 B
    a = oracle.cache_layout(8, 16, D, oracle.KV_TQ4)
    assert a["token_head_bytes"] == 128 and a["meta_offset_bytes"] == 16384 and a["cache_block_bytes"] == 17152
    w = wl.small(num_seqs=1, num_kv_heads=8, kv_block_size=16, ctx=(5,), kv_dtype=wl.KV_TQ4)
    assert w.cache_block_bytes == a["cache_block_bytes"] and w.data_region_bytes == a["data_region_bytes"]


# ---------------------------------------------------------------- closed forms from hand-written bytes
def _two_token_softmax(s0, s1, v0, v1):
    m = max(s0, s1)
    e0, e1 = math.exp(s0 - m), math.exp(s1 - m)
    return (e0 * v0 + e1 * v1) / (e0 + e1)


@pytest.mark.parametrize("BS", [16, 32])
def test_nibble_order_centroid_index_and_fields(oracle_mod, BS):
    """Token 0: every byte 0xBA (even dimensions code 10, odd code 11); token 1: every byte 0xAB.
    Q is 1 on even dimensions, 0 on odd ones, so s_t = scale * k_norm_t * 64 * c[code of the
    even dimensions]; V rows are constants given by v_zero alone (codes 0)."""
    w = _workload(ctx=(2,), BS=BS)
    hc = HandCache(w)
    knorm = (2.0, 3.0)
    vzero = (0.75, -1.25)
    for h in range(w.num_kv_heads):
        hc.put_row(0, 0, h, 0, [0xBA] * 64)
        hc.put_row(0, 1, h, 0, [0xAB] * 64)
        for t in range(2):
            hc.put_row(0, t, h, 1, [0x00] * 64)
            hc.put_field(0, t, h, 0, knorm[t])
            hc.put_field(0, t, h, 1, 0.5)          # v_scale (codes are 0: no effect)
            hc.put_field(0, t, h, 2, vzero[t])
    q = np.zeros((1, w.num_q_heads, D), np.float32)
    q[..., 0::2] = 1.0
    out = oh.run_oracle(hc.inputs(q, [2]))["out"]
    scale = 1.0 / math.sqrt(D)
    c = CENTROIDS.astype(np.float64)
    s0 = scale * knorm[0] * 64 * c[10]
    s1 = scale * knorm[1] * 64 * c[11]
    expect = _two_token_softmax(s0, s1, vzero[0], vzero[1])
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-12)


@pytest.mark.parametrize("d", [0, 1, 6, 7, 8, 31, 32, 63, 64, 100, 127])
def test_dimension_d_lives_in_byte_d_over_2(oracle_mod, d):
    """Q one-hot on dimension d: only the code of dimension d (byte d/2, nibble d%2) matters.
    Token 0 holds code 3 there, token 1 code 12; every other nibble of both rows is random."""
    w = _workload(ctx=(2,), Hk=1, seed=22)
    hc = HandCache(w)
    rng = np.random.default_rng(d)
    for t, code in ((0, 3), (1, 12)):
        row = rng.integers(0, 256, size=64).astype(np.uint8)
        byte = int(row[d // 2])
        byte = (byte & 0xF0) | code if d % 2 == 0 else (byte & 0x0F) | (code << 4)
        row[d // 2] = byte
        hc.put_row(0, t, 0, 0, row)
        hc.put_row(0, t, 0, 1, [0x00] * 64)
        hc.put_field(0, t, 0, 0, 4.0)
        hc.put_field(0, t, 0, 1, 1.0)
        hc.put_field(0, t, 0, 2, float(t))        # V row t is the constant t
    q = np.zeros((1, w.num_q_heads, D), np.float32)
    q[..., d] = 8.0
    out = oh.run_oracle(hc.inputs(q, [2]))["out"]
    scale = 1.0 / math.sqrt(D)
    c = CENTROIDS.astype(np.float64)
    expect = _two_token_softmax(scale * 8.0 * 4.0 * c[3], scale * 8.0 * 4.0 * c[12], 0.0, 1.0)
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-12)


def test_v_codes_by_hand(oracle_mod):
    """One-token context: the output is that token's V row, code(d) * v_scale + v_zero, with
    code(d) = d % 16 written as byte j = (2j % 16) | ((2j + 1) % 16) << 4."""
    w = _workload(ctx=(1,), Hk=2, seed=23)
    hc = HandCache(w)
    vbytes = [((2 * j) % 16) | (((2 * j + 1) % 16) << 4) for j in range(64)]
    for h, (vs, vz) in enumerate(((0.5, -1.0), (0.25, 2.0))):
        hc.put_row(0, 0, h, 0, [0x5A] * 64)
        hc.put_row(0, 0, h, 1, vbytes)
        hc.put_field(0, 0, h, 0, 1.0)
        hc.put_field(0, 0, h, 1, vs)
        hc.put_field(0, 0, h, 2, vz)
    q = np.random.default_rng(3).standard_normal((1, w.num_q_heads, D)).astype(np.float32)
    out = oh.run_oracle(hc.inputs(q, [1]))["out"][0].reshape(2, w.query_group_size, D)
    dims = np.arange(D) % 16
    assert np.array_equal(out[0], np.broadcast_to(dims * 0.5 - 1.0, out[0].shape))
    assert np.array_equal(out[1], np.broadcast_to(dims * 0.25 + 2.0, out[1].shape))


# ---------------------------------------------------------------- brute force on random codes
TQ_CASES = [
    dict(query_group_size=8, kv_block_size=16, ctx=(37, 5)),
    dict(query_group_size=6, kv_block_size=32, ctx=(1, 70)),
    dict(query_group_size=16, kv_block_size=16, ctx=(16, 33)),
]


def random_tq4_case(case, seed=5):
    """Random codes and fields, written through the generator's packer; also returns the float64
    K and V values computed from the codes directly (never from the cache bytes)."""
    w = wl.small(num_kv_heads=2, seed=seed, kv_dtype=wl.KV_TQ4, **case)
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((w.num_seqs, w.num_q_heads, D), dtype=np.float32)
    table = wl.draw_block_table(w, rng)
    cache = wl.empty_cache(w)
    Ks, Vs = [], []
    for b, n in enumerate(case["ctx"]):
        kc = rng.integers(0, 16, size=(n, 2, D)).astype(np.uint8)
        vc = rng.integers(0, 16, size=(n, 2, D)).astype(np.uint8)
        kn = wl.round_f16(rng.uniform(5, 15, size=(n, 2)))
        vs = wl.round_f16(rng.uniform(0.1, 0.6, size=(n, 2)))
        vz = wl.round_f16(rng.uniform(-3, 0, size=(n, 2)))
        wl.write_tq4_codes(w, cache, table[b], wl.pack_nibbles(kc), wl.pack_nibbles(vc), kn, vs, vz)
        Ks.append(oh.tq4_values(kc, centroids=CENTROIDS, k_norm_bits=kn))
        Vs.append(oh.tq4_values(vc, v_scale_bits=vs, v_zero_bits=vz))
    inp = wl.Inputs(w, wl.round_bf16(q), cache, table, np.asarray(case["ctx"], np.int32), {"centroids": CENTROIDS})
    return w, inp, Ks, Vs


@pytest.mark.parametrize("case", TQ_CASES)
def test_tq4_bruteforce_matches_sdpa(oracle_mod, case):
    w, inp, Ks, Vs = random_tq4_case(case)
    got = oh.run_oracle(inp)["out"]
    ref = oh.sdpa_reference(w, inp.query, Ks, Vs)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_tq4_partials_combine_to_unsplit(oracle_mod):
    w = wl.small(num_seqs=2, num_kv_heads=2, ctx=(700, 256), seed=24, kv_dtype=wl.KV_TQ4)
    inp = wl.generate(w)
    res = oh.run_oracle(inp, partials=True, G=1)
    for b in range(w.num_seqs):
        nv = -(-int(inp.context_lens[b]) // 256)
        m, l, o = res["part_m"][b, :, :nv], res["part_l"][b, :, :nv], res["part_o"][b, :, :nv]
        M = m.max(axis=1, keepdims=True)
        wgt = l * np.exp(m - M)
        comb = (wgt[..., None] * o).sum(axis=1) / wgt.sum(axis=1)[..., None]
        np.testing.assert_allclose(comb.reshape(w.num_q_heads, D), res["out"][b], rtol=0, atol=1e-12)


def test_tq4_block_relocation_is_bitwise_invariant(oracle_mod):
    w = wl.small(num_seqs=2, num_kv_heads=2, ctx=(100, 77), seed=25, extra_blocks=9, kv_dtype=wl.KV_TQ4)
    inp = wl.generate(w)
    base = oh.run_oracle(inp)["out"]
    perm = np.random.default_rng(0).permutation(w.num_cache_blocks)
    blocks = inp.cache.reshape(w.num_cache_blocks, w.cache_block_bytes)
    moved = np.empty_like(blocks)
    moved[perm] = blocks
    inp2 = wl.Inputs(w, inp.query, moved.reshape(-1), perm[inp.block_table].astype(np.int32), inp.context_lens,
                     inp.extra)
    assert np.array_equal(oh.run_oracle(inp2)["out"], base)


def test_generated_cache_decodes_to_the_quantised_rows(oracle_mod):
    """The generator's quantiser (not the oracle) against its own definition: a one-token context
    returns that token's dequantised V row, and it is within half a code step of the drawn row."""
    w = wl.small(num_seqs=1, num_kv_heads=2, ctx=(1,), seed=26, kv_dtype=wl.KV_TQ4)
    inp = wl.generate(w)
    rng = np.random.Generator(np.random.PCG64(w.seed))
    wl.draw_context_lens(w, rng)
    wl.draw_block_table(w, rng)
    rng.standard_normal((1, w.num_q_heads, D), dtype=np.float32)
    rng.standard_normal((1, w.num_kv_heads, D), dtype=np.float32)          # K
    V = rng.standard_normal((1, w.num_kv_heads, D), dtype=np.float32)
    out = oh.run_oracle(inp)["out"][0].reshape(2, w.query_group_size, D)
    step = (V.max(axis=-1) - V.min(axis=-1)) / 15.0
    for h in range(2):
        assert np.all(np.abs(out[h] - V[0, h]) <= 0.5 * step[0, h] + 2e-2)


def test_tq4_has_no_encoder(oracle_mod):
    w = wl.small(num_seqs=1, num_kv_heads=1, ctx=(3,), seed=27, kv_dtype=wl.KV_TQ4)
    inp = wl.generate(w)
    z = np.zeros((1, 1, D), np.uint16)
    with pytest.raises(ValueError):
        oracle.append_kv(oh.problem(w), inp.cache, z, z, inp.block_table, np.array([3], np.int32))


# ---------------------------------------------------------------- planted mistakes
SRC = os.path.join(os.path.dirname(oracle.__file__), "pda_oracle.c")
MUTATIONS = {
    "nibble_order": ("(row[d / 2] >> ((d % 2) * 4)) & 0xF", "(row[d / 2] >> ((1 - d % 2) * 4)) & 0xF"),
    "centroid_reversed": ("pr->centroids[code]", "pr->centroids[15 - code]"),
    "v_fields_swapped": ("(TQ4_V_SCALE * BS + slot) * 2", "(TQ4_V_ZERO * BS + slot) * 2"),
    "k_norm_from_v_scale": ("(TQ4_K_NORM * BS + slot) * 2", "(TQ4_V_SCALE * BS + slot) * 2"),
    "v_read_at_k_offset": ("(int64_t)which * (D / 2);", "0;"),
    "meta_head_stride": ("h * TQ4_FIELDS * BS * 2", "h * 2 * BS * 2"),
    "f16_bias_16": ("v = ldexp(1.0 + (double)m / 1024.0, e - 15);", "v = ldexp(1.0 + (double)m / 1024.0, e - 16);"),
    "f16_subnormal_exponent": ("v = ldexp((double)m / 1024.0, -14);", "v = ldexp((double)m / 1024.0, -15);"),
    "dim_byte_wraps_at_32": ("(row[d / 2] >> ((d % 2) * 4)) & 0xF", "(row[(d / 2) % 32] >> ((d % 2) * 4)) & 0xF"),
    "kv_head_offset_dropped": ("(slot * pr->num_kv_heads + h) * token_head_bytes", "slot * pr->num_kv_heads * token_head_bytes"),
}


def _battery(lib):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.f16_to_float64(bits, lib=lib)
    ref = bits.view(np.float16).astype(np.float64)
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    for case in TQ_CASES[:2]:
        w, inp, Ks, Vs = random_tq4_case(case)
        got = oh.run_oracle(inp, lib=lib)["out"]
        np.testing.assert_allclose(got, oh.sdpa_reference(w, inp.query, Ks, Vs), rtol=0, atol=1e-12)


def test_unmutated_copy_passes(tmp_path):
    c = tmp_path / "clean.c"
    so = tmp_path / "clean.so"
    c.write_text(open(SRC).read())
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", str(c), "-o", str(so),
                           "-lm"])
    _battery(oracle.load_library(str(so)))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_tq4_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor for {name} not found"
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(text.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", str(c), "-o", str(so),
                           "-lm"])
    with pytest.raises((AssertionError, ValueError)):
        _battery(oracle.load_library(str(so)))
