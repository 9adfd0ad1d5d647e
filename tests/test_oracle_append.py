"""Pins of the oracle's write side (no GPU): the e4m3 encoder and the append of one token."""
import numpy as np
import torch

import oracle
from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh


def test_encode_round_trips_every_finite_code(oracle_mod):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_to_float64(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_matches_torch_in_range(oracle_mod):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4000) * 40, rng.uniform(-448, 448, 2000),
                        rng.standard_normal(2000) * 1e-3]).astype(np.float32)
    # midpoints between neighbouring codes exercise ties to even
    pos = np.sort(oracle.e4m3_to_float64(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_encode_saturates_and_keeps_signed_zero(oracle_mod):
    got = oracle.e4m3_encode(np.array([500.0, -1e6, 448.0, 460.0, -0.0, 0.0, np.nan], np.float32))
    assert list(got) == [0x7E, 0xFE, 0x7E, 0x7E, 0x80, 0x00, 0x7F]


def test_append_writes_what_the_generator_writes(oracle_mod):
    """Appending token n of each sequence through the oracle gives the same bytes as generating a
    context of n + 1 tokens (the generator's quantiser is torch's float8 cast, a library routine)."""
    for kv in (wl.KV_BF16, wl.KV_FP8_E4M3):
        w = wl.small(num_seqs=3, num_kv_heads=2, kv_block_size=32, ctx=(5, 32, 70), kv_dtype=kv, seed=4)
        rng = np.random.default_rng(1)
        table = wl.draw_block_table(w, rng)
        # values already on the bf16 grid: the appended inputs are bf16
        K = [wl.bf16_bits_to_f32(wl.round_bf16(rng.standard_normal((c + 1, 2, 128)).astype(np.float32)))
             for c in (5, 32, 70)]
        V = [wl.bf16_bits_to_f32(wl.round_bf16(rng.standard_normal((c + 1, 2, 128)).astype(np.float32)))
             for c in (5, 32, 70)]
        q = np.zeros((3, w.num_q_heads, 128), np.float32)
        before = oh.build_from_values(w, q, [k[:-1] for k in K], [v[:-1] for v in V], table)
        after = oh.build_from_values(w, q, K, V, table)
        k_new = np.stack([wl.round_bf16(k[-1]) for k in K])
        v_new = np.stack([wl.round_bf16(v[-1]) for v in V])
        got = oracle.append_kv(oh.problem(w), before.cache, k_new, v_new, table, np.array([5, 32, 70], np.int32))
        assert np.array_equal(got, after.cache)


def test_append_skips_negative_positions_and_rejects_bad_ones(oracle_mod):
    w = wl.small(num_seqs=2, num_kv_heads=1, ctx=(3, 3), seed=5)
    inp = wl.generate(w)
    kn = np.zeros((2, 1, 128), np.uint16)
    same = oracle.append_kv(oh.problem(w), inp.cache, kn, kn, inp.block_table, np.array([-1, -5], np.int32))
    assert np.array_equal(same, inp.cache)
    import pytest
    with pytest.raises(ValueError):
        oracle.append_kv(oh.problem(w), inp.cache, kn, kn, inp.block_table,
                         np.array([w.max_blocks_per_seq * w.kv_block_size, 0], np.int32))
