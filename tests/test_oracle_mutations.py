"""Plants plausible mistakes in a copy of the oracle (on the CPU) and checks that the pins
of test_oracle_pins.py catch every one of them."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh
from tests.test_oracle_pins import CASES, _random_case, check_partials_by_brute_force

SRC = os.path.join(os.path.dirname(oracle.__file__), "pda_oracle.c")

MUTATIONS = {
    "slot_off_by_one": ("const int64_t slot = t % BS;", "const int64_t slot = (t + 1) % BS;"),
    "table_entry_per_16_tokens": ("block_table[b * MB + t / BS]", "block_table[b * MB + t / 16]"),
    "softmax_scale_dropped": ("s[t] = pr->softmax_scale * dot;", "s[t] = dot;"),
    "k_and_v_swapped": ("decode_row(pr, cache, blk, slot, h, 0, K + t * D);",
                        "decode_row(pr, cache, blk, slot, h, 1, K + t * D);"),
    "exponent_sign": ("const double e = exp(s[t] - m);", "const double e = exp(m - s[t]);"),
    "kv_head_offset_dropped": ("slot * pr->num_kv_heads * token_head_bytes + h * token_head_bytes",
                               "slot * pr->num_kv_heads * token_head_bytes"),
    "e4m3_bias_8": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "gqa_heads_interleaved": ("const int64_t qh = h * QG + r;", "const int64_t qh = r * Hk + h;"),
    "partition_starts_one_late": ("const int64_t lo = p * W,", "const int64_t lo = p * W + 1,"),
    "partial_sum_without_its_max": ("const double e = exp(s[t] - mp);", "const double e = exp(s[t]);"),
    "v_scale_read_from_k_field": ("((h * 2 + which) * pr->kv_block_size + slot) * 4",
                                  "((h * 2 + 0) * pr->kv_block_size + slot) * 4"),
}


def _battery(lib):
    for case in (CASES[0], CASES[1], CASES[3], CASES[4]):
        w, q, K, V, table = _random_case(case)
        inp = oh.build_from_values(w, q, K, V, table)
        got = oh.run_oracle(inp, lib=lib)["out"]
        ref = oh.sdpa_reference(w, inp.query, [oh.stored_values(w, k) for k in K], [oh.stored_values(w, v) for v in V])
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    case = dict(kv_dtype=wl.KV_BF16, query_group_size=8, kv_block_size=16, ctx=(700, 256))
    w, q, K, V, table = _random_case(case, seed=11)
    inp = oh.build_from_values(w, q, K, V, table)
    res = oh.run_oracle(inp, partials=True, G=1, lib=lib)
    check_partials_by_brute_force(w, inp, res, [oh.stored_values(w, k) for k in K],
                                  [oh.stored_values(w, v) for v in V], 256)
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_float64(codes, lib=lib)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def _compile(tmp_path, src_text, tag):
    c = tmp_path / f"{tag}.c"
    so = tmp_path / f"{tag}.so"
    c.write_text(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", str(c), "-o", str(so), "-lm"])
    return oracle.load_library(str(so))


def test_unmutated_copy_passes(tmp_path):
    _battery(_compile(tmp_path, open(SRC).read(), "clean"))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique"
    lib = _compile(tmp_path, text.replace(old, new), name)
    with pytest.raises((AssertionError, ValueError)):
        _battery(lib)
