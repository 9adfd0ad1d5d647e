"""The roofline's numerator: the bytes a step must move, worked by hand for a small batch (no GPU).

Two sequences of 40 and 17 tokens, 2 KV heads, QG 8, 16-token blocks, 256-token partitions:
57 tokens per head, one partition each, 3 + 2 block-table entries.
"""
import numpy as np
import pytest

import bench
from paged_kv_gqa_block_gb300 import workloads as wl

# KV bytes per (token, KV head): K and V of 128 dimensions, plus the format's per-token fields
PER_TOKEN_HEAD = {wl.KV_BF16: 2 * 128 * 2, wl.KV_FP8_E4M3: 2 * 128 + 2 * 4, wl.KV_TQ4: 64 + 64 + 3 * 2}


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_FP8_E4M3, wl.KV_TQ4])
def test_algorithmic_bytes_by_hand(kv):
    w = wl.small(num_seqs=2, num_kv_heads=2, query_group_size=8, kv_block_size=16, ctx=(40, 17), kv_dtype=kv)
    ab = bench.algorithmic_bytes(w, np.array([40, 17]), 256)
    kv_bytes = 57 * 2 * PER_TOKEN_HEAD[kv]
    q = 2 * 2 * 8 * 128 * 2                  # every Q row of the batch, bf16
    table = (3 + 2) * 4                      # entries of each sequence, read once for all its heads
    lengths = 2 * 4
    partials = 2 * 2 * 8 * (128 * 4 + 8)     # one partition per (sequence, head): o_p, m_p, l_p
    out = 2 * 2 * 8 * 128 * 2
    assert ab["kv"] == kv_bytes
    assert ab["decode"] == kv_bytes + q + table + lengths + partials
    assert ab["reduce"] == partials + out   # the reduce reads the partials and writes the output
    assert ab["tokens"] == 57 and ab["units"] == 4
