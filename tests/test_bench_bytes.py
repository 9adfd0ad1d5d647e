"""The roofline's numerator: the bytes a step must move, worked by hand for a small batch (no GPU).

Two sequences of 40 and 17 tokens, 2 KV heads, QG 8, 16-token blocks, 256-token partitions:
57 tokens per head, one partition each, 3 + 2 block-table entries.
"""
import types

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


def test_timing_mode_follows_the_kv_bytes_against_l2():
    # a step whose KV reads exceed L2 is timed back to back (no step finds the previous step's KV
    # in L2); a smaller one step by step after an L2 flush; the line's config says which
    expect = {"b1_hk1_qg8_bs16_ctx256": "flushed", "b8_hk8_qg8_bs16_ctx1-4096": "flushed",
              "b4_hk8_qg8_bs32_ctx32768_g5p32": "back_to_back", "b32_hk4_qg16_bs32_ctx2048-8192_kbias": "back_to_back",
              "b64_hk8_qg6_bs16_fp8_lognormal2048": "back_to_back", "b64_hk8_qg6_bs16_tq4_lognormal2048": "back_to_back"}
    for name, mode in expect.items():
        w = wl.WORKLOADS[name]
        # the workload's context lengths are the generator's first draw (no cache is built here)
        inp = types.SimpleNamespace(context_lens=wl.draw_context_lens(w, np.random.Generator(np.random.PCG64(w.seed))))
        W = 256 * max(1, w.tile_groups_per_partition)
        kv = bench.algorithmic_bytes(w, inp.context_lens, W)["kv"]
        assert (kv > bench.L2_BYTES) == (mode == "back_to_back"), name
        assert bench.timing_mode(w, inp, W) == mode, name
        note = bench.l2_note(mode, w, inp, W)
        assert ("back to back" in note) == (mode == "back_to_back")
        assert note.startswith("flushed") == (mode == "flushed")


def test_roofline_kernel_name_follows_the_variant():
    # the line's roofline names the kernel pda_decode launches for the plan (its ncu traffic entry
    # is looked up under that workload)
    import bench
    pda = types.SimpleNamespace(VARIANT_HEAD_WARPS=1, VARIANT_HEAD_GROUPS=2, VARIANT_ROW_HALVES=3)
    for v, want in ((1, "pda_partition_kernel"), (2, "pda_group_kernel"), (3, "pda_rows_kernel")):
        pda.kernel_variant = lambda p, v=v: v
        assert bench.kernel_name(pda, None) == want


def test_kernel_source_hash_covers_every_partition_kernel_source():
    # a change to any translation unit or header of the partition kernels must change the hash that
    # gates the committed DRAM traffic figures
    import glob
    import os
    import bench
    csrc = os.path.join(os.path.dirname(bench.__file__), "paged_kv_gqa_block_gb300", "csrc")
    kernel_files = {os.path.basename(f) for f in glob.glob(os.path.join(csrc, "*.cu*")) + glob.glob(os.path.join(csrc, "*.h"))}
    # the write side and the no-allocation wrapper launch no partition kernel of their own
    assert kernel_files - set(bench.PARTITION_KERNEL_SOURCES) <= {"pda_append.cu", "pda_noalloc.cu"}
