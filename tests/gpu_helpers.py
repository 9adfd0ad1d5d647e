"""Runs the CUDA path (through the C ABI) on generated inputs and hands back numpy arrays."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_gqa_block_gb300 import workloads as wl

SENTINEL_BITS = 0x7FBADBAD   # a NaN payload the kernels never produce


def to_device(inp: wl.Inputs, dev="cuda"):
    d = {
        "query": torch.from_numpy(inp.query.view(np.int16)).to(dev).view(torch.bfloat16),
        "cache": torch.from_numpy(inp.cache).to(dev),
        "block_table": torch.from_numpy(np.ascontiguousarray(inp.block_table)).to(dev),
        "context_lens": torch.from_numpy(np.ascontiguousarray(inp.context_lens)).to(dev),
    }
    if "centroids" in inp.extra:
        d["centroids"] = torch.from_numpy(np.ascontiguousarray(inp.extra["centroids"], dtype=np.float32)).to(dev)
    return d


def decode_any(p, w, d, ws, err=None):
    """The partition pass for any cache format (pda_decode_tq4 for TQ4, pda_decode otherwise)."""
    import paged_kv_gqa_block_gb300 as pda
    if w.kv_dtype == wl.KV_TQ4:
        pda.decode_tq4(p, d["query"], d["cache"], w.num_cache_blocks, d["centroids"], d["block_table"],
                       d["context_lens"], ws["partial_out"], ws["exp_sums"], ws["max_logits"], err_word=err)
    else:
        pda.decode(p, d["query"], d["cache"], w.num_cache_blocks, d["block_table"], d["context_lens"],
                   ws["partial_out"], ws["exp_sums"], ws["max_logits"], err_word=err)


def plan_for(w: wl.Workload, G=None, variant=0):
    """The plan of a workload; `variant` selects the partition kernel's layout (0 = automatic,
    1 = head warps, 2 = head groups, fp8 only)."""
    import paged_kv_gqa_block_gb300 as pda
    return pda.plan(w.num_seqs, w.num_kv_heads, w.query_group_size, w.kv_block_size, w.max_blocks_per_seq,
                    w.tile_groups_per_partition if G is None else G, w.max_partitions, w.kv_dtype, w.softmax_scale,
                    kernel_variant=variant)


def sentinel_ws(p, dev="cuda"):
    import paged_kv_gqa_block_gb300 as pda
    so, ss = pda.partial_shapes(p)
    mk = lambda s: torch.full(s, SENTINEL_BITS, dtype=torch.int32, device=dev).view(torch.float32)
    return {"partial_out": mk(so), "exp_sums": mk(ss), "max_logits": mk(ss)}


def run_gpu(inp: wl.Inputs, G=None, dev="cuda", d=None, variant=0):
    """Partition pass + reduce (fp32 and bf16 outputs).  Returns numpy arrays and the error word."""
    import paged_kv_gqa_block_gb300 as pda
    w = inp.workload
    p = plan_for(w, G, variant)
    d = d or to_device(inp, dev)
    ws = sentinel_ws(p, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    decode_any(p, w, d, ws, err)
    out32 = torch.empty((w.num_seqs, w.num_q_heads, 128), dtype=torch.float32, device=dev)
    out16 = torch.empty((w.num_seqs, w.num_q_heads, 128), dtype=torch.bfloat16, device=dev)
    pda.reduce(p, d["context_lens"], ws["partial_out"], ws["exp_sums"], ws["max_logits"], out32, err_word=err)
    pda.reduce(p, d["context_lens"], ws["partial_out"], ws["exp_sums"], ws["max_logits"], out16, err_word=err)
    torch.cuda.synchronize()
    return {
        "plan": p,
        "out": out32.cpu().numpy().astype(np.float64),
        "out_bf16": out16.float().cpu().numpy().astype(np.float64),
        "part_o": ws["partial_out"].cpu().numpy(),
        "part_m": ws["max_logits"].cpu().numpy(),
        "part_l": ws["exp_sums"].cpu().numpy(),
        "err": int(err.item()),
    }


def is_sentinel(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.int32) == SENTINEL_BITS


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 8)


# (KV format, partition-kernel variant) pairs that cover every kernel: fp8 runs on head warps and
# on head groups; bf16 and TQ4 have head warps only
KV_VARIANTS = [(wl.KV_BF16, 0), (wl.KV_FP8_E4M3, 1), (wl.KV_FP8_E4M3, 2), (wl.KV_TQ4, 0)]
