"""GPU robustness checks through the C ABI: the bounded-wait error path, cache blocks past 4 GiB,
guard words around every buffer the kernels write, and inputs and output in pinned host memory.

The timeout test makes the kernel's own waits run out (a 1 ns limit is shorter than any tile's
copy latency); nothing faults or hangs: a warp that gives up still waits, with the default 1 s
limit, for the copies it has in flight before it leaves, and the next call on the same context
must be correct.
"""
import numpy as np
import pytest
import torch

from paged_kv_gqa_block_gb300 import workloads as wl
from tests import oracle_helpers as oh
from tests.gpu_helpers import KV_VARIANTS, SENTINEL_BITS, decode_any, plan_for, run_gpu, to_device

pytestmark = pytest.mark.gpu

TOL = {wl.KV_BF16: 2e-3, wl.KV_FP8_E4M3: 1e-2, wl.KV_TQ4: 1e-2}


@pytest.fixture(scope="module")
def pda():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_block_gb300 as pda
    return pda


def _step(pda, p, d, nb, err=None, out_dtype=torch.float32, ws=None):
    B, Hq = p.num_seqs, p.num_kv_heads * p.query_group_size
    ws = ws or pda.workspace(p, "cuda")
    out = torch.empty((B, Hq, 128), dtype=out_dtype, device="cuda")
    if p.kv_dtype == wl.KV_TQ4:
        pda.decode_tq4(p, d["query"], d["cache"], nb, d["centroids"], d["block_table"], d["context_lens"],
                       ws["partial_out"], ws["exp_sums"], ws["max_logits"], err_word=err)
    else:
        pda.decode(p, d["query"], d["cache"], nb, d["block_table"], d["context_lens"], ws["partial_out"],
                   ws["exp_sums"], ws["max_logits"], err_word=err)
    pda.reduce(p, d["context_lens"], ws["partial_out"], ws["exp_sums"], ws["max_logits"], out, err_word=err)
    torch.cuda.synchronize()
    return out


# (not TQ4: its warps are bound by their own arithmetic, every 2 KB tile has landed before its
# wait begins, so even a 1 ns limit is not reached; the timeout path itself does not depend on
# the cache format)
@pytest.mark.parametrize("kv,variant", [(wl.KV_BF16, 0), (wl.KV_FP8_E4M3, 1), (wl.KV_FP8_E4M3, 2)])
def test_wait_timeout_sets_the_error_bit_and_the_next_call_is_correct(oracle_mod, pda, kv, variant):
    # a step big enough to load HBM (every copy then takes microseconds), each wait limited to 1 ns
    w = wl.small(num_seqs=16, num_kv_heads=8, ctx=(8192,) * 16, kv_dtype=kv, seed=61, extra_blocks=0)
    inp = wl.generate(w)
    d = to_device(inp)
    p = pda.plan(w.num_seqs, w.num_kv_heads, w.query_group_size, w.kv_block_size, w.max_blocks_per_seq,
                 kv_dtype=kv, wait_timeout_ns=1, kernel_variant=variant)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _step(pda, p, d, w.num_cache_blocks, err)
    assert int(err.item()) & pda.ERRW_PIPELINE_TIMEOUT
    assert torch.zeros(1, device="cuda").add_(1).item() == 1.0   # the context is usable
    res = run_gpu(inp, d=d, variant=variant)   # default limit, same inputs: no error bit, and correct
    assert res["err"] == 0
    units = [0, 37, 127]
    ref = oh.run_oracle(inp, units=units)["out"]
    for u in units:
        b, h = divmod(u, w.num_kv_heads)
        rows = slice(h * w.query_group_size, (h + 1) * w.query_group_size)
        assert np.abs(res["out"][b, rows] - ref[b, rows]).max() <= TOL[kv]


def test_cache_blocks_past_4_gib(oracle_mod, pda):
    # the referenced blocks sit at the end of a pool of more than 4 GiB, so their byte offsets
    # need 64 bits; the oracle reads the same blocks from the compact pool
    w = wl.small(num_seqs=2, num_kv_heads=2, ctx=(700, 300), seed=62, extra_blocks=3)
    inp = wl.generate(w)
    cbb = w.cache_block_bytes
    offset = ((4 << 30) + (256 << 20)) // cbb
    nb = offset + w.num_cache_blocks
    assert nb * cbb > (1 << 32) and nb < (1 << 31)
    d = to_device(inp)
    big = torch.full((nb * cbb,), 0xFF, dtype=torch.uint8, device="cuda")
    big[offset * cbb:] = d["cache"]
    d["cache"] = big
    d["block_table"] = d["block_table"] + offset
    p = plan_for(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _step(pda, p, d, nb, err)
    assert int(err.item()) == 0
    ref = oh.run_oracle(inp)["out"]
    assert np.abs(out.cpu().numpy() - ref).max() <= 2e-3
    del big


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_guard_words_around_every_written_buffer_stay_intact(pda, kv, variant):
    w = wl.small(num_seqs=3, num_kv_heads=8, ctx=(900, 17, 256), kv_dtype=kv, seed=63)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w, variant=variant)
    G = 64   # guard floats before and after each buffer (256 bytes keep the 16-byte alignment)

    def guarded(n):
        buf = torch.full((n + 2 * G,), SENTINEL_BITS, dtype=torch.int32, device="cuda").view(torch.float32)
        return buf, buf[G:G + n]

    (so, ss) = pda.partial_shapes(p)
    po_buf, po = guarded(int(np.prod(so)))
    es_buf, es = guarded(int(np.prod(ss)))
    ml_buf, ml = guarded(int(np.prod(ss)))
    out_n = w.num_seqs * w.num_q_heads * 128
    out_buf, out = guarded(out_n)
    err_buf = torch.full((3,), SENTINEL_BITS, dtype=torch.int32, device="cuda")
    err_buf[1] = 0
    decode_any(p, w, d, {"partial_out": po, "exp_sums": es, "max_logits": ml}, err_buf[1:2])
    pda.reduce(p, d["context_lens"], po, es, ml, out.view(w.num_seqs, w.num_q_heads, 128), err_word=err_buf[1:2])
    torch.cuda.synchronize()
    for name, buf, n in (("partial_out", po_buf, po.numel()), ("exp_sums", es_buf, es.numel()),
                         ("max_logits", ml_buf, ml.numel()), ("out", out_buf, out_n)):
        bits = buf.view(torch.int32).cpu().numpy()
        assert (bits[:G] == SENTINEL_BITS).all() and (bits[G + n:] == SENTINEL_BITS).all(), name
    assert int(err_buf[1].item()) == 0
    assert int(err_buf[0].item()) == SENTINEL_BITS and int(err_buf[2].item()) == SENTINEL_BITS
    # inputs are read only
    assert torch.equal(d["cache"], torch.from_numpy(inp.cache).to("cuda"))


@pytest.mark.parametrize("kv,variant", KV_VARIANTS)
def test_inputs_and_output_in_pinned_host_memory(pda, kv, variant):
    # query, block table and context lengths read by the kernels across the host link, the output
    # written back the same way: the same bits as with every buffer on the device
    w = wl.small(num_seqs=4, num_kv_heads=8, ctx=(700, 1, 300, 2000), kv_dtype=kv, seed=64)
    inp = wl.generate(w)
    d = to_device(inp)
    p = plan_for(w, variant=variant)
    ref = _step(pda, p, d, w.num_cache_blocks).cpu()
    h = {"query": d["query"].cpu().pin_memory(), "block_table": d["block_table"].cpu().pin_memory(),
         "context_lens": d["context_lens"].cpu().pin_memory(), "cache": d["cache"], "centroids": d.get("centroids")}
    ws = pda.workspace(p, "cuda")
    out = torch.empty(ref.shape, dtype=torch.float32).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    decode_any(p, w, h, ws, err)
    pda.reduce(p, h["context_lens"], ws["partial_out"], ws["exp_sums"], ws["max_logits"], out, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, ref)
