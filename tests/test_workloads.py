"""The seeded generator: determinism, layout, poison and the fp8 scale convention (no GPU)."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_block_gb300 import workloads as wl


def test_same_seed_same_bytes():
    w = wl.small(num_seqs=2, num_kv_heads=2, ctx=(33, 70), seed=21)
    a, b = wl.generate(w), wl.generate(w)
    for x, y in ((a.query, b.query), (a.cache, b.cache), (a.block_table, b.block_table), (a.context_lens, b.context_lens)):
        assert np.array_equal(x, y)


def test_token_bytes_sit_where_the_layout_says():
    """Token t of sequence b, KV head h: block table[b][t // BS], byte offset
    slot*Hk*2*D*e + h*2*D*e (K), + D*e (V) inside the block (data region [slot][head][K|V])."""
    w = wl.small(num_seqs=1, num_kv_heads=3, kv_block_size=32, ctx=(70,), seed=1)
    rng = np.random.default_rng(0)
    K = rng.standard_normal((70, 3, 128), dtype=np.float32)
    V = rng.standard_normal((70, 3, 128), dtype=np.float32)
    table = wl.draw_block_table(w, rng)
    cache = wl.empty_cache(w)
    wl.write_tokens(w, cache, table[0], K, V)
    t, h = 45, 2
    blk, slot = table[0, t // 32], t % 32
    off = blk * w.cache_block_bytes + slot * 3 * 512 + h * 512
    k = cache[off:off + 256].view(np.uint16)
    v = cache[off + 256:off + 512].view(np.uint16)
    assert np.array_equal(k, wl.round_bf16(K[t, h])) and np.array_equal(v, wl.round_bf16(V[t, h]))


def test_fp8_scale_layout_and_convention():
    w = wl.small(num_seqs=1, num_kv_heads=2, kv_block_size=16, ctx=(20,), kv_dtype=wl.KV_FP8_E4M3, seed=2)
    rng = np.random.default_rng(1)
    K = rng.standard_normal((20, 2, 128), dtype=np.float32)
    V = rng.standard_normal((20, 2, 128), dtype=np.float32)
    K[17, 1] = 0.0
    K[17, 1, 5] = -448.0           # absmax 448 -> scale exactly 1, codes are e4m3(x)
    V[17, 1] = 0.0                 # all-zero row -> scale 1, codes 0
    table = wl.draw_block_table(w, rng)
    cache = wl.empty_cache(w)
    wl.write_tokens(w, cache, table[0], K, V)
    t, h = 17, 1
    blk, slot = table[0, t // 16], t % 16
    base = blk * w.cache_block_bytes
    meta = base + w.data_region_bytes
    ks = cache[meta + ((h * 2 + 0) * 16 + slot) * 4: meta + ((h * 2 + 0) * 16 + slot) * 4 + 4].view(np.float32)[0]
    vs = cache[meta + ((h * 2 + 1) * 16 + slot) * 4: meta + ((h * 2 + 1) * 16 + slot) * 4 + 4].view(np.float32)[0]
    assert ks == 1.0 and vs == 1.0
    off = base + slot * 2 * 256 + h * 256
    kc = cache[off:off + 128]
    assert kc[5] == 0xFE and np.all(np.delete(kc, 5) == 0)       # -448 = S.1111.110
    assert np.all(cache[off + 128:off + 256] == 0)
    # another row: scale = absmax/448 in fp32 and |code * scale - x| within half an e4m3 step
    meta0 = table[0, 0] * w.cache_block_bytes + w.data_region_bytes       # token 3 lives in block table[0][0]
    ks2 = cache[meta0 + ((0 * 2 + 0) * 16 + 3) * 4: meta0 + ((0 * 2 + 0) * 16 + 3) * 4 + 4].view(np.float32)[0]
    assert ks2 == np.float32(np.abs(K[3, 0]).max() / np.float32(448.0))


def test_poison_outside_the_context():
    w = wl.small(num_seqs=1, num_kv_heads=1, kv_block_size=16, ctx=(20,), seed=3)
    inp = wl.generate(w)
    blk = inp.block_table[0, 1]
    blockbytes = inp.cache[blk * w.cache_block_bytes:(blk + 1) * w.cache_block_bytes].view(np.uint16).reshape(16, 2, 128)
    assert np.all(blockbytes[4:] == 0xFFFF)                 # slots 4..15 of the second block (tokens 20..31)
    assert not np.any(blockbytes[:4] == 0xFFFF)


def test_workload_shapes():
    w = wl.WORKLOADS["b1_hk1_qg8_bs16_ctx256"]
    inp = wl.generate(w)
    assert inp.block_table.shape == (1, 16) and len(set(inp.block_table.ravel())) == 16
    assert inp.block_table.max() < 64 and int(inp.context_lens[0]) == 256
    w2 = wl.WORKLOADS["b8_hk8_qg8_bs16_ctx1-4096"]
    rng = np.random.Generator(np.random.PCG64(w2.seed))
    ctx = wl.draw_context_lens(w2, rng)
    assert ctx.min() >= 1 and ctx.max() <= 4096
    w5 = wl.WORKLOADS["b64_hk8_qg6_bs16_fp8_lognormal2048"]
    ctx5 = wl.draw_context_lens(w5, np.random.Generator(np.random.PCG64(w5.seed)))
    assert ctx5.min() >= 16 and ctx5.max() <= 16384 and 1000 < np.median(ctx5) < 4000
    assert w5.cache_block_bytes == 16 * 8 * 256 + 8 * 2 * 16 * 4


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -3.14159], np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(wl.bf16_bits_to_f32(wl.round_bf16(x)), ref)
    assert wl.bf16_bits_to_f32(wl.round_bf16(np.float32(1.0 + 2 ** -8)))[()] == 1.0


# The input recipe of every workload, as the design notes state it: shapes, pool size, context
# range, tables drawn without replacement from the pool, the key-bias spread, seeds 1001..1006.
RECIPES = {
    # name: (B, Hk, QG, BS, MB, pool, kv dtype, ctx kind, lo, hi, k_bias_std, seed)
    "b1_hk1_qg8_bs16_ctx256": (1, 1, 8, 16, 16, 64, wl.KV_BF16, "fixed", 256, 256, 0.0, 1001),
    "b8_hk8_qg8_bs16_ctx1-4096": (8, 8, 8, 16, 256, 2048, wl.KV_BF16, "uniform", 1, 4096, 0.0, 1002),
    "b32_hk4_qg16_bs32_ctx2048-8192_kbias": (32, 4, 16, 32, 256, 8192, wl.KV_BF16, "uniform", 2048, 8192, 2.0, 1003),
    "b4_hk8_qg8_bs32_ctx32768_g5p32": (4, 8, 8, 32, 1280, 5120, wl.KV_BF16, "fixed", 32768, 32768, 0.0, 1004),
    "b64_hk8_qg6_bs16_fp8_lognormal2048": (64, 8, 6, 16, 1024, 65536, wl.KV_FP8_E4M3, "lognormal", 16, 16384, 0.0, 1005),
    "b64_hk8_qg6_bs16_tq4_lognormal2048": (64, 8, 6, 16, 1024, 65536, wl.KV_TQ4, "lognormal", 16, 16384, 0.0, 1006),
}


@pytest.mark.parametrize("name", sorted(RECIPES))
def test_every_workload_follows_its_recipe(name):
    B, Hk, QG, BS, MB, pool, kv, kind, lo, hi, kb, seed = RECIPES[name]
    w = wl.WORKLOADS[name]
    assert (w.num_seqs, w.num_kv_heads, w.query_group_size, w.kv_block_size, w.max_blocks_per_seq) == (B, Hk, QG, BS, MB)
    assert (w.num_cache_blocks, w.kv_dtype, w.ctx[0], w.k_bias_std, w.seed) == (pool, kv, kind, kb, seed)
    rng = np.random.Generator(np.random.PCG64(w.seed))    # the generator's own draw order: lengths, then tables
    ctx = wl.draw_context_lens(w, rng)
    table = wl.draw_block_table(w, rng)
    assert ctx.min() >= lo and ctx.max() <= hi and ctx.max() <= MB * BS
    assert table.shape == (B, MB) and table.min() >= 0 and table.max() < pool
    assert len(np.unique(table)) == table.size               # without replacement
    if kind == "uniform":                                     # both ends reachable, spread over the range
        assert ctx.max() - ctx.min() > (hi - lo) // 2
    if kind == "lognormal":                                   # median near exp(mu) = 2048, the clip respected
        assert 1200 < np.median(ctx) < 3500
