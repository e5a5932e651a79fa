"""GPU parity of the fp8 KV-cache path (decode_attn_paged_fp8 / _ring_fp8) against
the fp64 oracle over the same e4m3 codes and scales: attention within
4e-3 + 1e-2 |oracle|; the quantised append (K row, transposed V column, both
scales) bit-exact, every other byte of the 2176-byte blocks untouched; dead
cells hold NaN codes and NaN scales."""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
from cases import make_case, paged_identity, shuffle_pages
from paged_decode_attention_kv_gb300 import workloads as wl
from test_gpu_decode import DEV, assert_close, dev, dev_bits

pytestmark = pytest.mark.gpu


def pre(c):
    return np.maximum(c.lens - 1, 0)


def to_dev(cache):
    return torch.from_numpy(cache.blocks.copy()).to(DEV)


def from_dev(t):
    return oracle.Fp8Cache(t.cpu().numpy())


def assert_blocks_equal(got, want):
    """Bit-exact: every byte of every block (codes, and the scales' bit patterns)."""
    np.testing.assert_array_equal(got.blocks, want.blocks)


def check_paged_fp8(c, window, seed, fused=True):
    kp, vp, bt = paged_identity(c, c.lens if not fused else pre(c))
    kp, vp, bt = shuffle_pages(kp, vp, bt, seed, spare=4)
    blank = oracle.Fp8Cache.empty_paged(kp.shape[0], c.Hkv, 16, c.D)
    cache = oracle.scatter_fp8(c.hist_k, c.hist_v, c.lens if not fused else pre(c), blank,
                               block_table=bt)
    kv = to_dev(cache)
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_fp8(dev_bits(c.q), dev_bits(c.k_new) if fused else None,
                             dev_bits(c.v_new) if fused else None, kv, dev(bt),
                             dev(c.lens), dev(c.sinks), window, c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_paged_fp8(c.q, c.k_new if fused else None, c.v_new if fused else None,
                                  cache, bt, c.lens, c.sinks, window, c.scale)
    assert_close(out.double().cpu().numpy(), ref, f"paged fp8 window={window}")
    want = oracle.kv_append_fp8(c.k_new, c.v_new, cache, c.lens, block_table=bt) if fused else cache
    assert_blocks_equal(from_dev(kv), want)


EDGE = [1, 2, 15, 16, 17, 31, 33, 100, 257, 1000]


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (8, 8), (16, 1), (32, 4)])
@pytest.mark.parametrize("window", [0, 7, 100])
def test_paged_fp8_matches_oracle(Hq, Hkv, window):
    c = make_case(700 + Hq + Hkv + window, len(EDGE), Hq, Hkv, 64, EDGE)
    check_paged_fp8(c, window, seed=window + 1)


def test_paged_fp8_without_append_and_long_sequences():
    c = make_case(720, 3, 64, 8, 64, [40, 5000, 12000])
    check_paged_fp8(c, 0, seed=3, fused=False)
    check_paged_fp8(c, 0, seed=4, fused=True)


@pytest.mark.parametrize("W", [16, 128])
def test_ring_fp8_matches_oracle(W):
    lens = [1, 15, 16, 17, W - 1, W, W + 1, 3 * W + 5, 0]
    c = make_case(730 + W, len(lens), 64, 8, 64, lens)
    blank = oracle.Fp8Cache.empty_ring(c.B, c.Hkv, W, c.D)
    cache = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c), blank, window=W)
    kv = to_dev(cache)
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_ring_fp8(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), kv,
                            dev(c.lens), dev(c.sinks), c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_ring_fp8(c.q, c.k_new, c.v_new, cache, c.lens, c.sinks, W, c.scale)
    assert_close(out.double().cpu().numpy(), ref, f"ring fp8 W={W}")
    want = oracle.kv_append_fp8(c.k_new, c.v_new, cache, c.lens, window=W)
    assert_blocks_equal(from_dev(kv), want)


def test_paged_fp8_inactive_slots():
    c = make_case(740, 6, 64, 8, 64, [0, 50, 0, 0, 17, 0])
    check_paged_fp8(c, 0, seed=5)
    check_paged_fp8(c, 128, seed=6)
    c0 = make_case(741, 3, 64, 8, 64, [0, 0, 0])
    check_paged_fp8(c0, 0, seed=7)


def test_paged_fp8_many_segments_across_ctas():
    rng = np.random.default_rng(9)
    lens = list(rng.integers(1, 70, size=200)) + [3000, 700, 1]
    c = make_case(742, len(lens), 64, 8, 64, lens)
    check_paged_fp8(c, 0, seed=8)


@pytest.mark.parametrize("name", ["b64", "long1"])
def test_full_size_fp8(name):
    """Benchmark-size fp8 pools of random codes and scales; every output row against the
    oracle, the appended rows and scales bit-exact."""
    cfg = wl.config(name)
    lens = wl.seq_lens(name)
    gen = wl.cpu_generator(cfg["seed"])
    vgen = torch.Generator(device=DEV)
    vgen.manual_seed(cfg["seed"])
    B, Hq, Hkv, D, P = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["page_size"]
    inp = wl.draw_decode_inputs(B, Hq, Hkv, D, lens, gen)
    npages = wl.pool_size(name, lens)
    bt = wl.draw_block_table(lens, P, npages, wl.max_pages_per_seq(name, lens), gen)
    pool = wl.draw_fp8_paged_pool(npages, Hkv, P, D, vgen, device=DEV)
    before = from_dev(pool)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
    sl = np.asarray(lens, np.int32)
    da.decode_attn_paged_fp8(dev(inp.q), dev(inp.k_new), dev(inp.v_new), pool, dev(bt), dev(sl),
                             dev(inp.sinks), 0, inp.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_paged_fp8(wl.bits(inp.q), wl.bits(inp.k_new), wl.bits(inp.v_new), before,
                                  bt.numpy(), sl, inp.sinks.numpy(), 0, inp.scale)
    assert_close(out.double().cpu().numpy(), ref, f"{name} paged fp8")
    want = oracle.kv_append_fp8(wl.bits(inp.k_new), wl.bits(inp.v_new), before, sl,
                                block_table=bt.numpy())
    assert_blocks_equal(from_dev(pool), want)


@pytest.mark.parametrize("max_seq_len", [None, 1 << 20])
def test_paged_fp8_grid_choice(max_seq_len):
    """The host sizes the fp8 grid (one or two CTAs per SM) from an upper bound of the
    call's tiles, which grows with max_seq_len; a tight and a very loose bound give the
    two grids on the same sequences."""
    lens = [1000, 17, 0, 512, 999, 1, 300, 64, 16, 800, 33, 700, 5, 950, 128, 640]
    c = make_case(746, len(lens), 64, 8, 64, lens)
    kp, vp, bt = paged_identity(c, pre(c))
    kp, vp, bt = shuffle_pages(kp, vp, bt, 11, spare=4)
    width = bt.shape[1] if max_seq_len is None else max_seq_len // 16
    bt = np.pad(bt, ((0, 0), (0, width - bt.shape[1])), constant_values=-1)
    cache = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c),
                               oracle.Fp8Cache.empty_paged(kp.shape[0], c.Hkv, 16, c.D), block_table=bt)
    kv = to_dev(cache)
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_fp8(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), kv, dev(bt),
                             dev(c.lens), dev(c.sinks), 0, c.scale, out,
                             max_seq_len=max(lens) if max_seq_len is None else max_seq_len)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_paged_fp8(c.q, c.k_new, c.v_new, cache, bt, c.lens, c.sinks, 0, c.scale)
    assert_close(out.double().cpu().numpy(), ref, f"paged fp8 max_seq_len={max_seq_len}")
    assert_blocks_equal(from_dev(kv), oracle.kv_append_fp8(c.k_new, c.v_new, cache, c.lens, block_table=bt))


@pytest.mark.parametrize("W", [256, 512])
def test_ring_fp8_many_slots(W):
    """64 slots of 8 KV heads: at W = 512 the ring call is large enough for the two-CTA grid."""
    rng = np.random.default_rng(W)
    lens = [0 if rng.random() < 0.1 else int(rng.integers(1, 3 * W)) for _ in range(64)]
    lens[:4] = [W - 1, W, W + 1, 1]
    c = make_case(747 + W, len(lens), 64, 8, 64, lens)
    cache = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c), oracle.Fp8Cache.empty_ring(c.B, c.Hkv, W, c.D),
                               window=W)
    kv = to_dev(cache)
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_ring_fp8(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), kv,
                            dev(c.lens), dev(c.sinks), c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_ring_fp8(c.q, c.k_new, c.v_new, cache, c.lens, c.sinks, W, c.scale)
    assert_close(out.double().cpu().numpy(), ref, f"ring fp8 many slots W={W}")
    assert_blocks_equal(from_dev(kv), oracle.kv_append_fp8(c.k_new, c.v_new, cache, c.lens, window=W))


def test_paged_fp8_maximum_batch():
    rng = np.random.default_rng(9)
    lens = [0 if rng.random() < 0.25 else int(rng.integers(1, 48)) for _ in range(1024)]
    lens[3] = 700
    c = make_case(743, len(lens), 16, 2, 64, lens)
    check_paged_fp8(c, 0, seed=9)


def test_fp8_cuda_graph_capture_and_replay():
    """The fp8 paged and ring calls captured once and replayed after lengths, block table
    and inputs changed in place."""
    lens = [30, 500, 17, 0, 260]
    c = make_case(744, len(lens), 64, 8, 64, lens)
    kp, vp, bt = paged_identity(c, pre(c))
    kp, vp, bt = shuffle_pages(kp, vp, bt, 3, spare=4)
    cache = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c),
                               oracle.Fp8Cache.empty_paged(kp.shape[0], c.Hkv, 16, c.D), block_table=bt)
    ring = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c), oracle.Fp8Cache.empty_ring(c.B, c.Hkv, 128, c.D),
                              window=128)
    kv, rv = to_dev(cache), to_dev(ring)
    q, kn, vn, sl, sk, btd = dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), dev(c.lens), dev(c.sinks), dev(bt)
    out_p = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=DEV)
    out_r = torch.empty_like(out_p)
    da.decode_attn_reserve(da.decode_attn_workspace_bytes(c.B, c.Hq, c.Hkv, c.D))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        da.decode_attn_paged_fp8(q, kn, vn, kv.clone(), btd, sl, sk, 0, c.scale, out_p)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            da.decode_attn_paged_fp8(q, kn, vn, kv, btd, sl, sk, 0, c.scale, out_p)
            da.decode_attn_ring_fp8(q, kn, vn, rv, sl, sk, c.scale, out_r)
    torch.cuda.synchronize()
    lens2 = [31, 100, 0, 45, 261]
    c2 = make_case(745, len(lens2), 64, 8, 64, lens2)
    kp2, vp2, bt2 = paged_identity(c2, pre(c2))
    kp2, vp2, bt2 = shuffle_pages(kp2, vp2, bt2, 3, spare=kp.shape[0] - kp2.shape[0])  # captured pool size
    assert kp2.shape == kp.shape and bt2.shape[0] == bt.shape[0]
    bt2 = np.pad(bt2, ((0, 0), (0, bt.shape[1] - bt2.shape[1])), constant_values=-1)
    cache2 = oracle.scatter_fp8(c2.hist_k, c2.hist_v, pre(c2),
                                oracle.Fp8Cache.empty_paged(kp.shape[0], c.Hkv, 16, c.D), block_table=bt2)
    ring2 = oracle.scatter_fp8(c2.hist_k, c2.hist_v, pre(c2), oracle.Fp8Cache.empty_ring(c.B, c.Hkv, 128, c.D),
                               window=128)
    kv.copy_(to_dev(cache2)); rv.copy_(to_dev(ring2))
    for dst, src in ((q, c2.q), (kn, c2.k_new), (vn, c2.v_new)):
        dst.copy_(dev_bits(src))
    sl.copy_(dev(c2.lens)); btd.copy_(dev(bt2)); sk.copy_(dev(c2.sinks))
    g.replay()
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref_p = oracle.decode_paged_fp8(c2.q, c2.k_new, c2.v_new, cache2, bt2, c2.lens, c2.sinks, 0, c.scale)
    ref_r = oracle.decode_ring_fp8(c2.q, c2.k_new, c2.v_new, ring2, c2.lens, c2.sinks, 128, c.scale)
    assert_close(out_p.double().cpu().numpy(), ref_p, "graph fp8 paged")
    assert_close(out_r.double().cpu().numpy(), ref_r, "graph fp8 ring")
    assert_blocks_equal(from_dev(kv), oracle.kv_append_fp8(c2.k_new, c2.v_new, cache2, c2.lens, block_table=bt2))
    assert_blocks_equal(from_dev(rv), oracle.kv_append_fp8(c2.k_new, c2.v_new, ring2, c2.lens, window=128))


# ---------------------------------------------------------------- fp8 cache with the fused RoPE
def _tables(maxpos):
    cs, sn = wl.rope_tables(maxpos, 64)
    return cs, sn


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (64, 4), (8, 8)])
@pytest.mark.parametrize("window", [0, 100])
def test_paged_fp8_rope_matches_oracle(Hq, Hkv, window):
    """q and the new key rotated to position L - 1, the key rotated before it is quantised;
    the appended block bytes bit-exact against quantise(rope_k(k_new))."""
    c = make_case(760 + Hq + Hkv + window, len(EDGE), Hq, Hkv, 64, EDGE)
    kp, vp, bt = shuffle_pages(*paged_identity(c, pre(c)), window + 2, spare=4)
    cache = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c),
                               oracle.Fp8Cache.empty_paged(kp.shape[0], c.Hkv, 16, c.D), block_table=bt)
    cs, sn = _tables(int(c.lens.max()) + 3)
    kv = to_dev(cache)
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_fp8_rope(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), kv, dev(bt),
                                  dev(c.lens), dev(c.sinks), dev(cs), dev(sn), window, c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_paged_fp8_rope(c.q, c.k_new, c.v_new, cache, bt, c.lens, c.sinks, cs, sn,
                                       window, c.scale)
    assert_close(out.double().cpu().numpy(), ref, f"paged fp8 rope window={window}")
    krot = oracle.rope_k(c.k_new, c.lens, cs, sn)
    assert_blocks_equal(from_dev(kv), oracle.kv_append_fp8(krot, c.v_new, cache, c.lens, block_table=bt))


@pytest.mark.parametrize("W", [16, 128])
def test_ring_fp8_rope_matches_oracle(W):
    lens = [1, 15, 16, 17, W - 1, W, W + 1, 3 * W + 5, 0]
    c = make_case(780 + W, len(lens), 64, 8, 64, lens)
    cache = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c), oracle.Fp8Cache.empty_ring(c.B, c.Hkv, W, c.D),
                               window=W)
    cs, sn = _tables(int(c.lens.max()) + 1)
    kv = to_dev(cache)
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_ring_fp8_rope(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), kv, dev(c.lens),
                                 dev(c.sinks), dev(cs), dev(sn), c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_ring_fp8_rope(c.q, c.k_new, c.v_new, cache, c.lens, c.sinks, cs, sn, W, c.scale)
    assert_close(out.double().cpu().numpy(), ref, f"ring fp8 rope W={W}")
    krot = oracle.rope_k(c.k_new, c.lens, cs, sn)
    assert_blocks_equal(from_dev(kv), oracle.kv_append_fp8(krot, c.v_new, cache, c.lens, window=W))


def test_full_size_fp8_rope_two_ctas_per_sm():
    """The batch-64 workload on fp8 blocks with the RoPE: large enough for the two-CTA grid."""
    name = "b64"
    cfg = wl.config(name)
    lens = wl.seq_lens(name)
    gen = wl.cpu_generator(cfg["seed"] + 5)
    vgen = torch.Generator(device=DEV)
    vgen.manual_seed(cfg["seed"] + 5)
    B, Hq, Hkv, D, P = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["page_size"]
    inp = wl.draw_decode_inputs(B, Hq, Hkv, D, lens, gen)
    npages = wl.pool_size(name, lens)
    bt = wl.draw_block_table(lens, P, npages, wl.max_pages_per_seq(name, lens), gen)
    pool = wl.draw_fp8_paged_pool(npages, Hkv, P, D, vgen, device=DEV)
    before = from_dev(pool)
    cs, sn = _tables(max(lens) + 1)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
    sl = np.asarray(lens, np.int32)
    da.decode_attn_paged_fp8_rope(dev(inp.q), dev(inp.k_new), dev(inp.v_new), pool, dev(bt), dev(sl),
                                  dev(inp.sinks), dev(cs), dev(sn), 0, inp.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_paged_fp8_rope(wl.bits(inp.q), wl.bits(inp.k_new), wl.bits(inp.v_new), before,
                                       bt.numpy(), sl, inp.sinks.numpy(), cs, sn, 0, inp.scale)
    assert_close(out.double().cpu().numpy(), ref, "b64 paged fp8 rope")
    krot = oracle.rope_k(wl.bits(inp.k_new), sl, cs, sn)
    assert_blocks_equal(from_dev(pool), oracle.kv_append_fp8(krot, wl.bits(inp.v_new), before, sl,
                                                             block_table=bt.numpy()))
