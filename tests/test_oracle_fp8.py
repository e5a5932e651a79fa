"""Pins for the oracle's fp8 (e4m3) KV cache: the codec against torch's
float8_e4m3fn, the per-row quantisation rule in closed form, exact agreement
with the bf16 oracle when every stored value is representable in both, layouts
(paged and ring blocks of 16 tokens: K rows, transposed V, scales) agreeing,
the block layout byte by byte, and the quantised append."""
import numpy as np
import pytest
import torch

import oracle
from cases import make_case, paged_identity, shuffle_pages
from paged_decode_attention_kv_gb300 import workloads as wl


def pre(c):
    return np.maximum(c.lens - 1, 0)


def test_decode_every_code_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[m], ref[m])
    assert oracle.e4m3_decode(np.array([0x7E], np.uint8))[0] == 448.0


def test_encode_rounds_to_nearest_even_like_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.uniform(-448, 448, 20000),
        rng.standard_normal(20000) * 0.01,           # down to the subnormals (2^-9)
        rng.standard_normal(20000),
        oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)),   # exact codes
    ]).astype(np.float32)
    # exact midpoints between neighbouring codes: ties go to the even code
    vals = np.sort(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_encode_saturates():
    got = oracle.e4m3_encode(np.array([448.0, 460.0, 1e9, -500.0, 464.0], np.float32))
    np.testing.assert_array_equal(got, np.array([0x7E, 0x7E, 0x7E, 0xFE, 0x7E], np.uint8))


def test_quantisation_rule_closed_form():
    c = make_case(601, 4, 8, 2, 64, [3, 3, 3, 3])
    rows = c.hist_k.reshape(-1, 64)
    codes, scales = oracle.quantise_rows(rows)
    from cases import bf16_to_f64
    x = bf16_to_f64(rows).astype(np.float32)
    amax = np.abs(x).max(axis=1)
    np.testing.assert_array_equal(scales, (amax / np.float32(448)).astype(np.float32))
    # the largest element lands on +-448 exactly
    idx = np.abs(x).argmax(axis=1)
    top = codes[np.arange(len(idx)), idx]
    assert np.all((top == 0x7E) | (top == 0xFE))
    # and everything is within half an e4m3 step of the scaled value
    deq = oracle.e4m3_decode(codes) * scales[:, None]
    assert np.all(np.abs(deq - x) <= 2 ** -4 * np.abs(x) + 2 ** -10 * scales[:, None] + 1e-30)
    zc, zs = oracle.quantise_rows(np.zeros((2, 64), np.uint16))
    assert np.all(zc == 0) and np.all(zs == 1.0)


def _exact_fp8_cache(seed, num_pages, Hkv, P, D):
    """Random finite codes with power-of-two scales: every value is exact in bf16 too."""
    rng = np.random.default_rng(seed)
    mags = rng.integers(0, 0x7F, size=(num_pages, Hkv, P, D), dtype=np.uint8)  # no NaN
    signs = rng.integers(0, 2, size=mags.shape, dtype=np.uint8) << 7
    k = mags | signs
    vcodes = rng.integers(0, 0x7F, size=k.shape, dtype=np.uint8) | (
        rng.integers(0, 2, size=k.shape, dtype=np.uint8) << 7)
    ks = (2.0 ** rng.integers(-6, -2, size=(num_pages, Hkv, P))).astype(np.float32)
    vs = (2.0 ** rng.integers(-6, -2, size=(num_pages, Hkv, P))).astype(np.float32)
    cache = oracle.Fp8Cache.from_parts(k, vcodes.transpose(0, 1, 3, 2), ks, vs)
    kdeq = oracle.e4m3_decode(k) * ks[..., None]
    vdeq = oracle.e4m3_decode(vcodes) * vs[..., None]
    from cases import f64_to_bf16_bits
    return cache, f64_to_bf16_bits(kdeq), f64_to_bf16_bits(vdeq)


@pytest.mark.parametrize("window", [0, 20])
def test_fp8_equals_bf16_on_values_exact_in_both(window):
    lens = [5, 33, 64]
    c = make_case(602, 3, 8, 2, 64, lens)
    npages, P = 16, 16
    cache, kb, vb = _exact_fp8_cache(3, npages, 2, P, 64)
    bt = np.full((3, 4), -1, np.int32)
    perm = np.random.default_rng(1).permutation(npages)
    at = 0
    for b, L in enumerate(lens):
        n = -(-L // P)
        bt[b, :n] = perm[at:at + n]
        at += n
    f8 = oracle.decode_paged_fp8(c.q, None, None, cache, bt, c.lens, c.sinks, window, c.scale)
    bf = oracle.decode_paged(c.q, None, None, kb, vb, bt, c.lens, c.sinks, window, c.scale, P)
    np.testing.assert_allclose(f8, bf, rtol=0, atol=1e-14)


def test_paged_and_ring_agree_and_append_is_fused():
    lens = [1, 16, 17, 40]
    c = make_case(603, 4, 8, 2, 64, lens)
    W = 64                                   # >= every length: ring == full paged
    kp, vp, bt = paged_identity(c, pre(c))
    kp, vp, bt = shuffle_pages(kp, vp, bt, 2)
    paged = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c),
                               oracle.Fp8Cache.empty_paged(kp.shape[0], 2, 16, 64), block_table=bt)
    ring = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c), oracle.Fp8Cache.empty_ring(4, 2, W, 64),
                              window=W)
    a = oracle.decode_paged_fp8(c.q, c.k_new, c.v_new, paged, bt, c.lens, c.sinks, 0, c.scale)
    r = oracle.decode_ring_fp8(c.q, c.k_new, c.v_new, ring, c.lens, c.sinks, W, c.scale)
    np.testing.assert_array_equal(a, r)
    # appending first, then attending without the new token, is the same step
    app = oracle.kv_append_fp8(c.k_new, c.v_new, paged, c.lens, block_table=bt)
    b2 = oracle.decode_paged_fp8(c.q, None, None, app, bt, c.lens, c.sinks, 0, c.scale)
    np.testing.assert_array_equal(a, b2)
    # exactly one K row, one V column and two scales change per (active sequence, head)
    changed = (app.k != paged.k).any(axis=-1).sum()
    assert changed <= 4 * 2 and np.sum(app.ks != paged.ks) + np.sum(np.isnan(paged.ks) & ~np.isnan(app.ks)) >= 1
    # the fp8 step is close to the bf16 step on the same (unquantised) history
    bf = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, 0, c.scale, 16)
    assert np.all(np.abs(a - bf) <= 0.1 * np.abs(bf) + 0.1)   # loose: e4m3 keeps 3 mantissa bits


def test_block_layout_byte_by_byte():
    """One token written into an empty cache lands at the documented bytes: K codes at
    slot * 64, V codes at 1024 + d * 16 + slot, K scale at 2048 + 4 slot, V scale at
    2112 + 4 slot of block page * Hkv + g (paged) or (b * Hkv + g) * W/16 + cell/16 (ring)."""
    c = make_case(604, 2, 4, 2, 64, [21, 37])
    x = c.hist_k[1, 36, 1]                       # token 36 of sequence 1, head 1
    y = c.hist_v[1, 36, 1]
    kc, ksc = oracle.quantise_rows(x[None])
    vc, vsc = oracle.quantise_rows(y[None])
    bt = np.array([[5, 0, -1], [3, 1, 2]], np.int32)   # token 36 -> page bt[1][2] = 2, slot 4
    paged = oracle.kv_append_fp8(c.k_new, c.v_new, oracle.Fp8Cache.empty_paged(6, 2, 16, 64),
                                 c.lens, block_table=bt)
    blk = paged.blocks[2, 1]
    np.testing.assert_array_equal(blk[4 * 64:5 * 64], kc[0])
    np.testing.assert_array_equal(blk[1024 + np.arange(64) * 16 + 4], vc[0])
    assert blk[2048 + 16:2048 + 20].view(np.float32)[0] == ksc[0]
    assert blk[2112 + 16:2112 + 20].view(np.float32)[0] == vsc[0]
    # every other byte of the pool is untouched (the fill code, NaN scales): the append
    # writes slot 4 of page 2 (sequence 1, token 36) and of page 0 (sequence 0, token 20)
    touched = np.zeros(paged.blocks.shape, bool)
    for page in (2, 0):
        for g in range(2):
            t = touched[page, g]
            t[4 * 64:5 * 64] = True
            t[1024 + np.arange(64) * 16 + 4] = True
            t[2064:2068] = t[2128:2132] = True
    empty = oracle.Fp8Cache.empty_paged(6, 2, 16, 64).blocks
    np.testing.assert_array_equal(paged.blocks[~touched], empty[~touched])
    # ring of capacity 32: token 36 sits in cell 4 = block 0 of (1, 1), slot 4
    ring = oracle.kv_append_fp8(c.k_new, c.v_new, oracle.Fp8Cache.empty_ring(2, 2, 32, 64), c.lens,
                                window=32)
    rb = ring.blocks[1, 1, 0]
    np.testing.assert_array_equal(rb[4 * 64:5 * 64], kc[0])
    np.testing.assert_array_equal(rb[1024 + np.arange(64) * 16 + 4], vc[0])
    assert rb[2064:2068].view(np.float32)[0] == ksc[0] and rb[2128:2132].view(np.float32)[0] == vsc[0]


# ---------------------------------------------------------------- fp8 cache with the fused RoPE
def _rope_tables(kind, maxpos, D=64):
    if kind == "identity":
        return np.ones((maxpos, D // 2), np.float32), np.zeros((maxpos, D // 2), np.float32)
    if kind == "quarter":   # cos 0, sin 1: (x1, x2) -> (-x2, x1), exact on bf16 patterns
        return np.zeros((maxpos, D // 2), np.float32), np.ones((maxpos, D // 2), np.float32)
    return wl.rope_tables(maxpos, D)


def _half_swap(x):
    h = x.shape[-1] // 2
    return np.concatenate([x[..., h:] ^ np.uint16(0x8000), x[..., :h]], axis=-1)


def _fp8_rope_case(seed):
    lens = [1, 16, 17, 40]
    c = make_case(seed, 4, 8, 2, 64, lens)
    kp, vp, bt = shuffle_pages(*paged_identity(c, pre(c)), 3)
    paged = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c),
                               oracle.Fp8Cache.empty_paged(kp.shape[0], 2, 16, 64), block_table=bt)
    ring = oracle.scatter_fp8(c.hist_k, c.hist_v, pre(c), oracle.Fp8Cache.empty_ring(4, 2, 32, 64),
                              window=32)
    return c, bt, paged, ring


def test_fp8_rope_with_identity_tables_is_the_fp8_step():
    c, bt, paged, ring = _fp8_rope_case(611)
    cs, sn = _rope_tables("identity", 64)
    np.testing.assert_array_equal(
        oracle.decode_paged_fp8_rope(c.q, c.k_new, c.v_new, paged, bt, c.lens, c.sinks, cs, sn, 0, c.scale),
        oracle.decode_paged_fp8(c.q, c.k_new, c.v_new, paged, bt, c.lens, c.sinks, 0, c.scale))
    np.testing.assert_array_equal(
        oracle.decode_ring_fp8_rope(c.q, c.k_new, c.v_new, ring, c.lens, c.sinks, cs, sn, 32, c.scale),
        oracle.decode_ring_fp8(c.q, c.k_new, c.v_new, ring, c.lens, c.sinks, 32, c.scale))


def test_fp8_rope_quarter_turn_is_the_step_on_half_swapped_inputs():
    """A quarter turn rotates q and the new key into their signed half swaps exactly; the
    quantised new key of the swapped row is then the swapped codes (same amax, same scale)."""
    c, bt, paged, ring = _fp8_rope_case(612)
    cs, sn = _rope_tables("quarter", 64)
    qs, ks = _half_swap(c.q), _half_swap(c.k_new)
    np.testing.assert_array_equal(
        oracle.decode_paged_fp8_rope(c.q, c.k_new, c.v_new, paged, bt, c.lens, c.sinks, cs, sn, 0, c.scale),
        oracle.decode_paged_fp8(qs, ks, c.v_new, paged, bt, c.lens, c.sinks, 0, c.scale))
    np.testing.assert_array_equal(
        oracle.decode_ring_fp8_rope(c.q, c.k_new, c.v_new, ring, c.lens, c.sinks, cs, sn, 32, c.scale),
        oracle.decode_ring_fp8(qs, ks, c.v_new, ring, c.lens, c.sinks, 32, c.scale))


def test_fp8_rope_rotates_the_new_key_before_quantising_it():
    """At generic angles the fused step equals: store quantise(rotate(k_new)) first (the
    bf16 rotation of the RoPE pins, the quantisation of the fp8 pins), then attend with the
    rotated query and the token read back from the cache. Quantising first and rotating
    the codes would store different values."""
    c, bt, paged, ring = _fp8_rope_case(613)
    cs, sn = _rope_tables("plain", 64)
    krot = oracle.rope_k(c.k_new, c.lens, cs, sn)
    fused = oracle.decode_paged_fp8_rope(c.q, c.k_new, c.v_new, paged, bt, c.lens, c.sinks, cs, sn, 0,
                                         c.scale)
    app = oracle.kv_append_fp8(krot, c.v_new, paged, c.lens, block_table=bt)
    after = oracle.decode_paged_fp8_rope(c.q, None, None, app, bt, c.lens, c.sinks, cs, sn, 0, c.scale)
    np.testing.assert_array_equal(fused, after)
    wrong = oracle.decode_paged_fp8_rope(c.q, None, None,
                                         oracle.kv_append_fp8(c.k_new, c.v_new, paged, c.lens,
                                                              block_table=bt),
                                         bt, c.lens, c.sinks, cs, sn, 0, c.scale)
    assert np.abs(wrong - fused).max() > 1e-3
    fr = oracle.decode_ring_fp8_rope(c.q, c.k_new, c.v_new, ring, c.lens, c.sinks, cs, sn, 32, c.scale)
    ar = oracle.kv_append_fp8(krot, c.v_new, ring, c.lens, window=32)
    np.testing.assert_array_equal(
        fr, oracle.decode_ring_fp8_rope(c.q, None, None, ar, c.lens, c.sinks, cs, sn, 32, c.scale))
