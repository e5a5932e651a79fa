"""Pins for the oracle's several-token step over an fp8 cache (the several-token reading of
the chapters "Speculative Decoding" and "Chunked Prefill" composed with the fp8 cache reading
of "quantised KV pages"): one new token per sequence is the one-token fp8 step (a separate,
separately pinned function), paged and ring, with and without a window; when every stored
value and every new token is exact in both formats it is the bf16 several-token step; and the
quantised append of the n new tokens leaves the cache that quantising the whole history
(positions 0 .. L-1) builds."""
import numpy as np
import pytest

import oracle
from cases import f64_to_bf16_bits
from test_oracle_fp8 import _exact_fp8_cache
from test_oracle_multi import Multi

P, D = 16, 64


def fp8_paged(m, seed):
    """The history before the step (positions < L - n) quantised into shuffled pages."""
    kp, vp, bt = m.paged(seed)
    blank = oracle.Fp8Cache.empty_paged(kp.shape[0], m.c.Hkv, P, D)
    base = np.where(m.lens > 0, m.lens - m.n, 0).astype(np.int32)
    return oracle.scatter_fp8(m.c.hist_k, m.c.hist_v, base, blank, block_table=bt), bt, base


@pytest.mark.parametrize("window", [0, 20])
def test_one_new_token_is_the_one_token_fp8_step(window):
    lens = [1, 5, 33, 70, 0, 130]
    m = Multi(701, 8, 2, lens, [1 if L > 0 else 0 for L in lens], 1)
    cache, bt, _ = fp8_paged(m, 1)
    multi = oracle.decode_multi_fp8(m.q, m.k_new, m.v_new, cache, m.lens, m.sinks, window, m.c.scale,
                                    block_table=bt, q_lens=m.n)
    one = oracle.decode_paged_fp8(m.q[:, 0], m.k_new[:, 0], m.v_new[:, 0], cache, bt, m.lens, m.sinks,
                                  window, m.c.scale)
    np.testing.assert_allclose(multi[:, 0], one, rtol=0, atol=1e-15)


def test_one_new_token_ring():
    W = 32
    lens = [1, 16, 17, 40, 100]
    m = Multi(702, 8, 2, lens, [1] * len(lens), 1)
    base = (m.lens - 1).astype(np.int32)
    ring = oracle.scatter_fp8(m.c.hist_k, m.c.hist_v, base, oracle.Fp8Cache.empty_ring(m.c.B, 2, W, D),
                              window=W)
    multi = oracle.decode_multi_fp8(m.q, m.k_new, m.v_new, ring, m.lens, m.sinks, W, m.c.scale,
                                    q_lens=m.n)
    one = oracle.decode_ring_fp8(m.q[:, 0], m.k_new[:, 0], m.v_new[:, 0], ring, m.lens, m.sinks, W,
                                 m.c.scale)
    np.testing.assert_allclose(multi[:, 0], one, rtol=0, atol=1e-15)


def _exact_rows(rng, shape):
    """bf16 rows that quantise losslessly: random e4m3 codes times 2^k with one element of
    each row at +-448 * 2^k, so the row's scale is the power of two 2^k exactly."""
    mags = rng.integers(0, 0x7F, size=shape, dtype=np.uint8)
    mags[..., 0] = 0x7E
    codes = mags | (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7)
    k = rng.integers(-8, -4, size=shape[:-1])
    vals = oracle.e4m3_decode(codes) * (2.0 ** k)[..., None]
    return f64_to_bf16_bits(vals)


@pytest.mark.parametrize("window", [0, 24])
def test_exact_values_give_the_bf16_step(window):
    T, Hq, Hkv = 4, 8, 2
    lens = [5, 33, 20]
    n = [4, 2, 3]
    npages = 12
    cache, kb, vb = _exact_fp8_cache(7, npages, Hkv, P, D)
    bt = np.full((3, 3), -1, np.int32)
    perm = np.random.default_rng(2).permutation(npages)
    at = 0
    for b, L in enumerate(lens):
        k = -(-L // P)
        bt[b, :k] = perm[at:at + k]
        at += k
    rng = np.random.default_rng(3)
    m = Multi(703, Hq, Hkv, lens, n, T)
    kn = _exact_rows(rng, (3, T, Hkv, D))
    vn = _exact_rows(rng, (3, T, Hkv, D))
    lens_a, n_a = np.asarray(lens, np.int32), np.asarray(n, np.int32)
    f8 = oracle.decode_multi_fp8(m.q, kn, vn, cache, lens_a, m.sinks, window, m.c.scale,
                                 block_table=bt, q_lens=n_a)
    bf = oracle.decode_multi(m.q, kn, vn, kb, vb, lens_a, m.sinks, window, m.c.scale, block_table=bt,
                             q_lens=n_a)
    np.testing.assert_allclose(f8, bf, rtol=0, atol=1e-14)


@pytest.mark.parametrize("ring", [False, True])
def test_append_equals_quantising_the_whole_history(ring):
    T = 4
    lens = [4, 17, 33, 100, 0]
    n = [4, 3, 4, 1, 0]
    m = Multi(704, 8, 2, lens, n, T)
    if ring:
        W = 32
        base = np.where(m.lens > 0, m.lens - m.n, 0).astype(np.int32)
        before = oracle.scatter_fp8(m.c.hist_k, m.c.hist_v, base,
                                    oracle.Fp8Cache.empty_ring(m.c.B, 2, W, D), window=W)
        after = oracle.kv_append_multi_fp8(m.k_new, m.v_new, before, m.lens, window=W, q_lens=m.n)
        want = oracle.scatter_fp8(m.c.hist_k, m.c.hist_v, m.lens,
                                  oracle.Fp8Cache.empty_ring(m.c.B, 2, W, D), window=W)
    else:
        before, bt, _ = fp8_paged(m, 4)
        after = oracle.kv_append_multi_fp8(m.k_new, m.v_new, before, m.lens, block_table=bt, q_lens=m.n)
        want = oracle.scatter_fp8(m.c.hist_k, m.c.hist_v, m.lens,
                                  oracle.Fp8Cache.empty_paged(before.blocks.shape[0], 2, P, D),
                                  block_table=bt)
    np.testing.assert_array_equal(after.blocks, want.blocks)
