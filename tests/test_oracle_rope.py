"""Pins for the oracle's fused rotary position embedding (SimpleLLM README,
changes table, row "RoPE as one fused kernel at every batch size"): identity
and quarter-turn tables reduce it to closed forms, position 0 is the identity,
rotations keep norms, attention depends only on relative positions, and the
stored key's rounding matches fp32 arithmetic rounded by torch's bf16 cast."""
import numpy as np
import pytest
import torch

import oracle
from cases import NAN, make_case, paged_identity, ring_from_history, shuffle_pages
from paged_decode_attention_kv_gb300 import workloads as wl


def pre(c):
    return np.maximum(c.lens - 1, 0)


def tables(kind, maxpos, D):
    if kind == "identity":
        return np.ones((maxpos, D // 2), np.float32), np.zeros((maxpos, D // 2), np.float32)
    if kind == "quarter":
        return np.zeros((maxpos, D // 2), np.float32), np.ones((maxpos, D // 2), np.float32)
    return wl.rope_tables(maxpos, D)


def rot_half_quarter(x):
    """cos = 0, sin = 1: (x1, x2) -> (-x2, x1), exact on bf16 bit patterns."""
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x2 ^ np.uint16(0x8000), x1], axis=-1)


def test_identity_tables_change_nothing():
    c = make_case(401, 3, 8, 2, 64, [1, 30, 77])
    kp, vp, bt = shuffle_pages(*paged_identity(c, pre(c)), 1)
    cs, sn = tables("identity", 128, 64)
    plain = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, 0, c.scale, 16)
    rope = oracle.decode_paged_rope(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, cs, sn,
                                    0, c.scale, 16)
    np.testing.assert_array_equal(rope, plain)
    np.testing.assert_array_equal(oracle.rope_k(c.k_new, c.lens, cs, sn), c.k_new)


def test_quarter_turn_is_a_signed_half_swap():
    c = make_case(402, 3, 8, 2, 64, [2, 17, 64])
    cs, sn = tables("quarter", 128, 64)
    np.testing.assert_array_equal(oracle.rope_k(c.k_new, c.lens, cs, sn), rot_half_quarter(c.k_new))
    q64 = oracle.rope_q64(c.q, c.lens, cs, sn)
    from cases import bf16_to_f64
    np.testing.assert_array_equal(q64, bf16_to_f64(rot_half_quarter(c.q)))
    # the whole step equals the plain step on the swapped query and new key
    kp, vp, bt = shuffle_pages(*paged_identity(c, pre(c)), 2)
    rope = oracle.decode_paged_rope(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, cs, sn,
                                    0, c.scale, 16)
    plain = oracle.decode_paged(rot_half_quarter(c.q), rot_half_quarter(c.k_new), c.v_new, kp, vp,
                                bt, c.lens, c.sinks, 0, c.scale, 16)
    np.testing.assert_allclose(rope, plain, rtol=0, atol=1e-15)


def test_position_zero_is_the_identity():
    """A one-token sequence sits at position 0, where every angle is 0."""
    c = make_case(403, 4, 8, 2, 64, [1, 1, 1, 1])
    cs, sn = tables("real", 4096, 64)
    kp, vp, bt = paged_identity(c, pre(c))
    rope = oracle.decode_paged_rope(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, cs, sn,
                                    0, c.scale, 16)
    plain = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, 0, c.scale, 16)
    np.testing.assert_allclose(rope, plain, rtol=0, atol=1e-15)


def test_rotation_keeps_norms():
    c = make_case(404, 3, 8, 2, 64, [5, 900, 3000])
    cs, sn = tables("real", 4096, 64)
    from cases import bf16_to_f64
    q = bf16_to_f64(c.q)
    r = oracle.rope_q64(c.q, c.lens, cs, sn)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-6)
    # and it does rotate: positions > 0 change the vector
    assert np.abs(r[2] - q[2]).max() > 1e-2


def test_stored_key_rounding_is_fp32_then_bf16_nearest_even():
    c = make_case(405, 6, 8, 8, 64, [1, 2, 100, 513, 4000, 4095])
    cs, sn = tables("real", 4096, 64)
    got = oracle.rope_k(c.k_new, c.lens, cs, sn)
    from cases import bf16_to_f64
    k = bf16_to_f64(c.k_new).astype(np.float32)
    h = 32
    want = np.empty_like(k)
    for b in range(c.B):
        p = int(c.lens[b]) - 1
        cc, ss = cs[p], sn[p]
        k1, k2 = k[b, :, :h], k[b, :, h:]
        want[b, :, :h] = (k1 * cc) - (k2 * ss)          # numpy float32: each op rounded
        want[b, :, h:] = (k2 * cc) + (k1 * ss)
    want_bits = wl.bits(torch.from_numpy(want).to(torch.bfloat16))
    np.testing.assert_array_equal(got, want_bits)


@pytest.mark.parametrize("shift", [1, 37, 1000])
def test_attention_depends_only_on_relative_positions(shift):
    """The same raw keys at positions 0..L-1, or at shift..shift+L-1 behind a window of L
    (the first `shift` tokens fall out of the window): same outputs, up to the bf16
    rounding of keys rotated by different absolute angles."""
    L, Hq, Hkv, D = 50, 8, 2, 64
    c = make_case(406 + shift, 1, Hq, Hkv, D, [L])
    cs, sn = tables("real", 4096, D)
    # raw history keys rotated at their own positions (cache holds rotated keys)
    def rotated_history(offset, total):
        hk = np.full((1, total, Hkv, D), NAN, np.uint16)
        hv = np.full((1, total, Hkv, D), NAN, np.uint16)
        for j in range(L):
            pos = offset + j
            hk[0, pos] = oracle.rope_k(c.hist_k[0, j][None], np.array([pos + 1]), cs, sn)[0]
            hv[0, pos] = c.hist_v[0, j]
        return hk, hv
    outs = []
    for offset, window in ((0, 0), (shift, L)):
        total = offset + L
        hk, hv = rotated_history(offset, total)
        cc = make_case(406 + shift, 1, Hq, Hkv, D, [total])
        cc.q = c.q
        cc.hist_k, cc.hist_v = hk, hv
        lens = np.array([total], np.int32)
        cc.lens = lens
        kp, vp, bt = paged_identity(cc, lens - 1)
        raw_new_k, new_v = c.hist_k[:, L - 1], c.hist_v[:, L - 1]
        outs.append(oracle.decode_paged_rope(c.q, raw_new_k, new_v, kp, vp, bt, lens, c.sinks,
                                             cs, sn, window, c.scale, 16))
    np.testing.assert_allclose(outs[1], outs[0], rtol=2e-2, atol=5e-3)
