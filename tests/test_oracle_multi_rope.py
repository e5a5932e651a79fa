"""Pins for the oracle's several-token step with the rotary embedding (SimpleLLM README,
changes table, row "RoPE as one fused kernel at every batch size", composed with the
several-token reading of the chapters "Speculative Decoding" and "Chunked Prefill"): every
new token is rotated at its own position L - n + t, and the rotated query and key enter
the attention as the bf16 model holds them. Identity tables reduce it to the plain
several-token step; one new token per sequence reduces it to the plain one-token step on
the rows the separately pinned one-token rotation (rope_k) gives; a table that turns only
one position by a quarter turn rotates exactly the token at that position (a signed half
swap, exact on bf16 bits); and the rotated keys and queries round as fp32 arithmetic cast
to bf16 by torch."""
import numpy as np
import pytest
import torch

import oracle
from cases import bf16_to_f64, make_case, paged_identity, shuffle_pages
from paged_decode_attention_kv_gb300 import workloads as wl
from test_oracle_multi import Multi
from test_oracle_rope import rot_half_quarter, tables

D = 64


def test_identity_tables_give_the_plain_step():
    m = Multi(501, 8, 2, [3, 40, 17, 0, 90], [3, 2, 1, 0, 4], 4)
    kp, vp, bt = m.paged(1)
    cs, sn = tables("identity", 256, D)
    plain = oracle.decode_multi(m.q, m.k_new, m.v_new, kp, vp, m.lens, m.sinks, 0, m.c.scale,
                                block_table=bt, q_lens=m.n)
    rope = oracle.decode_multi_rope(m.q, m.k_new, m.v_new, kp, vp, m.lens, m.sinks, cs, sn, 0,
                                    m.c.scale, block_table=bt, q_lens=m.n)
    np.testing.assert_array_equal(rope, plain)
    _, krot, qrot = oracle.rope_multi(m.q, m.k_new, m.lens, cs, sn, q_lens=m.n, with_q_bf16=True)
    np.testing.assert_array_equal(krot, m.k_new)
    np.testing.assert_array_equal(qrot, m.q)


@pytest.mark.parametrize("window", [0, 20])
def test_one_new_token_is_the_one_token_step(window):
    """n = 1 everywhere: the several-token rotation is the one-token one (position L - 1):
    the plain one-token step on the rows rope_k rotates (queries and keys alike)."""
    lens = [1, 5, 33, 70, 0, 130]
    m = Multi(502, 8, 2, lens, [1 if L > 0 else 0 for L in lens], 1)
    kp, vp, bt = m.paged(2)
    cs, sn = tables("real", 4096, D)
    multi = oracle.decode_multi_rope(m.q, m.k_new, m.v_new, kp, vp, m.lens, m.sinks, cs, sn,
                                     window, m.c.scale, block_table=bt, q_lens=m.n)
    q1 = oracle.rope_k(m.q[:, 0], m.lens, cs, sn)       # per-row rotation at L - 1, to bf16
    k1 = oracle.rope_k(m.k_new[:, 0], m.lens, cs, sn)
    one = oracle.decode_paged(q1, k1, m.v_new[:, 0], kp, vp, bt, m.lens, m.sinks, window,
                              m.c.scale, 16)
    np.testing.assert_allclose(multi[:, 0], one, rtol=0, atol=1e-15)
    _, krot, qrot = oracle.rope_multi(m.q, m.k_new, m.lens, cs, sn, q_lens=m.n, with_q_bf16=True)
    np.testing.assert_array_equal(krot[:, 0], k1)
    np.testing.assert_array_equal(qrot[:, 0], q1)


def test_each_token_is_rotated_at_its_own_position():
    """Identity everywhere except one position p*, turned by a quarter: only the new token
    that sits at p* (query rows and key) is changed, by the exact signed half swap."""
    T = 4
    lens = [10, 10, 12, 7]
    n = [4, 3, 4, 2]
    m = Multi(503, 8, 2, lens, n, T)
    p_star = 8
    cs, sn = tables("identity", 64, D)
    cs[p_star], sn[p_star] = 0.0, 1.0
    q64, krot = oracle.rope_multi(m.q, m.k_new, m.lens, cs, sn, q_lens=m.n)
    want_q = m.q.copy()
    want_k = m.k_new.copy()
    hit = 0
    for b in range(m.c.B):
        base = int(m.lens[b]) - int(m.n[b])
        for t in range(int(m.n[b])):
            if base + t == p_star:
                want_q[b, t] = rot_half_quarter(m.q[b, t])
                want_k[b, t] = rot_half_quarter(m.k_new[b, t])
                hit += 1
    assert hit == 3  # b = 0 (t = 2), b = 1 (t = 1), b = 2 (t = 0)
    active = np.zeros(want_q.shape[:2], bool)
    for b in range(m.c.B):
        active[b, :int(m.n[b])] = True
    np.testing.assert_array_equal(q64[active], bf16_to_f64(want_q)[active])
    assert not q64[~active].any()
    np.testing.assert_array_equal(krot[active], want_k[active])
    # and the whole step equals the plain step on those inputs
    kp, vp, bt = m.paged(3)
    rope = oracle.decode_multi_rope(m.q, m.k_new, m.v_new, kp, vp, m.lens, m.sinks, cs, sn, 0,
                                    m.c.scale, block_table=bt, q_lens=m.n)
    plain = oracle.decode_multi(want_q, want_k, m.v_new, kp, vp, m.lens, m.sinks, 0, m.c.scale,
                                block_table=bt, q_lens=m.n)
    np.testing.assert_allclose(rope, plain, rtol=0, atol=1e-15)


def test_ring_form_matches_the_paged_form():
    """The same history in a ring of capacity W and in pages behind a window of W."""
    W = 32
    lens = [5, 40, 77, 33]
    n = [3, 4, 2, 4]
    m = Multi(504, 8, 2, lens, n, 4)
    cs, sn = tables("real", 4096, D)
    kp, vp, bt = m.paged(4)
    kr, vr = m.ring(W)
    paged = oracle.decode_multi_rope(m.q, m.k_new, m.v_new, kp, vp, m.lens, m.sinks, cs, sn, W,
                                     m.c.scale, block_table=bt, q_lens=m.n)
    ring = oracle.decode_multi_rope(m.q, m.k_new, m.v_new, kr, vr, m.lens, m.sinks, cs, sn, W,
                                    m.c.scale, q_lens=m.n)
    np.testing.assert_allclose(ring, paged, rtol=0, atol=1e-15)


def test_rotated_rows_round_as_fp32_then_bf16():
    T = 3
    lens = [3, 200, 4000]
    m = Multi(505, 8, 8, lens, [3, 3, 2], T)
    cs, sn = tables("real", 4096, D)
    _, krot, qrot = oracle.rope_multi(m.q, m.k_new, m.lens, cs, sn, q_lens=m.n, with_q_bf16=True)
    h = D // 2
    for x, got in ((m.k_new, krot), (m.q, qrot)):
        xf = bf16_to_f64(x).astype(np.float32)
        for b in range(m.c.B):
            base = int(m.lens[b]) - int(m.n[b])
            for t in range(int(m.n[b])):
                p = base + t
                x1, x2 = xf[b, t, :, :h], xf[b, t, :, h:]
                want = np.concatenate([(x1 * cs[p]) - (x2 * sn[p]), (x2 * cs[p]) + (x1 * sn[p])], axis=-1)
                np.testing.assert_array_equal(got[b, t], wl.bits(torch.from_numpy(want).to(torch.bfloat16)))
