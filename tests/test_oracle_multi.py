"""Pins for the oracle's multi-token step (several query tokens per sequence with a
causal mask: the teaching repo's chapters "Chunked Prefill" and "Speculative
Decoding", table "The files" on the page "Run it locally"), checked against things
other than itself: the pure-Python brute force over the logical history (token t is
a single-token step on the history up to its own position), torch's fp64
scaled-dot-product attention with an explicit causal mask, the single-token oracle
at T = 1, ring = windowed paged, zero rows beyond q_lens, and the append against
caches built with plain array operations."""
import numpy as np
import pytest
import torch

import oracle
from brute import attend as brute_attend
from cases import NAN, bf16_to_f64, make_case, paged_identity, ring_from_history, shuffle_pages
from paged_decode_attention_kv_gb300 import workloads as wl


class Multi:
    """A multi-token step built from a make_case history: sequence b has L_b tokens after
    the step, the last n_b of them new."""

    def __init__(self, seed, Hq, Hkv, lens, n, T, D=64):
        self.c = c = make_case(seed, len(lens), Hq, Hkv, D, lens)
        self.T, self.n = T, np.asarray(n, np.int32)
        self.lens = c.lens
        self.base = np.where(self.lens > 0, self.lens - self.n, 0).astype(np.int32)
        gen = wl.cpu_generator(seed + 5000)
        self.q = wl.bits(wl.randn_bf16((c.B, T, Hq, D), gen))
        self.k_new = np.full((c.B, T, Hkv, D), NAN, np.uint16)   # padding rows stay NaN
        self.v_new = np.full((c.B, T, Hkv, D), NAN, np.uint16)
        for b in range(c.B):
            for t in range(int(self.n[b])):
                self.k_new[b, t] = c.hist_k[b, self.base[b] + t]
                self.v_new[b, t] = c.hist_v[b, self.base[b] + t]
        self.sinks = c.sinks

    def paged(self, seed=1, after=False, total_pages=None, table_width=None):
        """Pools of the history (before the step, or after its append) behind a shuffled
        block table; optionally exactly total_pages pages and table_width table columns."""
        kp, vp, bt = paged_identity(self.c, self.lens if after else self.base)
        spare = 3 if total_pages is None else total_pages - kp.shape[0]
        kp, vp, bt = shuffle_pages(kp, vp, bt, seed, spare=spare)
        if table_width is not None:
            bt = np.pad(bt, ((0, 0), (0, table_width - bt.shape[1])), constant_values=-1)
        return kp, vp, bt

    def ring(self, W, after=False):
        return ring_from_history(self.c, self.lens if after else self.base, W)

    def run(self, window, paged=True, sinks=True, q_lens=True, seed=1):
        if paged:
            kp, vp, bt = self.paged(seed)
            return oracle.decode_multi(self.q, self.k_new, self.v_new, kp, vp, self.lens,
                                       self.sinks if sinks else None, window, self.c.scale,
                                       block_table=bt, q_lens=self.n if q_lens else None)
        kr, vr = self.ring(window)
        return oracle.decode_multi(self.q, self.k_new, self.v_new, kr, vr, self.lens,
                                   self.sinks if sinks else None, window, self.c.scale,
                                   q_lens=self.n if q_lens else None)

    def brute(self, window, sinks=True):
        c = self.c
        out = np.zeros((c.B, self.T, c.Hq, c.D))
        for b in range(c.B):
            for t in range(int(self.n[b])):
                p = int(self.base[b]) + t
                out[b, t] = brute_attend(self.q[b, t].tolist(), c.hist_k[b].tolist(),
                                         c.hist_v[b].tolist(), p + 1,
                                         list(self.sinks) if sinks else None, window,
                                         c.scale, c.Hq // c.Hkv)
        return out


CASES = [
    # (Hq, Hkv, lens, n, T)
    (4, 2, [5, 17, 33], [3, 1, 4], 4),
    (8, 1, [2, 40, 16], [2, 5, 0], 5),
    (6, 3, [7, 20], [7, 6], 7),
]


# ---------------------------------------------------------------- brute force (logical history)
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("window", [0, 3, 16])
def test_multi_brute_force_paged(case, window):
    Hq, Hkv, lens, n, T = CASES[case]
    m = Multi(40 + case, Hq, Hkv, lens, n, T, D=8)
    np.testing.assert_allclose(m.run(window), m.brute(window), rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("W", [8, 16, 40])
def test_multi_brute_force_ring(case, W):
    Hq, Hkv, lens, n, T = CASES[case]
    m = Multi(50 + case, Hq, Hkv, lens, n, T, D=8)
    np.testing.assert_allclose(m.run(W, paged=False), m.brute(W), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- textbook causal attention
def test_multi_equals_torch_sdpa_with_causal_mask():
    m = Multi(60, 8, 2, [9, 30, 64], [4, 4, 2], 4)
    out = m.run(0, sinks=False)
    c, G = m.c, 8 // 2
    for b in range(c.B):
        L, n, base = int(m.lens[b]), int(m.n[b]), int(m.base[b])
        q = torch.from_numpy(bf16_to_f64(m.q[b, :n])).permute(1, 0, 2)[None]        # [1,Hq,n,D]
        k = torch.from_numpy(bf16_to_f64(c.hist_k[b, :L])).permute(1, 0, 2)         # [Hkv,L,D]
        v = torch.from_numpy(bf16_to_f64(c.hist_v[b, :L])).permute(1, 0, 2)
        k = k.repeat_interleave(G, dim=0)[None]
        v = v.repeat_interleave(G, dim=0)[None]
        mask = torch.arange(L)[None, :] <= (base + torch.arange(n))[:, None]        # [n, L]
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                               scale=c.scale)
        np.testing.assert_allclose(out[b, :n], ref[0].permute(1, 0, 2).numpy(), rtol=0,
                                   atol=1e-10)


# ---------------------------------------------------------------- relations to other oracles
def test_one_token_equals_the_single_token_step():
    c = make_case(61, 4, 8, 2, 64, [1, 16, 17, 50])
    pre = np.maximum(c.lens - 1, 0)
    kp, vp, bt = shuffle_pages(*paged_identity(c, pre), 2)
    single = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, 20,
                                 c.scale, 16)
    multi = oracle.decode_multi(c.q[:, None], c.k_new[:, None], c.v_new[:, None], kp, vp,
                                c.lens, c.sinks, 20, c.scale, block_table=bt)
    np.testing.assert_array_equal(multi[:, 0], single)


def test_ring_equals_windowed_paged():
    m = Multi(62, 8, 2, [3, 20, 45, 70], [3, 4, 4, 1], 4)
    for W in (16, 32):
        np.testing.assert_array_equal(m.run(W, paged=False), m.run(W, paged=True))


def test_rows_beyond_q_lens_and_inactive_slots_are_zero():
    m = Multi(63, 4, 2, [0, 12, 5], [0, 2, 5], 5)
    out = m.run(0)
    assert np.all(out[0] == 0)            # inactive slot
    assert np.all(out[1, 2:] == 0)        # rows t >= n
    assert np.all(np.isfinite(out)) and np.any(out[1, :2] != 0)
    # q_lens = None means all T rows are new tokens
    m2 = Multi(64, 4, 2, [9, 12], [3, 3], 3)
    np.testing.assert_array_equal(m2.run(0, q_lens=True), m2.run(0, q_lens=False))


# ---------------------------------------------------------------- the append
@pytest.mark.parametrize("paged", [True, False])
def test_append_is_bit_exact_and_touches_only_the_new_cells(paged):
    m = Multi(65, 8, 2, [4, 16, 17, 45, 0], [4, 3, 1, 5, 0], 5)
    W = 16
    if paged:
        kp, vp, bt = m.paged(seed=4)
        ek, ev, _ = m.paged(seed=4, after=True)
        gk, gv = oracle.kv_append_multi(m.k_new, m.v_new, kp, vp, m.lens, block_table=bt,
                                        q_lens=m.n)
    else:
        kr, vr = m.ring(W)
        ek, ev = m.ring(W, after=True)
        gk, gv = oracle.kv_append_multi(m.k_new, m.v_new, kr, vr, m.lens, window=W, q_lens=m.n)
    np.testing.assert_array_equal(gk, ek)
    np.testing.assert_array_equal(gv, ev)
