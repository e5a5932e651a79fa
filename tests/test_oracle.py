"""Pins for the fp64 CPU oracle, checked against things other than itself:
a pure-Python brute force, torch's fp64 scaled-dot-product attention, closed
forms, layout identities built with plain array ops, GQA = repeated-KV MHA,
bit-exact append, permutation invariance and a hand-worked example.

The definition being pinned: SimpleLLM README, changes table, row "one
decode-attention kernel for sinks, sliding window, GQA and the KV append"
(plus the rows on the paged KV cache and the sliding-window ring buffer).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from brute import attend as brute_attend
from cases import (NAN, bf16_to_f64, f64_to_bf16_bits, make_case, paged_identity,
                   ring_from_history, shuffle_pages)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def pre(c):
    return np.maximum(c.lens - 1, 0)


def o_paged(c, kp, vp, bt, window=0, sinks="case", fused=True, items=None):
    s = c.sinks if isinstance(sinks, str) else sinks
    return oracle.decode_paged(c.q, c.k_new if fused else None, c.v_new if fused else None,
                               kp, vp, bt, c.lens, s, window, c.scale, c.P, items=items)


def o_ring(c, kr, vr, W, sinks="case", fused=True):
    s = c.sinks if isinstance(sinks, str) else sinks
    return oracle.decode_ring(c.q, c.k_new if fused else None, c.v_new if fused else None,
                              kr, vr, c.lens, s, W, c.scale)


def o_contig(c, window=0, sinks="case"):
    s = c.sinks if isinstance(sinks, str) else sinks
    return oracle.decode_contig(c.q, c.hist_k, c.hist_v, c.lens, s, window, c.scale)


# ---------------------------------------------------------------- P1 brute force
@pytest.mark.parametrize("seed,B,Hq,Hkv,D,lens,W", [
    (11, 2, 4, 2, 8, [5, 17], 0),
    (12, 3, 6, 3, 4, [1, 16, 33], 7),
    (13, 2, 8, 1, 16, [40, 2], 16),
    (14, 1, 2, 2, 64, [31], 0),
])
def test_brute_force_matches_all_layouts(seed, B, Hq, Hkv, D, lens, W):
    c = make_case(seed, B, Hq, Hkv, D, lens, P=4)
    G = Hq // Hkv
    ref = np.array([brute_attend(c.q[b].tolist(), c.hist_k[b].tolist(), c.hist_v[b].tolist(),
                                 int(c.lens[b]), c.sinks.tolist(), W, c.scale, G)
                    for b in range(B)])
    np.testing.assert_allclose(o_contig(c, W), ref, rtol=0, atol=1e-12)
    kp, vp, bt = paged_identity(c, pre(c))
    kp, vp, bt = shuffle_pages(kp, vp, bt, seed)
    np.testing.assert_allclose(o_paged(c, kp, vp, bt, W), ref, rtol=0, atol=1e-12)
    if W > 0:
        kr, vr = ring_from_history(c, pre(c), W)
        np.testing.assert_allclose(o_ring(c, kr, vr, W), ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- P2 textbook softmax attention
@pytest.mark.parametrize("window", [0, 9])
def test_no_sink_equals_torch_sdpa_fp64(window):
    c = make_case(21, 3, 8, 2, 64, [1, 30, 77])
    out = o_contig(c, window, sinks=None)
    G = c.Hq // c.Hkv
    for b in range(c.B):
        L = int(c.lens[b])
        lo = max(0, L - window) if window else 0
        q = torch.from_numpy(bf16_to_f64(c.q[b]))[None, :, None, :]          # [1,Hq,1,D]
        k = torch.from_numpy(bf16_to_f64(c.hist_k[b, lo:L])).permute(1, 0, 2)  # [Hkv,n,D]
        v = torch.from_numpy(bf16_to_f64(c.hist_v[b, lo:L])).permute(1, 0, 2)
        k = k.repeat_interleave(G, dim=0)[None]
        v = v.repeat_interleave(G, dim=0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=c.scale)
        np.testing.assert_allclose(out[b], ref[0, :, 0, :].numpy(), rtol=0, atol=1e-10)


# ---------------------------------------------------------------- P3 closed forms
def test_single_token_is_sigmoid_weighted_value():
    c = make_case(31, 4, 8, 2, 64, [1, 1, 1, 1])
    kp, vp, bt = paged_identity(c, pre(c))
    out = o_paged(c, kp, vp, bt)
    G = c.Hq // c.Hkv
    for b in range(c.B):
        for h in range(c.Hq):
            g = h // G
            s = c.scale * float(bf16_to_f64(c.q[b, h]) @ bf16_to_f64(c.k_new[b, g]))
            expect = bf16_to_f64(c.v_new[b, g]) / (1.0 + math.exp(float(c.sinks[h]) - s))
            np.testing.assert_allclose(out[b, h], expect, rtol=1e-13, atol=1e-15)
    # and with no sink the single token's value comes back exactly
    out0 = o_paged(c, kp, vp, bt, sinks=None)
    for b in range(c.B):
        np.testing.assert_array_equal(out0[b], np.repeat(bf16_to_f64(c.v_new[b]), G, axis=0))


def test_zero_query_is_windowed_mean_with_sink():
    """q = 0 makes every score 0: out = sum_{j in window} v_j / (n + e^sigma).
    Pins the window bounds, the GQA head map and the sink term at once."""
    c = make_case(32, 3, 8, 4, 64, [5, 40, 129])
    c.q[:] = 0
    G = c.Hq // c.Hkv
    for W in (0, 16, 200):
        out = o_contig(c, W)
        kp, vp, bt = paged_identity(c, pre(c))
        outp = o_paged(c, kp, vp, bt, W)
        for b in range(c.B):
            L = int(c.lens[b])
            lo = max(0, L - W) if W else 0
            vsum = bf16_to_f64(c.hist_v[b, lo:L]).sum(axis=0)        # [Hkv, D]
            for h in range(c.Hq):
                expect = vsum[h // G] / ((L - lo) + math.exp(float(c.sinks[h])))
                np.testing.assert_allclose(out[b, h], expect, rtol=1e-12, atol=1e-14)
                np.testing.assert_allclose(outp[b, h], expect, rtol=1e-12, atol=1e-14)


def test_equal_keys_equal_values_closed_form():
    """All keys equal (score c) and all values equal v: out = v * n e^c / (n e^c + e^sigma)."""
    c = make_case(33, 2, 4, 1, 64, [3, 50])
    key = c.hist_k[0, 0, 0].copy()
    val = c.hist_v[0, 0, 0].copy()
    c.hist_k[:] = key
    c.hist_v[:] = val
    c.k_new[:] = key
    c.v_new[:] = val
    kp, vp, bt = paged_identity(c, pre(c))
    out = o_paged(c, kp, vp, bt)
    for b in range(c.B):
        n = int(c.lens[b])
        for h in range(c.Hq):
            s = c.scale * float(bf16_to_f64(c.q[b, h]) @ bf16_to_f64(key))
            frac = n * math.exp(s) / (n * math.exp(s) + math.exp(float(c.sinks[h])))
            np.testing.assert_allclose(out[b, h], bf16_to_f64(val) * frac, rtol=1e-12, atol=1e-15)


def test_large_sink_absorbs_everything_and_tiny_sink_vanishes():
    c = make_case(34, 2, 8, 2, 64, [20, 33])
    kp, vp, bt = paged_identity(c, pre(c))
    big = o_paged(c, kp, vp, bt, sinks=np.full(c.Hq, 60.0, np.float32))
    assert np.abs(big).max() < 1e-15
    tiny = o_paged(c, kp, vp, bt, sinks=np.full(c.Hq, -1e4, np.float32))
    none = o_paged(c, kp, vp, bt, sinks=None)
    np.testing.assert_allclose(tiny, none, rtol=0, atol=1e-15)


def test_inactive_slot_is_zero():
    c = make_case(35, 3, 8, 2, 64, [0, 9, 0])
    kp, vp, bt = paged_identity(c, pre(c))
    out = o_paged(c, kp, vp, bt)
    assert np.all(out[0] == 0) and np.all(out[2] == 0) and np.all(np.isfinite(out[1]))
    kr, vr = ring_from_history(c, pre(c), 8)
    outr = o_ring(c, kr, vr, 8)
    assert np.all(outr[0] == 0) and np.all(outr[2] == 0)


# ---------------------------------------------------------------- P4 window >= L
def test_window_at_or_beyond_length_equals_full():
    c = make_case(41, 3, 8, 2, 64, [7, 64, 100])
    kp, vp, bt = paged_identity(c, pre(c))
    full = o_paged(c, kp, vp, bt, 0)
    for W in (100, 101, 4096):
        np.testing.assert_allclose(o_paged(c, kp, vp, bt, W), full, rtol=0, atol=1e-14)
        kr, vr = ring_from_history(c, pre(c), W)
        np.testing.assert_allclose(o_ring(c, kr, vr, W), full, rtol=0, atol=1e-14)
    # a window shorter than some lengths must change those rows
    part = o_paged(c, kp, vp, bt, 50)
    np.testing.assert_allclose(part[0], full[0], rtol=0, atol=1e-14)
    assert np.abs(part[2] - full[2]).max() > 1e-6


# ---------------------------------------------------------------- P5 layouts agree
@pytest.mark.parametrize("W", [16, 13, 128])
def test_ring_paged_contig_agree(W):
    c = make_case(51, 4, 8, 2, 64, [1, 15, 16, 300])
    ref = o_contig(c, W)
    kp, vp, bt = paged_identity(c, pre(c))
    np.testing.assert_allclose(o_paged(c, kp, vp, bt, W), ref, rtol=0, atol=1e-14)
    k2, v2, bt2 = shuffle_pages(kp, vp, bt, 5, spare=7)
    np.testing.assert_allclose(o_paged(c, k2, v2, bt2, W), ref, rtol=0, atol=1e-14)
    kr, vr = ring_from_history(c, pre(c), W)
    np.testing.assert_allclose(o_ring(c, kr, vr, W), ref, rtol=0, atol=1e-14)


def test_oracle_scatter_matches_array_built_layouts():
    c = make_case(52, 3, 8, 2, 64, [3, 31, 90])
    kp, vp, bt = paged_identity(c, pre(c))
    k2, v2, bt2 = shuffle_pages(kp, vp, bt, 9, spare=4)
    blank_k = np.full_like(k2, NAN)
    sk, sv = oracle.scatter_paged(c.hist_k, c.hist_v, pre(c), bt2, blank_k, blank_k)
    np.testing.assert_array_equal(sk, k2)
    np.testing.assert_array_equal(sv, v2)
    W = 32
    kr, vr = ring_from_history(c, pre(c), W)
    blank_r = np.full_like(kr, NAN)
    rk, rv = oracle.scatter_ring(c.hist_k, c.hist_v, pre(c), W, blank_r, blank_r)
    np.testing.assert_array_equal(rk, kr)
    np.testing.assert_array_equal(rv, vr)


# ---------------------------------------------------------------- P6 GQA
def test_gqa_equals_mha_on_repeated_kv():
    c = make_case(61, 2, 8, 2, 64, [12, 45])
    G = c.Hq // c.Hkv
    out = o_contig(c, 0)
    m = make_case(61, 2, 8, 2, 64, [12, 45])
    m.Hkv = c.Hq
    m.hist_k = np.ascontiguousarray(np.repeat(c.hist_k, G, axis=2))
    m.hist_v = np.ascontiguousarray(np.repeat(c.hist_v, G, axis=2))
    np.testing.assert_allclose(o_contig(m, 0), out, rtol=0, atol=1e-14)
    # a wrong head map (h % Hkv instead of h // G) must be distinguishable
    wrong = np.ascontiguousarray(np.tile(c.hist_k, (1, 1, G, 1)))
    m.hist_k = wrong
    m.hist_v = np.ascontiguousarray(np.tile(c.hist_v, (1, 1, G, 1)))
    assert np.abs(o_contig(m, 0) - out).max() > 1e-3


# ---------------------------------------------------------------- P7 append
def test_append_is_bit_exact_and_touches_only_target_cells():
    c = make_case(71, 4, 8, 2, 64, [1, 16, 17, 40])
    kp, vp, bt = paged_identity(c, pre(c), extra_pages_per_seq=1)
    kp, vp, bt = shuffle_pages(kp, vp, bt, 3, spare=5)
    ak, av = oracle.kv_append_paged(c.k_new, c.v_new, kp, vp, bt, c.lens)
    # the appended pool equals the one materialised with L tokens
    kl, vl, btl = paged_identity(c, c.lens, extra_pages_per_seq=1)
    kl, vl, _ = shuffle_pages(kl, vl, btl, 3, spare=5)
    np.testing.assert_array_equal(ak, kl)
    np.testing.assert_array_equal(av, vl)
    changed = int((ak != kp).sum() + (av != vp).sum())
    assert changed == 2 * int((c.lens > 0).sum()) * c.Hkv * c.D
    # fused append+attend equals attend on the appended cache without k_new
    np.testing.assert_allclose(o_paged(c, kp, vp, bt, fused=True),
                               o_paged(c, ak, av, bt, fused=False), rtol=0, atol=0)


@pytest.mark.parametrize("W", [16, 24])
def test_ring_append_evicts_oldest(W):
    c = make_case(72, 3, 8, 2, 64, [5, 16, 70])
    kr, vr = ring_from_history(c, pre(c), W)
    ak, av = oracle.kv_append_ring(c.k_new, c.v_new, kr, vr, c.lens, W)
    ek, ev = ring_from_history(c, c.lens, W)
    np.testing.assert_array_equal(ak, ek)
    np.testing.assert_array_equal(av, ev)
    np.testing.assert_allclose(o_ring(c, kr, vr, W, fused=True),
                               o_ring(c, ak, av, W, fused=False), rtol=0, atol=0)


# ---------------------------------------------------------------- P8 permutation invariance
def test_token_order_does_not_matter():
    c = make_case(81, 2, 8, 2, 64, [33, 64])
    out = o_contig(c, 0)
    rng = np.random.default_rng(0)
    for b in range(c.B):
        L = int(c.lens[b])
        perm = rng.permutation(L)
        c.hist_k[b, :L] = c.hist_k[b, perm]
        c.hist_v[b, :L] = c.hist_v[b, perm]
    np.testing.assert_allclose(o_contig(c, 0), out, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- hand-worked example
def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        g = json.load(f)
    enc = lambda x: f64_to_bf16_bits(np.asarray(x, np.float64))
    q = enc(g["q"])[None]                                  # [1, Hq, D]
    hk = enc(g["k"])[None, :, None, :]                     # [1, L, 1, D]
    hv = enc(g["v"])[None, :, None, :]
    L = hk.shape[1]
    lens = np.array([L], np.int32)
    sinks = np.asarray(g["sinks"], np.float32)
    expect = np.array([[eval(e, {"math": math}) for e in row] for row in g["expected"]])
    out = oracle.decode_contig(q, hk, hv, lens, sinks, 0, g["scale"])
    np.testing.assert_allclose(out[0], expect, rtol=1e-15, atol=1e-15)
    # the same example through the paged (page 2) and ring (W = L) readers
    kp = hk[0, :L - 1].reshape(1, L - 1, 1, -1).transpose(0, 2, 1, 3)
    pad_k = np.full((1, 1, 2, kp.shape[-1]), NAN, np.uint16)
    pad_v = pad_k.copy()
    pad_k[0, 0, :L - 1] = hk[0, :L - 1, 0]
    pad_v[0, 0, :L - 1] = hv[0, :L - 1, 0]
    outp = oracle.decode_paged(q, hk[:, L - 1], hv[:, L - 1], pad_k, pad_v,
                               np.array([[0]], np.int32), lens, sinks, 0, g["scale"], 2)
    np.testing.assert_allclose(outp[0], expect, rtol=1e-15, atol=1e-15)
