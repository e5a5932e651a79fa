"""The early-input levels (decode_attn_set_early_inputs): at level 1 each attention kernel
reads the lengths, block table and sinks and works out its split before it waits for the
kernel launched just before it, at level 2 it also fetches its first cache tiles into L2; the
query rows, new tokens and output (and the append) come after the wait.

Checked against the oracle: calls whose q / k_new / v_new and output buffer are written by
the kernel launched directly before them (so a read or write on the wrong side of the wait
would show), the edge-length, many-segment and long-sequence cases of the default order,
several-token and fp8 calls, and a captured multi-layer step; and the outputs of both
orders equal bit for bit on one mixed batch.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
import test_gpu_decode as gd
import test_gpu_fp8 as gf
import test_gpu_graph_step as gg
import test_gpu_multi as gm
from cases import make_case
from paged_decode_attention_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = gd.DEV


@pytest.fixture(params=[1, 2])
def early(request):
    prev = da.decode_attn_set_early_inputs(request.param)
    yield request.param
    da.decode_attn_set_early_inputs(prev)


def test_switch_returns_the_previous_level():
    prev = da.decode_attn_set_early_inputs(2)
    try:
        assert da.decode_attn_set_early_inputs(1) == 2
        assert da.decode_attn_set_early_inputs(0) == 1
        with pytest.raises(da.DecodeAttnError):
            da.decode_attn_set_early_inputs(3)
        assert da.decode_attn_set_early_inputs(0) == 0
    finally:
        da.decode_attn_set_early_inputs(prev)


def produced(src_bits):
    """A device bf16 tensor whose values an elementwise kernel writes just before use: the
    destination is first filled with NaN, then a conversion kernel writes the values."""
    src = gd.dev_bits(src_bits).float()
    dst = torch.full(src.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    return src, dst


@pytest.mark.parametrize("last", ["q", "k_new", "out"])
@pytest.mark.parametrize("ring", [False, True])
def test_inputs_written_by_the_kernel_just_before(early, ring, last):
    lens = [0, 1, 17, 300, 4100, 0, 129, 2000]
    c = make_case(900 + ring, len(lens), 64, 8, 64, lens)
    if ring:
        W = 128
        kr, vr = gd.ring_from_history(c, gd.pre(c), W)
        kc, vc = gd.dev_bits(kr), gd.dev_bits(vr)
        bt = None
    else:
        kp, vp, btn = gd.paged_setup(c, 11)
        kc, vc, bt = gd.dev_bits(kp), gd.dev_bits(vp), gd.dev(btn)
    sl = gd.dev(c.lens)
    sk = gd.dev(c.sinks)
    qs, q = produced(c.q)
    ks, kn = produced(c.k_new)
    vs, vn = produced(c.v_new)
    out = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)  # the producers queue up behind a spin
    producers = {"q": lambda: q.copy_(qs), "k_new": lambda: (kn.copy_(ks), vn.copy_(vs)),
                 "out": lambda: out.fill_(float("nan"))}
    for name in [n for n in producers if n != last] + [last]:  # `last` runs directly before
        producers[name]()
    if ring:
        da.decode_attn_ring(q, kn, vn, kc, vc, sl, sk, c.scale, out)
    else:
        da.decode_attn_paged(q, kn, vn, kc, vc, bt, sl, sk, 0, c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    got = out.double().cpu().numpy()
    if ring:
        ref = oracle.decode_ring(c.q, c.k_new, c.v_new, kr, vr, c.lens, c.sinks, W, c.scale)
        ek, ev = oracle.kv_append_ring(c.k_new, c.v_new, kr, vr, c.lens, W)
    else:
        ref = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, btn, c.lens, c.sinks, 0, c.scale, c.P)
        ek, ev = oracle.kv_append_paged(c.k_new, c.v_new, kp, vp, btn, c.lens)
    gd.assert_close(got, ref, "early inputs, producer kernels just before")
    np.testing.assert_array_equal(wl.bits(kc), ek)
    np.testing.assert_array_equal(wl.bits(vc), ev)


def test_edge_lengths(early):
    gd.test_paged_edge_lengths_all_groups(64, 8, 0)
    gd.test_paged_edge_lengths_all_groups(16, 4, 100)
    gd.test_ring_edge_lengths(128)
    gd.test_ring_other_groups(16, 1)


def test_inactive_slots_and_no_append(early):
    gd.test_inactive_slots()
    gd.test_no_sinks_and_no_append()


def test_many_segments_and_one_long_sequence(early):
    gd.test_many_short_and_a_few_long_sequences()
    gd.test_single_long_sequence_spans_every_cta()
    gd.test_repeated_calls_are_identical()


def test_same_bits_at_every_level():
    rng = np.random.default_rng(31)
    lens = [0] * 4 + list(rng.integers(1, 9000, size=40)) + [60000]
    c = make_case(920, len(lens), 64, 8, 64, lens)
    kp, vp, bt = gd.paged_setup(c, 13)
    outs = {}
    for level in (0, 1, 2):
        prev = da.decode_attn_set_early_inputs(level)
        try:
            outs[level], _, _ = gd.run_paged(c, kp, vp, bt, 0)
        finally:
            da.decode_attn_set_early_inputs(prev)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    ref = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, 0, c.scale, c.P)
    gd.assert_close(outs[2], ref, "early inputs, mixed batch")


@pytest.mark.parametrize("T", [2, 4])
def test_several_tokens(early, T):
    gm.test_paged_multi_matches_oracle(64, 8, T, 0)
    gm.test_paged_multi_matches_oracle(16, 4, T, 100)


def test_fp8(early):
    gf.test_paged_fp8_matches_oracle(64, 8, 0)
    gf.test_ring_fp8_matches_oracle(128)


def test_captured_step(early):
    gg.test_one_graph_serves_every_active_slot_set()


@pytest.mark.parametrize("W", [1000, 1024])
def test_long_ring_windows_prefetched_by_runs(W):
    """Level 2 on ring calls whose workers hold more tiles than their pipeline: each run of a
    worker's tiles in one window is prefetched as one range, up to the window's end (W = 1000
    ends inside a tile), then read as usual."""
    rng = np.random.default_rng(W)
    lens = [int(x) for x in rng.integers(W // 2, 3 * W, size=24)] + [0, W, W + 1]
    c = make_case(940 + W, len(lens), 64, 8, 64, lens)
    prev = da.decode_attn_set_early_inputs(2)
    try:
        gd.check_ring(c, W)
    finally:
        da.decode_attn_set_early_inputs(prev)


def test_long_fp8_ring_windows_prefetched_by_runs():
    W = 1024
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(W // 2, 3 * W, size=24)] + [0, W - 1]
    c = make_case(960, len(lens), 64, 8, 64, lens)
    blank = oracle.Fp8Cache.empty_ring(c.B, c.Hkv, W, c.D)
    cache = oracle.scatter_fp8(c.hist_k, c.hist_v, gf.pre(c), blank, window=W)
    kv = gf.to_dev(cache)
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    prev = da.decode_attn_set_early_inputs(2)
    try:
        da.decode_attn_ring_fp8(gd.dev_bits(c.q), gd.dev_bits(c.k_new), gd.dev_bits(c.v_new), kv,
                                gd.dev(c.lens), gd.dev(c.sinks), c.scale, out)
        torch.cuda.synchronize()
    finally:
        da.decode_attn_set_early_inputs(prev)
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_ring_fp8(c.q, c.k_new, c.v_new, cache, c.lens, c.sinks, W, c.scale)
    gd.assert_close(out.double().cpu().numpy(), ref, "ring fp8 W=1024, level 2")
    gf.assert_blocks_equal(gf.from_dev(kv), oracle.kv_append_fp8(c.k_new, c.v_new, cache, c.lens, window=W))
