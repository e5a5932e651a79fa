"""Calls on several streams at once (decode_attn_stream_reserve): each stream with workspaces
of its own, the calls of two or three streams queued behind a GPU spin so that they run at
the same time, every output checked against the oracle; the caches' appends bit-exact.
Also: a release returns the stream to the device workspace, a graph captured on a reserved
stream replays correctly, and reserving during a capture is refused."""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
import test_gpu_decode as gd
from cases import make_case
from paged_decode_attention_kv_gb300 import workloads as wl
from test_oracle_multi import Multi

pytestmark = pytest.mark.gpu
DEV = gd.DEV
REPEAT = 6  # calls per stream, each into an output buffer of its own


class PagedJob:
    """One paged one-token call, repeated: the fused append rewrites the same cell with the
    same values, so every repetition must give the same output."""

    def __init__(self, seed, lens, Hq=64, Hkv=8, window=0):
        self.c = c = make_case(seed, len(lens), Hq, Hkv, 64, lens)
        self.window = window
        self.kp, self.vp, self.bt = gd.paged_setup(c, seed)
        self.kd, self.vd = gd.dev_bits(self.kp), gd.dev_bits(self.vp)
        self.args = (gd.dev_bits(c.q), gd.dev_bits(c.k_new), gd.dev_bits(c.v_new), self.kd, self.vd,
                     gd.dev(self.bt), gd.dev(c.lens), gd.dev(c.sinks))
        self.outs = [torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
                     for _ in range(REPEAT)]
        torch.cuda.synchronize()  # made on the default stream, used on others

    def launch(self, i, stream):
        q, kn, vn, kd, vd, bt, sl, sk = self.args
        da.decode_attn_paged(q, kn, vn, kd, vd, bt, sl, sk, self.window, self.c.scale, self.outs[i],
                             stream=stream)

    def check(self):
        c = self.c
        ref = oracle.decode_paged(c.q, c.k_new, c.v_new, self.kp, self.vp, self.bt, c.lens, c.sinks,
                                  self.window, c.scale, c.P)
        for i, o in enumerate(self.outs):
            gd.assert_close(o.double().cpu().numpy(), ref, f"paged stream call {i}")
        ek, ev = oracle.kv_append_paged(c.k_new, c.v_new, self.kp, self.vp, self.bt, c.lens)
        np.testing.assert_array_equal(wl.bits(self.kd), ek)
        np.testing.assert_array_equal(wl.bits(self.vd), ev)


class RingJob:
    def __init__(self, seed, lens, W=128):
        self.c = c = make_case(seed, len(lens), 64, 8, 64, lens)
        self.W = W
        self.kr, self.vr = gd.ring_from_history(c, gd.pre(c), W)
        self.kd, self.vd = gd.dev_bits(self.kr), gd.dev_bits(self.vr)
        self.args = (gd.dev_bits(c.q), gd.dev_bits(c.k_new), gd.dev_bits(c.v_new), self.kd, self.vd,
                     gd.dev(c.lens), gd.dev(c.sinks))
        self.outs = [torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
                     for _ in range(REPEAT)]
        torch.cuda.synchronize()  # made on the default stream, used on others

    def launch(self, i, stream):
        q, kn, vn, kd, vd, sl, sk = self.args
        da.decode_attn_ring(q, kn, vn, kd, vd, sl, sk, self.c.scale, self.outs[i], stream=stream)

    def check(self):
        c = self.c
        ref = oracle.decode_ring(c.q, c.k_new, c.v_new, self.kr, self.vr, c.lens, c.sinks, self.W, c.scale)
        for i, o in enumerate(self.outs):
            gd.assert_close(o.double().cpu().numpy(), ref, f"ring stream call {i}")
        ek, ev = oracle.kv_append_ring(c.k_new, c.v_new, self.kr, self.vr, c.lens, self.W)
        np.testing.assert_array_equal(wl.bits(self.kd), ek)
        np.testing.assert_array_equal(wl.bits(self.vd), ev)


class MultiJob:
    """A several-token paged call (T = 2: the decode kernel's form; T = 8: the tcgen05
    kernel and its split fold)."""

    def __init__(self, seed, lens, T):
        n = [min(T, L) for L in lens]
        self.m = m = Multi(seed, 64, 8, lens, n, T)
        self.kp, self.vp, self.bt = m.paged(seed)
        self.kd, self.vd = gd.dev_bits(self.kp), gd.dev_bits(self.vp)
        c = m.c
        self.args = (gd.dev_bits(m.q), gd.dev_bits(m.k_new), gd.dev_bits(m.v_new), self.kd, self.vd,
                     gd.dev(self.bt), gd.dev(m.lens), gd.dev(m.sinks), gd.dev(m.n))
        self.outs = [torch.full((c.B, T, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
                     for _ in range(REPEAT)]
        torch.cuda.synchronize()

    def launch(self, i, stream):
        q, kn, vn, kd, vd, bt, sl, sk, ql = self.args
        da.decode_attn_paged_multi(q, kn, vn, kd, vd, bt, sl, sk, 0, self.m.c.scale, self.outs[i],
                                   q_lens=ql, stream=stream)

    def check(self):
        m = self.m
        ref = oracle.decode_multi(m.q, m.k_new, m.v_new, self.kp, self.vp, m.lens, m.sinks, 0, m.c.scale,
                                  block_table=self.bt, q_lens=m.n)
        for i, o in enumerate(self.outs):
            gd.assert_close(o.double().cpu().numpy(), ref, f"multi T={m.T} stream call {i}")
        ek, ev = oracle.kv_append_multi(m.k_new, m.v_new, self.kp, self.vp, m.lens, block_table=self.bt,
                                        q_lens=m.n)
        np.testing.assert_array_equal(wl.bits(self.kd), ek)
        np.testing.assert_array_equal(wl.bits(self.vd), ev)


def run_concurrently(jobs):
    """Each job on a stream of its own with its own workspaces; all streams held behind a
    spin, then their calls interleaved at launch so the kernels of different streams run
    side by side."""
    streams = [torch.cuda.Stream() for _ in jobs]
    try:
        for s in streams:
            da.decode_attn_stream_reserve(s)
            with torch.cuda.stream(s):
                torch.cuda._sleep(1_000_000)
        for i in range(REPEAT):
            for job, s in zip(jobs, streams):
                job.launch(i, s)
        torch.cuda.synchronize()
        assert da.decode_attn_device_status() == 0
    finally:
        for s in streams:
            da.decode_attn_stream_release(s)
    for job in jobs:
        job.check()


def test_paged_and_ring_layers_on_two_streams():
    rng = np.random.default_rng(3)
    lens_a = [0, 1, 17, 4100, 129, 2000] + [int(x) for x in rng.integers(1, 3000, size=18)]
    lens_b = [int(x) for x in rng.integers(1, 700, size=40)] + [0, 128, 129]
    run_concurrently([PagedJob(1201, lens_a), RingJob(1202, lens_b)])


def test_three_paged_streams_with_long_sequences():
    """Long sequences spread over every CTA, so each call's segments cross CTAs and use
    the arrival counters of its workspace."""
    run_concurrently([PagedJob(1211, [30000, 5, 70]), PagedJob(1212, [20000, 20000], window=1000),
                      PagedJob(1213, [1, 9000, 12000, 3], Hq=32, Hkv=2)])


@pytest.mark.parametrize("T", [2, 8])
def test_several_tokens_beside_a_one_token_call(T):
    run_concurrently([MultiJob(1220 + T, [3000, 17, 1, 9000, 640, 0], T),
                      PagedJob(1230 + T, [8000, 1, 200, 4096, 33])])


def test_release_returns_to_the_device_workspace():
    s = torch.cuda.Stream()
    assert da.decode_attn_stream_release(s) is None  # nothing reserved: fine
    da.decode_attn_stream_reserve(s, 1 << 20, 1 << 20)
    da.decode_attn_stream_reserve(s, 1 << 16)  # already large enough: kept
    job = PagedJob(1240, [5000, 3, 1000])
    job.launch(0, s)
    da.decode_attn_stream_release(s)
    for i in range(1, REPEAT):
        job.launch(i, s)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    job.check()


def test_graph_captured_on_a_reserved_stream():
    s = torch.cuda.Stream()
    job = PagedJob(1250, [7000, 12, 300, 2500])
    da.decode_attn_stream_reserve(
        s, da.decode_attn_workspace_bytes(job.c.B, job.c.Hq, job.c.Hkv))
    try:
        with torch.cuda.stream(s):
            job.launch(0, s)  # warm the library's per-kernel set-up outside the capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(1, REPEAT):
                job.launch(i, s)
        with torch.cuda.stream(s):
            for o in job.outs[1:]:
                o.fill_(float("nan"))
            g.replay()
        s.synchronize()
        assert da.decode_attn_device_status() == 0
        job.check()
        del g
    finally:
        da.decode_attn_stream_release(s)


def test_reserving_during_a_capture_is_refused():
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    x = torch.zeros(4, device=DEV)
    with torch.cuda.graph(g, stream=s):
        x.add_(1)
        with pytest.raises(da.DecodeAttnError) as e:
            da.decode_attn_stream_reserve(s, 1 << 20)
        assert e.value.code == da.DA_ERR_WORKSPACE
    del g
