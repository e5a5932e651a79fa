"""GPU parity of the several-token steps with the rotary embedding
(decode_attn_paged_multi_rope / _ring_multi_rope) against the fp64 oracle
(oracle.decode_multi_rope): every output row within 4e-3 + 1e-2 |oracle| (rows beyond q_lens
and inactive slots exactly zero), the rotated new keys stored bit-exactly (both sides round
them the same way), every route of the several-token step (the decode kernel's forms at 2-4
tokens, the row-block kernel, tcgen05 and its split fold), identity tables equal to the plain
call, q and k_new left untouched, a position beyond the tables reported, a captured graph."""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
from paged_decode_attention_kv_gb300 import workloads as wl
from test_gpu_decode import DEV, assert_close, dev, dev_bits
from test_oracle_multi import Multi

pytestmark = pytest.mark.gpu


def _tables(maxpos, kind="real"):
    if kind == "identity":
        return np.ones((maxpos, 32), np.float32), np.zeros((maxpos, 32), np.float32)
    return wl.rope_tables(maxpos, 64)


def run_paged(m, window, cs, sn, seed=1):
    kp, vp, bt = m.paged(seed)
    kd, vd = dev_bits(kp), dev_bits(vp)
    c = m.c
    q, kn = dev_bits(m.q), dev_bits(m.k_new)
    out = torch.full((c.B, m.T, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_multi_rope(q, kn, dev_bits(m.v_new), kd, vd, dev(bt), dev(m.lens),
                                    dev(m.sinks), dev(cs), dev(sn), window, c.scale, out,
                                    q_lens=dev(m.n))
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    np.testing.assert_array_equal(wl.bits(q), m.q)        # inputs untouched
    np.testing.assert_array_equal(wl.bits(kn), m.k_new)
    ref = oracle.decode_multi_rope(m.q, m.k_new, m.v_new, kp, vp, m.lens, m.sinks, cs, sn, window,
                                   c.scale, block_table=bt, q_lens=m.n)
    assert_close(out.double().cpu().numpy(), ref, f"paged multi rope T={m.T} window={window}")
    _, krot = oracle.rope_multi(m.q, m.k_new, m.lens, cs, sn, q_lens=m.n)
    ek, ev = oracle.kv_append_multi(krot, m.v_new, kp, vp, m.lens, block_table=bt, q_lens=m.n)
    np.testing.assert_array_equal(wl.bits(kd), ek)         # the rotated keys, bit for bit
    np.testing.assert_array_equal(wl.bits(vd), ev)
    return out


def run_ring(m, W, cs, sn):
    kr, vr = m.ring(W)
    kd, vd = dev_bits(kr), dev_bits(vr)
    c = m.c
    out = torch.full((c.B, m.T, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_ring_multi_rope(dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new), kd, vd,
                                   dev(m.lens), dev(m.sinks), dev(cs), dev(sn), c.scale, out,
                                   q_lens=dev(m.n))
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_multi_rope(m.q, m.k_new, m.v_new, kr, vr, m.lens, m.sinks, cs, sn, W,
                                   c.scale, q_lens=m.n)
    assert_close(out.double().cpu().numpy(), ref, f"ring multi rope T={m.T} W={W}")
    _, krot = oracle.rope_multi(m.q, m.k_new, m.lens, cs, sn, q_lens=m.n)
    ek, ev = oracle.kv_append_multi(krot, m.v_new, kr, vr, m.lens, window=W, q_lens=m.n)
    np.testing.assert_array_equal(wl.bits(kd), ek)
    np.testing.assert_array_equal(wl.bits(vd), ev)


def counts(T, lens, seed):
    rng = np.random.default_rng(seed)
    n = [int(rng.integers(1, min(T, L) + 1)) if L > 0 else 0 for L in lens]
    for i, L in enumerate(lens):
        if L >= T:
            n[i] = T
            break
    return n


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (16, 1), (32, 4)])
@pytest.mark.parametrize("T", [2, 3, 4, 5, 16])
@pytest.mark.parametrize("window", [0, 100])
def test_paged_multi_rope_matches_oracle(Hq, Hkv, T, window):
    lens = [1, 4, 15, 16, 17, 33, 100, 257, 0, 1500]
    m = Multi(1300 + Hq + T + window, Hq, Hkv, lens, counts(T, lens, T), T)
    run_paged(m, window, *_tables(2048))


@pytest.mark.parametrize("T", [3, 16])
@pytest.mark.parametrize("W", [16, 128])
def test_ring_multi_rope_matches_oracle(W, T):
    lens = [1, 16, 17, W + 1, 700, 0]
    m = Multi(1340 + W + T, 64, 8, lens, counts(T, lens, W + T), T)
    run_ring(m, W, *_tables(1024))


@pytest.mark.parametrize("T", [4, 16])
def test_long_history_many_splits(T):
    """A 20k-token sequence: its keys split over many CTAs (the 32-row decode form at 4
    tokens; tcgen05 and its fold kernel at 16), each new token at its own position."""
    m = Multi(1360 + T, 64, 8, [20000, 3000], [T, T - 1], T)
    run_paged(m, 0, *_tables(20100))
    run_paged(m, 1000, *_tables(20100))


def test_identity_tables_equal_the_plain_call():
    lens = [3, 40, 700, 0]
    m = Multi(1370, 64, 8, lens, [3, 4, 2, 0], 4)
    kp, vp, bt = m.paged(2)
    got = run_paged(m, 0, *_tables(1024, "identity"), seed=2)
    out = torch.full_like(got, float("nan"))
    kd, vd = dev_bits(kp), dev_bits(vp)
    da.decode_attn_paged_multi(dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new), kd, vd, dev(bt),
                               dev(m.lens), dev(m.sinks), 0, m.c.scale, out, q_lens=dev(m.n))
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), out.view(torch.int16))


def test_position_beyond_the_tables_is_reported():
    m = Multi(1380, 64, 8, [10, 300], [2, 3], 3)
    kp, vp, bt = m.paged(1)
    cs, sn = _tables(100)   # positions 297..299 are beyond the 100 rows
    out = torch.empty((2, 3, 64, 64), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_multi_rope(dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new), dev_bits(kp),
                                    dev_bits(vp), dev(bt), dev(m.lens), dev(m.sinks), dev(cs), dev(sn),
                                    0, m.c.scale, out, q_lens=dev(m.n))
    assert da.decode_attn_device_status() & da.DA_STATUS_BAD_POSITION


def test_null_tables_are_refused():
    m = Multi(1381, 8, 8, [10], [2], 2)
    kp, vp, bt = m.paged(1)
    out = torch.empty((1, 2, 8, 64), dtype=torch.bfloat16, device=DEV)
    cs, _ = _tables(64)
    with pytest.raises(da.DecodeAttnError):
        lib = da.load_library()
        rc = lib.decode_attn_paged_multi_rope(
            da._ptr(dev_bits(m.q)), da._ptr(dev_bits(m.k_new)), da._ptr(dev_bits(m.v_new)),
            da._ptr(dev_bits(kp)), da._ptr(dev_bits(vp)), da._ptr(dev(bt)), da._ptr(dev(m.lens)), None,
            da._ptr(dev(m.sinks)), da._ptr(dev(cs)), None, 64, 0, m.c.scale, da._ptr(out),
            da.da_shape(1, 8, 8, 64), 2, 16, bt.shape[1], kp.shape[0], bt.shape[1] * 16, None)
        da._check(rc)


def test_captured_graph_replays():
    """A graph captured once (the workspace reserved first, so the capture allocates
    nothing) and replayed on fresh pools: the rotation kernel and the attention are both in
    the graph."""
    T = 4
    lens = [40, 900, 5, 300]
    m = Multi(1390, 64, 8, lens, [4, 4, 4, 2], T)
    cs, sn = _tables(2048)
    kp, vp, bt = m.paged(3)
    c = m.c
    da.decode_attn_multi_reserve(da.decode_attn_multi_workspace_bytes(c.B, c.Hq, c.Hkv, T, 0,
                                                                     bt.shape[1] * 16))
    q, kn, vn = dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new)
    kd, vd = dev_bits(kp), dev_bits(vp)
    tb, sl, ql, sk, dcs, dsn = dev(bt), dev(m.lens), dev(m.n), dev(m.sinks), dev(cs), dev(sn)
    out = torch.full((c.B, T, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    call = lambda: da.decode_attn_paged_multi_rope(q, kn, vn, kd, vd, tb, sl, sk, dcs, dsn, 0,
                                                   c.scale, out, q_lens=ql)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    # the same step again on fresh pools, through the graph
    kd.copy_(dev_bits(kp))
    vd.copy_(dev_bits(vp))
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_multi_rope(m.q, m.k_new, m.v_new, kp, vp, m.lens, m.sinks, cs, sn, 0,
                                   c.scale, block_table=bt, q_lens=m.n)
    assert_close(out.double().cpu().numpy(), ref, "graph replay, multi rope")
