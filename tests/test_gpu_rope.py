"""GPU parity of the fused rotary embedding (decode_attn_paged_rope / _ring_rope)
against the fp64 oracle: attention within 4e-3 + 1e-2 |oracle|, the rotated
new key stored bit-exactly (both sides round it the same way), identity
tables equal to the plain call, full-size workloads on sampled heads."""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
from paged_decode_attention_kv_gb300 import workloads as wl
from cases import make_case, paged_identity, ring_from_history, shuffle_pages
from test_gpu_decode import DEV, assert_close, dev, dev_bits, full_workload, pre

pytestmark = pytest.mark.gpu


def _tables(maxpos, D=64, kind="real"):
    if kind == "identity":
        return np.ones((maxpos, D // 2), np.float32), np.zeros((maxpos, D // 2), np.float32)
    return wl.rope_tables(maxpos, D)


def run_paged_rope(c, kp, vp, bt, window, cs, sn):
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    kd, vd = dev_bits(kp), dev_bits(vp)
    da.decode_attn_paged_rope(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), kd, vd, dev(bt),
                              dev(c.lens), dev(c.sinks), dev(cs), dev(sn), window, c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    return out.double().cpu().numpy(), wl.bits(kd), wl.bits(vd)


@pytest.mark.parametrize("Hq,Hkv,window", [(64, 8, 0), (8, 8, 0), (16, 1, 0), (64, 8, 100)])
def test_paged_rope_matches_oracle(Hq, Hkv, window):
    lens = [1, 2, 15, 17, 100, 257, 3000]
    c = make_case(500 + Hq + window, len(lens), Hq, Hkv, 64, lens)
    cs, sn = _tables(4096)
    kp, vp, bt = shuffle_pages(*paged_identity(c, pre(c)), 3)
    got, ak, av = run_paged_rope(c, kp, vp, bt, window, cs, sn)
    ref = oracle.decode_paged_rope(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, cs, sn,
                                   window, c.scale, 16)
    assert_close(got, ref, "paged rope")
    krot = oracle.rope_k(c.k_new, c.lens, cs, sn)
    ek, ev = oracle.kv_append_paged(krot, c.v_new, kp, vp, bt, c.lens)
    np.testing.assert_array_equal(ak, ek)   # the rotated key, bit for bit
    np.testing.assert_array_equal(av, ev)


@pytest.mark.parametrize("W", [16, 128])
def test_ring_rope_matches_oracle(W):
    lens = [1, 16, 17, W + 1, 5000]
    c = make_case(520 + W, len(lens), 64, 8, 64, lens)
    cs, sn = _tables(8192)
    kr, vr = ring_from_history(c, pre(c), W)
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    kd, vd = dev_bits(kr), dev_bits(vr)
    da.decode_attn_ring_rope(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), kd, vd,
                             dev(c.lens), dev(c.sinks), dev(cs), dev(sn), c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_ring_rope(c.q, c.k_new, c.v_new, kr, vr, c.lens, c.sinks, cs, sn, W,
                                  c.scale)
    assert_close(out.double().cpu().numpy(), ref, "ring rope")
    krot = oracle.rope_k(c.k_new, c.lens, cs, sn)
    ek, ev = oracle.kv_append_ring(krot, c.v_new, kr, vr, c.lens, W)
    np.testing.assert_array_equal(wl.bits(kd), ek)
    np.testing.assert_array_equal(wl.bits(vd), ev)


def test_identity_tables_equal_the_plain_call():
    lens = [3, 40, 700]
    c = make_case(530, len(lens), 64, 8, 64, lens)
    cs, sn = _tables(1024, kind="identity")
    kp, vp, bt = shuffle_pages(*paged_identity(c, pre(c)), 4)
    got, ak, _ = run_paged_rope(c, kp, vp, bt, 0, cs, sn)
    out = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=DEV)
    kd, vd = dev_bits(kp), dev_bits(vp)
    da.decode_attn_paged(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), kd, vd, dev(bt),
                         dev(c.lens), dev(c.sinks), 0, c.scale, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got, out.double().cpu().numpy())
    np.testing.assert_array_equal(ak, wl.bits(kd))


def test_position_beyond_the_tables_is_reported():
    c = make_case(540, 2, 64, 8, 64, [10, 300])
    cs, sn = _tables(100)     # position 299 is beyond the 100 rows
    kp, vp, bt = paged_identity(c, pre(c))
    out = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_rope(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), dev_bits(kp),
                              dev_bits(vp), dev(bt), dev(c.lens), dev(c.sinks), dev(cs), dev(sn),
                              0, c.scale, out)
    assert da.decode_attn_device_status() & da.DA_STATUS_BAD_POSITION


@pytest.mark.parametrize("name", ["b64", "long1"])
def test_full_size_workload_with_rope(name):
    cfg, lens, inp, pool, ring = full_workload(name)
    Hq, W = cfg["Hq"], cfg["window"]
    cs, sn = _tables(max(lens) + 1)
    q, kn, vn = dev(inp.q), dev(inp.k_new), dev(inp.v_new)
    sl, sk = dev(inp.seq_lens), dev(inp.sinks)
    k_pre, v_pre = wl.bits(pool.k_cache), wl.bits(pool.v_cache)
    out = torch.empty((cfg["B"], Hq, cfg["D"]), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_rope(q, kn, vn, pool.k_cache, pool.v_cache, pool.block_table, sl, sk,
                              dev(cs), dev(sn), 0, inp.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_paged_rope(wl.bits(inp.q), wl.bits(inp.k_new), wl.bits(inp.v_new), k_pre,
                                   v_pre, pool.block_table.cpu().numpy(), np.asarray(lens, np.int32),
                                   inp.sinks.numpy(), cs, sn, 0, inp.scale, cfg["page_size"])
    assert_close(out.double().cpu().numpy(), ref, f"{name} paged rope")
    krot = oracle.rope_k(wl.bits(inp.k_new), np.asarray(lens, np.int32), cs, sn)
    ek, _ = oracle.kv_append_paged(krot, wl.bits(inp.v_new), k_pre, v_pre,
                                   pool.block_table.cpu().numpy(), np.asarray(lens, np.int32))
    assert np.array_equal(wl.bits(pool.k_cache), ek)
