"""GPU parity of the fused decode-attention path against the fp64 CPU oracle,
called through the C ABI (via the thin Python binding).

Bar: attention outputs within |gpu - oracle| <= 4e-3 + 1e-2 |oracle| on bf16
inputs; the KV append bit-exact, with every other cache byte unchanged
(dead cells are NaN-poisoned, so a stray read shows up as NaN and a stray
write as a changed byte).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
from paged_decode_attention_kv_gb300 import workloads as wl
from cases import NAN, make_case, paged_identity, ring_from_history, shuffle_pages

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1e-2
DEV = "cuda"


def dev_bits(a):
    return wl.from_bits(a, DEV)


def dev(t):
    return torch.as_tensor(t).to(DEV).contiguous()


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: |gpu-oracle| exceeds tolerance at {worst}: "
                               f"gpu {got[worst]:.6f} oracle {ref[worst]:.6f}")


def run_paged(c, kp, vp, bt, window, fused=True, sinks=True, max_seq_len=None):
    """Run the GPU path; returns (out as float64, k pool after, v pool after)."""
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    kd, vd = dev_bits(kp), dev_bits(vp)
    da.decode_attn_paged(dev_bits(c.q), dev_bits(c.k_new) if fused else None,
                         dev_bits(c.v_new) if fused else None, kd, vd, dev(bt), dev(c.lens),
                         dev(c.sinks) if sinks else None, window, c.scale, out,
                         max_seq_len=max_seq_len)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    return out.double().cpu().numpy(), wl.bits(kd), wl.bits(vd)


def run_ring(c, kr, vr, W, fused=True, sinks=True):
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    kd, vd = dev_bits(kr), dev_bits(vr)
    da.decode_attn_ring(dev_bits(c.q), dev_bits(c.k_new) if fused else None,
                        dev_bits(c.v_new) if fused else None, kd, vd, dev(c.lens),
                        dev(c.sinks) if sinks else None, c.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    return out.double().cpu().numpy(), wl.bits(kd), wl.bits(vd)


def pre(c):
    return np.maximum(c.lens - 1, 0)


def paged_setup(c, seed, spare=5, appended=False):
    """Pools before this step's append (fused calls) or after it (calls without k_new)."""
    kp, vp, bt = paged_identity(c, c.lens if appended else pre(c))
    return shuffle_pages(kp, vp, bt, seed, spare=spare)


def check_paged(c, window, seed=0, fused=True, sinks=True):
    kp, vp, bt = paged_setup(c, seed, appended=not fused)
    got, ak, av = run_paged(c, kp, vp, bt, window, fused=fused, sinks=sinks)
    ref = oracle.decode_paged(c.q, c.k_new if fused else None, c.v_new if fused else None, kp, vp,
                              bt, c.lens, c.sinks if sinks else None, window, c.scale, c.P)
    assert_close(got, ref, f"paged window={window}")
    if fused:
        ek, ev = oracle.kv_append_paged(c.k_new, c.v_new, kp, vp, bt, c.lens)
        np.testing.assert_array_equal(ak, ek)
        np.testing.assert_array_equal(av, ev)
    else:
        np.testing.assert_array_equal(ak, kp)
        np.testing.assert_array_equal(av, vp)


def check_ring(c, W, fused=True, sinks=True):
    kr, vr = ring_from_history(c, pre(c) if fused else c.lens, W)
    got, ak, av = run_ring(c, kr, vr, W, fused=fused, sinks=sinks)
    ref = oracle.decode_ring(c.q, c.k_new if fused else None, c.v_new if fused else None, kr, vr,
                             c.lens, c.sinks if sinks else None, W, c.scale)
    assert_close(got, ref, f"ring W={W}")
    if fused:
        ek, ev = oracle.kv_append_ring(c.k_new, c.v_new, kr, vr, c.lens, W)
        np.testing.assert_array_equal(ak, ek)
        np.testing.assert_array_equal(av, ev)


# ------------------------------------------------------------------ the tiny workload
def test_tiny_workload_paged_and_ring():
    cfg = wl.config("tiny")
    c = make_case(cfg["seed"], cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["lens"],
                  P=cfg["page_size"])
    check_paged(c, 0, seed=cfg["seed"])
    check_ring(c, cfg["window"])


# ------------------------------------------------------------------ edge lengths, every G
EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 100, 257]


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (16, 4), (64, 8), (32, 2)])
@pytest.mark.parametrize("window", [0, 1, 7, 16, 100])
def test_paged_edge_lengths_all_groups(Hq, Hkv, window):
    c = make_case(100 + Hq + Hkv + window, len(EDGE_LENS), Hq, Hkv, 64, EDGE_LENS)
    check_paged(c, window, seed=window)


@pytest.mark.parametrize("W", [16, 24, 128, 130])
def test_ring_edge_lengths(W):
    lens = [1, 15, 16, 17, W - 1, W, W + 1, 3 * W + 5]
    c = make_case(200 + W, len(lens), 64, 8, 64, lens)
    check_ring(c, W)


@pytest.mark.parametrize("Hq,Hkv", [(16, 1), (8, 8), (4, 2)])
def test_ring_other_groups(Hq, Hkv):
    lens = [3, 40, 200]
    c = make_case(250 + Hq, len(lens), Hq, Hkv, 64, lens)
    check_ring(c, 32)


def test_no_sinks_and_no_append():
    c = make_case(300, 4, 64, 8, 64, [5, 64, 65, 300])
    check_paged(c, 0, sinks=False)
    check_paged(c, 0, fused=False)
    check_paged(c, 0, fused=False, sinks=False)
    check_ring(c, 128, sinks=False)
    check_ring(c, 128, fused=False)


def test_inactive_slots():
    c = make_case(310, 6, 64, 8, 64, [0, 50, 0, 0, 17, 0])
    check_paged(c, 0)
    check_paged(c, 128)
    check_ring(c, 128)
    c0 = make_case(311, 3, 64, 8, 64, [0, 0, 0])
    check_paged(c0, 0)
    check_ring(c0, 16)


# ------------------------------------------------------------------ work decomposition
def test_many_short_and_a_few_long_sequences():
    """Hundreds of segments per CTA, segments split across warps and across CTAs."""
    rng = np.random.default_rng(7)
    lens = list(rng.integers(1, 70, size=300)) + [1500, 700, 1]
    c = make_case(320, len(lens), 16, 2, 64, lens)
    check_paged(c, 0, seed=1)
    check_paged(c, 128, seed=2)
    check_ring(c, 128)


def test_single_long_sequence_spans_every_cta():
    c = make_case(330, 1, 64, 8, 64, [40000])
    check_paged(c, 0, seed=3)
    check_paged(c, 1000, seed=4)


def test_repeated_calls_are_identical():
    """Arrival counters must be back at zero after every call."""
    rng = np.random.default_rng(9)
    lens = list(rng.integers(1000, 9000, size=12))
    c = make_case(340, len(lens), 64, 8, 64, lens)
    kp, vp, bt = paged_setup(c, 5)
    outs = []
    for _ in range(3):
        got, _, _ = run_paged(c, kp, vp, bt, 0)
        outs.append(got)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


# ------------------------------------------------------------------ the append alone
def test_kv_append_kernel_bit_exact():
    c = make_case(350, 5, 64, 8, 64, [1, 16, 17, 200, 0])
    kp, vp, bt = paged_setup(c, 6)
    kd, vd = dev_bits(kp), dev_bits(vp)
    da.kv_append(dev_bits(c.k_new), dev_bits(c.v_new), kd, vd, dev(c.lens), block_table=dev(bt))
    torch.cuda.synchronize()
    ek, ev = oracle.kv_append_paged(c.k_new, c.v_new, kp, vp, bt, c.lens)
    np.testing.assert_array_equal(wl.bits(kd), ek)
    np.testing.assert_array_equal(wl.bits(vd), ev)
    for W in (16, 128):
        kr, vr = ring_from_history(c, pre(c), W)
        kd, vd = dev_bits(kr), dev_bits(vr)
        da.kv_append(dev_bits(c.k_new), dev_bits(c.v_new), kd, vd, dev(c.lens))
        torch.cuda.synchronize()
        ek, ev = oracle.kv_append_ring(c.k_new, c.v_new, kr, vr, c.lens, W)
        np.testing.assert_array_equal(wl.bits(kd), ek)
        np.testing.assert_array_equal(wl.bits(vd), ev)
    assert da.decode_attn_device_status() == 0


def test_append_then_attend_equals_fused():
    c = make_case(360, 3, 64, 8, 64, [9, 33, 400])
    kp, vp, bt = paged_setup(c, 7)
    fused, _, _ = run_paged(c, kp, vp, bt, 0, fused=True)
    kd, vd = dev_bits(kp), dev_bits(vp)
    da.kv_append(dev_bits(c.k_new), dev_bits(c.v_new), kd, vd, dev(c.lens), block_table=dev(bt))
    out = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged(dev_bits(c.q), None, None, kd, vd, dev(bt), dev(c.lens), dev(c.sinks), 0,
                         c.scale, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.double().cpu().numpy(), fused)


# ------------------------------------------------------------------ device status word
def test_bad_lengths_and_pages_are_reported_not_faulted():
    c = make_case(370, 3, 64, 8, 64, [20, 40, 60])
    kp, vp, bt = paged_setup(c, 8)
    # a length beyond the declared max_seq_len -> that slot is inactive, status bit set
    out = torch.full((c.B, c.Hq, c.D), 1.0, dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), dev_bits(kp),
                         dev_bits(vp), dev(bt), dev(c.lens), dev(c.sinks), 0, c.scale, out,
                         max_seq_len=50)
    assert da.decode_attn_device_status() & da.DA_STATUS_BAD_SEQ_LEN
    assert torch.all(out[2] == 0)
    # a block-table entry outside the pool -> read as zeros, status bit set, no fault
    bt2 = bt.copy()
    bt2[1, 0] = kp.shape[0] + 1000
    out2 = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), dev_bits(kp),
                         dev_bits(vp), dev(bt2), dev(c.lens), dev(c.sinks), 0, c.scale, out2)
    assert da.decode_attn_device_status() & da.DA_STATUS_BAD_PAGE
    assert da.decode_attn_device_status() == 0  # cleared by the read


# ------------------------------------------------------------------ full-size workloads
def full_workload(name, device=DEV):
    """Benchmark-style inputs: random pools, shuffled block tables, the recipe's lengths."""
    cfg = wl.config(name)
    lens = wl.seq_lens(name)
    gen = wl.cpu_generator(cfg["seed"])
    vgen = torch.Generator(device=device)
    vgen.manual_seed(cfg["seed"])
    B, Hq, Hkv, D, P, W = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["page_size"], cfg["window"]
    inp = wl.draw_decode_inputs(B, Hq, Hkv, D, lens, gen)
    pool = wl.draw_paged_pool(wl.pool_size(name, lens), Hkv, P, D, lens,
                              wl.max_pages_per_seq(name, lens), gen, device=device,
                              value_gen=vgen)
    ring = wl.draw_ring_pool(B, Hkv, W, D, vgen, device=device)
    return cfg, lens, inp, pool, ring


@pytest.mark.parametrize("name", ["b1", "b64", "long1", "long8", "serve"])
def test_full_size_workload(name):
    cfg, lens, inp, pool, ring = full_workload(name)
    Hq, W = cfg["Hq"], cfg["window"]
    q, kn, vn = dev(inp.q), dev(inp.k_new), dev(inp.v_new)
    sl, sk = dev(inp.seq_lens), dev(inp.sinks)
    k_pre, v_pre = wl.bits(pool.k_cache), wl.bits(pool.v_cache)
    out = torch.empty((cfg["B"], Hq, cfg["D"]), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged(q, kn, vn, pool.k_cache, pool.v_cache, pool.block_table, sl, sk, 0,
                         inp.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    # every output row against the oracle (well under a second of host time per workload)
    ref = oracle.decode_paged(wl.bits(inp.q), wl.bits(inp.k_new), wl.bits(inp.v_new), k_pre, v_pre,
                              pool.block_table.cpu().numpy(), np.asarray(lens, np.int32),
                              inp.sinks.numpy(), 0, inp.scale, cfg["page_size"])
    assert_close(out.double().cpu().numpy(), ref, f"{name} paged")
    ek, ev = oracle.kv_append_paged(wl.bits(inp.k_new), wl.bits(inp.v_new), k_pre, v_pre,
                                    pool.block_table.cpu().numpy(), np.asarray(lens, np.int32))
    assert np.array_equal(wl.bits(pool.k_cache), ek) and np.array_equal(wl.bits(pool.v_cache), ev)
    del k_pre, v_pre, ek, ev
    # the window-128 ring layer of the same step
    rk_pre, rv_pre = wl.bits(ring.k_cache), wl.bits(ring.v_cache)
    da.decode_attn_ring(q, kn, vn, ring.k_cache, ring.v_cache, sl, sk, inp.scale, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_ring(wl.bits(inp.q), wl.bits(inp.k_new), wl.bits(inp.v_new), rk_pre,
                             rv_pre, np.asarray(lens, np.int32), inp.sinks.numpy(), W, inp.scale)
    assert_close(out.double().cpu().numpy(), ref, f"{name} ring")
    ek, ev = oracle.kv_append_ring(wl.bits(inp.k_new), wl.bits(inp.v_new), rk_pre, rv_pre,
                                   np.asarray(lens, np.int32), W)
    assert np.array_equal(wl.bits(ring.k_cache), ek) and np.array_equal(wl.bits(ring.v_cache), ev)


# ------------------------------------------------------------------ CUDA graph capture
def test_cuda_graph_capture_and_replay_with_new_lengths():
    """Serving-mix shapes (256 slots, block tables of 2048 pages) captured once;
    lengths, block tables and inputs then change in place between replays."""
    cfg, lens, inp, pool, ring = full_workload("serve")
    B, Hq, Hkv, D, W = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["window"]
    q, kn, vn = dev(inp.q), dev(inp.k_new), dev(inp.v_new)
    sl, sk, bt = dev(inp.seq_lens), dev(inp.sinks), pool.block_table
    out_p = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
    out_r = torch.empty_like(out_p)
    da.decode_attn_reserve(da.decode_attn_workspace_bytes(B, Hq, Hkv, D))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture: module load, kernel attributes
        da.decode_attn_paged(q, kn, vn, pool.k_cache, pool.v_cache, bt, sl, sk, 0, inp.scale, out_p)
        da.decode_attn_ring(q, kn, vn, ring.k_cache, ring.v_cache, sl, sk, inp.scale, out_r)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            da.decode_attn_paged(q, kn, vn, pool.k_cache, pool.v_cache, bt, sl, sk, 0, inp.scale,
                                 out_p)
            da.decode_attn_ring(q, kn, vn, ring.k_cache, ring.v_cache, sl, sk, inp.scale, out_r)
    torch.cuda.synchronize()
    # new step: shorter lengths (every sequence shrinks, some slots go idle), new inputs
    rng = np.random.default_rng(21)
    new_lens = np.array([int(rng.integers(0, L + 1)) if L > 0 else 0 for L in lens], np.int32)
    new_lens[rng.choice(B, 16, replace=False)] = 0
    gen = wl.cpu_generator(99)
    new = wl.draw_decode_inputs(B, Hq, Hkv, D, new_lens.tolist(), gen)
    q.copy_(new.q.to(DEV)); kn.copy_(new.k_new.to(DEV)); vn.copy_(new.v_new.to(DEV))
    sl.copy_(torch.from_numpy(new_lens).to(DEV))
    # and a rewritten block table (pages handed out again from a new shuffle)
    bt_new = wl.draw_block_table(new_lens.tolist(), cfg["page_size"], pool.num_pages,
                                 pool.max_pages_per_seq, gen)
    bt.copy_(bt_new.to(DEV))
    k_pre, v_pre = wl.bits(pool.k_cache), wl.bits(pool.v_cache)
    rk_pre, rv_pre = wl.bits(ring.k_cache), wl.bits(ring.v_cache)
    g.replay()
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_paged(wl.bits(new.q), wl.bits(new.k_new), wl.bits(new.v_new), k_pre,
                              v_pre, bt_new.numpy(), new_lens, inp.sinks.numpy(), 0, inp.scale,
                              cfg["page_size"])
    assert_close(out_p.double().cpu().numpy(), ref, "graph paged")
    ref = oracle.decode_ring(wl.bits(new.q), wl.bits(new.k_new), wl.bits(new.v_new), rk_pre,
                             rv_pre, new_lens, inp.sinks.numpy(), W, inp.scale)
    assert_close(out_r.double().cpu().numpy(), ref, "graph ring")
    for b in np.nonzero(new_lens == 0)[0][:4]:
        assert torch.all(out_p[b] == 0) and torch.all(out_r[b] == 0)


def test_maximum_batch():
    """1024 slots (the largest batch the library takes), a quarter of them inactive, the rest
    short with a few long ones, 16 query heads over 2 KV heads: the device-side prefix over
    every slot, thousands of segments, the append into every active slot."""
    rng = np.random.default_rng(8)
    lens = [0 if rng.random() < 0.25 else int(rng.integers(1, 48)) for _ in range(1024)]
    lens[5], lens[700] = 600, 900
    c = make_case(340, len(lens), 16, 2, 64, lens)
    check_paged(c, 0, seed=4)
    check_ring(c, 32)
