"""The allocation-free entry point, decode_attn_paged_noalloc.

It exists for callers that cannot allocate device memory when they run decode
attention (a runtime that hands out all GPU memory from its own pool, a plugin
host that forbids cudaMalloc, code that must not risk the synchronisation an
allocation can cause): its scratch lives in a fixed array inside the library.
These tests call it through the C ABI, twice in a row on the same inputs (the
second call finds the array as the first one left it), and check every output
row against the fp64 oracle and against decode_attn_paged, which uses the
library workspace. The cases cover 8- and 16-head query groups, full attention
and a 128-token window, and a shape exactly at the array's limit of 4096
(sequence, KV head) pairs, at early-input level 0 and, for the mixed lengths, level 2
(lengths, tables and the first cache tiles read before the wait for the kernel just
before the call, which in these tests never writes them). The file is named to be
collected last; it passes in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
from paged_decode_attention_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1e-2
DA_ERR_SCRATCH_LIMIT = -5
P = 16


def _entry():
    lib = da.load_library()
    fn = lib.decode_attn_paged_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_float, vp, da.da_shape,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp]
    fn.restype = ctypes.c_int
    return fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(fn, q, kn, vn, kc, vc, bt, sl, sk, window, scale, out):
    B, Hq, D = q.shape
    num_pages, Hkv, page, _ = kc.shape
    maxp = bt.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(_p(q), _p(kn), _p(vn), _p(kc), _p(vc), _p(bt), _p(sl), _p(sk), window, scale,
              _p(out), da.da_shape(B, Hq, Hkv, D), page, maxp, num_pages, maxp * page, stream)


def _inputs(lens, seed, Hq, Hkv, D=64):
    B = len(lens)
    gen = wl.cpu_generator(seed)
    vgen = torch.Generator(device="cuda")
    vgen.manual_seed(seed)
    inp = wl.draw_decode_inputs(B, Hq, Hkv, D, lens, gen)
    npages = sum(wl.pages_needed(L, P) for L in lens) + 8
    maxp = max(1, max(wl.pages_needed(L, P) for L in lens))
    pool = wl.draw_paged_pool(npages, Hkv, P, D, lens, maxp, gen, device="cuda", value_gen=vgen)
    return inp, pool


def _close(got, want, what):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    excess = np.abs(got - want) - (ATOL + RTOL * np.abs(want))
    assert excess.max() <= 0, f"{what}: worst excess {excess.max():.3e}"


def _lens_mixed():
    # long sequences split across many CTAs (partials + tickets in the scratch), short ones
    # finished inside one warp, an inactive slot
    return [3000, 17000, 40, 0, 9000, 1]


def _lens_at_limit():
    # 512 slots x 8 KV heads = 4096 (sequence, KV head) pairs, the most the array holds
    rng = np.random.default_rng(31)
    lens = [int(x) for x in rng.integers(1, 300, size=512)]
    lens[7], lens[300], lens[511] = 5000, 0, 2500
    return lens


@pytest.mark.parametrize("lens_fn,Hq,Hkv,window,level", [
    (_lens_mixed, 64, 8, 0, 0),
    (_lens_mixed, 64, 8, 128, 0),
    (_lens_mixed, 64, 4, 0, 0),      # 16 query heads per KV head: the widest partial slot
    (_lens_mixed, 64, 4, 128, 0),
    (_lens_at_limit, 64, 8, 0, 0),
    (_lens_mixed, 64, 8, 0, 2),
    (_lens_mixed, 64, 4, 128, 2),
])
def test_noalloc_matches_oracle_and_workspace_entry_on_two_calls(lens_fn, Hq, Hkv, window, level):
    prev = da.decode_attn_set_early_inputs(level)
    try:
        _check_two_calls(lens_fn, Hq, Hkv, window)
    finally:
        da.decode_attn_set_early_inputs(prev)


def _check_two_calls(lens_fn, Hq, Hkv, window):
    fn = _entry()
    lens = lens_fn()
    inp, pool = _inputs(lens, 7 + Hkv + window, Hq, Hkv)
    d = lambda t: t.to("cuda").contiguous()
    q, kn, vn, sl, sk = d(inp.q), d(inp.k_new), d(inp.v_new), d(inp.seq_lens), d(inp.sinks)
    kc, vc, bt = pool.k_cache, pool.v_cache, pool.block_table
    k_pre, v_pre = wl.bits(kc), wl.bits(vc)
    bt_h, sl_h = bt.cpu().numpy(), np.asarray(lens, np.int32)
    want = oracle.decode_paged(wl.bits(inp.q), wl.bits(inp.k_new), wl.bits(inp.v_new), k_pre, v_pre,
                               bt_h, sl_h, inp.sinks.numpy(), window, inp.scale, P)
    ek, ev = oracle.kv_append_paged(wl.bits(inp.k_new), wl.bits(inp.v_new), k_pre, v_pre, bt_h, sl_h)
    # the workspace entry point on its own copy of the caches
    ref = torch.empty_like(q)
    da.decode_attn_paged(q, kn, vn, kc.clone(), vc.clone(), bt, sl, sk, window, inp.scale, ref)
    torch.cuda.synchronize()
    ref = ref.double().cpu().numpy()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _call_noalloc(fn, q, kn, vn, kc, vc, bt, sl, sk, window, inp.scale, out)
        assert rc == 0, da.decode_attn_error_string(rc)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        _close(got, want, f"call {call} vs oracle")
        _close(got, ref, f"call {call} vs decode_attn_paged")
        # the fused append wrote exactly the oracle's cells (the second call rewrites them)
        assert np.array_equal(wl.bits(kc), ek) and np.array_equal(wl.bits(vc), ev)
    assert da.decode_attn_device_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    fn = _entry()
    B, Hq, Hkv, D = 1024, 64, 8, 64   # 8192 (sequence, kv head) pairs > 4096
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = fn(p, p, p, p, p, p, p, None, 0, 0.125, p, da.da_shape(B, Hq, Hkv, D), 16, 1, 1, 16,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == DA_ERR_SCRATCH_LIMIT
    assert "scratch" in da.decode_attn_error_string(rc)
