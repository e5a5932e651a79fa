"""The allocation-free entry point, decode_attn_paged_noalloc.

It exists for callers that cannot allocate device memory when they run decode
attention (a runtime that hands out all GPU memory from its own pool, a plugin
host that forbids cudaMalloc, code that must not risk the synchronisation an
allocation can cause): its scratch lives in a fixed array inside the library.
This test calls it through the C ABI and checks it against decode_attn_paged,
which uses the library workspace, on two calls in a row (the second call finds
the array as the first one left it). It is in a file of its own, named to be
collected last, and it passes in a fresh process as well as after the others.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_decode_attention_kv_gb300 as da
from paged_decode_attention_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1e-2
DA_ERR_SCRATCH_LIMIT = -5


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
    num_pages, Hkv, P, _ = kc.shape
    maxp = bt.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(_p(q), _p(kn), _p(vn), _p(kc), _p(vc), _p(bt), _p(sl), _p(sk), window, scale,
              _p(out), da.da_shape(B, Hq, Hkv, D), P, maxp, num_pages, maxp * P, stream)


def _inputs(lens, seed):
    B, Hq, Hkv, D, P = len(lens), 64, 8, 64, 16
    gen = wl.cpu_generator(seed)
    vgen = torch.Generator(device="cuda")
    vgen.manual_seed(seed)
    inp = wl.draw_decode_inputs(B, Hq, Hkv, D, lens, gen)
    npages = sum(wl.pages_needed(L, P) for L in lens) + 8
    maxp = max(wl.pages_needed(L, P) for L in lens)
    pool = wl.draw_paged_pool(npages, Hkv, P, D, lens, maxp, gen, device="cuda", value_gen=vgen)
    d = lambda t: t.to("cuda").contiguous()
    return (d(inp.q), d(inp.k_new), d(inp.v_new), pool.k_cache, pool.v_cache, pool.block_table,
            d(inp.seq_lens), d(inp.sinks), inp.scale)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    fn = _entry()
    # long sequences split across many CTAs (partials + tickets in the scratch), short ones
    # finished inside one warp, an inactive slot
    lens = [3000, 17000, 40, 0, 9000, 1]
    q, kn, vn, kc, vc, bt, sl, sk, scale = _inputs(lens, 7)
    ref = torch.empty_like(q)
    da.decode_attn_paged(q, kn, vn, kc, vc, bt, sl, sk, 0, scale, ref)
    torch.cuda.synchronize()
    k_after, v_after = kc.clone(), vc.clone()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _call_noalloc(fn, q, kn, vn, kc, vc, bt, sl, sk, 0, scale, out)
        assert rc == 0, da.decode_attn_error_string(rc)
        torch.cuda.synchronize()
        got, want = out.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        excess = np.abs(got - want) - (ATOL + RTOL * np.abs(want))
        assert excess.max() <= 0, f"call {call}: worst excess {excess.max():.3e}"
        # the fused append wrote the same cells as the workspace entry point did
        assert torch.equal(kc, k_after) and torch.equal(vc, v_after)
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
