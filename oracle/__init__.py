"""fp64 CPU oracle for decode attention with KV append, GQA, window and sinks.

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
baseline leg use this package. It shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (see its header for the definition and the
passage it follows: SimpleLLM README, changes table, rows "one decode-attention
kernel for sinks, sliding window, GQA and the KV append", "paged KV cache for
full-attention layers" and "ring buffer for sliding-window layers"). This module
only marshals numpy arrays into it. bf16 tensors travel as their raw 16-bit
patterns (``numpy.uint16``).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None
_FUNCS = ("oracle_decode_paged", "oracle_decode_ring", "oracle_decode_contig",
          "oracle_kv_append_paged", "oracle_kv_append_ring", "oracle_scatter_paged",
          "oracle_scatter_ring", "oracle_rope_q64", "oracle_rope_k", "oracle_decode_paged_rope",
          "oracle_decode_ring_rope", "oracle_e4m3_decode", "oracle_e4m3_encode",
          "oracle_quantise_rows", "oracle_decode_paged_fp8", "oracle_decode_ring_fp8",
          "oracle_kv_append_fp8", "oracle_scatter_fp8", "oracle_decode_multi",
          "oracle_kv_append_multi", "oracle_decode_paged_fp8_rope", "oracle_decode_ring_fp8_rope",
          "oracle_rope_multi", "oracle_decode_multi_rope", "oracle_decode_multi_fp8",
          "oracle_kv_append_multi_fp8")

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        c_int, c_double = ctypes.c_int, ctypes.c_double
        lib.oracle_decode_paged.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, _f32p, c_int, c_double, _f64p,
            c_int, c_int, c_int, c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_decode_ring.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _u16p, _i32p, _f32p, c_int, c_double, _f64p,
            c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_decode_contig.argtypes = [
            _u16p, _u16p, _u16p, _i32p, c_int, _f32p, c_int, c_double, _f64p,
            c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_kv_append_paged.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, c_int, c_int, c_int, c_int, c_int, c_int]
        lib.oracle_kv_append_ring.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _i32p, c_int, c_int, c_int, c_int]
        lib.oracle_scatter_paged.argtypes = [
            _u16p, _u16p, _i32p, c_int, _i32p, _u16p, _u16p, c_int, c_int, c_int, c_int, c_int,
            c_int]
        lib.oracle_scatter_ring.argtypes = [
            _u16p, _u16p, _i32p, c_int, c_int, _u16p, _u16p, c_int, c_int, c_int]
        lib.oracle_rope_q64.argtypes = [_u16p, _i32p, _f32p, _f32p, c_int, c_int, c_int, c_int,
                                        _f64p]
        lib.oracle_rope_k.argtypes = [_u16p, _i32p, _f32p, _f32p, c_int, c_int, c_int, c_int, _u16p]
        lib.oracle_decode_paged_rope.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, _f32p, _f32p, _f32p, c_int, c_int,
            c_double, _f64p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_decode_ring_rope.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _u16p, _i32p, _f32p, _f32p, _f32p, c_int, c_int, c_double,
            _f64p, c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_e4m3_decode.argtypes = [_u8p, c_int, _f64p]
        lib.oracle_e4m3_encode.argtypes = [_f32p, c_int, _u8p]
        lib.oracle_quantise_rows.argtypes = [_u16p, c_int, c_int, _u8p, _f32p]
        lib.oracle_decode_paged_fp8.argtypes = [
            _u16p, _u16p, _u16p, _u8p, _i32p, _i32p, _f32p, c_int, c_double,
            _f64p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_decode_ring_fp8.argtypes = [
            _u16p, _u16p, _u16p, _u8p, _i32p, _f32p, c_int, c_double, _f64p,
            c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_decode_paged_fp8_rope.argtypes = [
            _u16p, _u16p, _u16p, _u8p, _i32p, _i32p, _f32p, _f32p, _f32p, c_int, c_int, c_double,
            _f64p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_decode_ring_fp8_rope.argtypes = [
            _u16p, _u16p, _u16p, _u8p, _i32p, _f32p, _f32p, _f32p, c_int, c_int, c_double, _f64p,
            c_int, c_int, c_int, c_int, _i32p, c_int, c_int]
        lib.oracle_kv_append_fp8.argtypes = [
            _u16p, _u16p, _u8p, _i32p, _i32p, c_int, c_int, c_int, c_int, c_int, c_int, c_int]
        lib.oracle_scatter_fp8.argtypes = [
            _u16p, _u16p, _i32p, c_int, _i32p, c_int, _u8p, c_int, c_int, c_int, c_int, c_int,
            c_int]
        lib.oracle_decode_multi.argtypes = [
            c_int, _u16p, _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p, _f32p, c_int, c_double,
            _f64p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int]
        lib.oracle_kv_append_multi.argtypes = [
            c_int, _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p, c_int, c_int, c_int, c_int,
            c_int, c_int, c_int, c_int]
        lib.oracle_rope_multi.argtypes = [
            _u16p, _u16p, _i32p, _i32p, _f32p, _f32p, c_int, c_int, c_int, c_int, c_int, c_int,
            _f64p, _u16p, _u16p]
        lib.oracle_decode_multi_fp8.argtypes = [
            c_int, _u16p, _u16p, _u16p, _u8p, _i32p, _i32p, _i32p, _f32p, c_int, c_double, _f64p,
            c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int]
        lib.oracle_kv_append_multi_fp8.argtypes = [
            c_int, _u16p, _u16p, _u8p, _i32p, _i32p, _i32p, c_int, c_int, c_int, c_int, c_int, c_int,
            c_int, c_int]
        lib.oracle_decode_multi_rope.argtypes = [
            c_int, _u16p, _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p, _f32p, _f32p, _f32p,
            c_int, c_int, c_double, _f64p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
            c_int]
        for name in _FUNCS:
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def load_library(path):
    """Point this wrapper at another build of the oracle (used by the tests
    that plant mistakes in a copy of oracle.c). Returns the previous handle."""
    global _lib
    prev = _lib
    ref = _load()
    lib = ctypes.CDLL(path)
    for fn in _FUNCS:
        f_new, f_ref = getattr(lib, fn), getattr(ref, fn)
        f_new.argtypes, f_new.restype = f_ref.argtypes, f_ref.restype
    _lib = lib
    return prev


def restore_library(prev):
    global _lib
    _lib = prev


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count())


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctype)


def _u16(a, name):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name}: expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _items(items):
    if items is None:
        return None, 0
    arr = np.ascontiguousarray(np.asarray(items, dtype=np.int32).reshape(-1, 2))
    return arr, arr.shape[0]


def _check(status, what):
    if status != 0:
        raise ValueError(f"{what}: oracle returned {status} (bad argument or index)")


def decode_paged(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks, window, scale,
                 page_size, items=None, nthreads=None):
    """Attention output in fp64, shape [B, Hq, D] (or [n_items, D] for sampled items).

    q: [B, Hq, D] u16; k_new/v_new: [B, Hkv, D] u16 or None (no append: token p
    is read from the cache); k_cache/v_cache: [num_pages, Hkv, P, D] u16;
    block_table: [B, max_pages] int32; seq_lens: [B] int32 (post-append);
    sinks: [Hq] float32 or None; window: 0 = full attention.
    """
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    k_cache, v_cache = _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    bt, sl, sk = _i32(block_table), _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_cache.shape
    assert D2 == D and P == page_size and v_cache.shape == k_cache.shape
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_paged(
        _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(k_cache, _u16p),
        _ptr(v_cache, _u16p), _ptr(bt, _i32p), _ptr(sl, _i32p), _ptr(sk, _f32p), int(window),
        float(scale), _ptr(out, _f64p), B, Hq, Hkv, D, P, bt.shape[1], num_pages,
        _ptr(it, _i32p), n_items, nthreads or default_threads())
    _check(st, "decode_paged")
    return out


def decode_ring(q, k_new, v_new, k_cache, v_cache, seq_lens, sinks, window, scale, items=None,
                nthreads=None):
    """Attention over a ring cache k_cache [B, Hkv, W, D] (W = window = capacity)."""
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    k_cache, v_cache = _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    sl, sk = _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    B2, Hkv, W, D2 = k_cache.shape
    assert B2 == B and D2 == D and W == window
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_ring(
        _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(k_cache, _u16p),
        _ptr(v_cache, _u16p), _ptr(sl, _i32p), _ptr(sk, _f32p), int(window), float(scale),
        _ptr(out, _f64p), B, Hq, Hkv, D, _ptr(it, _i32p), n_items,
        nthreads or default_threads())
    _check(st, "decode_ring")
    return out


def decode_contig(q, hist_k, hist_v, seq_lens, sinks, window, scale, items=None, nthreads=None):
    """Attention over a contiguous history hist [B, Tmax, Hkv, D] that already
    holds the new token at position L - 1. window = 0 means full attention."""
    lib = _load()
    q, hist_k, hist_v = _u16(q, "q"), _u16(hist_k, "hist_k"), _u16(hist_v, "hist_v")
    sl, sk = _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    B2, Tmax, Hkv, D2 = hist_k.shape
    assert B2 == B and D2 == D
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_contig(
        _ptr(q, _u16p), _ptr(hist_k, _u16p), _ptr(hist_v, _u16p), _ptr(sl, _i32p), Tmax,
        _ptr(sk, _f32p), int(window), float(scale), _ptr(out, _f64p), B, Hq, Hkv, D,
        _ptr(it, _i32p), n_items, nthreads or default_threads())
    _check(st, "decode_contig")
    return out


def kv_append_paged(k_new, v_new, k_cache, v_cache, block_table, seq_lens):
    """Return copies of the paged caches with each active sequence's new token written."""
    lib = _load()
    k_new, v_new = _u16(k_new, "k_new"), _u16(v_new, "v_new")
    kc, vc = np.array(k_cache, dtype=np.uint16, copy=True), np.array(v_cache, dtype=np.uint16,
                                                                      copy=True)
    bt, sl = _i32(block_table), _i32(seq_lens)
    num_pages, Hkv, P, D = kc.shape
    st = lib.oracle_kv_append_paged(
        _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(kc, _u16p), _ptr(vc, _u16p),
        _ptr(bt, _i32p), _ptr(sl, _i32p), sl.shape[0], Hkv, D, P, bt.shape[1], num_pages)
    _check(st, "kv_append_paged")
    return kc, vc


def kv_append_ring(k_new, v_new, k_cache, v_cache, seq_lens, window):
    """Return copies of the ring caches with each active sequence's new token written."""
    lib = _load()
    k_new, v_new = _u16(k_new, "k_new"), _u16(v_new, "v_new")
    kc, vc = np.array(k_cache, dtype=np.uint16, copy=True), np.array(v_cache, dtype=np.uint16,
                                                                      copy=True)
    sl = _i32(seq_lens)
    B, Hkv, W, D = kc.shape
    assert W == window
    st = lib.oracle_kv_append_ring(
        _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(kc, _u16p), _ptr(vc, _u16p),
        _ptr(sl, _i32p), int(window), B, Hkv, D)
    _check(st, "kv_append_ring")
    return kc, vc


def scatter_paged(hist_k, hist_v, n_tokens, block_table, k_cache, v_cache):
    """Write tokens 0..n[b]-1 of each history into (copies of) the paged caches."""
    lib = _load()
    hist_k, hist_v = _u16(hist_k, "hist_k"), _u16(hist_v, "hist_v")
    kc, vc = np.array(k_cache, dtype=np.uint16, copy=True), np.array(v_cache, dtype=np.uint16,
                                                                      copy=True)
    n, bt = _i32(n_tokens), _i32(block_table)
    B, Tmax, Hkv, D = hist_k.shape
    num_pages, Hkv2, P, D2 = kc.shape
    assert Hkv2 == Hkv and D2 == D
    st = lib.oracle_scatter_paged(
        _ptr(hist_k, _u16p), _ptr(hist_v, _u16p), _ptr(n, _i32p), Tmax, _ptr(bt, _i32p),
        _ptr(kc, _u16p), _ptr(vc, _u16p), B, Hkv, D, P, bt.shape[1], num_pages)
    _check(st, "scatter_paged")
    return kc, vc


def scatter_ring(hist_k, hist_v, n_tokens, window, k_cache, v_cache):
    """Write the ring state after n[b] tokens into (copies of) the ring caches."""
    lib = _load()
    hist_k, hist_v = _u16(hist_k, "hist_k"), _u16(hist_v, "hist_v")
    kc, vc = np.array(k_cache, dtype=np.uint16, copy=True), np.array(v_cache, dtype=np.uint16,
                                                                      copy=True)
    n = _i32(n_tokens)
    B, Tmax, Hkv, D = hist_k.shape
    st = lib.oracle_scatter_ring(
        _ptr(hist_k, _u16p), _ptr(hist_v, _u16p), _ptr(n, _i32p), Tmax, int(window),
        _ptr(kc, _u16p), _ptr(vc, _u16p), B, Hkv, D)
    _check(st, "scatter_ring")
    return kc, vc


# ---------------------------------------------------------------- rotary position embedding
def _tables(rope_cos, rope_sin, D):
    c = np.ascontiguousarray(rope_cos, dtype=np.float32)
    sn = np.ascontiguousarray(rope_sin, dtype=np.float32)
    assert c.shape == sn.shape and c.ndim == 2 and c.shape[1] == D // 2
    return c, sn, c.shape[0]


def rope_q64(q, seq_lens, rope_cos, rope_sin):
    """Queries rotated to position L - 1, fp64 [B, Hq, D] (rotate-half pairs (i, i + D/2))."""
    lib = _load()
    q = _u16(q, "q")
    sl = _i32(seq_lens)
    B, Hq, D = q.shape
    c, sn, maxpos = _tables(rope_cos, rope_sin, D)
    out = np.zeros((B, Hq, D), np.float64)
    _check(lib.oracle_rope_q64(_ptr(q, _u16p), _ptr(sl, _i32p), _ptr(c, _f32p), _ptr(sn, _f32p),
                               maxpos, B, Hq, D, _ptr(out, _f64p)), "rope_q64")
    return out


def rope_k(k_new, seq_lens, rope_cos, rope_sin):
    """New keys rotated to position L - 1 as stored in a bf16 cache (fp32 arithmetic,
    round to nearest even), uint16 [B, Hkv, D]."""
    lib = _load()
    k = _u16(k_new, "k_new")
    sl = _i32(seq_lens)
    B, Hkv, D = k.shape
    c, sn, maxpos = _tables(rope_cos, rope_sin, D)
    out = np.zeros_like(k)
    _check(lib.oracle_rope_k(_ptr(k, _u16p), _ptr(sl, _i32p), _ptr(c, _f32p), _ptr(sn, _f32p),
                             maxpos, B, Hkv, D, _ptr(out, _u16p)), "rope_k")
    return out


def decode_paged_rope(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks, rope_cos,
                      rope_sin, window, scale, page_size, items=None, nthreads=None):
    """decode_paged with q and k_new rotated to position L - 1 first."""
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    k_cache, v_cache = _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    bt, sl, sk = _i32(block_table), _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_cache.shape
    assert P == page_size
    c, sn, maxpos = _tables(rope_cos, rope_sin, D)
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_paged_rope(
        _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(k_cache, _u16p),
        _ptr(v_cache, _u16p), _ptr(bt, _i32p), _ptr(sl, _i32p), _ptr(sk, _f32p), _ptr(c, _f32p),
        _ptr(sn, _f32p), maxpos, int(window), float(scale), _ptr(out, _f64p), B, Hq, Hkv, D, P,
        bt.shape[1], num_pages, _ptr(it, _i32p), n_items, nthreads or default_threads())
    _check(st, "decode_paged_rope")
    return out


def decode_ring_rope(q, k_new, v_new, k_cache, v_cache, seq_lens, sinks, rope_cos, rope_sin,
                     window, scale, items=None, nthreads=None):
    """decode_ring with q and k_new rotated to position L - 1 first."""
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    k_cache, v_cache = _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    sl, sk = _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    _, Hkv, W, _ = k_cache.shape
    assert W == window
    c, sn, maxpos = _tables(rope_cos, rope_sin, D)
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_ring_rope(
        _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(k_cache, _u16p),
        _ptr(v_cache, _u16p), _ptr(sl, _i32p), _ptr(sk, _f32p), _ptr(c, _f32p), _ptr(sn, _f32p),
        maxpos, int(window), float(scale), _ptr(out, _f64p), B, Hq, Hkv, D, _ptr(it, _i32p),
        n_items, nthreads or default_threads())
    _check(st, "decode_ring_rope")
    return out


# ---------------------------------------------------------------- fp8 (e4m3) KV cache
def e4m3_decode(codes):
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(c.shape, np.float64)
    lib.oracle_e4m3_decode(_ptr(c, _u8p), c.size, _ptr(out, _f64p))
    return out


def e4m3_encode(x):
    lib = _load()
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(f.shape, np.uint8)
    lib.oracle_e4m3_encode(_ptr(f, _f32p), f.size, _ptr(out, _u8p))
    return out


def quantise_rows(rows):
    """bf16 rows [..., D] -> (e4m3 codes [..., D], fp32 scales [...])."""
    lib = _load()
    r = _u16(rows, "rows")
    D = r.shape[-1]
    n = r.size // D
    codes = np.zeros(r.shape, np.uint8)
    scales = np.zeros(r.shape[:-1], np.float32)
    lib.oracle_quantise_rows(_ptr(r, _u16p), n, D, _ptr(codes, _u8p), _ptr(scales, _f32p))
    return codes, scales


class Fp8Cache:
    """An fp8 cache: numpy uint8 blocks [..., 2*P*D + 8*P], one per P = 16 tokens of one KV
    head (paged: [num_pages, Hkv, bytes]; ring of capacity W: [B, Hkv, W / P, bytes]), each
    K codes [P][D], V codes transposed [D][P], K scales [P] and V scales [P] (fp32). The
    properties k, vt, ks, vs are views of those parts."""

    def __init__(self, blocks, P=16, D=64):
        assert blocks.dtype == np.uint8 and blocks.shape[-1] == 2 * P * D + 8 * P
        self.blocks, self.P, self.D = blocks, P, D

    @property
    def k(self):
        P, D = self.P, self.D
        return self.blocks[..., :P * D].reshape(self.blocks.shape[:-1] + (P, D))

    @property
    def vt(self):
        P, D = self.P, self.D
        return self.blocks[..., P * D:2 * P * D].reshape(self.blocks.shape[:-1] + (D, P))

    @property
    def ks(self):
        o = 2 * self.P * self.D
        return self.blocks[..., o:o + 4 * self.P].view(np.float32)

    @property
    def vs(self):
        o = 2 * self.P * self.D + 4 * self.P
        return self.blocks[..., o:o + 4 * self.P].view(np.float32)

    @staticmethod
    def _filled(lead, P, D, fill_code, fill_scale):
        c = Fp8Cache(np.full(tuple(lead) + (2 * P * D + 8 * P,), fill_code, np.uint8), P, D)
        c.ks[...] = fill_scale
        c.vs[...] = fill_scale
        return c

    @staticmethod
    def empty_paged(num_pages, Hkv, P, D, fill_code=0x7F, fill_scale=np.nan):
        return Fp8Cache._filled((num_pages, Hkv), P, D, fill_code, fill_scale)

    @staticmethod
    def empty_ring(B, Hkv, W, D, fill_code=0x7F, fill_scale=np.nan, P=16):
        assert W % P == 0, "the fp8 ring capacity is a multiple of 16"
        return Fp8Cache._filled((B, Hkv, W // P), P, D, fill_code, fill_scale)

    @staticmethod
    def from_parts(k, vt, ks, vs):
        """Pack K codes [..., P, D], V^T codes [..., D, P] and scales [..., P] into blocks."""
        P, D = k.shape[-2], k.shape[-1]
        c = Fp8Cache._filled(k.shape[:-2], P, D, 0, 0.0)
        c.k[...] = k
        c.vt[...] = vt
        c.ks[...] = ks
        c.vs[...] = vs
        return c

    def copy(self):
        return Fp8Cache(self.blocks.copy(), self.P, self.D)

    def ptr(self):
        assert self.blocks.flags.c_contiguous
        return _ptr(self.blocks, _u8p)


def scatter_fp8(hist_k, hist_v, n_tokens, cache, block_table=None, window=0):
    """Quantise tokens 0..n[b]-1 of each history into (a copy of) an fp8 cache: paged when a
    block table is given, else the ring state of capacity `window`."""
    lib = _load()
    hk, hv = _u16(hist_k, "hist_k"), _u16(hist_v, "hist_v")
    n = _i32(n_tokens)
    out = cache.copy()
    B, Tmax, Hkv, D = hk.shape
    if block_table is not None:
        bt = _i32(block_table)
        maxp, npages = bt.shape[1], out.blocks.shape[0]
    else:
        bt, maxp, npages = None, 0, 0
    _check(lib.oracle_scatter_fp8(_ptr(hk, _u16p), _ptr(hv, _u16p), _ptr(n, _i32p), Tmax,
                                  _ptr(bt, _i32p), int(window), out.ptr(), B, Hkv, D, out.P, maxp,
                                  npages), "scatter_fp8")
    return out


def kv_append_fp8(k_new, v_new, cache, seq_lens, block_table=None, window=0):
    lib = _load()
    kn, vn = _u16(k_new, "k_new"), _u16(v_new, "v_new")
    sl = _i32(seq_lens)
    out = cache.copy()
    B, Hkv, D = kn.shape
    if block_table is not None:
        bt = _i32(block_table)
        maxp, npages = bt.shape[1], out.blocks.shape[0]
    else:
        bt, maxp, npages = None, 0, 0
    _check(lib.oracle_kv_append_fp8(_ptr(kn, _u16p), _ptr(vn, _u16p), out.ptr(), _ptr(bt, _i32p),
                                    _ptr(sl, _i32p), int(window), B, Hkv, D, out.P, maxp, npages),
           "kv_append_fp8")
    return out


def decode_paged_fp8(q, k_new, v_new, cache, block_table, seq_lens, sinks, window, scale,
                     items=None, nthreads=None):
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    bt, sl, sk = _i32(block_table), _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    num_pages, Hkv = cache.blocks.shape[:2]
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    _check(lib.oracle_decode_paged_fp8(
        _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), cache.ptr(), _ptr(bt, _i32p),
        _ptr(sl, _i32p), _ptr(sk, _f32p), int(window), float(scale), _ptr(out, _f64p), B, Hq, Hkv,
        D, cache.P, bt.shape[1], num_pages, _ptr(it, _i32p), n_items, nthreads or default_threads()),
        "decode_paged_fp8")
    return out


def decode_ring_fp8(q, k_new, v_new, cache, seq_lens, sinks, window, scale, items=None,
                    nthreads=None):
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    sl, sk = _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    Hkv = cache.blocks.shape[1]
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    _check(lib.oracle_decode_ring_fp8(
        _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), cache.ptr(), _ptr(sl, _i32p),
        _ptr(sk, _f32p), int(window), float(scale), _ptr(out, _f64p), B, Hq, Hkv, D,
        _ptr(it, _i32p), n_items, nthreads or default_threads()), "decode_ring_fp8")
    return out


def decode_paged_fp8_rope(q, k_new, v_new, cache, block_table, seq_lens, sinks, rope_cos, rope_sin,
                          window, scale, items=None, nthreads=None):
    """decode_paged_fp8 with q and k_new rotated to position L - 1 first (the new key is
    rotated as stored in bf16, then quantised on append)."""
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    bt, sl, sk = _i32(block_table), _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    num_pages, Hkv = cache.blocks.shape[:2]
    c, sn, maxpos = _tables(rope_cos, rope_sin, D)
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    _check(lib.oracle_decode_paged_fp8_rope(
        _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), cache.ptr(), _ptr(bt, _i32p),
        _ptr(sl, _i32p), _ptr(sk, _f32p), _ptr(c, _f32p), _ptr(sn, _f32p), maxpos, int(window),
        float(scale), _ptr(out, _f64p), B, Hq, Hkv, D, cache.P, bt.shape[1], num_pages,
        _ptr(it, _i32p), n_items, nthreads or default_threads()), "decode_paged_fp8_rope")
    return out


def decode_ring_fp8_rope(q, k_new, v_new, cache, seq_lens, sinks, rope_cos, rope_sin, window, scale,
                         items=None, nthreads=None):
    """decode_ring_fp8 with q and k_new rotated to position L - 1 first."""
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    sl, sk = _i32(seq_lens), _f32(sinks)
    B, Hq, D = q.shape
    Hkv = cache.blocks.shape[1]
    c, sn, maxpos = _tables(rope_cos, rope_sin, D)
    it, n_items = _items(items)
    out = np.zeros((n_items, D) if it is not None else (B, Hq, D), dtype=np.float64)
    _check(lib.oracle_decode_ring_fp8_rope(
        _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), cache.ptr(), _ptr(sl, _i32p),
        _ptr(sk, _f32p), _ptr(c, _f32p), _ptr(sn, _f32p), maxpos, int(window), float(scale),
        _ptr(out, _f64p), B, Hq, Hkv, D, _ptr(it, _i32p), n_items, nthreads or default_threads()),
        "decode_ring_fp8_rope")
    return out


# ---------------------------------------------------------------- several query tokens
def decode_multi(q, k_new, v_new, k_cache, v_cache, seq_lens, sinks, window, scale,
                 block_table=None, q_lens=None, page_size=16, nthreads=None):
    """q [B, T, Hq, D], k_new / v_new [B, T, Hkv, D] (bf16 bits); caches hold the history
    before the step (paged when a block table is given, else the ring of capacity `window`).
    Returns out [B, T, Hq, D] float64."""
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    kc, vc = _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    sl, ql, sk = _i32(seq_lens), _i32(q_lens), _f32(sinks)
    B, T, Hq, D = q.shape
    Hkv = k_new.shape[2]
    ring = block_table is None
    bt = None if ring else _i32(block_table)
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    _check(lib.oracle_decode_multi(
        int(ring), _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(kc, _u16p),
        _ptr(vc, _u16p), _ptr(bt, _i32p), _ptr(sl, _i32p), _ptr(ql, _i32p), _ptr(sk, _f32p),
        int(window), float(scale), _ptr(out, _f64p), B, T, Hq, Hkv, D, page_size,
        0 if ring else bt.shape[1], 0 if ring else kc.shape[0], nthreads or default_threads()),
        "decode_multi")
    return out


def rope_multi(q, k_new, seq_lens, rope_cos, rope_sin, q_lens=None, with_q_bf16=False):
    """Several-token rotary embedding: query row (t, h) and new key (t, g), t < n, rotated to
    their own position L - n + t. Returns (q64 [B, T, Hq, D] float64, the exact rotation, zero
    rows for t >= n; k_rot [B, T, Hkv, D] uint16 as stored, rows t >= n copied), and with
    with_q_bf16 also q_rot [B, T, Hq, D] uint16: the query as the bf16 model holds it after
    the rotation (rounded like the key; rows t >= n copied)."""
    lib = _load()
    q, kn = _u16(q, "q"), _u16(k_new, "k_new")
    sl, ql = _i32(seq_lens), _i32(q_lens)
    B, T, Hq, D = q.shape
    Hkv = kn.shape[2]
    c, sn, maxpos = _tables(rope_cos, rope_sin, D)
    q64 = np.zeros((B, T, Hq, D), np.float64)
    qrot = np.zeros_like(q)
    krot = np.zeros_like(kn)
    _check(lib.oracle_rope_multi(_ptr(q, _u16p), _ptr(kn, _u16p), _ptr(sl, _i32p), _ptr(ql, _i32p),
                                 _ptr(c, _f32p), _ptr(sn, _f32p), maxpos, B, T, Hq, Hkv, D,
                                 _ptr(q64, _f64p), _ptr(qrot, _u16p), _ptr(krot, _u16p)), "rope_multi")
    return (q64, krot, qrot) if with_q_bf16 else (q64, krot)


def decode_multi_rope(q, k_new, v_new, k_cache, v_cache, seq_lens, sinks, rope_cos, rope_sin,
                      window, scale, block_table=None, q_lens=None, page_size=16, nthreads=None):
    """decode_multi with q and k_new rotated first (rope_multi), both as the bf16 model holds
    them (the query rounded to bf16 like the stored key): the several-token step of a model
    whose keys are stored rotated. The append of the step stores the rotated keys
    (kv_append_multi of rope_multi's k_rot)."""
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    kc, vc = _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    sl, ql, sk = _i32(seq_lens), _i32(q_lens), _f32(sinks)
    B, T, Hq, D = q.shape
    Hkv = k_new.shape[2]
    c, sn, maxpos = _tables(rope_cos, rope_sin, D)
    ring = block_table is None
    bt = None if ring else _i32(block_table)
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    _check(lib.oracle_decode_multi_rope(
        int(ring), _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(kc, _u16p),
        _ptr(vc, _u16p), _ptr(bt, _i32p), _ptr(sl, _i32p), _ptr(ql, _i32p), _ptr(sk, _f32p),
        _ptr(c, _f32p), _ptr(sn, _f32p), maxpos, int(window), float(scale), _ptr(out, _f64p), B, T,
        Hq, Hkv, D, page_size, 0 if ring else bt.shape[1], 0 if ring else kc.shape[0],
        nthreads or default_threads()), "decode_multi_rope")
    return out


def kv_append_multi(k_new, v_new, k_cache, v_cache, seq_lens, window=0, block_table=None,
                    q_lens=None, page_size=16):
    """Copies of the caches with the step's n = q_lens[b] (or T) new tokens appended."""
    lib = _load()
    kn, vn = _u16(k_new, "k_new"), _u16(v_new, "v_new")
    kc, vc = _u16(k_cache, "k_cache").copy(), _u16(v_cache, "v_cache").copy()
    sl, ql = _i32(seq_lens), _i32(q_lens)
    B, T, Hkv, D = kn.shape
    ring = block_table is None
    bt = None if ring else _i32(block_table)
    _check(lib.oracle_kv_append_multi(
        int(ring), _ptr(kn, _u16p), _ptr(vn, _u16p), _ptr(kc, _u16p), _ptr(vc, _u16p),
        _ptr(bt, _i32p), _ptr(sl, _i32p), _ptr(ql, _i32p), int(window), B, T, Hkv, D, page_size,
        0 if ring else bt.shape[1], 0 if ring else kc.shape[0]), "kv_append_multi")
    return kc, vc


# ---------------------------------------------------------------- several query tokens, fp8 cache
def decode_multi_fp8(q, k_new, v_new, cache, seq_lens, sinks, window, scale, block_table=None,
                     q_lens=None, nthreads=None):
    """decode_multi over an fp8 cache (Fp8Cache: paged when a block table is given, else the
    ring of capacity `window`): history rows dequantised from their blocks, each new token
    quantised as its append stores it. Returns out [B, T, Hq, D] float64."""
    lib = _load()
    q, k_new, v_new = _u16(q, "q"), _u16(k_new, "k_new"), _u16(v_new, "v_new")
    sl, ql, sk = _i32(seq_lens), _i32(q_lens), _f32(sinks)
    B, T, Hq, D = q.shape
    Hkv = k_new.shape[2]
    ring = block_table is None
    bt = None if ring else _i32(block_table)
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    _check(lib.oracle_decode_multi_fp8(
        int(ring), _ptr(q, _u16p), _ptr(k_new, _u16p), _ptr(v_new, _u16p), cache.ptr(),
        _ptr(bt, _i32p), _ptr(sl, _i32p), _ptr(ql, _i32p), _ptr(sk, _f32p), int(window),
        float(scale), _ptr(out, _f64p), B, T, Hq, Hkv, D, cache.P,
        0 if ring else bt.shape[1], 0 if ring else cache.blocks.shape[0],
        nthreads or default_threads()), "decode_multi_fp8")
    return out


def kv_append_multi_fp8(k_new, v_new, cache, seq_lens, block_table=None, window=0, q_lens=None):
    """A copy of the fp8 cache with the step's n = q_lens[b] (or T) new tokens quantised into
    their blocks."""
    lib = _load()
    kn, vn = _u16(k_new, "k_new"), _u16(v_new, "v_new")
    sl, ql = _i32(seq_lens), _i32(q_lens)
    out = cache.copy()
    B, T, Hkv, D = kn.shape
    ring = block_table is None
    bt = None if ring else _i32(block_table)
    _check(lib.oracle_kv_append_multi_fp8(
        int(ring), _ptr(kn, _u16p), _ptr(vn, _u16p), out.ptr(), _ptr(bt, _i32p), _ptr(sl, _i32p),
        _ptr(ql, _i32p), int(window), B, T, Hkv, D, out.P, 0 if ring else bt.shape[1],
        0 if ring else out.blocks.shape[0]), "kv_append_multi_fp8")
    return out
