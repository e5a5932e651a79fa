"""Fused decode-step attention for GB300: KV append + GQA over a paged cache or a
sliding-window ring + per-head attention sinks.

A thin ctypes binding over the C ABI in ``include/decode_attn.h`` (library
``libdecode_attn.so`` next to this file, built by ``build.py``). Every step of
the computation runs in the library's CUDA kernels; this module only turns
torch tensors into device pointers, sizes and the current CUDA stream, and
turns error codes into exceptions. There is no CPU fallback: if the library
is missing, every call raises.

Tensor layouts (all contiguous, bf16 unless noted):
  q, out            [B, Hq, D]
  k_new, v_new      [B, Hkv, D]
  paged caches      [num_pages, Hkv, page_size, D]
  ring caches       [B, Hkv, window, D]
  block_table       [B, max_pages_per_seq] int32
  seq_lens          [B] int32, length after this step's append (0 = inactive)
  sinks             [Hq] float32, or None
"""
import ctypes
import os

import torch

__all__ = [
    "da_shape",
    "DecodeAttnError", "decode_attn_paged", "decode_attn_ring", "kv_append",
    "decode_attn_workspace_bytes", "decode_attn_reserve", "decode_attn_device_status",
    "decode_attn_error_string", "library_path", "load_library",
    "DA_STATUS_BAD_SEQ_LEN", "DA_STATUS_BAD_PAGE", "DA_STATUS_TIMEOUT", "DA_STATUS_BAD_POSITION",
    "decode_attn_paged_rope", "decode_attn_ring_rope", "decode_attn_paged_fp8", "decode_attn_ring_fp8",
    "decode_attn_paged_multi", "decode_attn_ring_multi", "decode_attn_multi_workspace_bytes",
    "decode_attn_multi_reserve", "decode_attn_multi_launches", "decode_attn_test_expire_wait",
    "decode_attn_paged_fp8_rope", "decode_attn_ring_fp8_rope", "decode_attn_set_early_inputs",
    "decode_attn_stream_reserve", "decode_attn_stream_release",
    "decode_attn_paged_multi_rope", "decode_attn_ring_multi_rope",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libdecode_attn.so"

DA_OK = 0
DA_ERR_INVALID_ARG = -1
DA_ERR_UNSUPPORTED = -2
DA_ERR_WORKSPACE = -3
DA_ERR_CUDA = -4
DA_STATUS_BAD_SEQ_LEN = 1
DA_STATUS_BAD_PAGE = 2
DA_STATUS_TIMEOUT = 4
DA_STATUS_BAD_POSITION = 8


class da_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int)]


class DecodeAttnError(RuntimeError):
    def __init__(self, code, message):
        super().__init__(f"decode_attn error {code}: {message}")
        self.code = code


_lib = None


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load_library():
    """Load the CUDA library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    c_int, c_float = ctypes.c_int, ctypes.c_float
    lib.decode_attn_paged.argtypes = [vp, vp, vp, vp, vp, i32p, i32p, f32p, c_int, c_float, vp,
                                      da_shape, c_int, c_int, c_int, c_int, vp]
    lib.decode_attn_ring.argtypes = [vp, vp, vp, vp, vp, i32p, f32p, c_int, c_float, vp,
                                     da_shape, vp]
    lib.kv_append.argtypes = [vp, vp, vp, vp, i32p, i32p, c_int, da_shape, c_int, c_int, c_int, vp]
    lib.decode_attn_paged_rope.argtypes = [vp, vp, vp, vp, vp, i32p, i32p, f32p, f32p, f32p, c_int,
                                           c_int, c_float, vp, da_shape, c_int, c_int, c_int, c_int,
                                           vp]
    lib.decode_attn_ring_rope.argtypes = [vp, vp, vp, vp, vp, i32p, f32p, f32p, f32p, c_int, c_int,
                                          c_float, vp, da_shape, vp]
    lib.decode_attn_paged_fp8.argtypes = [vp, vp, vp, vp, i32p, i32p, f32p, c_int, c_float, vp,
                                          da_shape, c_int, c_int, c_int, c_int, vp]
    lib.decode_attn_ring_fp8.argtypes = [vp, vp, vp, vp, i32p, f32p, c_int, c_float, vp, da_shape,
                                         vp]
    lib.decode_attn_paged_fp8_rope.argtypes = [vp, vp, vp, vp, i32p, i32p, f32p, f32p, f32p,
                                               c_int, c_int, c_float, vp, da_shape, c_int, c_int,
                                               c_int, c_int, vp]
    lib.decode_attn_ring_fp8_rope.argtypes = [vp, vp, vp, vp, i32p, f32p, f32p, f32p, c_int, c_int,
                                              c_float, vp, da_shape, vp]
    lib.decode_attn_paged_multi.argtypes = [vp, vp, vp, vp, vp, i32p, i32p, i32p, f32p, c_int,
                                            c_float, vp, da_shape, c_int, c_int, c_int, c_int,
                                            c_int, vp]
    lib.decode_attn_ring_multi.argtypes = [vp, vp, vp, vp, vp, i32p, i32p, f32p, c_int, c_float,
                                           vp, da_shape, c_int, vp]
    lib.decode_attn_paged_multi_rope.argtypes = [vp, vp, vp, vp, vp, i32p, i32p, i32p, f32p, f32p,
                                                 f32p, c_int, c_int, c_float, vp, da_shape, c_int,
                                                 c_int, c_int, c_int, c_int, vp]
    lib.decode_attn_ring_multi_rope.argtypes = [vp, vp, vp, vp, vp, i32p, i32p, f32p, f32p, f32p,
                                                c_int, c_int, c_float, vp, da_shape, c_int, vp]
    lib.decode_attn_multi_workspace_bytes.argtypes = [da_shape, c_int, c_int, c_int]
    lib.decode_attn_multi_workspace_bytes.restype = ctypes.c_size_t
    lib.decode_attn_multi_launches.argtypes = [da_shape, c_int, c_int, c_int]
    lib.decode_attn_multi_launches.restype = c_int
    lib.decode_attn_multi_reserve.argtypes = [ctypes.c_size_t]
    lib.decode_attn_workspace_bytes.argtypes = [da_shape, c_int]
    lib.decode_attn_workspace_bytes.restype = ctypes.c_size_t
    lib.decode_attn_reserve.argtypes = [ctypes.c_size_t]
    lib.decode_attn_stream_reserve.argtypes = [vp, ctypes.c_size_t, ctypes.c_size_t]
    lib.decode_attn_stream_release.argtypes = [vp]
    lib.decode_attn_device_status.argtypes = [vp]
    lib.decode_attn_test_expire_wait.argtypes = [c_int]
    lib.decode_attn_set_early_inputs.argtypes = [c_int]
    lib.decode_attn_error_string.argtypes = [c_int]
    lib.decode_attn_error_string.restype = ctypes.c_char_p
    for fn in (lib.decode_attn_paged, lib.decode_attn_ring, lib.kv_append, lib.decode_attn_reserve,
               lib.decode_attn_device_status, lib.decode_attn_paged_rope, lib.decode_attn_ring_rope,
               lib.decode_attn_paged_fp8, lib.decode_attn_ring_fp8, lib.decode_attn_paged_multi,
               lib.decode_attn_ring_multi, lib.decode_attn_multi_reserve,
               lib.decode_attn_test_expire_wait, lib.decode_attn_paged_fp8_rope,
               lib.decode_attn_ring_fp8_rope, lib.decode_attn_set_early_inputs,
               lib.decode_attn_stream_reserve, lib.decode_attn_stream_release,
               lib.decode_attn_paged_multi_rope, lib.decode_attn_ring_multi_rope):
        fn.restype = c_int
    _lib = lib
    return lib


def decode_attn_error_string(code: int) -> str:
    return load_library().decode_attn_error_string(int(code)).decode()


def _check(code):
    if code != 0:
        raise DecodeAttnError(code, decode_attn_error_string(code))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _shape(q, k_cache_heads):
    B, Hq, D = q.shape
    return da_shape(B, Hq, k_cache_heads, D)


def decode_attn_paged(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks, window,
                      scale, out, max_seq_len=None, stream=None):
    """One decode step over a paged cache, with the KV append fused in.

    k_new/v_new None = no append. window 0 = full attention. max_seq_len
    defaults to the block table's capacity (max_pages_per_seq * page_size).
    """
    num_pages, Hkv, P, _ = k_cache.shape
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * P
    lib = load_library()
    _check(lib.decode_attn_paged(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(sinks), int(window), float(scale), _ptr(out), _shape(q, Hkv), P,
        max_pages, num_pages, int(max_seq_len), _stream(stream)))
    return out


def decode_attn_ring(q, k_new, v_new, k_cache, v_cache, seq_lens, sinks, scale, out,
                     stream=None):
    """One decode step over a sliding-window ring [B, Hkv, W, D] (W = its capacity)."""
    B, Hkv, W, _ = k_cache.shape
    lib = load_library()
    _check(lib.decode_attn_ring(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
        _ptr(sinks), int(W), float(scale), _ptr(out), _shape(q, Hkv), _stream(stream)))
    return out


def decode_attn_paged_rope(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks,
                           rope_cos, rope_sin, window, scale, out, max_seq_len=None, stream=None):
    """decode_attn_paged with the rotary embedding of position L - 1 applied to q and k_new
    first; rope_cos/rope_sin are fp32 [max_position, D/2] device tables."""
    num_pages, Hkv, P, _ = k_cache.shape
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * P
    lib = load_library()
    _check(lib.decode_attn_paged_rope(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(sinks), _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]),
        int(window), float(scale), _ptr(out), _shape(q, Hkv), P, max_pages, num_pages,
        int(max_seq_len), _stream(stream)))
    return out


def decode_attn_ring_rope(q, k_new, v_new, k_cache, v_cache, seq_lens, sinks, rope_cos, rope_sin,
                          scale, out, stream=None):
    """decode_attn_ring with the rotary embedding of position L - 1 applied first."""
    B, Hkv, W, _ = k_cache.shape
    lib = load_library()
    _check(lib.decode_attn_ring_rope(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
        _ptr(sinks), _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]), int(W), float(scale),
        _ptr(out), _shape(q, Hkv), _stream(stream)))
    return out


FP8_BLOCK_BYTES = 2176  # 16 tokens of one KV head: K codes, V^T codes, K and V scales


def decode_attn_paged_fp8(q, k_new, v_new, kv_cache, block_table, seq_lens, sinks, window, scale,
                          out, max_seq_len=None, stream=None):
    """decode_attn_paged over an fp8 cache: kv_cache uint8 [num_pages, Hkv, 2176], one block
    per page and KV head (K codes [16][64], V codes [64][16], K scales [16], V scales [16])."""
    num_pages, Hkv, nb = kv_cache.shape
    if nb != FP8_BLOCK_BYTES:
        raise ValueError(f"kv_cache blocks must be {FP8_BLOCK_BYTES} bytes, got {nb}")
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * 16
    lib = load_library()
    _check(lib.decode_attn_paged_fp8(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(sinks), int(window), float(scale), _ptr(out), _shape(q, Hkv), 16, max_pages,
        num_pages, int(max_seq_len), _stream(stream)))
    return out


def decode_attn_ring_fp8(q, k_new, v_new, kv_cache, seq_lens, sinks, scale, out, stream=None):
    """decode_attn_ring over an fp8 ring: kv_cache uint8 [B, Hkv, W / 16, 2176]."""
    B, Hkv, nblk, nb = kv_cache.shape
    if nb != FP8_BLOCK_BYTES:
        raise ValueError(f"kv_cache blocks must be {FP8_BLOCK_BYTES} bytes, got {nb}")
    lib = load_library()
    _check(lib.decode_attn_ring_fp8(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kv_cache), _ptr(seq_lens), _ptr(sinks),
        int(nblk * 16), float(scale), _ptr(out), _shape(q, Hkv), _stream(stream)))
    return out


def decode_attn_paged_fp8_rope(q, k_new, v_new, kv_cache, block_table, seq_lens, sinks, rope_cos,
                               rope_sin, window, scale, out, max_seq_len=None, stream=None):
    """decode_attn_paged_fp8 with the rotary embedding of position L - 1 applied to q and
    k_new first (the key before it is quantised); rope_cos/rope_sin fp32 [max_position, 32]."""
    num_pages, Hkv, nb = kv_cache.shape
    if nb != FP8_BLOCK_BYTES:
        raise ValueError(f"kv_cache blocks must be {FP8_BLOCK_BYTES} bytes, got {nb}")
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * 16
    lib = load_library()
    _check(lib.decode_attn_paged_fp8_rope(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(sinks), _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]), int(window),
        float(scale), _ptr(out), _shape(q, Hkv), 16, max_pages, num_pages, int(max_seq_len),
        _stream(stream)))
    return out


def decode_attn_ring_fp8_rope(q, k_new, v_new, kv_cache, seq_lens, sinks, rope_cos, rope_sin, scale,
                              out, stream=None):
    """decode_attn_ring_fp8 with the rotary embedding of position L - 1 applied first."""
    B, Hkv, nblk, nb = kv_cache.shape
    if nb != FP8_BLOCK_BYTES:
        raise ValueError(f"kv_cache blocks must be {FP8_BLOCK_BYTES} bytes, got {nb}")
    lib = load_library()
    _check(lib.decode_attn_ring_fp8_rope(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kv_cache), _ptr(seq_lens), _ptr(sinks),
        _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]), int(nblk * 16), float(scale),
        _ptr(out), _shape(q, Hkv), _stream(stream)))
    return out


def kv_append(k_new, v_new, k_cache, v_cache, seq_lens, block_table=None, stream=None):
    """Append alone: paged when block_table is given, else ring [B, Hkv, W, D]."""
    B, Hkv, D = k_new.shape
    lib = load_library()
    if block_table is not None:
        num_pages, _, P, _ = k_cache.shape
        args = (0, da_shape(B, Hkv, Hkv, D), P, block_table.shape[1], num_pages)
    else:
        W = k_cache.shape[2]
        args = (W, da_shape(B, Hkv, Hkv, D), 0, 0, 0)
    _check(lib.kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                         _ptr(block_table), _ptr(seq_lens), *args, _stream(stream)))


def decode_attn_paged_multi(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks, window,
                            scale, out, q_lens=None, max_seq_len=None, stream=None):
    """Several query tokens per sequence: q / out [B, T, Hq, 64], k_new / v_new [B, T, Hkv, 64]
    bf16; seq_lens counts the cached tokens plus the q_lens[b] (or T) new ones. Attention is
    causal over the cache and the new tokens, which are then appended to the pages."""
    B, T, Hq, D = q.shape
    num_pages, Hkv = k_cache.shape[0], k_cache.shape[1]
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * 16
    lib = load_library()
    _check(lib.decode_attn_paged_multi(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(q_lens), _ptr(sinks), int(window), float(scale), _ptr(out),
        da_shape(B, Hq, Hkv, D), T, 16, max_pages, num_pages, int(max_seq_len), _stream(stream)))
    return out


def decode_attn_ring_multi(q, k_new, v_new, k_cache, v_cache, seq_lens, sinks, scale, out,
                           q_lens=None, stream=None):
    """decode_attn_paged_multi over a ring of capacity W = k_cache.shape[2]; the ring holds
    the window of the history before the step."""
    B, T, Hq, D = q.shape
    Hkv, W = k_cache.shape[1], k_cache.shape[2]
    lib = load_library()
    _check(lib.decode_attn_ring_multi(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
        _ptr(q_lens), _ptr(sinks), int(W), float(scale), _ptr(out), da_shape(B, Hq, Hkv, D), T,
        _stream(stream)))
    return out


def decode_attn_paged_multi_rope(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks,
                                 rope_cos, rope_sin, window, scale, out, q_lens=None, max_seq_len=None,
                                 stream=None):
    """decode_attn_paged_multi with the rotary embedding: each new token's query rows and key
    rotated to its own position (rope_cos / rope_sin fp32 [max_position, 32] device tables)."""
    B, T, Hq, D = q.shape
    num_pages, Hkv = k_cache.shape[0], k_cache.shape[1]
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * 16
    lib = load_library()
    _check(lib.decode_attn_paged_multi_rope(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(q_lens), _ptr(sinks), _ptr(rope_cos), _ptr(rope_sin),
        int(rope_cos.shape[0]), int(window), float(scale), _ptr(out), da_shape(B, Hq, Hkv, D), T,
        16, max_pages, num_pages, int(max_seq_len), _stream(stream)))
    return out


def decode_attn_ring_multi_rope(q, k_new, v_new, k_cache, v_cache, seq_lens, sinks, rope_cos,
                                rope_sin, scale, out, q_lens=None, stream=None):
    """decode_attn_ring_multi with the rotary embedding (see decode_attn_paged_multi_rope)."""
    B, T, Hq, D = q.shape
    Hkv, W = k_cache.shape[1], k_cache.shape[2]
    lib = load_library()
    _check(lib.decode_attn_ring_multi_rope(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
        _ptr(q_lens), _ptr(sinks), _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]), int(W),
        float(scale), _ptr(out), da_shape(B, Hq, Hkv, D), T, _stream(stream)))
    return out


def decode_attn_multi_workspace_bytes(batch, num_q_heads, num_kv_heads, q_tokens, ring_window=0,
                                      max_seq_len=0, head_dim=64):
    return int(load_library().decode_attn_multi_workspace_bytes(
        da_shape(batch, num_q_heads, num_kv_heads, head_dim), int(q_tokens), int(ring_window),
        int(max_seq_len)))


def decode_attn_multi_launches(batch, num_q_heads, num_kv_heads, q_tokens, ring_window=0,
                               max_seq_len=0, head_dim=64):
    """Kernel launches of one multi-token call of this shape (0: invalid, or no device)."""
    return int(load_library().decode_attn_multi_launches(
        da_shape(batch, num_q_heads, num_kv_heads, head_dim), int(q_tokens), int(ring_window),
        int(max_seq_len)))


def decode_attn_multi_reserve(nbytes: int):
    _check(load_library().decode_attn_multi_reserve(int(nbytes)))


def decode_attn_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim=64, max_seq_len=0):
    return int(load_library().decode_attn_workspace_bytes(
        da_shape(batch, num_q_heads, num_kv_heads, head_dim), int(max_seq_len)))


def decode_attn_reserve(nbytes: int):
    _check(load_library().decode_attn_reserve(int(nbytes)))


def decode_attn_stream_reserve(stream, nbytes: int = 0, multi_nbytes: int = 0):
    """Workspaces of its own for the attention calls issued on `stream` (a torch.cuda.Stream
    or a raw handle), so that they may overlap calls on other streams; held until
    decode_attn_stream_release(stream)."""
    _check(load_library().decode_attn_stream_reserve(_stream(stream), int(nbytes), int(multi_nbytes)))


def decode_attn_stream_release(stream):
    """Synchronise `stream` and free its own workspaces (no-op if it has none)."""
    _check(load_library().decode_attn_stream_release(_stream(stream)))


def decode_attn_device_status(stream=None) -> int:
    """Wait for the stream, return and clear the device status bits."""
    rc = load_library().decode_attn_device_status(_stream(stream))
    if rc < 0:
        _check(rc)
    return rc


def decode_attn_set_early_inputs(level: int) -> int:
    """Process-wide: what the attention kernels read before waiting for the kernel launched
    just before each call; returns the previous level. 0 (default): nothing. 1: seq_lens,
    q_lens, block_table and sinks (they must have been written before that kernel started).
    2: as 1, and the first cache tiles of each long worker share are prefetched into L2 (a
    hint to the GPU-wide cache: the same conditions as level 1)."""
    rc = load_library().decode_attn_set_early_inputs(int(level))
    if rc < 0:
        _check(rc)
    return rc


def decode_attn_test_expire_wait(tile: int):
    """Testing aid: the next one-token attention call gives up at its first worker's tile
    wait number `tile` (after the tile landed) as if the wait had expired; < 0 disarms."""
    _check(load_library().decode_attn_test_expire_wait(int(tile)))
