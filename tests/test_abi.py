"""CPU-only checks of the C ABI: the library loads without a GPU, exports every
entry point the header declares, and its host-side argument validation
returns the documented error codes before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "decode_attn.h")


@pytest.fixture(scope="module")
def lib():
    from paged_decode_attention_kv_gb300 import build
    build.build()
    import paged_decode_attention_kv_gb300 as da
    return da.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^DA_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"decode_attn_paged", "decode_attn_ring", "kv_append", "decode_attn_workspace_bytes",
            "decode_attn_reserve", "decode_attn_device_status",
            "decode_attn_error_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in the header but not exported"


def _shape(B=2, Hq=8, Hkv=1, D=64):
    from paged_decode_attention_kv_gb300 import da_shape
    return da_shape(B, Hq, Hkv, D)


P = ctypes.c_void_p(0x10000)      # a fake, 16-byte-aligned device address
BAD = ctypes.c_void_p(0x10008)    # misaligned


def paged(lib, **kw):
    a = dict(q=P, k_new=P, v_new=P, kc=P, vc=P, bt=P, sl=P, sinks=P, window=0, scale=0.125,
             out=P, s=_shape(), page=16, maxp=16, npages=64, maxlen=200, stream=None)
    a.update(kw)
    return lib.decode_attn_paged(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"], a["bt"],
                                 a["sl"], a["sinks"], a["window"], a["scale"], a["out"], a["s"],
                                 a["page"], a["maxp"], a["npages"], a["maxlen"], a["stream"])


def ring(lib, **kw):
    a = dict(q=P, k_new=P, v_new=P, kc=P, vc=P, sl=P, sinks=P, window=128, scale=0.125, out=P,
             s=_shape(), stream=None)
    a.update(kw)
    return lib.decode_attn_ring(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"], a["sl"],
                                a["sinks"], a["window"], a["scale"], a["out"], a["s"], a["stream"])


def test_paged_argument_validation(lib):
    assert paged(lib, q=None) == -1
    assert paged(lib, out=None) == -1
    assert paged(lib, bt=None) == -1
    assert paged(lib, k_new=None) == -1                # k_new without v_new
    assert paged(lib, q=BAD) == -1                     # misaligned
    assert paged(lib, s=_shape(Hq=6, Hkv=4)) == -1     # Hq % Hkv != 0
    assert paged(lib, s=_shape(D=128)) == -2           # head dim
    assert paged(lib, s=_shape(Hq=24, Hkv=1)) == -2    # G = 24
    assert paged(lib, s=_shape(B=2048)) == -2          # batch
    assert paged(lib, page=32) == -2                   # page size
    assert paged(lib, window=-1) == -1
    assert paged(lib, maxlen=16 * 16 + 1) == -1        # beyond the block table row
    assert paged(lib, scale=float("nan")) == -1
    assert paged(lib, s=_shape(B=0)) == 0              # empty batch: nothing to do


def test_ring_argument_validation(lib):
    assert ring(lib, window=0) == -1
    assert ring(lib, window=8) == -2
    assert ring(lib, kc=None) == -1
    assert ring(lib, s=_shape(D=32)) == -2
    assert ring(lib, s=_shape(B=0)) == 0


def multi(lib, ring_=False, **kw):
    a = dict(q=P, k_new=P, v_new=P, kc=P, vc=P, bt=P, sl=P, ql=None, sinks=P, window=0,
             scale=0.125, out=P, s=_shape(), T=4, page=16, maxp=16, npages=64, maxlen=200,
             stream=None)
    if ring_:
        a["window"] = 128
    a.update(kw)
    if ring_:
        return lib.decode_attn_ring_multi(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"], a["sl"],
                                          a["ql"], a["sinks"], a["window"], a["scale"], a["out"],
                                          a["s"], a["T"], a["stream"])
    return lib.decode_attn_paged_multi(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"], a["bt"],
                                       a["sl"], a["ql"], a["sinks"], a["window"], a["scale"], a["out"],
                                       a["s"], a["T"], a["page"], a["maxp"], a["npages"], a["maxlen"],
                                       a["stream"])


def test_multi_argument_validation(lib):
    assert multi(lib, k_new=None) == -1                # the new tokens are required
    assert multi(lib, v_new=None) == -1
    assert multi(lib, T=0) == -1
    assert multi(lib, T=5000) == -2                    # beyond 4096 query tokens
    assert multi(lib, q=BAD) == -1
    assert multi(lib, bt=None) == -1
    assert multi(lib, page=32) == -2
    assert multi(lib, maxlen=16 * 16 + 1) == -1
    assert multi(lib, s=_shape(Hq=24, Hkv=1)) == -2
    assert multi(lib, s=_shape(B=0)) == 0
    assert multi(lib, ring_=True, window=8) == -2
    assert multi(lib, ring_=True, window=0) == -1
    assert multi(lib, ring_=True, s=_shape(B=0)) == 0


def test_append_argument_validation(lib):
    s = _shape()
    assert lib.kv_append(None, P, P, P, P, P, 0, s, 16, 16, 64, None) == -1
    assert lib.kv_append(P, P, P, P, None, P, 0, s, 16, 16, 64, None) == -1   # ring, window 0
    assert lib.kv_append(P, P, P, P, P, P, 0, s, 0, 16, 64, None) == -1       # page size 0
    assert lib.kv_append(P, P, P, P, P, P, 0, _shape(B=0), 16, 16, 64, None) == 0


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -99):
        assert lib.decode_attn_error_string(code)
    assert b"unsupported" in lib.decode_attn_error_string(-2)
