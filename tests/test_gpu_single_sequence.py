"""Single-sequence paged calls (one sequence slot, every KV head's tiles spread over many CTAs
and combined across them) against the oracle, the append bit-exact: lengths from one token
(heads with fewer tiles than CTAs leave CTAs without keys) to 16384, every group size up to
8, windows, sinks on and off, calls without the append, the early-input levels, repeated
calls. (These calls were also run on a thread-block-cluster variant that combined through
distributed shared memory; it measured slower and was dropped.)"""
import numpy as np
import pytest

import oracle
import paged_decode_attention_kv_gb300 as da
import test_gpu_decode as gd
from cases import make_case

pytestmark = pytest.mark.gpu

LENS = [1, 2, 15, 16, 17, 100, 255, 256, 257, 4096, 5000, 16384]


def check(c, window, seed, fused=True, sinks=True, max_seq_len=None):
    kp, vp, bt = gd.paged_setup(c, seed, appended=not fused)
    got, ak, av = gd.run_paged(c, kp, vp, bt, window, fused=fused, sinks=sinks,
                               max_seq_len=max_seq_len if max_seq_len is not None else int(c.lens[0]))
    ref = oracle.decode_paged(c.q, c.k_new if fused else None, c.v_new if fused else None, kp, vp, bt,
                              c.lens, c.sinks if sinks else None, window, c.scale, c.P)
    gd.assert_close(got, ref, f"cluster path L={c.lens[0]} window={window}")
    if fused:
        ek, ev = oracle.kv_append_paged(c.k_new, c.v_new, kp, vp, bt, c.lens)
        np.testing.assert_array_equal(ak, ek)
        np.testing.assert_array_equal(av, ev)
    return got


@pytest.mark.parametrize("L", LENS)
@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (8, 8), (16, 4), (32, 16)])
def test_single_sequence_matches_oracle(L, Hq, Hkv):
    c = make_case(1000 + L + Hq, 1, Hq, Hkv, 64, [L])
    check(c, 0, seed=L)


@pytest.mark.parametrize("L", [17, 300, 4096, 9000])
@pytest.mark.parametrize("window", [1, 100, 1000])
def test_windows(L, window):
    c = make_case(1100 + L + window, 1, 64, 8, 64, [L])
    check(c, window, seed=window)


def test_no_sinks_and_no_append():
    c = make_case(1200, 1, 64, 8, 64, [3000])
    check(c, 0, seed=1, sinks=False)
    check(c, 0, seed=2, fused=False)
    check(c, 128, seed=3, fused=False, sinks=False)


def test_inactive_slot():
    c = make_case(1210, 1, 64, 8, 64, [0])
    check(c, 0, seed=4, max_seq_len=16)


def test_repeated_calls_are_identical():
    c = make_case(1220, 1, 64, 8, 64, [7000])
    kp, vp, bt = gd.paged_setup(c, 5)
    outs = [gd.run_paged(c, kp, vp, bt, 0, max_seq_len=7000)[0] for _ in range(3)]
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


@pytest.mark.parametrize("level", [1, 2])
def test_early_input_levels(level):
    prev = da.decode_attn_set_early_inputs(level)
    try:
        for L in (5, 4096, 12000):
            c = make_case(1230 + L, 1, 64, 8, 64, [L])
            check(c, 0, seed=L)
    finally:
        da.decode_attn_set_early_inputs(prev)


def test_max_seq_len_above_the_length():
    c = make_case(1240, 1, 64, 8, 64, [16385])
    check(c, 0, seed=6, max_seq_len=16385)
