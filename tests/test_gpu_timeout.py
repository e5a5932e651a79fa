"""The bounded-wait failure path of the one-token kernel, driven without a real stall.

decode_attn_test_expire_wait makes the first worker of the next call give up at one of
its tile waits after that tile has landed, as an expired wait would: the call must
report DA_STATUS_TIMEOUT, leave no fault and no copy in flight, and leave the arrival
counters at zero, which the next normal call proves by matching the oracle on a case
whose segments are split across warps and across CTAs.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
from cases import make_case, ring_from_history
from test_gpu_decode import (DEV, assert_close, dev, dev_bits, paged_setup, pre, run_paged,
                             run_ring)

pytestmark = pytest.mark.gpu


def _expired_paged(c, kp, vp, bt, tile):
    out = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_test_expire_wait(tile)
    da.decode_attn_paged(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), dev_bits(kp),
                         dev_bits(vp), dev(bt), dev(c.lens), dev(c.sinks), 0, c.scale, out)
    return da.decode_attn_device_status()


@pytest.mark.parametrize("tile", [0, 1, 3, 6])
def test_expired_wait_is_reported_and_the_next_call_is_clean(tile):
    # one long sequence shares every KV head's segment among many warps and CTAs; the
    # short ones put several segments into one warp's share
    c = make_case(380 + tile, 4, 64, 8, 64, [40000, 3000, 70, 5])
    kp, vp, bt = paged_setup(c, 9)
    status = _expired_paged(c, kp, vp, bt, tile)
    assert status & da.DA_STATUS_TIMEOUT, status
    assert da.decode_attn_device_status() == 0  # cleared by the read
    for _ in range(2):  # the following calls are right and leave a clean status
        got, _, _ = run_paged(c, kp, vp, bt, 0)
        ref = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, 0, c.scale, c.P)
        assert_close(got, ref, f"after an expired wait at tile {tile}")


def test_expired_wait_in_the_ring_and_many_segments_per_worker():
    rng = np.random.default_rng(12)
    lens = [int(x) for x in rng.integers(1, 60, size=200)] + [900]
    c = make_case(390, len(lens), 16, 2, 64, lens)
    kr, vr = ring_from_history(c, pre(c), 128)
    out = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_test_expire_wait(0)  # (the first worker's share may be two tiles: one pass)
    da.decode_attn_ring(dev_bits(c.q), dev_bits(c.k_new), dev_bits(c.v_new), dev_bits(kr),
                        dev_bits(vr), dev(c.lens), dev(c.sinks), c.scale, out)
    assert da.decode_attn_device_status() & da.DA_STATUS_TIMEOUT
    got, _, _ = run_ring(c, kr, vr, 128)
    ref = oracle.decode_ring(c.q, c.k_new, c.v_new, kr, vr, c.lens, c.sinks, 128, c.scale)
    assert_close(got, ref, "ring after an expired wait")
    kp, vp, bt = paged_setup(c, 3)
    got, _, _ = run_paged(c, kp, vp, bt, 0)
    ref = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, 0, c.scale, c.P)
    assert_close(got, ref, "paged after an expired wait in the ring")


def test_disarmed_expiry_does_nothing():
    c = make_case(395, 2, 64, 8, 64, [3000, 40])
    kp, vp, bt = paged_setup(c, 4)
    da.decode_attn_test_expire_wait(0)
    da.decode_attn_test_expire_wait(-1)
    got, _, _ = run_paged(c, kp, vp, bt, 0)  # asserts a clean status
    ref = oracle.decode_paged(c.q, c.k_new, c.v_new, kp, vp, bt, c.lens, c.sinks, 0, c.scale, c.P)
    assert_close(got, ref, "disarmed")
