"""A whole decode step (several full and windowed layers) captured once as a CUDA
graph and replayed for different sets of active slots, lengths and block tables,
checked layer by layer against the oracle on sampled heads."""
import numpy as np
import pytest
import torch

import oracle
from paged_decode_attention_kv_gb300 import decode_attn_paged, decode_attn_ring
from paged_decode_attention_kv_gb300 import workloads as wl
from paged_decode_attention_kv_gb300.graph import DecodeStepGraph
from test_gpu_decode import DEV, assert_close, dev

pytestmark = pytest.mark.gpu


def test_one_graph_serves_every_active_slot_set():
    cfg = wl.config("serve")
    B, Hq, Hkv, D, P, W = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["page_size"], cfg["window"]
    lens0 = wl.seq_lens("serve")
    n_layers = 4   # full, ring, full, ring
    gen = wl.cpu_generator(77)
    vgen = torch.Generator(device=DEV)
    vgen.manual_seed(77)
    maxp = cfg["max_pages_per_seq"]
    npages = wl.pool_size("serve", lens0)
    # static buffers the graph is captured on
    q = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
    kn = torch.empty((B, Hkv, D), dtype=torch.bfloat16, device=DEV)
    vn = torch.empty_like(kn)
    sl = torch.zeros(B, dtype=torch.int32, device=DEV)
    bt = torch.full((B, maxp), -1, dtype=torch.int32, device=DEV)
    sinks = torch.randn(Hq, generator=gen).to(DEV)
    layers = []
    for li in range(n_layers):
        if li % 2 == 0:
            pool = wl.draw_paged_pool(npages, Hkv, P, D, lens0, maxp, gen, device=DEV, value_gen=vgen)
            layers.append(("full", pool.k_cache, pool.v_cache))
        else:
            ring = wl.draw_ring_pool(B, Hkv, W, D, vgen, device=DEV)
            layers.append(("ring", ring.k_cache, ring.v_cache))
    outs = [torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV) for _ in layers]

    def make_call(li):
        kind, kc, vc = layers[li]
        if kind == "full":
            return lambda: decode_attn_paged(q, kn, vn, kc, vc, bt, sl, sinks, 0, wl.SCALE, outs[li])
        return lambda: decode_attn_ring(q, kn, vn, kc, vc, sl, sinks, wl.SCALE, outs[li])

    step = DecodeStepGraph([make_call(i) for i in range(n_layers)], (B, Hq, Hkv, D)).capture()

    rng = np.random.default_rng(5)
    for replay in range(3):
        # a new set of active slots with new lengths, pages handed out again, new inputs
        lens = np.array([int(rng.integers(1, L + 1)) if L > 0 and rng.random() > 0.2 else 0
                         for L in lens0], np.int32)
        new = wl.draw_decode_inputs(B, Hq, Hkv, D, lens.tolist(), gen)
        bt_new = wl.draw_block_table(lens.tolist(), P, npages, maxp, gen)
        q.copy_(new.q.to(DEV)); kn.copy_(new.k_new.to(DEV)); vn.copy_(new.v_new.to(DEV))
        sl.copy_(torch.from_numpy(lens).to(DEV)); bt.copy_(bt_new.to(DEV))
        pre = [(wl.bits(kc), wl.bits(vc)) for _, kc, vc in layers]
        step.replay()
        torch.cuda.synchronize()
        for li, (kind, kc, vc) in enumerate(layers):
            kpre, vpre = pre[li]
            if kind == "full":
                ref = oracle.decode_paged(wl.bits(new.q), wl.bits(new.k_new), wl.bits(new.v_new), kpre,
                                          vpre, bt_new.numpy(), lens, sinks.cpu().numpy(), 0, wl.SCALE,
                                          P)
            else:
                ref = oracle.decode_ring(wl.bits(new.q), wl.bits(new.k_new), wl.bits(new.v_new), kpre,
                                         vpre, lens, sinks.cpu().numpy(), W, wl.SCALE)
            assert_close(outs[li].double().cpu().numpy(), ref, f"replay {replay} layer {li}")
        for b in np.nonzero(lens == 0)[0][:3]:
            assert all(torch.all(o[b] == 0) for o in outs)
