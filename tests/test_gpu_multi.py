"""GPU parity of the multi-token step (decode_attn_paged_multi / _ring_multi) against the
fp64 oracle: every output row within 4e-3 + 1e-2 |oracle| (rows beyond q_lens and
inactive slots exactly zero), and the caches after the call bit-exact against the
oracle's append, whole pools compared. Dead cache cells and the padding rows of
k_new / v_new hold NaN, so reading any of them shows."""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_kv_gb300 as da
from paged_decode_attention_kv_gb300 import workloads as wl
from test_gpu_decode import DEV, assert_close, dev, dev_bits
from test_oracle_multi import Multi

pytestmark = pytest.mark.gpu


def run_paged(m, window, seed=1, q_lens=True, sinks=True):
    kp, vp, bt = m.paged(seed)
    kd, vd = dev_bits(kp), dev_bits(vp)
    c = m.c
    out = torch.full((c.B, m.T, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_multi(dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new), kd, vd, dev(bt),
                               dev(m.lens), dev(m.sinks) if sinks else None, window, c.scale, out,
                               q_lens=dev(m.n) if q_lens else None)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_multi(m.q, m.k_new, m.v_new, kp, vp, m.lens, m.sinks if sinks else None,
                              window, c.scale, block_table=bt, q_lens=m.n if q_lens else None)
    assert_close(out.double().cpu().numpy(), ref, f"paged multi window={window}")
    ek, ev = oracle.kv_append_multi(m.k_new, m.v_new, kp, vp, m.lens, block_table=bt,
                                    q_lens=m.n if q_lens else None)
    np.testing.assert_array_equal(wl.bits(kd), ek)
    np.testing.assert_array_equal(wl.bits(vd), ev)


def run_ring(m, W, q_lens=True):
    kr, vr = m.ring(W)
    kd, vd = dev_bits(kr), dev_bits(vr)
    c = m.c
    out = torch.full((c.B, m.T, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_ring_multi(dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new), kd, vd,
                              dev(m.lens), dev(m.sinks), c.scale, out,
                              q_lens=dev(m.n) if q_lens else None)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref = oracle.decode_multi(m.q, m.k_new, m.v_new, kr, vr, m.lens, m.sinks, W, c.scale,
                              q_lens=m.n if q_lens else None)
    assert_close(out.double().cpu().numpy(), ref, f"ring multi W={W}")
    ek, ev = oracle.kv_append_multi(m.k_new, m.v_new, kr, vr, m.lens, window=W,
                                    q_lens=m.n if q_lens else None)
    np.testing.assert_array_equal(wl.bits(kd), ek)
    np.testing.assert_array_equal(wl.bits(vd), ev)


LENS = [1, 4, 15, 16, 17, 33, 100, 257, 0]


def counts(T, lens, seed):
    """Per-sequence new-token counts in [0, min(T, L)], with T itself and 1 present."""
    rng = np.random.default_rng(seed)
    n = [int(rng.integers(0, min(T, L) + 1)) if L > 0 else 0 for L in lens]
    for i, L in enumerate(lens):
        if L >= T:
            n[i] = T
            break
    for i, L in enumerate(lens):
        if L > 0 and n[i] == 0:
            n[i] = 1
            break
    return n


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (8, 8), (16, 1), (32, 4)])
@pytest.mark.parametrize("T", [2, 3, 4, 5, 16])
@pytest.mark.parametrize("window", [0, 7, 100])
def test_paged_multi_matches_oracle(Hq, Hkv, T, window):
    """Up to 4 tokens and 32 query rows per KV head run in the decode kernel (over 16 rows:
    two row groups, e.g. G = 8 at T = 3 and 4, G = 16 at T = 2), more on the row-block or
    tcgen05 kernels."""
    n = counts(T, LENS, Hq + T + window)
    m = Multi(800 + Hq + T + window, Hq, Hkv, LENS, n, T)
    run_paged(m, window, seed=T + 1)


@pytest.mark.parametrize("W", [16, 128, 1024])
@pytest.mark.parametrize("T", [3, 16, 40])
def test_ring_multi_matches_oracle(W, T):
    """Windows of one and eight tiles run unsplit; a 1024-token window splits its keys over
    several CTAs at 3 and 16 tokens, whose partials the last one combines."""
    lens = [1, 15, 16, 17, W - 1, W, W + 1, 3 * W + 5, 60, 0]
    n = counts(T, lens, W + T)
    m = Multi(850 + W + T, 64, 8, lens, n, T)
    run_ring(m, W)


@pytest.mark.parametrize("Hq,Hkv,T", [(64, 8, 2), (32, 8, 2), (64, 8, 4), (128, 8, 2)])
def test_segments_spanning_whole_pipelines(Hq, Hkv, T):
    """Sequences whose key tiles fill a warp's stage ring exactly (4, 5, 8, 10, 12, 15, 16,
    20 tiles): the next sequence's first tile then lands in the stage whose slot held this
    one's query rows before this one's last tiles (which hold the new tokens) are processed.
    Two and four tokens, 16 and 32 query rows per KV head (one and two row groups)."""
    lens = [64, 80, 128, 160, 192, 240, 256, 320, 63, 65, 2, 17]
    m = Multi(865 + Hq + T, Hq, Hkv, lens, [min(T, L) for L in lens], T)
    run_paged(m, 0)
    run_paged(m, 48)


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (16, 1)])
def test_one_token_through_the_multi_calls(Hq, Hkv):
    """T = 1 (one warp per CTA at G = 8, two at G = 16): the multi-token calls reduce to
    the single-token step, paged and ring, with and without the token counts."""
    lens = [1, 16, 17, 300, 0, 129]
    m = Multi(860 + Hq, Hq, Hkv, lens, [1 if L > 0 else 0 for L in lens], 1)
    run_paged(m, 0)
    run_paged(m, 100, q_lens=False)
    run_ring(m, 128)


def test_all_rows_new_without_q_lens_and_no_sinks():
    m = Multi(870, 64, 8, [8, 40, 300], [8, 8, 8], 8)
    run_paged(m, 0, q_lens=False)
    run_paged(m, 0, sinks=False)
    run_ring(m, 32, q_lens=False)


def test_chunked_prefill_sized_step():
    """A run of 200 tokens appended behind a 1000-token history, and a first chunk (no
    history at all): many query-row blocks per KV head."""
    m = Multi(871, 64, 8, [1200, 200], [200, 200], 200)
    run_paged(m, 0)
    run_paged(m, 128)
    run_ring(m, 128)


@pytest.mark.parametrize("T", [4, 6, 16])
def test_long_history_uses_many_splits(T):
    """One sequence of 20k tokens: its keys are split over many CTAs and the last one
    combines the partials (the decode kernel's row groups at 4 tokens, the row-block kernel
    at 6, tcgen05 at 16)."""
    m = Multi(872 + T, 64, 8, [20000, 3000], [T, T - 1], T)
    run_paged(m, 0)
    run_paged(m, 1000)


def test_repeated_calls_are_identical_and_counters_return_to_zero():
    m = Multi(873, 64, 8, [5000, 70], [4, 4], 4)
    kp, vp, bt = m.paged(2)
    outs = []
    for _ in range(3):
        kd, vd = dev_bits(kp), dev_bits(vp)
        out = torch.empty((m.c.B, m.T, m.c.Hq, m.c.D), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_paged_multi(dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new), kd, vd,
                                   dev(bt), dev(m.lens), dev(m.sinks), 0, m.c.scale, out,
                                   q_lens=dev(m.n))
        outs.append(out.cpu())
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))


def test_bad_counts_are_reported_not_faulted():
    m = Multi(874, 8, 8, [10, 20], [2, 2], 2)
    kp, vp, bt = m.paged(1)
    out = torch.empty((2, 2, 8, 64), dtype=torch.bfloat16, device=DEV)
    bad_q = torch.tensor([3, 2], dtype=torch.int32, device=DEV)   # 3 > T
    da.decode_attn_paged_multi(dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new), dev_bits(kp),
                               dev_bits(vp), dev(bt), dev(m.lens), dev(m.sinks), 0, m.c.scale, out,
                               q_lens=bad_q)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() & da.DA_STATUS_BAD_SEQ_LEN
    assert torch.all(out[0].float() == 0)                          # treated as inactive


@pytest.mark.parametrize("T", [2, 4, 8])
def test_full_size_speculative_step(T):
    """The batch-64 workload with T draft tokens per sequence (lengths from the benchmark
    recipe, random pools): a sample of sequences against the oracle, the append
    bit-exact over the whole pool."""
    cfg = wl.config("b64")
    lens = [L + T for L in wl.seq_lens("b64")]
    B, Hq, Hkv, D, P = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["page_size"]
    gen = wl.cpu_generator(cfg["seed"])
    vgen = torch.Generator(device=DEV)
    vgen.manual_seed(cfg["seed"])
    npages = sum(-(-L // P) for L in lens) + 64
    maxp = max(-(-L // P) for L in lens)
    pool = wl.draw_paged_pool(npages, Hkv, P, D, lens, maxp, gen, device=DEV, value_gen=vgen)
    q = wl.randn_bf16((B, T, Hq, D), gen)
    kn = wl.randn_bf16((B, T, Hkv, D), gen)
    vn = wl.randn_bf16((B, T, Hkv, D), gen)
    sinks = torch.randn((Hq,), generator=gen, dtype=torch.float32)
    sl = np.asarray(lens, np.int32)
    k_pre, v_pre = wl.bits(pool.k_cache), wl.bits(pool.v_cache)
    out = torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_paged_multi(dev(q), dev(kn), dev(vn), pool.k_cache, pool.v_cache,
                               pool.block_table, dev(sl), dev(sinks), 0, wl.SCALE, out)
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    bt = pool.block_table.cpu().numpy()
    pick = sorted({0, int(np.argmax(lens)), int(np.argmin(lens)), 17, 40})
    ref = oracle.decode_multi(wl.bits(q)[pick], wl.bits(kn)[pick], wl.bits(vn)[pick], k_pre, v_pre,
                              sl[pick], sinks.numpy(), 0, wl.SCALE, block_table=bt[pick])
    assert_close(out.double().cpu().numpy()[pick], ref, f"b64 T={T}")
    ek, ev = oracle.kv_append_multi(wl.bits(kn), wl.bits(vn), k_pre, v_pre, sl, block_table=bt)
    assert np.array_equal(wl.bits(pool.k_cache), ek) and np.array_equal(wl.bits(pool.v_cache), ev)


@pytest.mark.parametrize("T", [6, 16])
@pytest.mark.parametrize("B,deferred", [(24, False), (2, True)])
def test_split_combine_in_kernel_and_deferred(T, B, deferred):
    """Few key splits per row block are folded by the row block's last CTA; many by a
    kernel of their own after the attention (three launches in all). Both paths, on the
    row-block kernel (6 tokens) and on tcgen05 (16)."""
    rng = np.random.default_rng(880 + T + B)
    lens = [int(x) for x in rng.integers(700, 3000, size=B)]
    lens[0] = 2900  # at 2 sequences: over 8 splits of at least 16 tiles
    m = Multi(880 + T + B, 64, 8, lens, [T] * B, T)
    _, _, bt = m.paged(1)
    launches = da.decode_attn_multi_launches(B, 64, 8, T, 0, bt.shape[1] * 16)
    assert launches == (3 if deferred else 2)
    run_paged(m, 0)
    run_paged(m, 300)


@pytest.mark.parametrize("T", [4, 6])
def test_workspace_reuse_across_shapes(T):
    """A call with few (sequence, head, row-block) groups and many splits writes split
    partials; a following call with more groups must still find its arrival counters at
    zero (the counters live in a region of their own)."""
    few = Multi(875, 64, 8, [9000, 4000], [T, 2], T)        # few groups, many splits
    run_paged(few, 0)
    lens = [int(x) for x in np.random.default_rng(5).integers(600, 2000, size=48)]
    many = Multi(876, 64, 8, lens, [T] * 48, T)              # many groups, a few splits each
    run_paged(many, 0)
    run_paged(few, 0)
    run_paged(many, 0)


def ramp_keys(m, top):
    """Scale key j of every sequence by 1 + (top - 1) j / Tmax (rounded to bf16): scores grow
    along the sequence, so later key blocks raise the running maximum by many octaves."""
    from cases import bf16_to_f64, f64_to_bf16_bits
    hk = bf16_to_f64(m.c.hist_k)
    Tmax = hk.shape[1]
    hk = hk * (1.0 + (top - 1.0) * np.arange(Tmax) / Tmax)[None, :, None, None]
    m.c.hist_k = f64_to_bf16_bits(hk)
    for b in range(m.c.B):
        for t in range(int(m.n[b])):
            m.k_new[b, t] = m.c.hist_k[b, m.base[b] + t]


@pytest.mark.parametrize("T", [4, 16])
def test_growing_scores_force_rescales(T):
    m = Multi(877, 64, 8, [900, 300, 2000], [T, T, T], T)
    ramp_keys(m, 12.0)
    run_paged(m, 0)
    run_paged(m, 200)
    run_ring(m, 128)


def test_multi_many_slots():
    """256 slots, a quarter inactive, 8 query tokens each (counts from 0 to 8): the tcgen05
    kernel on the paged layer, many groups and splits."""
    rng = np.random.default_rng(10)
    lens = [0 if rng.random() < 0.25 else int(rng.integers(8, 400)) for _ in range(256)]
    n = [0 if L == 0 else int(rng.integers(0, 9)) for L in lens]
    m = Multi(878, 64, 8, lens, n, 8)
    run_paged(m, 0)
    run_ring(m, 128)


@pytest.mark.parametrize("T", [4, 16])
def test_cuda_graph_capture_and_replay(T):
    """A multi-token step captured once in a CUDA graph (workspace reserved ahead, nothing on
    the host depends on lengths) and replayed after the lengths, the counts and the inputs
    changed in place: both layers against the oracle, both appends bit-exact."""
    lens = [300, 40, 1200, 0, 77, 900]
    m = Multi(879, 64, 8, lens, [T, 1, T, 0, 3, T], T)
    kp, vp, bt = m.paged(5)
    kr, vr = m.ring(128)
    kd, vd, krd, vrd = dev_bits(kp), dev_bits(vp), dev_bits(kr), dev_bits(vr)
    q, kn, vn = dev_bits(m.q), dev_bits(m.k_new), dev_bits(m.v_new)
    sl, ql, sk, btd = dev(m.lens), dev(m.n), dev(m.sinks), dev(bt)
    B, Hq, D = m.c.B, m.c.Hq, m.c.D
    out_p = torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device=DEV)
    out_r = torch.empty_like(out_p)
    need = max(da.decode_attn_multi_workspace_bytes(B, Hq, 8, T, 0, bt.shape[1] * 16),
               da.decode_attn_multi_workspace_bytes(B, Hq, 8, T, 128, 0))
    da.decode_attn_multi_reserve(need)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture (the caches are rewritten below)
        da.decode_attn_paged_multi(q, kn, vn, kd, vd, btd, sl, sk, 0, m.c.scale, out_p, q_lens=ql)
        da.decode_attn_ring_multi(q, kn, vn, krd, vrd, sl, sk, m.c.scale, out_r, q_lens=ql)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            da.decode_attn_paged_multi(q, kn, vn, kd, vd, btd, sl, sk, 0, m.c.scale, out_p, q_lens=ql)
            da.decode_attn_ring_multi(q, kn, vn, krd, vrd, sl, sk, m.c.scale, out_r, q_lens=ql)
    torch.cuda.synchronize()
    # a new step in place: other lengths and counts, new queries and new tokens
    m2 = Multi(880, 64, 8, [250, 45, 1100, 60, 0, 800], [T, 2, 1, T, 0, T], T)
    kp2, vp2, bt2 = m2.paged(5, total_pages=kp.shape[0], table_width=bt.shape[1])  # the captured sizes
    kr2, vr2 = m2.ring(128)
    assert kp2.shape == kp.shape and bt2.shape == bt.shape
    for dst, src in ((kd, kp2), (vd, vp2), (krd, kr2), (vrd, vr2), (q, m2.q), (kn, m2.k_new),
                     (vn, m2.v_new)):
        dst.copy_(dev_bits(src))
    for dst, src in ((sl, m2.lens), (ql, m2.n), (btd, bt2), (sk, m2.sinks)):
        dst.copy_(dev(src))
    g.replay()
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    ref_p = oracle.decode_multi(m2.q, m2.k_new, m2.v_new, kp2, vp2, m2.lens, m2.sinks, 0, m2.c.scale,
                                block_table=bt2, q_lens=m2.n)
    ref_r = oracle.decode_multi(m2.q, m2.k_new, m2.v_new, kr2, vr2, m2.lens, m2.sinks, 128, m2.c.scale,
                                q_lens=m2.n)
    assert_close(out_p.double().cpu().numpy(), ref_p, "graph multi paged")
    assert_close(out_r.double().cpu().numpy(), ref_r, "graph multi ring")
    ek, ev = oracle.kv_append_multi(m2.k_new, m2.v_new, kp2, vp2, m2.lens, block_table=bt2, q_lens=m2.n)
    np.testing.assert_array_equal(wl.bits(kd), ek)
    np.testing.assert_array_equal(wl.bits(vd), ev)
    ek, ev = oracle.kv_append_multi(m2.k_new, m2.v_new, kr2, vr2, m2.lens, window=128, q_lens=m2.n)
    np.testing.assert_array_equal(wl.bits(krd), ek)
    np.testing.assert_array_equal(wl.bits(vrd), ev)
