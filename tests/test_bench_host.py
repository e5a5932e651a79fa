"""Host-side pieces of bench.py that run without a GPU: the staging of a step's inputs
in one buffer (one copy per direction in the end-to-end loop), the algorithmic byte
counts, and the recorded-traffic lookup."""
import os

import numpy as np
import pytest
import torch

import bench


def test_packed_views_are_aligned_and_round_trip():
    rng = np.random.default_rng(3)
    tensors = [torch.from_numpy(rng.standard_normal((5, 7)).astype(np.float32)).to(torch.bfloat16),
               torch.arange(13, dtype=torch.int32),
               torch.from_numpy(rng.standard_normal(3).astype(np.float32)),
               torch.zeros((0,), dtype=torch.int32)]
    buf, views = bench.packed(tensors)
    assert buf.dtype == torch.uint8 and buf.dim() == 1
    base = buf.data_ptr()
    ends = []
    for v, t in zip(views, tensors):
        assert v.dtype == t.dtype and v.shape == t.shape and v.is_contiguous()
        if t.numel() == 0:  # an empty view has no meaningful address
            continue
        off = v.data_ptr() - base
        assert off % 256 == 0
        ends.append((off, off + t.numel() * t.element_size()))
        v.copy_(t)
    # the views do not overlap and lie inside the buffer
    for (a0, a1), (b0, b1) in zip(ends, ends[1:]):
        assert a1 <= b0
    assert ends[-1][1] <= buf.numel()
    for v, t in zip(views, tensors):
        assert torch.equal(v, t)
    # one copy of the whole buffer carries every tensor
    buf2, views2 = bench.packed(tensors)
    buf2.copy_(buf)
    for v, t in zip(views2, tensors):
        assert torch.equal(v, t)


def test_algorithmic_bytes_scale_with_the_cache_format():
    lens = [1000, 17, 0, 4096]
    args = (64, 8, 64, 16, 128)
    bf = bench.algorithmic_bytes(lens, "paged_full", *args, kv="bf16")
    f8 = bench.algorithmic_bytes(lens, "paged_full", *args, kv="fp8")
    # per cached token and KV head: 256 bytes of bf16 K + V against 136 of e4m3 codes + scales
    cached = sum(max(0, L - 1) for L in lens) * 8
    assert bf - f8 == pytest.approx(cached * (256 - 136), rel=0.05)
    assert bench.algorithmic_bytes([0, 0], "paged_full", *args, kv="bf16") < 4096


def test_recorded_traffic_is_ignored_for_another_source(tmp_path, monkeypatch):
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\nb64 paged %s 123456\nb64 paged 0000000000000000 999\n" % bench.source_hash())
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("b64", "paged") == 123456.0
    assert bench.recorded_traffic("b64", "ring") is None
    f.write_text("b64 paged 0000000000000000 999\n")
    assert bench.recorded_traffic("b64", "paged") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", os.path.join(str(tmp_path), "missing.txt"))
    assert bench.recorded_traffic("b64", "paged") is None


def test_the_code_hash_ignores_comments_only():
    src = 'int a = 1; // one\nconst char *s = "// kept /* kept */"; /* two\nlines */ char c = \'"\';'
    out = bench.strip_comments(src)
    assert "one" not in out and "two" not in out and "lines" not in out
    assert '"// kept /* kept */"' in out and "char c = '\"';" in out and "int a = 1;" in out
    assert bench.strip_comments(src.replace("// one", "// another")) == out
    assert bench.strip_comments(src.replace("a = 1", "a = 2")) != out


def test_launch_count_sums_the_library_answer_per_layer(monkeypatch):
    import paged_decode_attention_kv_gb300 as da
    cfg = {"B": 64, "Hq": 64, "Hkv": 8, "page_size": 16, "window": 128}
    seen = []

    def fake(B, Hq, Hkv, T, ring_window, max_seq_len):
        seen.append((B, Hq, Hkv, T, ring_window, max_seq_len))
        return 1 if ring_window == 0 else 2  # paged call fused, ring call attention + append

    monkeypatch.setattr(da, "decode_attn_multi_launches", fake)
    assert bench.launches_per_step(1, cfg, 495) == 2  # one token: one launch per layer
    assert seen == []
    assert bench.launches_per_step(4, cfg, 495) == 3
    assert seen == [(64, 64, 8, 4, 0, 495 * 16), (64, 64, 8, 4, 128, 0)]
    # with the rotary embedding each layer's call launches its rotation kernel first
    assert bench.launches_per_step(4, cfg, 495, rope=True) == 5
    monkeypatch.setattr(da, "decode_attn_multi_launches", lambda *a: 0)
    with pytest.raises(RuntimeError):
        bench.launches_per_step(4, cfg, 495)
