"""Seeded synthetic inputs for decode attention.

This module only draws random numbers: values, lengths, page permutations. It
holds none of the attention arithmetic and none of the cache address maps, so
the CUDA path and the CPU oracle can both be fed from it.

Recipe (shapes from the gpt-oss attention used by the SimpleLLM engine: 64
query heads, 8 KV heads, head dim 64, page 16, window 128):
  * q, k, v values ~ N(0, 1) drawn in fp32 and rounded to bf16 (nearest-even);
  * sink logits ~ N(0, 1) in fp32; scale = 1/8 (= 1/sqrt(64));
  * block tables hand out pages from a shuffled free list; unused table entries
    are -1;
  * pools are either fully random (benchmark) or NaN-filled (tests, where the
    oracle writes the live tokens in and every dead cell stays NaN);
  * fp8 pools (benchmark) are 2176-byte blocks of uniform random finite e4m3
    codes and per-token scales uniform in [2/448, 3/448).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

BF16_NAN_BITS = 0x7FC0

# name -> recipe. "lens" is either a list or a rule resolved by seq_lens().
CONFIGS = {
    "tiny": dict(seed=0, B=2, Hq=8, Hkv=1, D=64, page_size=16, window=16,
                 lens=[37, 200], spare_pages=4),
    "b1": dict(seed=1, B=1, Hq=64, Hkv=8, D=64, page_size=16, window=128,
               lens=[4096], pool_pages=512),
    "b64": dict(seed=2, B=64, Hq=64, Hkv=8, D=64, page_size=16, window=128,
                lens="uniform", lo=1024, hi=8192, spare_frac=0.10),
    "long1": dict(seed=3, B=1, Hq=64, Hkv=8, D=64, page_size=16, window=128,
                  lens=[131072], spare_frac=0.0),
    "long8": dict(seed=3, B=8, Hq=64, Hkv=8, D=64, page_size=16, window=128,
                  lens=[131072] * 8, spare_frac=0.0),
    "serve": dict(seed=4, B=256, Hq=64, Hkv=8, D=64, page_size=16, window=128,
                  lens="lognormal", median=2048, sigma=1.0, max_len=32768, inactive=64,
                  max_pages_per_seq=2048, spare_frac=0.10),
}

SCALE = 0.125


def config(name: str) -> dict:
    if name not in CONFIGS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}")
    return dict(CONFIGS[name])


def cpu_generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def seq_lens(name: str) -> list[int]:
    """Post-append sequence lengths of a named workload (0 = inactive slot)."""
    c = config(name)
    lens = c["lens"]
    if isinstance(lens, list):
        return list(lens)
    g = cpu_generator(c["seed"] + 1000)
    B = c["B"]
    if lens == "uniform":
        return torch.randint(c["lo"], c["hi"] + 1, (B,), generator=g).tolist()
    if lens == "lognormal":
        z = torch.randn(B, generator=g, dtype=torch.float64)
        raw = torch.exp(math.log(c["median"]) + c["sigma"] * z)
        active = torch.clamp(torch.ceil(raw), 1, c["max_len"]).to(torch.int64)
        inactive = torch.randperm(B, generator=g)[: c["inactive"]]
        active[inactive] = 0
        return active.tolist()
    raise ValueError(lens)


def randn_bf16(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """N(0,1) drawn in fp32, rounded to bf16 (round-to-nearest-even)."""
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)


def nan_bf16(shape, device="cpu") -> torch.Tensor:
    t = torch.full(shape, BF16_NAN_BITS, dtype=torch.int16, device=device)
    return t.view(torch.bfloat16)


def pages_needed(n_tokens: int, page_size: int) -> int:
    """Pages a sequence of n_tokens occupies (allocation bookkeeping)."""
    return -(-n_tokens // page_size)


@dataclass
class DecodeInputs:
    """Per-step inputs of one attention layer for a batch of sequences."""
    q: torch.Tensor          # [B, Hq, D] bf16
    k_new: torch.Tensor      # [B, Hkv, D] bf16
    v_new: torch.Tensor      # [B, Hkv, D] bf16
    sinks: torch.Tensor      # [Hq] fp32
    seq_lens: torch.Tensor   # [B] int32, post-append
    scale: float = SCALE


@dataclass
class PagedPool:
    k_cache: torch.Tensor       # [num_pages, Hkv, P, D] bf16
    v_cache: torch.Tensor
    block_table: torch.Tensor   # [B, max_pages_per_seq] int32, -1 = unused
    page_size: int
    max_pages_per_seq: int

    @property
    def num_pages(self) -> int:
        return self.k_cache.shape[0]


@dataclass
class RingPool:
    k_cache: torch.Tensor       # [B, Hkv, W, D] bf16
    v_cache: torch.Tensor
    window: int


def draw_decode_inputs(B, Hq, Hkv, D, lens, gen, device="cpu") -> DecodeInputs:
    q = randn_bf16((B, Hq, D), gen, device)
    k_new = randn_bf16((B, Hkv, D), gen, device)
    v_new = randn_bf16((B, Hkv, D), gen, device)
    sinks = torch.randn((Hq,), generator=gen, dtype=torch.float32, device=device)
    sl = torch.tensor(lens, dtype=torch.int32, device=device)
    return DecodeInputs(q, k_new, v_new, sinks, sl)


def draw_block_table(lens, page_size, num_pages, max_pages_per_seq, gen) -> torch.Tensor:
    """Hand each sequence pages_needed(L) distinct pages from a shuffled free list."""
    need = [pages_needed(L, page_size) for L in lens]
    if sum(need) > num_pages:
        raise ValueError("pool too small")
    if max(need, default=0) > max_pages_per_seq:
        raise ValueError("max_pages_per_seq too small")
    free = torch.randperm(num_pages, generator=gen).to(torch.int32)
    bt = torch.full((len(lens), max_pages_per_seq), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        bt[b, :n] = free[at:at + n]
        at += n
    return bt


def pool_size(name: str, lens) -> int:
    c = config(name)
    P = c["page_size"]
    used = sum(pages_needed(L, P) for L in lens)
    if "pool_pages" in c:
        return max(c["pool_pages"], used)
    if "spare_pages" in c:
        return used + c["spare_pages"]
    return used + int(math.ceil(used * c.get("spare_frac", 0.0)))


def max_pages_per_seq(name: str, lens) -> int:
    c = config(name)
    if "max_pages_per_seq" in c:
        return c["max_pages_per_seq"]
    return max(1, max(pages_needed(L, c["page_size"]) for L in lens))


def draw_paged_pool(num_pages, Hkv, P, D, lens, max_pages, gen, device="cpu",
                    fill="randn", value_gen=None) -> PagedPool:
    """Block table from `gen` (CPU); pool contents random (fill='randn', drawn from
    value_gen or gen on `device`) or NaN (fill='nan')."""
    bt = draw_block_table(lens, P, num_pages, max_pages, gen)
    shape = (num_pages, Hkv, P, D)
    if fill == "randn":
        vg = value_gen or gen
        k = randn_bf16(shape, vg, device)
        v = randn_bf16(shape, vg, device)
    elif fill == "nan":
        k, v = nan_bf16(shape, device), nan_bf16(shape, device)
    else:
        raise ValueError(fill)
    return PagedPool(k, v, bt.to(device), P, max_pages)


def draw_ring_pool(B, Hkv, W, D, gen, device="cpu", fill="randn") -> RingPool:
    shape = (B, Hkv, W, D)
    if fill == "randn":
        k, v = randn_bf16(shape, gen, device), randn_bf16(shape, gen, device)
    elif fill == "nan":
        k, v = nan_bf16(shape, device), nan_bf16(shape, device)
    else:
        raise ValueError(fill)
    return RingPool(k, v, W)


FP8_BLOCK_BYTES = 2176  # 16 tokens of one KV head: K codes, V^T codes, K and V scales


def draw_fp8_codes(shape, gen, device="cpu") -> torch.Tensor:
    """Uniform random e4m3 byte patterns with the two NaN patterns (0x7F, 0xFF)
    redrawn as their neighbours 0x7E / 0xFE: every finite code, both signs."""
    c = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32, device=device)
    c = torch.where((c & 0x7F) == 0x7F, c - 1, c)
    return c.to(torch.uint8)


def draw_fp8_scales(shape, gen, device="cpu") -> torch.Tensor:
    """Per-token scales in [2/448, 3/448): what a row of N(0,1) values with an
    absolute maximum of 2 to 3 would get."""
    u = torch.rand(shape, generator=gen, dtype=torch.float32, device=device)
    return (2.0 + u) / 448.0


def draw_fp8_blocks(lead, gen, P=16, D=64, device="cpu") -> torch.Tensor:
    """fp8 cache blocks [*lead, 2PD + 8P] bytes: random codes (K rows, V^T) then random
    per-token K and V scales."""
    codes = draw_fp8_codes(tuple(lead) + (2 * P * D,), gen, device)
    scales = draw_fp8_scales(tuple(lead) + (2 * P,), gen, device)
    return torch.cat([codes, scales.view(torch.uint8)], dim=-1).contiguous()


def draw_fp8_paged_pool(num_pages, Hkv, P, D, gen, device="cpu") -> torch.Tensor:
    """[num_pages, Hkv, 2176]: one block per page and KV head."""
    return draw_fp8_blocks((num_pages, Hkv), gen, P, D, device)


def draw_fp8_ring_pool(B, Hkv, W, D, gen, device="cpu", P=16) -> torch.Tensor:
    """[B, Hkv, W / 16, 2176]: the ring of capacity W as blocks of 16 cells."""
    return draw_fp8_blocks((B, Hkv, W // P), gen, P, D, device)


def draw_history(B, Tmax, Hkv, D, gen, device="cpu"):
    """Contiguous per-sequence K/V histories [B, Tmax, Hkv, D] bf16."""
    return randn_bf16((B, Tmax, Hkv, D), gen, device), randn_bf16((B, Tmax, Hkv, D), gen, device)


def bits(t: torch.Tensor):
    """Raw 16-bit patterns of a bf16 tensor as a numpy uint16 array (host copy)."""
    import numpy as np
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a, device="cpu") -> torch.Tensor:
    """bf16 tensor from a numpy uint16 array of raw patterns."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def rope_tables(max_position: int, D: int, base: float = 150000.0):
    """cos/sin tables [max_position, D/2] fp32 of the plain rotary schedule
    angle(pos, i) = pos * base^(-2i/D), computed in fp64 and rounded once. These
    are caller inputs (the model's frequency schedule; a scaled schedule such as
    YaRN would be folded into the same tables)."""
    import numpy as np
    pos = np.arange(max_position, dtype=np.float64)[:, None]
    inv = base ** (-np.arange(0, D, 2, dtype=np.float64) / D)[None, :]
    ang = pos * inv
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
