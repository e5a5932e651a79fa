"""Small seeded decode-attention cases for tests (host side, numpy/torch CPU).

A case starts from a logical history of tokens per sequence; the caches are
materialised from it by plain array operations (reshape, transpose, roll,
page permutation) -- not by the oracle's address loops -- so comparing the
oracle's paged/ring readers against its contiguous reader pins the address
maps. Dead cells (slots past the last live token, unused and spare pages,
ring cells not yet written) hold bf16 NaN.
"""
from dataclasses import dataclass

import numpy as np
import torch

from paged_decode_attention_kv_gb300 import workloads as wl

NAN = np.uint16(wl.BF16_NAN_BITS)


@dataclass
class Case:
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    lens: np.ndarray        # [B] int32, post-append
    hist_k: np.ndarray      # [B, Tmax, Hkv, D] u16 (token L-1 is the new one)
    hist_v: np.ndarray
    q: np.ndarray           # [B, Hq, D] u16
    sinks: np.ndarray       # [Hq] f32
    k_new: np.ndarray       # [B, Hkv, D] u16
    v_new: np.ndarray
    scale: float = wl.SCALE


def make_case(seed, B, Hq, Hkv, D, lens, P=16) -> Case:
    gen = wl.cpu_generator(seed)
    lens = np.asarray(lens, dtype=np.int32)
    Tmax = max(1, int(lens.max()))
    hk, hv = wl.draw_history(B, Tmax, Hkv, D, gen)
    q = wl.randn_bf16((B, Hq, D), gen)
    sinks = torch.randn((Hq,), generator=gen, dtype=torch.float32).numpy()
    hk, hv, q = wl.bits(hk), wl.bits(hv), wl.bits(q)
    k_new = np.zeros((B, Hkv, D), np.uint16)
    v_new = np.zeros((B, Hkv, D), np.uint16)
    for b in range(B):
        if lens[b] > 0:
            k_new[b] = hk[b, lens[b] - 1]
            v_new[b] = hv[b, lens[b] - 1]
    return Case(B, Hq, Hkv, D, P, lens, hk, hv, q, sinks, k_new, v_new)


def paged_identity(c: Case, n_tokens, extra_pages_per_seq=0):
    """Pool where sequence b owns consecutive pages holding tokens 0..n[b]-1 in
    order (reshape of the history); pages cover ceil(L/P) so the append target
    page exists. Returns (k_pool, v_pool, block_table)."""
    P, Hkv, D = c.P, c.Hkv, c.D
    pages_k, pages_v, rows = [], [], []
    at = 0
    need = [max(1, -(-int(L) // P)) + extra_pages_per_seq for L in c.lens]
    maxp = max(need)
    for b in range(c.B):
        npg = need[b]
        buf_k = np.full((npg * P, Hkv, D), NAN, np.uint16)
        buf_v = np.full((npg * P, Hkv, D), NAN, np.uint16)
        n = int(n_tokens[b])
        buf_k[:n] = c.hist_k[b, :n]
        buf_v[:n] = c.hist_v[b, :n]
        pages_k.append(buf_k.reshape(npg, P, Hkv, D).transpose(0, 2, 1, 3))
        pages_v.append(buf_v.reshape(npg, P, Hkv, D).transpose(0, 2, 1, 3))
        row = np.full(maxp, -1, np.int32)
        row[:npg] = np.arange(at, at + npg)
        rows.append(row)
        at += npg
    return (np.ascontiguousarray(np.concatenate(pages_k)),
            np.ascontiguousarray(np.concatenate(pages_v)), np.stack(rows))


def shuffle_pages(k_pool, v_pool, block_table, seed, spare=3):
    """Move every page to a random physical slot of a larger NaN pool and
    rewrite the block table to match."""
    rng = np.random.default_rng(seed)
    n = k_pool.shape[0]
    total = n + spare
    perm = rng.permutation(total)[:n]          # old page i -> new page perm[i]
    k2 = np.full((total,) + k_pool.shape[1:], NAN, np.uint16)
    v2 = np.full_like(k2, NAN)
    k2[perm] = k_pool
    v2[perm] = v_pool
    bt = np.where(block_table >= 0, perm[np.maximum(block_table, 0)], -1).astype(np.int32)
    return k2, v2, bt


def ring_from_history(c: Case, n_tokens, W):
    """Ring [B, Hkv, W, D] after n[b] tokens, built with a roll: token j sits in
    cell j % W for the last min(n, W) tokens; never-written cells are NaN."""
    k = np.full((c.B, W, c.Hkv, c.D), NAN, np.uint16)
    v = np.full_like(k, NAN)
    for b in range(c.B):
        n = int(n_tokens[b])
        if n >= W:
            k[b] = np.roll(c.hist_k[b, n - W:n], shift=n % W, axis=0)
            v[b] = np.roll(c.hist_v[b, n - W:n], shift=n % W, axis=0)
        elif n > 0:
            k[b, :n] = c.hist_k[b, :n]
            v[b, :n] = c.hist_v[b, :n]
    return (np.ascontiguousarray(k.transpose(0, 2, 1, 3)),
            np.ascontiguousarray(v.transpose(0, 2, 1, 3)))


def bf16_to_f64(a):
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Round fp64 values to bf16 bit patterns (nearest-even via torch)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return wl.bits(t)
