"""CPU model of the one-token kernel's work split (host logic, no GPU), checked for the
invariants the kernel relies on: the units (one 16-token tile of one (sequence, KV head)
segment) are ordered (b, g, tile); CTA c takes [cta_start(c), cta_start(c + 1)), the even
split's boundary moved to the nearer edge of a short segment; its warps split that range
evenly. Every unit belongs to exactly one warp, every working CTA and warp has at least one
unit, a segment of at most `snap` units never spans two CTAs, and the CTA found for a unit
by searching near the even split is the CTA that owns it. The merge plan each warp works
out before its loop (head and tail segment, the consecutive warps holding each) is checked
against a walk over the warp's units, as the loop meets them.

The arithmetic mirrors the kernel's (32-bit integer formulas); the GPU parity tests run the
kernel itself on the same kinds of length mixes."""
import math

import numpy as np
import pytest

WARPS, MIN_TILES, MIN_TILES_SMALL, SNAP_UNITS, PAGE = 8, 4, 2, 32, 16


def units_prefix(lens, Hkv, window=0, ring=False):
    tiles = []
    for L in lens:
        if L <= 0:
            tiles.append(0)
        elif ring:
            tiles.append(math.ceil(min(L, window) / PAGE))
        else:
            lo = L - window if (window > 0 and L > window) else 0
            tiles.append((L - 1) // PAGE - lo // PAGE + 1)
    pre = np.concatenate([[0], np.cumsum(np.asarray(tiles) * Hkv)]).astype(np.int64)
    return pre, tiles


def segment_of_unit(pre, Hkv, x):
    b = int(np.searchsorted(pre, x, side="right") - 1)
    tiles = (pre[b + 1] - pre[b]) // Hkv
    g = (x - pre[b]) // tiles
    first = pre[b] + g * tiles
    return b * Hkv + g, int(first), int(first + tiles)


def split(pre, Hkv, ncta, min_tiles=None):
    U = int(pre[-1])
    if min_tiles is None:  # the kernel's rule: 2 tiles per worker for a call of <= 2 per grid worker
        min_tiles = MIN_TILES_SMALL if U <= 2 * ncta * WARPS else MIN_TILES
    nwork = min(ncta * WARPS, (U + min_tiles - 1) // min_tiles)
    if nwork >= WARPS:
        nwork -= nwork % WARPS
    q, r = divmod(U, nwork)
    wst = lambda w: w * q + (w * r) // nwork
    snap_max = min(SNAP_UNITS, 4 * q)

    def cta_start(c):
        x = wst(min(c * WARPS, nwork))
        if x <= 0 or x >= U:
            return x
        _, f, e = segment_of_unit(pre, Hkv, x)
        if x == f or e - f > snap_max:
            return x
        return f if x - f <= e - x else e

    n_cta = (nwork + WARPS - 1) // WARPS
    warps = []
    for c in range(n_cta):
        R0, R1 = cta_start(c), cta_start(c + 1)
        nw = min(WARPS, nwork - c * WARPS)
        qw, rw = divmod(R1 - R0, nw)
        for w in range(nw):
            warps.append((c, R0 + w * qw + (w * rw) // nw, R0 + (w + 1) * qw + ((w + 1) * rw) // nw))

    def cta_of(x):  # an fp32 estimate, then the search
        c = min(n_cta - 1, int(np.float32(x) * (np.float32(n_cta) / np.float32(U))))
        while c > 0 and cta_start(c) > x:
            c -= 1
        while c + 1 < n_cta and cta_start(c + 1) <= x:
            c += 1
        return c

    return U, n_cta, cta_start, warps, cta_of, snap_max


LEN_MIXES = {
    "b64": lambda rng: list(rng.integers(1024, 8193, 64)),
    "b1": lambda rng: [4096],
    "long1": lambda rng: [131072],
    "serve": lambda rng: [0 if rng.random() < 0.25 else int(min(32768, max(1, math.ceil(
        math.exp(math.log(2048) + rng.standard_normal()))))) for _ in range(256)],
    "short_many": lambda rng: list(rng.integers(1, 70, 300)) + [1500, 700, 1],
    "max_batch": lambda rng: [0 if rng.random() < 0.25 else int(rng.integers(1, 48)) for _ in range(1024)],
}


@pytest.mark.parametrize("mix", sorted(LEN_MIXES))
@pytest.mark.parametrize("ring", [False, True])
@pytest.mark.parametrize("min_tiles", [None, 2, 4])
def test_split_invariants(mix, ring, min_tiles):
    rng = np.random.default_rng(sum(map(ord, mix)) + ring)
    lens = LEN_MIXES[mix](rng)
    Hkv = 8 if mix != "short_many" else 2
    pre, _ = units_prefix(lens, Hkv, window=128, ring=ring)
    U = int(pre[-1])
    if U == 0:
        return
    U2, n_cta, cta_start, warps, cta_of, snap_max = split(pre, Hkv, ncta=152, min_tiles=min_tiles)
    # CTA boundaries strictly increasing from 0 to U: every working CTA has units
    bounds = [cta_start(c) for c in range(n_cta + 1)]
    assert bounds[0] == 0 and bounds[-1] == U
    assert all(a < b for a, b in zip(bounds, bounds[1:]))
    # warps tile [0, U) exactly, in order, each with at least one unit
    at = 0
    for c, ua, ue in warps:
        assert ua == at and ue > ua and bounds[c] <= ua and ue <= bounds[c + 1]
        at = ue
    assert at == U
    # a short segment never spans two CTAs; cta_of finds the owner
    for c in range(1, n_cta):
        x = bounds[c]
        _, f, e = segment_of_unit(pre, Hkv, x)
        if e - f <= snap_max:
            assert x in (f, e)
    for x in list(range(0, U, max(1, U // 500))) + [U - 1] + bounds[1:-1]:
        c = cta_of(x)
        assert bounds[c] <= x < bounds[c + 1]
    # balance: a CTA boundary moves by at most snap_max / 2 from the even split
    share = U / (len(warps))
    for c in range(n_cta):
        nw = sum(1 for w in warps if w[0] == c)
        assert bounds[c + 1] - bounds[c] <= nw * share + snap_max + 2


def test_ring_segments_of_the_serving_mix_stay_in_one_cta():
    """The window-128 ring layer of the serving mix: 8-tile segments and a worker share of
    about 10 units, so every CTA boundary sits on a segment edge."""
    rng = np.random.default_rng(4)
    lens = LEN_MIXES["serve"](rng)
    pre, _ = units_prefix(lens, 8, window=128, ring=True)
    U, n_cta, cta_start, warps, cta_of, snap_max = split(pre, 8, ncta=152)
    assert snap_max >= 8
    for c in range(1, n_cta):
        x = cta_start(c)
        _, f, e = segment_of_unit(pre, 8, x)
        assert x == f


def merge_plan(pre, Hkv, ua, ue):
    """The kernel's merge plan for a warp with units [ua, ue), from the split alone: its
    head segment (the first one, when it starts before ua) and its tail segment (the last one,
    when it goes on after ue; a single segment crossing either edge counts as the tail)."""
    sF, fF, eF = segment_of_unit(pre, Hkv, ua)
    sL, fL, eL = segment_of_unit(pre, Hkv, ue - 1)
    head = tail = None
    if sF == sL:
        if fF < ua or eL > ue:
            tail = (sL, fL, eL)
    else:
        if fF < ua:
            head = (sF, fF, eF)
        if eL > ue:
            tail = (sL, fL, eL)
    return head, tail


def walked_plan(pre, Hkv, ua, ue):
    """The same two segments as the main loop finds them, walking the warp's units in order:
    a segment left at a switch is kept (the head) when it began before ua, and the segment open
    at the end is kept (the tail) when it began before ua or goes on after ue."""
    head = None
    cur = None
    for x in range(ua, ue):
        seg, f, e = segment_of_unit(pre, Hkv, x)
        if cur is None or seg != cur[0]:
            if cur is not None and cur[1] < ua:
                head = cur
            cur = (seg, f, e)
    tail = cur if (cur[1] < ua or cur[2] > ue) else None
    return head, tail


@pytest.mark.parametrize("mix", sorted(LEN_MIXES))
@pytest.mark.parametrize("ring", [False, True])
def test_merge_plan_matches_the_walk_and_holders_are_consecutive(mix, ring):
    """The plan worked out before the loop names the same head and tail segments the loop's
    walk keeps, every warp of a CTA holding a unit of a shared segment has it in its plan, and
    the holders of each segment within a CTA are consecutive warps (first warp and count are
    what the merge uses)."""
    rng = np.random.default_rng(7 + sum(map(ord, mix)) + ring)
    lens = LEN_MIXES[mix](rng)
    Hkv = 8 if mix != "short_many" else 2
    pre, _ = units_prefix(lens, Hkv, window=128, ring=ring)
    if int(pre[-1]) == 0:
        return
    U, n_cta, cta_start, warps, cta_of, snap_max = split(pre, Hkv, ncta=152)
    by_cta = {}
    for c, ua, ue in warps:
        by_cta.setdefault(c, []).append((ua, ue))
    checked = 0
    for c, ranges in by_cta.items():
        if checked > 40 and mix in ("serve", "max_batch", "b64"):
            break
        checked += 1
        plans = [merge_plan(pre, Hkv, ua, ue) for ua, ue in ranges]
        for (ua, ue), plan in zip(ranges, plans):
            assert plan == walked_plan(pre, Hkv, ua, ue)
        # every segment a warp shares (with another warp or CTA) is in that warp's plan
        for w, (ua, ue) in enumerate(ranges):
            x = ua
            while x < ue:
                seg, f, e = segment_of_unit(pre, Hkv, x)
                shared = f < ua or e > ue
                in_plan = any(p is not None and p[0] == seg for p in plans[w])
                assert in_plan == shared, (c, w, seg)
                x = e
        # holders: the warps whose ranges meet the segment, consecutive
        for plan in plans:
            for p in plan:
                if p is None:
                    continue
                seg, f, e = p
                holders = [w for w, (ua, ue) in enumerate(ranges) if ua < e and ue > f]
                assert holders == list(range(holders[0], holders[-1] + 1))
                for w in holders:
                    assert any(q is not None and q[0] == seg for q in plans[w])
