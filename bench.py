"""Benchmark of the fused decode-attention step on GB300.

A step is one decode step of attention for one full-attention layer (paged KV
cache, page 16) and one sliding-window layer (ring of 128 cells), each with
its fused 1-token KV append, for the gpt-oss head shape (64 query heads, 8 KV
heads, head dim 64). Default workload: batch 64, lengths uniform in
[1024, 8192]. Prints one JSON line.

  value     achieved HBM GB/s of the step (algorithmic bytes / device time),
            summed over all ranks (replicas; the path needs no exchange)
  roofline  the paged kernel's own GB/s against the measured HBM copy peak
  e2e       the same metric end to end through the public API, with the
            step's inputs copied from pinned host memory and outputs read back
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/call and achieved HBM GB/s (% of GB300 peak) per config"
UNIT = "GB/s"
KERNEL_SRC = os.path.join(ROOT, "paged_decode_attention_kv_gb300", "csrc", "decode_attn.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
FALLBACK_HBM_GBS = 6800.0
HBM_BUS_BITS = 8192  # 8 HBM3e stacks x 1024 bits


# ---------------------------------------------------------------- bytes the method must move
def algorithmic_bytes(lens, kind, Hq, Hkv, D, P, W, kv="bf16", q_tokens=1):
    """Per call: cached K+V of the attended positions (each read once per sequence and KV
    head, however many query tokens see it), the n = q_tokens new tokens' k/v read and
    written into the cache, q read and out written for the n rows, block-table entries
    read, seq_lens, sinks. A cached token costs 2*2*D bytes per KV head in bf16, or 2*D
    codes + two fp32 scales in fp8."""
    tok = 4 * D if kv == "bf16" else 2 * D + 8
    total = 0
    for L in lens:
        if L <= 0:
            continue
        n = min(q_tokens, L)
        base = L - n
        if kind == "paged_full":
            cached, tiles = base, math.ceil(L / P)
        elif kind == "paged_window":
            lo = max(0, base - W + 1)
            cached, tiles = base - lo, (L - 1) // P - lo // P + 1
        else:  # ring: the union of the n windows reaches W - 1 positions behind the first
            cached, tiles = min(base, W - 1), 0
        total += cached * tok * Hkv + n * (2 * 2 * Hkv * D + tok * Hkv) + 2 * Hq * D * n \
            + 2 * Hq * D * n + 4 * tiles
    return total + 4 * len(lens) + 4 * Hq


# ---------------------------------------------------------------- ranks (replicas)
def max_over_ranks(x: float, device) -> float:
    """The slowest rank's value (all ranks get it); x itself on a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank: float, ms_per_step_max: float, world: int) -> float:
    """Whole-job throughput: every rank moves the same bytes per step (weak scaling),
    divided by the slowest rank's time per step."""
    return world * bytes_per_step_per_rank / (ms_per_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------- environment helpers
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def nominal_hbm_peak():
    """Memory clock x 2 (double data rate) x bus width, for context next to the measured peak."""
    mhz = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("mem_max_mhz") or 0) or None
    except Exception:
        pass
    if mhz is None:
        try:
            out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.memory",
                                  "--format=csv,noheader,nounits"], capture_output=True,
                                 text=True, timeout=10).stdout.split()
            mhz = float(out[0])
        except Exception:
            return None
    return mhz * 1e6 * 2 * HBM_BUS_BITS / 8 / 1e9


def strip_comments(src: str) -> str:
    """C/C++ source without its // and /* */ comments (string and character literals kept),
    so that editing a comment does not change what the code hash identifies."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # a literal: copy through its closing quote
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join(out)


def source_hash():
    """sha256[:16] of the kernel sources' code (every .cu / .cuh of csrc, in name order,
    comments removed)."""
    h = hashlib.sha256()
    csrc = os.path.dirname(KERNEL_SRC)
    for name in sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh"))):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kind):
    """DRAM bytes per launch from an ncu capture, if taken on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload \
                        and parts[1] == kind and parts[2] == source_hash():
                    return float(parts[3])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 8:
                    continue
                if self.uuid and self.uuid not in p[0]:
                    continue
                rows.append(p)
        os.unlink(self.tmp.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------- workload construction
class StepInputs:
    """One independent copy of a step's inputs and caches on the device."""

    def __init__(self, name, device, seed_offset=0, batch_limit=None, kv="bf16", q_tokens=1):
        import torch
        from paged_decode_attention_kv_gb300 import workloads as wl
        cfg = wl.config(name)
        # T new tokens per sequence behind the same cached history as the 1-token step
        self.T = q_tokens
        self.lens = [L + q_tokens - 1 if L > 0 else 0 for L in wl.seq_lens(name)[:batch_limit]]
        cfg["B"] = len(self.lens)
        self.cfg = cfg
        seed = cfg["seed"] + seed_offset
        gen = wl.cpu_generator(seed)
        vgen = torch.Generator(device=device)
        vgen.manual_seed(seed)
        B, Hq, Hkv, D, P, W = (cfg[k] for k in ("B", "Hq", "Hkv", "D", "page_size", "window"))
        self.kv = kv
        self.inp = wl.draw_decode_inputs(B, Hq, Hkv, D, self.lens, gen)
        npages = wl.pool_size(name, self.lens)
        if kv == "bf16":
            self.pool = wl.draw_paged_pool(npages, Hkv, P, D, self.lens,
                                           wl.max_pages_per_seq(name, self.lens), gen,
                                           device=device, value_gen=vgen)
            self.ring = wl.draw_ring_pool(B, Hkv, W, D, vgen, device=device)
            self.block_table = self.pool.block_table
        else:
            self.block_table = wl.draw_block_table(self.lens, P, npages,
                                                   wl.max_pages_per_seq(name, self.lens),
                                                   gen).to(device)
            self.pool = wl.draw_fp8_paged_pool(npages, Hkv, P, D, vgen, device=device)
            self.ring = wl.draw_fp8_ring_pool(B, Hkv, W, D, vgen, device=device)
        d = lambda t: t.to(device).contiguous()
        if q_tokens > 1:  # [B, T, heads, D] rows instead
            self.inp.q = wl.randn_bf16((B, q_tokens, Hq, D), gen)
            self.inp.k_new = wl.randn_bf16((B, q_tokens, Hkv, D), gen)
            self.inp.v_new = wl.randn_bf16((B, q_tokens, Hkv, D), gen)
        self.q, self.k_new, self.v_new = d(self.inp.q), d(self.inp.k_new), d(self.inp.v_new)
        self.seq_lens, self.sinks = d(self.inp.seq_lens), d(self.inp.sinks)
        self.out_full = torch.empty(tuple(self.q.shape), dtype=torch.bfloat16, device=device)
        self.out_ring = torch.empty_like(self.out_full)
        cs, sn = wl.rope_tables(max(self.lens) + 1, D)
        self.rope_cos = torch.from_numpy(cs).to(device)
        self.rope_sin = torch.from_numpy(sn).to(device)

    def cache_tensors(self):
        if self.kv == "bf16":
            return [self.pool.k_cache, self.pool.v_cache, self.ring.k_cache, self.ring.v_cache]
        return [self.pool, self.ring]

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in self.cache_tensors())


def call_paged(s, rope, q=None, k_new=None, v_new=None, bt=None, sl=None, sinks=None, out=None):
    import paged_decode_attention_kv_gb300 as da
    out = s.out_full if out is None else out
    q = s.q if q is None else q
    k_new = s.k_new if k_new is None else k_new
    v_new = s.v_new if v_new is None else v_new
    bt = s.block_table if bt is None else bt
    sl = s.seq_lens if sl is None else sl
    sinks = s.sinks if sinks is None else sinks
    if s.T > 1 and rope:
        da.decode_attn_paged_multi_rope(q, k_new, v_new, s.pool.k_cache, s.pool.v_cache, bt, sl, sinks,
                                        s.rope_cos, s.rope_sin, 0, s.inp.scale, out)
    elif s.T > 1:
        da.decode_attn_paged_multi(q, k_new, v_new, s.pool.k_cache, s.pool.v_cache, bt, sl, sinks, 0,
                                   s.inp.scale, out)
    elif s.kv == "fp8" and rope:
        da.decode_attn_paged_fp8_rope(q, k_new, v_new, s.pool, bt, sl, sinks, s.rope_cos, s.rope_sin, 0,
                                      s.inp.scale, out)
    elif s.kv == "fp8":
        da.decode_attn_paged_fp8(q, k_new, v_new, s.pool, bt, sl, sinks, 0, s.inp.scale, out)
    elif rope:
        da.decode_attn_paged_rope(q, k_new, v_new, s.pool.k_cache, s.pool.v_cache, bt, sl, sinks,
                                  s.rope_cos, s.rope_sin, 0, s.inp.scale, out)
    else:
        da.decode_attn_paged(q, k_new, v_new, s.pool.k_cache, s.pool.v_cache, bt, sl, sinks, 0,
                             s.inp.scale, out)


def call_ring(s, rope, q=None, k_new=None, v_new=None, sl=None, sinks=None, out=None):
    import paged_decode_attention_kv_gb300 as da
    out = s.out_ring if out is None else out
    q = s.q if q is None else q
    k_new = s.k_new if k_new is None else k_new
    v_new = s.v_new if v_new is None else v_new
    sl = s.seq_lens if sl is None else sl
    sinks = s.sinks if sinks is None else sinks
    if s.T > 1 and rope:
        da.decode_attn_ring_multi_rope(q, k_new, v_new, s.ring.k_cache, s.ring.v_cache, sl, sinks,
                                       s.rope_cos, s.rope_sin, s.inp.scale, out)
    elif s.T > 1:
        da.decode_attn_ring_multi(q, k_new, v_new, s.ring.k_cache, s.ring.v_cache, sl, sinks,
                                  s.inp.scale, out)
    elif s.kv == "fp8" and rope:
        da.decode_attn_ring_fp8_rope(q, k_new, v_new, s.ring, sl, sinks, s.rope_cos, s.rope_sin,
                                     s.inp.scale, out)
    elif s.kv == "fp8":
        da.decode_attn_ring_fp8(q, k_new, v_new, s.ring, sl, sinks, s.inp.scale, out)
    elif rope:
        da.decode_attn_ring_rope(q, k_new, v_new, s.ring.k_cache, s.ring.v_cache, sl, sinks,
                                 s.rope_cos, s.rope_sin, s.inp.scale, out)
    else:
        da.decode_attn_ring(q, k_new, v_new, s.ring.k_cache, s.ring.v_cache, sl, sinks,
                            s.inp.scale, out)


def decode_route(q_tokens, cfg):
    """Whether the library runs a paged multi-token call in the decode kernel (up to four
    query tokens, at most 32 query rows per KV head), append fused."""
    return 1 < q_tokens <= 4 and q_tokens * cfg["Hq"] // cfg["Hkv"] <= 32


def launches_per_step(q_tokens, cfg, max_pages, rope=False):
    """Kernel launches of one step (a paged and a ring layer): one per layer for a single
    query token; for several, what the library reports for each layer's call (the attention,
    the append unless fused, and a kernel that folds many key splits' partials), plus the
    rotation kernel of each layer's call with the rotary embedding."""
    if q_tokens == 1:
        return 2
    import paged_decode_attention_kv_gb300 as da
    n = [da.decode_attn_multi_launches(cfg["B"], cfg["Hq"], cfg["Hkv"], q_tokens, 0, max_pages * cfg["page_size"]),
         da.decode_attn_multi_launches(cfg["B"], cfg["Hq"], cfg["Hkv"], q_tokens, cfg["window"], 0)]
    if min(n) <= 0:
        raise RuntimeError("the library reported no launch count for this shape")
    return sum(n) + (2 if rope else 0)


def step_bytes(name, lens, kv="bf16", q_tokens=1):
    from paged_decode_attention_kv_gb300 import workloads as wl
    c = wl.config(name)
    args = (c["Hq"], c["Hkv"], c["D"], c["page_size"], c["window"])
    return (algorithmic_bytes(lens, "paged_full", *args, kv=kv, q_tokens=q_tokens),
            algorithmic_bytes(lens, "ring", *args, kv=kv, q_tokens=q_tokens))


# ---------------------------------------------------------------- the CPU oracle on a sample
def oracle_sample(name, s: "StepInputs", budget_s):
    """Time the fp64 oracle on whole sequences (all heads, both layers) of this workload,
    adding sequences until about budget_s of CPU work. Returns (GB/s, cores, description)."""
    import numpy as np
    import oracle
    from paged_decode_attention_kv_gb300 import workloads as wl
    c = s.cfg
    Hq, P, W = c["Hq"], c["page_size"], c["window"]
    if s.kv == "bf16":
        kp, vp = wl.bits(s.pool.k_cache), wl.bits(s.pool.v_cache)
        rk, rv = wl.bits(s.ring.k_cache), wl.bits(s.ring.v_cache)
    else:
        pool8, ring8 = oracle.Fp8Cache(s.pool.cpu().numpy()), oracle.Fp8Cache(s.ring.cpu().numpy())
    q, kn, vn = wl.bits(s.inp.q), wl.bits(s.inp.k_new), wl.bits(s.inp.v_new)
    bt = s.block_table.cpu().numpy()
    lens = np.asarray(s.lens, np.int32)
    sinks = s.inp.sinks.numpy()
    cores = oracle.default_threads()
    done_bytes, elapsed, seqs = 0, 0.0, 0
    order = [b for b in range(len(lens)) if lens[b] > 0]
    passes = 0
    while elapsed < budget_s and order:
        for b in order:
            items = [(b, h) for h in range(Hq)]
            t0 = time.perf_counter()
            if s.T > 1 and getattr(s, "rope", False):
                one = slice(b, b + 1)
                cs, sn = s.rope_cos.cpu().numpy(), s.rope_sin.cpu().numpy()
                oracle.decode_multi_rope(q[one], kn[one], vn[one], kp, vp, lens[one], sinks, cs, sn, 0,
                                         s.inp.scale, block_table=bt[one], nthreads=cores)
                oracle.decode_multi_rope(q[one], kn[one], vn[one], rk[one], rv[one], lens[one], sinks,
                                         cs, sn, W, s.inp.scale, nthreads=cores)
            elif s.T > 1:
                one = slice(b, b + 1)
                oracle.decode_multi(q[one], kn[one], vn[one], kp, vp, lens[one], sinks, 0,
                                    s.inp.scale, block_table=bt[one], nthreads=cores)
                oracle.decode_multi(q[one], kn[one], vn[one], rk[one], rv[one], lens[one], sinks,
                                    W, s.inp.scale, nthreads=cores)
            elif s.kv == "fp8" and getattr(s, "rope", False):
                cs, sn = s.rope_cos.cpu().numpy(), s.rope_sin.cpu().numpy()
                oracle.decode_paged_fp8_rope(q, kn, vn, pool8, bt, lens, sinks, cs, sn, 0, s.inp.scale,
                                             items=items, nthreads=cores)
                oracle.decode_ring_fp8_rope(q, kn, vn, ring8, lens, sinks, cs, sn, W, s.inp.scale,
                                            items=items, nthreads=cores)
            elif s.kv == "fp8":
                oracle.decode_paged_fp8(q, kn, vn, pool8, bt, lens, sinks, 0, s.inp.scale,
                                        items=items, nthreads=cores)
                oracle.decode_ring_fp8(q, kn, vn, ring8, lens, sinks, W, s.inp.scale,
                                       items=items, nthreads=cores)
            elif getattr(s, "rope", False):
                cs, sn = s.rope_cos.cpu().numpy(), s.rope_sin.cpu().numpy()
                oracle.decode_paged_rope(q, kn, vn, kp, vp, bt, lens, sinks, cs, sn, 0,
                                         s.inp.scale, P, items=items, nthreads=cores)
                oracle.decode_ring_rope(q, kn, vn, rk, rv, lens, sinks, cs, sn, W, s.inp.scale,
                                        items=items, nthreads=cores)
            else:
                oracle.decode_paged(q, kn, vn, kp, vp, bt, lens, sinks, 0, s.inp.scale, P,
                                    items=items, nthreads=cores)
                oracle.decode_ring(q, kn, vn, rk, rv, lens, sinks, W, s.inp.scale, items=items,
                                   nthreads=cores)
            elapsed += time.perf_counter() - t0
            pb, rb = step_bytes(name, [int(lens[b])], s.kv, s.T)
            done_bytes += pb + rb
            seqs += 1
            if elapsed >= budget_s:
                break
        passes += 1
    desc = (f"{seqs} sequence-steps ({passes} pass(es) over the {len(order)} active sequences), "
            f"all {Hq} heads" + (f" x {s.T} query tokens" if s.T > 1 else "") +
            f", full + ring layer; {elapsed:.1f} s on {cores} threads")
    return done_bytes / elapsed / 1e9, cores, desc


# ---------------------------------------------------------------- arms
def run_reference(args, rank, world):
    """The oracle as the reference arm: timed on the host cores, rank 0 only."""
    if rank != 0:
        return None
    import torch
    device = "cuda" if torch.cuda.is_available() else "cpu"
    s = StepInputs(args.workload, device, batch_limit=args.batch_limit, kv=args.kv,
                   q_tokens=args.q_tokens)
    s.rope = args.rope
    # each step is a bounded sample: calibrate so that warmup+steps fit ~90 s
    per_step = max(0.02, min(10.0, 90.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(args.workload, s, per_step)
    vals, descs = [], []
    for _ in range(args.steps):
        v, cores, desc = oracle_sample(args.workload, s, per_step)
        vals.append(v)
        descs.append(desc)
    value = statistics.median(vals)
    pbytes, rbytes = step_bytes(args.workload, s.lens, args.kv, args.q_tokens)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round((pbytes + rbytes) / (value * 1e9) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(args.workload, s),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": descs[-1]},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def workload_config(name, s):
    c = s.cfg
    lens = [L for L in s.lens if L > 0]
    return {"workload": name, "batch": c["B"], "active": len(lens), "q_heads": c["Hq"],
            "kv_heads": c["Hkv"], "head_dim": c["D"], "page_size": c["page_size"],
            "window": c["window"], "mean_len": round(sum(lens) / max(1, len(lens)), 1),
            "max_len": max(lens) if lens else 0,
            "layers_per_step": ["paged full attention", f"ring window {c['window']}"],
            "rope": bool(getattr(s, "rope", False)),
            "kv_cache": "bf16" if s.kv == "bf16" else "fp8 e4m3 codes + per-token fp32 scales",
            "q_tokens": s.T,
            "parallelism": "replicas", **({"note": c["workload_note"]} if "workload_note" in c else {})}


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_decode_attention_kv_gb300 as da
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    da.decode_attn_set_early_inputs(args.early_inputs)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    # one set = the layer pairs of one step (each pair: a full layer and a ring layer with
    # their own caches); more sets rotate when one step's inputs would fit in L2
    def make_set(k):
        return [StepInputs(args.workload, dev, seed_offset=k * 10007 + 101 * li,
                           batch_limit=args.batch_limit, kv=args.kv, q_tokens=args.q_tokens)
                for li in range(args.layers)]
    sets = [make_set(0)]
    first = sets[0][0]
    first.rope = args.rope
    set_bytes = sum(l.nbytes() for l in sets[0])
    n_sets = 1 if set_bytes >= 2 * l2 else min(64, math.ceil(2 * l2 / set_bytes))
    sets += [make_set(k) for k in range(1, n_sets)]
    cfg = first.cfg
    B, Hq, Hkv, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"]
    da.decode_attn_reserve(da.decode_attn_workspace_bytes(B, Hq, Hkv, D))
    pbytes, rbytes = step_bytes(args.workload, first.lens, args.kv, args.q_tokens)
    pbytes_call, rbytes_call = pbytes, rbytes
    pbytes, rbytes = pbytes * args.layers, rbytes * args.layers
    if args.batch_limit is not None:
        first.cfg["workload_note"] = f"first {args.batch_limit} sequences only"
    stream = torch.cuda.current_stream()

    def step(layer_set):
        for s in layer_set:
            call_paged(s, args.rope)
            call_ring(s, args.rope)

    for i in range(args.warmup):
        step(sets[i % n_sets])
    torch.cuda.synchronize()
    assert da.decode_attn_device_status() == 0
    graphs = None
    if args.graph:  # the whole step captured once per input set
        from paged_decode_attention_kv_gb300.graph import DecodeStepGraph
        graphs = []
        for st in sets:
            calls = []
            for s in st:
                calls.append(lambda s=s: call_paged(s, args.rope))
                calls.append(lambda s=s: call_ring(s, args.rope))
            graphs.append(DecodeStepGraph(calls, (B, Hq, Hkv, D), dev).capture())
        for i in range(args.warmup):
            graphs[i % n_sets].replay()
        torch.cuda.synchronize()

    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(uuid)
    sampler.start()
    # Region A (value, ms_per_step): K steps back to back, events only at the ends.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        if graphs is not None:
            graphs[i % n_sets].replay()
        else:
            step(sets[i % n_sets])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # Region B (roofline): the same steps, each paged launch bracketed by events on its
    # stream; the bracket also holds the launch gap before the kernel, so this is the
    # conservative per-launch duration.
    ev_p0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_p1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_r1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        s = sets[i % n_sets][0]
        ev_p0[i].record(stream)
        call_paged(s, args.rope)
        ev_p1[i].record(stream)
        call_ring(s, args.rope)
        ev_r1[i].record(stream)
    torch.cuda.synchronize()
    per_config = per_config_fp8 = None
    if args.per_config == "on" or (args.per_config == "auto" and args.q_tokens == 1 and not args.rope
                                   and args.layers == 1):
        per_config = per_config_block(args, dev, l2, measured_hbm_peak()[0], nominal_hbm_peak())
        if args.kv == "bf16":  # the fp8 cache on the two target shapes, the same way
            per_config_fp8 = per_config_block(args, dev, l2, measured_hbm_peak()[0], nominal_hbm_peak(),
                                              workloads=("b64", "long1"), kv="fp8")
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    paged_ms = sum(a.elapsed_time(b) for a, b in zip(ev_p0, ev_p1)) / args.steps
    ms_step = max_over_ranks(total_ms / args.steps, dev)
    assert da.decode_attn_device_status() == 0
    value = whole_job_gbs(pbytes + rbytes, ms_step, world)
    ring_ms = sum(a.elapsed_time(b) for a, b in zip(ev_p1, ev_r1)) / args.steps

    # end to end through the public API with host buffers
    e2e = run_e2e(args, first, pbytes_call + rbytes_call, dev)

    peak, peak_kind = measured_hbm_peak()
    nominal = nominal_hbm_peak()
    achieved = pbytes_call / (paged_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload, ("paged" if args.kv == "bf16" else "paged_fp8")
                               if args.q_tokens == 1 else f"paged_multi{args.q_tokens}")
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if args.kv == "bf16" else "fp8 e4m3 cache, f16 mma, fp32 softmax",
        "data": "synthetic",
        "config": dict(workload_config(args.workload, first),
                       l2=("inputs larger than L2: %.0f MB per step" % (set_bytes / 1e6))
                       if n_sets == 1 else f"rotating {n_sets} input sets, {n_sets * set_bytes / 1e6:.0f} MB > 2x L2"),
        "us_per_call": {"paged_full": round(paged_ms * 1e3, 2), "ring": round(ring_ms * 1e3, 2)},
        "gb_per_s_per_call": {"paged_full": round(achieved, 1),
                              "ring": round(rbytes_call / (ring_ms * 1e-3) / 1e9, 1)},
        "algorithmic_bytes_per_step": {"paged_full": pbytes, "ring": rbytes},
        "layers_per_step": 2 * args.layers, "graph_replay": bool(args.graph),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "traffic": traffic,
                     "kernel": ("decode_attn_kernel (paged, full attention%s)" % (
                         "" if args.kv == "bf16" else ", fp8 cache")) if args.q_tokens == 1 else
                     (("decode_attn_kernel (paged, full attention, %d query tokens, fused append)"
                       % args.q_tokens) if decode_route(args.q_tokens, first.cfg) else
                      "%s + kv_append_multi_kernel (paged, full attention, "
                      "%d query tokens; one bracket around both)" % (
                          # the library runs 64+ query rows per KV head on tcgen05
                          "multi_tc_kernel" if args.q_tokens * first.cfg["Hq"] // first.cfg["Hkv"] >= 64
                          else "multi_attn_kernel", args.q_tokens)),
                     "nominal_peak": round(nominal, 1) if nominal else None,
                     "frac_of_nominal": round(achieved / nominal, 4) if nominal else None},
        "e2e": e2e,
        "gpu_launches": launches_per_step(args.q_tokens, first.cfg, first.block_table.shape[1], args.rope)
                        * args.layers * args.steps,
        "timing": ("value: steps back to back, events at the ends; us_per_call and roofline: "
                   "events around every launch in a second pass (includes the launch gap)"),
        "clocks": clocks,
        "launch": {"early_inputs": args.early_inputs,
                   "note": ("level 1: each attention kernel reads the lengths, block table and "
                            "sinks and works out its split before waiting for the previous "
                            "kernel; level 2: it also starts L2 prefetches of its first cache "
                            "tiles. The step's lengths and tables are written before its "
                            "kernels; the kernel before each call (the other layer) does not "
                            "write them")},
    }
    if per_config is not None:
        result["per_config"] = per_config
        if per_config_fp8 is not None:
            result["per_config_fp8"] = per_config_fp8
        result["per_config_timing"] = (
            "per workload, the paged (full attention) and the ring (window 128) call of the "
            "step, 128 timed calls of each kind: 16 batches of 8 calls of one kind queued back "
            "to back (input sets rotating, > 2x L2), CUDA events around each batch, every batch "
            "queued behind a GPU spin so the host never starves the device; us = the per-call "
            "mean of a batch (median, p10, p90 over the 16 batches); direct = launches through "
            "the public API, graph = the replay of a CUDA graph holding the batch's 8 calls, "
            "direct_wait_first = the direct launches with every input read after the wait for "
            "the previous kernel (decode_attn_set_early_inputs level 0)")
    if world == 1 and not args.no_cpu_baseline:
        v, cores, desc = oracle_sample(args.workload, first, args.cpu_seconds)
        result["cpu_baseline"] = {"value": round(v, 4), "unit": UNIT, "cores": cores,
                                  "kind": "oracle", "sample": desc}
    return result


# ---------------------------------------------------------------- every config, per call
PER_CONFIG = ("b1", "b64", "long1", "long8", "serve")


def quantiles(xs):
    """Median, 10th and 90th percentile (nearest rank) of a list of floats."""
    ys = sorted(xs)
    at = lambda f: ys[min(len(ys) - 1, max(0, int(round(f * (len(ys) - 1)))))]
    return at(0.5), at(0.1), at(0.9)


def timed_batches(n_sets, fn, n_batches, per_batch, gate_cycles):
    """Device µs per call of one kind of call: n_batches batches of per_batch calls queued
    back to back (rotating over n_sets input sets), CUDA events on the current stream around
    each batch, each batch queued behind a timed spin of the GPU (torch.cuda._sleep) so that
    the host's launch rate never starves the device. fn(i, k) launches the k-th call of
    batch i (or, for graphs, the whole batch at k == 0). Returns the per-call mean of every
    batch."""
    import torch
    stream = torch.cuda.current_stream()
    out = []
    for i in range(n_batches):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(gate_cycles)
        e0.record(stream)
        fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3 / per_batch)
    return out


def per_config_block(args, dev, l2, peak, nominal, n_batches=16, per_batch=8, workloads=PER_CONFIG, kv=None):
    """µs per call (median, p10 and p90 over n_batches batches of per_batch calls, each batch
    queued back to back: n_batches * per_batch >= 100 timed calls), algorithmic GB/s and the
    fractions of the measured and nominal HBM peaks for the paged and the ring call of every
    workload, by direct launch and by the replay of a CUDA graph holding one batch. Inputs
    are larger than L2 per call or rotate over sets totalling more than twice L2."""
    import torch
    import paged_decode_attention_kv_gb300 as da
    from paged_decode_attention_kv_gb300.graph import DecodeStepGraph
    gate = int(3e-3 * 2.07e9)  # about 3 ms of spin ahead of each batch
    out = {}
    kv = kv or args.kv
    for name in workloads:
        first = StepInputs(name, dev, kv=kv)
        set_bytes = first.nbytes() + sum(t.numel() * t.element_size() for t in
                                         (first.q, first.k_new, first.v_new, first.out_full, first.out_ring))
        n_sets = 1 if set_bytes >= 2 * l2 else min(64, math.ceil(2 * l2 / set_bytes))
        # calls of one kind back to back: at level 2 no call prefetches the cache that the
        # call just before it is appending to (the sets alternate)
        if args.early_inputs == 2:
            n_sets = max(2, n_sets)
        sets = [first] + [StepInputs(name, dev, seed_offset=k * 10007, kv=kv) for k in range(1, n_sets)]
        c = first.cfg
        shape = (c["B"], c["Hq"], c["Hkv"], c["D"])
        da.decode_attn_reserve(da.decode_attn_workspace_bytes(*shape))
        pb, rb = step_bytes(name, first.lens, kv)
        entry = {"timed_calls": n_batches * per_batch, "input_sets": n_sets,
                 "algorithmic_bytes": {"paged_full": pb, "ring": rb},
                 "max_len": max(first.lens), "active": sum(1 for L in first.lens if L > 0)}
        for kind, nbytes, call in (("paged_full", pb, call_paged), ("ring", rb, call_ring)):
            for k in range(2 * n_sets + 3):  # warm-up, module and attribute set-up before capture
                call(sets[k % n_sets], False)
            torch.cuda.synchronize()

            def direct(i):
                for k in range(per_batch):
                    call(sets[(i * per_batch + k) % n_sets], False)
            # one graph per distinct run of per_batch sets
            n_graphs = n_sets // math.gcd(n_sets, per_batch) if n_sets > 1 else 1
            graphs = [DecodeStepGraph([lambda s=sets[(g * per_batch + k) % n_sets]: call(s, False)
                                       for k in range(per_batch)], shape, dev).capture()
                      for g in range(n_graphs)]
            res = {"direct": timed_batches(n_sets, direct, n_batches, per_batch, gate),
                   "graph": timed_batches(n_sets, lambda i: graphs[i % n_graphs].replay(), n_batches,
                                          per_batch, gate)}
            if args.early_inputs > 0:  # the same direct launches, every read after the wait
                da.decode_attn_set_early_inputs(0)
                res["direct_wait_first"] = timed_batches(n_sets, direct, n_batches, per_batch, gate)
                da.decode_attn_set_early_inputs(args.early_inputs)
            e = {}
            for mode, xs in res.items():
                med, p10, p90 = quantiles(xs)
                gbs = nbytes / (med * 1e-6) / 1e9
                e[mode] = {"us_median": round(med, 2), "us_p10": round(p10, 2), "us_p90": round(p90, 2),
                           "gb_s": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
                           "frac_of_nominal": round(gbs / nominal, 4) if nominal else None}
            entry[kind] = e
            del graphs
        torch.cuda.synchronize()
        status = da.decode_attn_device_status()
        if status != 0:
            raise RuntimeError(f"{name}: device status {status}")
        out[name] = entry
        del sets, first
        torch.cuda.empty_cache()
    return out


def packed(tensors, dev=None, pin=False):
    """One byte buffer holding the given tensors back to back (each at a 256-byte aligned
    offset) and a view of each one into it, so that a step moves them in one copy."""
    import torch
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off += -(-t.numel() * t.element_size() // 256) * 256
    buf = torch.empty(off, dtype=torch.uint8, device=dev)
    if pin:
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def run_e2e(args, s, step_bytes_total, dev):
    """Per step: one H2D copy of q, k_new, v_new, seq_lens, block table and sinks, staged
    back to back in one pinned host buffer (as a serving loop stages a step's inputs); both
    layer calls; one D2H copy of both outputs, which the calls write into one device buffer.
    Wall clock around the whole loop."""
    import torch
    names = ("q", "k_new", "v_new", "seq_lens", "sinks", "block_table")
    src = [getattr(s, k) for k in names]
    host_in, host_views = packed(src, pin=True)
    for v, t in zip(host_views, src):
        v.copy_(t.cpu())
    dev_in, dev_views = packed(src, dev=dev)
    dst = dict(zip(names, dev_views))
    dev_out, (out_full, out_ring) = packed([s.out_full, s.out_ring], dev=dev)
    host_out = torch.empty_like(dev_out, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in src)
    d2h = s.out_full.numel() * s.out_full.element_size() + s.out_ring.numel() * s.out_ring.element_size()
    n = max(3, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        dev_in.copy_(host_in, non_blocking=True)
        call_paged(s, args.rope, dst["q"], dst["k_new"], dst["v_new"], dst["block_table"],
                   dst["seq_lens"], dst["sinks"], out=out_full)
        call_ring(s, args.rope, dst["q"], dst["k_new"], dst["v_new"], dst["seq_lens"], dst["sinks"],
                  out=out_ring)
        host_out.copy_(dev_out, non_blocking=True)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    return {"value": round(step_bytes_total * n / dt / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "us_per_step": round(dt / n * 1e6, 2)}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="b64",
                    choices=["tiny", "b1", "b64", "long1", "long8", "serve"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--layers", type=int, default=1,
                    help="full+ring layer pairs per step, each with its own caches")
    ap.add_argument("--graph", action="store_true",
                    help="capture the whole step once as a CUDA graph and time its replays")
    ap.add_argument("--rope", action="store_true",
                    help="fuse the rotary embedding of position L-1 (q and the new key) into both calls")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="cache storage: bf16, or e4m3 codes with per-token scales (quantised on append)")
    ap.add_argument("--q-tokens", type=int, default=1,
                    help="new tokens per sequence per step (speculative verification / chunked "
                         "prefill): > 1 runs the multi-token calls")
    ap.add_argument("--per-config", default="auto", choices=["auto", "on", "off"],
                    help="time the paged and ring calls of every workload (b1, b64, long1, long8, "
                         "serve) per call; auto: on for one-token steps without --rope")
    ap.add_argument("--early-inputs", type=int, default=2, choices=[0, 1, 2],
                    help="what the attention kernels read before waiting for the previous kernel "
                         "(decode_attn_set_early_inputs): 0 nothing, 1 lengths, block tables and "
                         "sinks, 2 those and L2 prefetches of the first cache tiles. The step's "
                         "lengths and tables are written before its kernels")
    ap.add_argument("--batch-limit", type=int, default=None,
                    help="keep only the first N sequences (smaller cases for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.q_tokens > 1 and (args.kv == "fp8" or args.graph):
        ap.error("--q-tokens > 1 runs the bf16 multi-token calls (with or without --rope), not --kv fp8 or --graph")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")

    if args.impl == "reference":
        result = run_reference(args, rank, world)
    else:
        result = run_ours(args, rank, world, local_rank)
    if rank == 0 and result is not None:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
