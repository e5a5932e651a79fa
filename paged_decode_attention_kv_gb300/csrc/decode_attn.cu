// decode_attn.cu -- fused decode-step attention for GB300 (sm_103a).
//
// One launch per call does the whole step described in the SimpleLLM README,
// changes table, row "one decode-attention kernel for sinks, sliding window,
// GQA and the KV append": it appends the new token's K/V into a paged cache
// (row "paged KV cache for full-attention layers") or a ring buffer (row "ring
// buffer for sliding-window layers"), attends with all query heads of a KV
// head at once (GQA), and folds the per-head sink logit into the softmax
// denominator when the per-split partials are combined.
//
// Work decomposition (graph-capturable, no host read of seq_lens):
//   * unit = one 16-token tile (one page) of one (sequence b, KV head g);
//     units are ordered (b, g, tile), so a "segment" (b, g) is a contiguous
//     run of units. Every CTA recomputes the prefix of units over b from
//     seq_lens in shared memory.
//   * the grid is one CTA per SM (two on large fp8 calls with 8-head groups,
//     whose instruction chains need the extra warps), 8 warps each; every warp is a worker that
//     takes an equal contiguous share of all units (split-KV with perfect
//     balance, whatever the length mix). A warp streams its tiles through a
//     private TMA/mbarrier pipeline and keeps an online-softmax state (running
//     max m, sum l, accumulator acc) per segment in registers.
//   * a segment a warp owns entirely is finished by that warp (sink + 1/den +
//     bf16 store). Segments shared by several warps are merged in shared
//     memory; segments shared by several CTAs leave one fp32 partial per CTA
//     in the workspace, and the last CTA to arrive (atomic ticket, no waiting)
//     combines them with the sink.
//   * the QK^T and PV products of a 16-token tile run on tensor cores
//     (mma.sync m16n8k16 bf16 -> fp32): keys are the M dimension and the G <= 8
//     query heads of the group the N dimension, so nothing is padded; the
//     probabilities are moved from the accumulator layout into the B-operand
//     layout with movmatrix.
//   * K/V tiles (2 KiB each) arrive by TMA with 128-byte swizzle, so the
//     ldmatrix reads are free of bank conflicts.
#include <cuda.h>  // CUtensorMap and its enums (types only; resolved at run time)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <unordered_map>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <type_traits>

#include "decode_attn.h"

namespace {

constexpr int kD = 64;             // head dim
constexpr int kPage = 16;          // tokens per page = per tile
constexpr int kWarps = 8;          // workers per CTA
constexpr int kThreads = kWarps * 32;
// tiles in flight per warp: the deepest pipeline the 227 KiB of shared memory allows
#ifndef DA_STAGES_G8
#define DA_STAGES_G8 5
#endif
#ifndef DA_STAGES_G8_ROPE
#define DA_STAGES_G8_ROPE 4
#endif
#ifndef DA_STAGES_G16
#define DA_STAGES_G16 4
#endif
// several query tokens, 32 rows per KV head in one warp (four 8-row n-tiles): the tiles and
// the 4 KiB of query rows per stage leave room for 3 stages
#ifndef DA_STAGES_MT32
#define DA_STAGES_MT32 3
#endif
// n-tiles up to which a warp holds its query rows' sink logits in registers through the loop
#ifndef DA_SINKS_REGS_MAX_NT
#define DA_SINKS_REGS_MAX_NT 2
#endif
// CPS = CTAs resident per SM (1 or 2). On large calls the fp8 kernel with 8-head groups is
// bound by the latency of its per-warp convert / MMA / softmax chain, not by HBM: two CTAs
// (16 warps, 128 registers each, 3 stages per warp) hide it better than one CTA with 7
// stages. Small calls, whose warps own a few tiles each, are bound by the first tiles'
// arrival and keep the deeper single-CTA pipeline. The host picks CPS per call from an
// upper bound of the call's tiles.
#ifndef DA_STAGES_FP8_2CTA
#define DA_STAGES_FP8_2CTA 3
#endif
#ifndef DA_FP8_2CTA_MIN_TILES
#define DA_FP8_2CTA_MIN_TILES 16384
#endif
constexpr int kMaxCtasPerSm = 2;
constexpr int kMaxSms = 160;  // the one-token grid is one (or two) CTAs per SM, up to this many SMs
template <int NT, bool ROPE, bool KV8, int CPS>
__host__ __device__ constexpr int stages_for() {
    // fp8 tiles are half the size: more of them in flight for the same bytes; with two
    // CTAs per SM each gets half the shared memory
    return KV8 ? (NT == 1 ? (CPS > 1 ? DA_STAGES_FP8_2CTA : 7) : (ROPE ? 5 : 6))
               : (NT == 1 ? (ROPE ? DA_STAGES_G8_ROPE : DA_STAGES_G8) : NT == 2 ? DA_STAGES_G16 : DA_STAGES_MT32);
}
#ifndef DA_PAIR_BF16
#define DA_PAIR_BF16 1
#endif
#ifndef DA_PAIR_FP8
#define DA_PAIR_FP8 1
#endif
// Refills of several tiles issued by several lanes at once (measured: faster for fp8
// blocks, one bulk copy each; slower for bf16 tiles, two tensor copies each)
#ifndef DA_PAR_ISSUE_FP8
#define DA_PAR_ISSUE_FP8 1
#endif
#ifndef DA_PAR_ISSUE_BF16
#define DA_PAR_ISSUE_BF16 0
#endif
#ifndef DA_MULTI_CTAS_PER_SM  // multi-token calls: key splits aim at this many CTAs per SM
#define DA_MULTI_CTAS_PER_SM 4
#endif
// Two-tile passes wholly inside a segment skip the append and the masks (measured: faster for
// the instruction-bound fp8 path, 1% slower for the memory-bound bf16 one)
#ifndef DA_FAST_PASS_FP8
#define DA_FAST_PASS_FP8 1
#endif
#ifndef DA_FAST_PASS_BF16
#define DA_FAST_PASS_BF16 0
#endif
// Lazy softmax maximum (bf16 tiles): a column's reference maximum moves only when a score
// exceeds it by more than 2^kLazyLog2 (one warp vote per n-tile and pass instead of the
// three-round shuffle reduction and the accumulator rescale); the probabilities then stay
// below 2^kLazyLog2, and m, l and O share the reference, so O / l is unchanged
#ifndef DA_LAZY_MAX_MT
#define DA_LAZY_MAX_MT 1
#endif
#ifndef DA_LAZY_MAX_BF16
#define DA_LAZY_MAX_BF16 0
#endif
// fp8 tiles: the probabilities are multiplied by the tokens' V scales and a power of two
// before the fp16 conversion; with the lazy maximum (probabilities below 2^4) that factor is
// 2^4 instead of 2^8, so the largest product stays the same as with exact maxima
#ifndef DA_LAZY_MAX_FP8
#define DA_LAZY_MAX_FP8 1
#endif
constexpr float kLazyLog2 = 8.f, kLazyLog2Fp8 = 4.f;
// Tiles per worker at least: 4, or 2 for a call of at most two tiles per worker of the grid
// (such a call cannot fill the grid anyway; two tiles are one loop pass)
#ifndef DA_MIN_TILES
#define DA_MIN_TILES 4
#endif
#ifndef DA_MIN_TILES_SMALL
#define DA_MIN_TILES_SMALL 2
#endif
// The first kStages copies of a warp issued by several lanes at once
#ifndef DA_PAR_FILL
#define DA_PAR_FILL 0
#endif

constexpr int kMinTilesPerWorker = DA_MIN_TILES;
constexpr int kMinTilesSmall = DA_MIN_TILES_SMALL;
// CTA boundaries move to the nearer edge of a segment of at most this many units (and of at
// most a worker's share), so that short segments are not split between CTAs
#ifndef DA_SNAP_UNITS
#define DA_SNAP_UNITS 32
#endif
constexpr int kSnapUnits = DA_SNAP_UNITS;
constexpr int kTileBytes = kPage * kD * 2;  // 2048 B of K (or V) per tile
// fp8 cache block: 16 tokens of one KV head, K codes [16][64], V codes transposed [64][16],
// K scales [16] and V scales [16] (fp32)
constexpr int kBlk8V = kPage * kD;            // offset of the V^T codes
constexpr int kBlk8S = 2 * kPage * kD;        // offset of the K scales (V scales follow)
constexpr int kBlk8Bytes = kBlk8S + 8 * kPage;  // 2176
constexpr int kMaxBatch = 1024;
constexpr int kMaxSegments = 65536;         // B * Hkv
constexpr int kMaxQHeads = 1024;
constexpr int kMaxNewMT = 4;   // query tokens per sequence of the MT kernel at most
constexpr int kWinfo = 16;     // ints of per-warp bookkeeping in shared memory
constexpr int kCounterBytes = kMaxSegments * 4;
constexpr long long kWaitLimitCycles = 4000000000ll;  // about 2 s of SM clock per tile wait
constexpr int kMaxSmem = 232448;                       // opt-in shared memory per block
constexpr float kLog2e = 1.4426950408889634f;

__device__ unsigned int g_status;  // DA_STATUS_* bits, read and cleared by the host

struct Params {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    __nv_bfloat16 *k_cache;
    __nv_bfloat16 *v_cache;
    const int *block_table;
    const int *seq_lens;
    const float *sinks;
    __nv_bfloat16 *out;
    float *part;     // [gridDim.x][2][slot floats] CTA partials
    int *counters;   // [B*Hkv] arrival tickets, zero at rest
    int B, Hq, Hkv, G, window, max_pages, num_pages, max_seq_len;
    float scale_log2;  // scale * log2(e)
    const float *rope_cos;  // [max_position][D/2] fp32, or null: no rotary embedding
    const float *rope_sin;
    int max_position;
    // several query tokens (the MT kernel): q / out [B][T][Hq][D], k_new / v_new
    // [B][T][Hkv][D]; the n = q_lens[b] (T if null) newest positions are new tokens
    int T;
    const int *q_lens;
    // query-row groups of the MT kernel: CTA c takes rows [16 (c % ngrp), + 16) of every
    // (sequence, KV head) over the units of CTA c / ngrp of a grid of gridDim.x / ngrp (the
    // CTAs of one unit range read the same tiles, all but the first from L2); 1 otherwise
    // (also for 32 rows in one warp's four n-tiles, the default)
    int ngrp;
    // testing aid: worker 0 gives up at its first tile wait from this tile on (after the tile
    // has landed), as if the wait had expired; -1 = never
    int expire_at;
    // 32 query rows (four n-tiles): a warp's saved first-segment state goes here instead of
    // registers, SegState<4> per warp of the grid (lane-interleaved); null otherwise
    float *head_scratch;
    // 1: seq_lens, q_lens, block_table and sinks were final before the previous kernel in the
    // stream started, so the lengths, the split and the first block-table entries are read
    // and worked out before waiting for that kernel (the rest, from the first query row and
    // cache tile on, after the wait); 2: as 1, and the cache rows the call reads were too,
    // so each worker's first cache tiles are also fetched into L2 before the wait (into
    // shared memory after it, with its query rows and new tokens); 0: every input is read
    // after the wait
    int early;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// Wait for phase `parity` of an mbarrier, giving up after kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > kWaitLimitCycles) return false;
    }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// L2 prefetches: no shared memory, no barrier
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void flag_status(unsigned bits) { atomicOr(&g_status, bits); }

// Shared-memory loads by address (of data that is no longer written while they run)
__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds_f32x4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v));
}

// Rotate two element pairs (x1 = elements d, d+1; x2 = elements d+32, d+33) by the
// table angles of d, d+1: x1' = x1 c - x2 s, x2' = x2 c + x1 s, every operation
// rounded to fp32 separately (no fused multiply-add), results rounded to bf16.
__device__ __forceinline__ void rope_pair(uint32_t &x1, uint32_t &x2, const float *c, const float *s) {
    const float2 a = unpack_bf16(x1), b = unpack_bf16(x2);
    const float o1x = __fsub_rn(__fmul_rn(a.x, c[0]), __fmul_rn(b.x, s[0]));
    const float o1y = __fsub_rn(__fmul_rn(a.y, c[1]), __fmul_rn(b.y, s[1]));
    const float o2x = __fadd_rn(__fmul_rn(b.x, c[0]), __fmul_rn(a.x, s[0]));
    const float o2y = __fadd_rn(__fmul_rn(b.y, c[1]), __fmul_rn(a.y, s[1]));
    x1 = pack_bf16(o1x, o1y);
    x2 = pack_bf16(o2x, o2y);
}

// One half of the rotation: `mine` holds elements d, d+1 and `other` their partners
// d +- 32; the first half gets mine*c - other*s, the second half mine*c + other*s.
__device__ __forceinline__ uint32_t rope_half(uint32_t mine, uint32_t other, const float *c, const float *s,
                                              bool first_half) {
    const float2 a = unpack_bf16(mine), b = unpack_bf16(other);
    float ox, oy;
    if (first_half) {
        ox = __fsub_rn(__fmul_rn(a.x, c[0]), __fmul_rn(b.x, s[0]));
        oy = __fsub_rn(__fmul_rn(a.y, c[1]), __fmul_rn(b.y, s[1]));
    } else {
        ox = __fadd_rn(__fmul_rn(a.x, c[0]), __fmul_rn(b.x, s[0]));
        oy = __fadd_rn(__fmul_rn(a.y, c[1]), __fmul_rn(b.y, s[1]));
    }
    return pack_bf16(ox, oy);
}

// ------------------------------------------------------------------ layout helpers
template <bool RING>
__device__ __forceinline__ int tiles_of(int L, int window) {
    if (L <= 0) return 0;
    if (RING) {
        const int n = L < window ? L : window;
        return (n + kPage - 1) / kPage;
    }
    const int lo = (window > 0 && L > window) ? L - window : 0;
    return ((L - 1) / kPage) - (lo / kPage) + 1;
}

// Largest b in [0, B) with pre[b] <= x (pre is non-decreasing, x < pre[B]).
__device__ __forceinline__ int find_seq(const int *pre, int B, int x) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The segment (b Hkv + g) holding unit x and its unit range [first, end).
__device__ __forceinline__ int segment_of_unit(const int *pre, int B, int Hkv, int x, int &first, int &end) {
    const int b = find_seq(pre, B, x);
    const int tiles = (pre[b + 1] - pre[b]) / Hkv;
    const int g = (x - pre[b]) / tiles;
    first = pre[b] + g * tiles;
    end = first + tiles;
    return b * Hkv + g;
}


template <int NT>
struct SegState {
    float acc[NT][4][4];  // O^T fragments: [n-tile][d m-tile][c0..c3]
    float m[NT][2];       // running max (log2 units) of heads 2(lane%4), +1
    float l[NT][2];       // running sum, this lane's token rows only until reduced
};

// A lane's state in global memory, value k of lane l at base[32 k + l] (coalesced per value).
template <int NT>
__device__ __forceinline__ void state_store_lanes(const SegState<NT> &s, float *base, int lane) {
    const float *v = reinterpret_cast<const float *>(&s);
#pragma unroll
    for (int k = 0; k < static_cast<int>(sizeof(SegState<NT>) / 4); ++k) base[32 * k + lane] = v[k];
}

template <int NT>
__device__ __forceinline__ void state_load_lanes(SegState<NT> &s, const float *base, int lane) {
    float *v = reinterpret_cast<float *>(&s);
#pragma unroll
    for (int k = 0; k < static_cast<int>(sizeof(SegState<NT>) / 4); ++k) v[k] = base[32 * k + lane];
}

template <int NT>
__device__ __forceinline__ void state_reset(SegState<NT> &s) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int k = 0; k < 4; ++k) s.acc[n][mt][k] = 0.f;
        s.m[n][0] = s.m[n][1] = -INFINITY;
        s.l[n][0] = s.l[n][1] = 0.f;
    }
}

// Sum the per-lane l over the 8 lanes holding the same heads (token rows).
template <int NT>
__device__ __forceinline__ void state_reduce_l(SegState<NT> &s) {
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float v = s.l[n][j];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            s.l[n][j] = v;
        }
}

template <int NT>
__device__ __forceinline__ void state_scale_acc(SegState<NT> &s, float f) {
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int k = 0; k < 4; ++k) s.acc[n][mt][k] *= f;
}

// Slot in shared memory holding one warp's partial state of a segment.
template <int NT>
struct Slot {
    static constexpr int GP = NT * 8;
    static constexpr int LD = kD + 4;  // padded row: conflict-free fragment stores
    float m[GP];
    float l[GP];
    float acc[GP][LD];
};

template <int NT>
__device__ __forceinline__ void state_to_slot(const SegState<NT> &s, Slot<NT> *slot, int lane) {
    const int r = lane >> 2, c = (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        if (lane < 4) {
            slot->m[n * 8 + c] = s.m[n][0];
            slot->m[n * 8 + c + 1] = s.m[n][1];
            slot->l[n * 8 + c] = s.l[n][0];
            slot->l[n * 8 + c + 1] = s.l[n][1];
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            slot->acc[n * 8 + c][mt * 16 + r] = s.acc[n][mt][0];
            slot->acc[n * 8 + c + 1][mt * 16 + r] = s.acc[n][mt][1];
            slot->acc[n * 8 + c][mt * 16 + r + 8] = s.acc[n][mt][2];
            slot->acc[n * 8 + c + 1][mt * 16 + r + 8] = s.acc[n][mt][3];
        }
    }
}

// Final output of a segment finished by one warp: sink, normalise, bf16, store.
template <int NT>
__device__ __forceinline__ void state_write_out(SegState<NT> &s, const float (&sig)[NT][2],
                                                __nv_bfloat16 *out_bg, int G, int lane) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        float f[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float M = fmaxf(s.m[n][j], sig[n][j]);
            const float a = fast_exp2(s.m[n][j] - M);
            const float den = s.l[n][j] * a + fast_exp2(sig[n][j] - M);
            f[j] = a / den;
        }
        const int head = n * 8 + (lane >> 2);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const uint32_t lo = movmatrix_t(pack_bf16(s.acc[n][mt][0] * f[0], s.acc[n][mt][1] * f[1]));
            const uint32_t hi = movmatrix_t(pack_bf16(s.acc[n][mt][2] * f[0], s.acc[n][mt][3] * f[1]));
            if (head < G) {
                uint32_t *row = reinterpret_cast<uint32_t *>(out_bg + head * kD);
                row[(mt * 16 + (lane & 3) * 2) >> 1] = lo;
                row[(mt * 16 + 8 + (lane & 3) * 2) >> 1] = hi;
            }
        }
    }
}

// The same for several query tokens: column c holds query row r = r0 + c = t G + h of the
// group, which goes to out[b][t][g G + h]; rows t >= n (no query token) are written as zeros.
template <int NT>
__device__ __forceinline__ void state_write_out_mt(SegState<NT> &s, const float (&sig)[NT][2], __nv_bfloat16 *out,
                                                   int b, int g, int T, int G, int Hq, int nq, int r0, int lane) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        float f[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float M = fmaxf(s.m[n][j], sig[n][j]);
            if (M == -INFINITY) {  // a column that saw no key and has no sink (not a query row)
                f[j] = 0.f;
                continue;
            }
            const float a = fast_exp2(s.m[n][j] - M);
            const float den = s.l[n][j] * a + fast_exp2(sig[n][j] - M);
            f[j] = a / den;
        }
        const int r = r0 + n * 8 + (lane >> 2), t = r / G, h = r - t * G;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            uint32_t lo = movmatrix_t(pack_bf16(s.acc[n][mt][0] * f[0], s.acc[n][mt][1] * f[1]));
            uint32_t hi = movmatrix_t(pack_bf16(s.acc[n][mt][2] * f[0], s.acc[n][mt][3] * f[1]));
            if (r < T * G) {
                if (t >= nq) lo = hi = 0u;
                uint32_t *row = reinterpret_cast<uint32_t *>(out + ((static_cast<size_t>(b) * T + t) * Hq + g * G + h) * kD);
                row[(mt * 16 + (lane & 3) * 2) >> 1] = lo;
                row[(mt * 16 + 8 + (lane & 3) * 2) >> 1] = hi;
            }
        }
    }
}

// ---- fp8 (e4m3) helpers
// Four e4m3 codes (bytes 0..3 of w) to two fp16 pairs: bytes 0,1 -> lo, bytes 2,3 -> hi
// (lower byte to the lower half). Exact: every e4m3 value is an fp16 value.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi) : "r"(w));
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    const float2 f = unpack_bf16(v);
    const __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two values to e4m3 codes (nearest, ties to even, saturating at +-448), low byte first.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Token held by row g (< 8) of a 16-token fp8 K tile in the QK product; row g + 8 holds
// that token + 2. The permutation makes the transposed probabilities of each lane
// cover the four consecutive tokens 4t..4t+3 that one 32-bit word of a V^T row holds.
__device__ __forceinline__ int fp8_row_token(int g) { return 4 * (g >> 1) + (g & 1); }

// Shared-memory layout of decode_attn_kernel<NT, ., ROPE, KV8, CPS>: byte offsets from a 1024-byte
// aligned base. The kernel carves its buffers from these offsets and the launch
// requests `bytes`, so the two cannot drift apart.
template <int NT, bool ROPE, bool KV8, int CPS, bool MT = false>
struct SmemLayout {
    static constexpr int kStages = stages_for<NT, ROPE || MT, KV8, CPS>();  // MT: the RoPE build's room
    static constexpr int GP = NT * 8;
    // a stage holds a K and a V tile (bf16: 2 KiB each, kept 1024-byte aligned for the
    // 128-byte swizzle; all K tiles first, then all V tiles) or one fp8 block
    static constexpr int kStageBytes = KV8 ? kBlk8Bytes : 2 * kTileBytes;
    // per stage: the group's q rows, the new token's k and v rows, the rotary cos and sin
    // rows, the fp8 tile's K and V scale rows
    static constexpr int kRopeOff = GP * kD * 2 + 2 * kD * 2;
    // several query tokens: the GP query rows of this CTA's row group (the new tokens' k/v
    // rows go to registers straight from global memory)
    static constexpr int kQBytes = MT ? GP * kD * 2 : kRopeOff + (ROPE ? 2 * (kD / 2) * 4 : 0);
    static constexpr int kWarpTileBytes = kStages * kStageBytes;  // the tiles of one warp
    static constexpr int kInts = (kMaxBatch + 1) + kMaxBatch + 2 * kWarps + kWarps * kWinfo + 16 +
                                 (kMaxCtasPerSm * kMaxSms + 1) + (MT ? kMaxBatch : 0);
    static constexpr size_t qarea = static_cast<size_t>(kWarps) * kWarpTileBytes;
    static constexpr size_t bars = qarea + static_cast<size_t>(kWarps) * kStages * kQBytes;
    static constexpr size_t meta = bars + static_cast<size_t>(kWarps) * kStages * 8;
    static constexpr size_t ints = meta + static_cast<size_t>(kWarps) * kStages * 16;
    static constexpr size_t sinks = ints + static_cast<size_t>(kInts) * 4;
    static constexpr size_t end = sinks + static_cast<size_t>(kMaxQHeads) * 4;
    static constexpr size_t bytes = 1024 + end;  // plus the slack to align the base
    static_assert(KV8 || kWarpTileBytes % 1024 == 0, "bf16 tiles stay 1024-byte aligned");
    static_assert(kWarpTileBytes % 16 == 0 && kStageBytes % 16 == 0, "bulk copies need 16-byte alignment");
    static_assert(kQBytes % 16 == 0 && meta % 16 == 0, "bulk copies and int4 need 16-byte alignment");
    static_assert(bytes <= kMaxSmem, "shared memory budget");
    // every resident CTA also takes 1 KiB of reserved shared memory (228 KiB per SM)
    static_assert(CPS == 1 || CPS * (bytes + 1024) <= 233472, "shared memory budget of the CTAs on one SM");
};

// ------------------------------------------------------------------ the kernel
// MT: several query tokens per sequence (paged, bf16, T <= kMaxNewMT): the query rows of a
// KV head are (token t, head h) pairs r = t G + h, one column of the products each; row t
// sees the positions lo_t .. base + t (base = L - n, lo_t its window start), the n new tokens
// are appended in the same pass, rows t >= n are zero. With more than 16 rows per KV head the
// rows are cut into groups of 16 (p.ngrp), one per CTA of a pair that covers the same units.
template <int NT, bool RING, bool ROPE, bool KV8, int CPS, bool MT = false>
__global__ void __launch_bounds__(kThreads, CPS)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const Params p) {
    static_assert(!MT || (!RING && !ROPE && !KV8 && CPS == 1), "several query tokens: paged bf16 only");
    using Lay = SmemLayout<NT, ROPE, KV8, CPS, MT>;
    constexpr int kTileB = KV8 ? kBlk8V : kTileBytes;  // bytes of one K (or V) tile
    constexpr int kStages = Lay::kStages;
    constexpr int GP = Lay::GP;
    constexpr int kQBytes = Lay::kQBytes;
    constexpr int kWarpBytes = Lay::kWarpTileBytes;
    // a warp's two merge slots (head and tail states) go to its drained tile area, or, when
    // they do not both fit there (32 rows), the tail slot to its drained query-row area
    constexpr bool kSlotsInTiles = 2 * sizeof(Slot<NT>) <= kWarpBytes;
    static_assert(kSlotsInTiles || (sizeof(Slot<NT>) <= kWarpBytes && sizeof(Slot<NT>) <= kStages * kQBytes),
                  "merge slots must fit a drained warp area");
    constexpr int kSlotFloats = 2 * GP + GP * kD;  // global partial: m, l, acc
    // two tiles per loop pass (single 8-head n-tile only: the registers of two 16-head passes
    // would not fit)
    constexpr bool kPair = NT == 1 && (KV8 ? DA_PAIR_FP8 : DA_PAIR_BF16);
    constexpr bool kLazy = KV8 ? DA_LAZY_MAX_FP8 : (MT ? DA_LAZY_MAX_MT : DA_LAZY_MAX_BF16);
    constexpr float kLazyT = KV8 ? kLazyLog2Fp8 : kLazyLog2;  // log2 of the largest probability
    // fp8: the power of two the V scales carry (taken out when a segment closes)
    constexpr float kV8Factor = kLazy ? 16.f : 256.f;
    constexpr bool kParIssue = KV8 ? DA_PAR_ISSUE_FP8 : DA_PAR_ISSUE_BF16;

    extern __shared__ uint8_t smem_raw[];
    // the 1024-byte aligned base, derived from the shared array itself so that every access
    // through it compiles to a shared-memory instruction (not a generic one)
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    // the unit split runs over ncta CTAs; this CTA is number cta of row group rgrp, whose
    // columns are the query rows r0g .. r0g + GP - 1 of each (sequence, KV head)
    const int ngrp = MT ? p.ngrp : 1;
    const int rgrp = MT ? static_cast<int>(blockIdx.x) % ngrp : 0;
    const int cta = MT ? static_cast<int>(blockIdx.x) / ngrp : static_cast<int>(blockIdx.x);
    const int ncta = MT ? static_cast<int>(gridDim.x) / ngrp : static_cast<int>(gridDim.x);
    const int r0g = rgrp * GP;
    uint8_t *qarea = smem + Lay::qarea;  // [kWarps][kStages] q / k_new / v_new / cos / sin slots
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::bars);
    int4 *meta = reinterpret_cast<int4 *>(smem + Lay::meta);
    int *s_pre = reinterpret_cast<int *>(smem + Lay::ints);  // [B + 1]
    int *s_len = s_pre + (kMaxBatch + 1);                             // [B]
    int *s_wsum = s_len + kMaxBatch;                                  // [kWarps]
    int *s_wmin = s_wsum + kWarps;                                    // [kWarps]
    int *s_winfo = s_wmin + kWarps;                                   // [kWarps][kWinfo]
    int *s_flag = s_winfo + kWarps * kWinfo;                          // [16]
    int *s_bnd = s_flag + 16;                                         // [CTAs + 1] CTA boundaries
    int *s_n = s_bnd + kMaxCtasPerSm * kMaxSms + 1;                   // [B] new tokens (MT)
    float *s_sink = reinterpret_cast<float *>(smem + Lay::sinks);     // [Hq], log2 units

    // Set-up that reads no input: it overlaps the previous kernel in the stream when this
    // grid is launched as a programmatic dependent.
    if (!KV8 && tid == 0) {  // fp8 blocks are plain bulk copies: no tensor maps
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    const uint32_t bar0 = smem_addr(bars + warp * kStages);
    if (lane == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(bar0 + 8 * st, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < 4) s_flag[tid] = -1;  // [0,1] segments this CTA combines; [2,3] its boundary segments
    // Inputs may come from the previous kernel: wait for it before the first read of one it
    // may have written (at once, or after the split when the step's lengths and tables were
    // final before it started). With an early level the next kernel may start its own set-up
    // as soon as this grid has waited (its early reads then overlap this call); at level 0
    // it is let start only when this grid's loops are done (measured: about 4 µs less per
    // alternating full / window step than letting it start at once).
    const bool early = p.early != 0;
    auto wait_previous = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (tid == 0 && early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    };
    if (!early) wait_previous();

    const int B = p.B, Hkv = p.Hkv;

    // ---- 1. lengths, validation, prefix of units over sequences
    {
        for (int h = tid; h < p.Hq; h += kThreads)
            s_sink[h] = p.sinks != nullptr ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
        int v[4], tsum = 0, tmin = 0x7fffffff;  // (tmin: the fewest units of a segment)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b = tid * 4 + k;
            int L = 0, nq = 1;
            if (b < B) {
                L = __ldg(p.seq_lens + b);
                bool bad = L < 0;
                if (!RING) bad = bad || L > p.max_seq_len || L > p.max_pages * kPage;
                if constexpr (MT) {
                    nq = p.q_lens != nullptr ? __ldg(p.q_lens + b) : p.T;
                    bad = bad || nq < 0 || nq > p.T || (L > 0 && nq > L);
                }
                if (bad) {
                    if (blockIdx.x == 0) flag_status(DA_STATUS_BAD_SEQ_LEN);
                    L = 0;
                }
                if (MT && nq == 0) L = 0;  // no query row: an inactive slot
                s_len[b] = L;
                if constexpr (MT) s_n[b] = nq;
            }
            if constexpr (MT) {  // positions lo_0 .. L - 1, lo_0 the first query token's window start
                const int lo0 = (p.window > 0 && L > 0) ? max(0, L - nq - p.window + 1) : 0;
                v[k] = (L > 0 ? (L - 1) / kPage - lo0 / kPage + 1 : 0) * Hkv;
            } else {
                v[k] = tiles_of<RING>(L, p.window) * Hkv;
            }
            tsum += v[k];
            if (v[k] > 0) tmin = min(tmin, v[k] / Hkv);
        }
        int incl = tsum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
            tmin = min(tmin, __shfl_xor_sync(0xffffffffu, tmin, off));
        }
        if (lane == 31) {
            s_wsum[warp] = incl;
            s_wmin[warp] = tmin;
        }
        __syncthreads();
        int woff = 0;
        for (int w = 0; w < warp; ++w) woff += s_wsum[w];
        int run = woff + incl - tsum;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b = tid * 4 + k;
            if (b < B) s_pre[b] = run;
            run += v[k];
        }
        if (tid == kThreads - 1) s_pre[B] = run;  // total (all later b are beyond B)
        __syncthreads();
    }
    const int U = s_pre[B];

    // ---- 2. inactive slots get a zero output (after the wait: the previous kernel may still
    // use the output buffer)
    auto zero_inactive = [&]() {
        for (int b = blockIdx.x; b < B; b += gridDim.x) {
            if (s_len[b] != 0) continue;
            const int rows_b = MT ? p.T : 1;  // query tokens per slot
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + static_cast<size_t>(b) * rows_b * p.Hq * kD);
            const int n16 = rows_b * p.Hq * kD * 2 / 16;
            for (int i = tid; i < n16; i += kThreads) dst[i] = make_uint4(0, 0, 0, 0);
        }
    };
    if (U == 0) {
        if (early) wait_previous();
        zero_inactive();
        return;
    }

    // ---- 3. workers and their unit ranges
    // (whole CTAs of workers once there are eight or more: every CTA then holds 8 shares)
    const int min_tiles = U <= 2 * ncta * kWarps ? kMinTilesSmall : kMinTilesPerWorker;
    long long nwork = min(static_cast<long long>(ncta) * kWarps, static_cast<long long>((U + min_tiles - 1) / min_tiles));
    if (nwork >= kWarps) nwork -= nwork % kWarps;
    if (static_cast<long long>(cta) * kWarps >= nwork) {  // whole CTA idle
        if (early) wait_previous();
        zero_inactive();
        return;
    }
    const long long wid = static_cast<long long>(cta) * kWarps + warp;
    // Two levels. CTA c takes the units from cta_start(c): worker c kWarps's start in an even
    // split over all nwork workers, floor(w U / nwork) = w q + floor(w r / nwork) with
    // U = q nwork + r (32-bit: w r < nwork^2 < 2^23), moved to the nearer edge of the segment
    // it falls in when that segment is at most four workers' shares (and kSnapUnits) long: a
    // segment that short is then never shared between CTAs, which would cost it a partial, a
    // ticket and a combine (more than the few tiles of imbalance). The CTA's warps split its
    // range evenly.
    const int nw32 = static_cast<int>(nwork);
    const int q_nw = U / nw32, r_nw = U - q_nw * nw32;
    auto wst = [&](int w) { return w * q_nw + (w * r_nw) / nw32; };
    // a boundary moves by at most snap_max / 2 <= 2 q, and a CTA holds 8 shares of q (or is
    // the only one): every CTA keeps units
    const int snap_max = min(kSnapUnits, 4 * q_nw);
    const int n_cta = (nw32 + kWarps - 1) / kWarps;  // CTAs with work
    int min_seg = s_wmin[0];  // the shortest segment of the call, in units
#pragma unroll
    for (int w = 1; w < kWarps; ++w) min_seg = min(min_seg, s_wmin[w]);
    const bool snapping = min_seg <= snap_max;  // (else no boundary can move)
    if (snapping) {  // every CTA boundary of the call, one lookup per thread, into shared memory
        for (int c = tid; c <= n_cta; c += kThreads) {
            int x = wst(min(c * kWarps, nw32));
            if (x > 0 && x < U) {
                int f, e;
                segment_of_unit(s_pre, B, Hkv, x, f, e);
                if (x != f && e - f <= snap_max) x = (x - f <= e - x) ? f : e;
            }
            s_bnd[c] = x;
        }
        __syncthreads();
    }
    auto cta_start = [&](int c) { return snapping ? s_bnd[c] : wst(min(c * kWarps, nw32)); };
    const int nw_cta = min(kWarps, nw32 - cta * kWarps);  // active warps of this CTA
    const bool active = warp < nw_cta;
    const int R0 = cta_start(cta), R1 = cta_start(cta + 1);  // this CTA's units
    const int q_w = (R1 - R0) / nw_cta, r_w = (R1 - R0) - q_w * nw_cta;
    const int ua = active ? R0 + warp * q_w + (warp * r_w) / nw_cta : 0;
    const int ue = active ? R0 + (warp + 1) * q_w + ((warp + 1) * r_w) / nw_cta : 0;
    const int n_tiles = ue - ua;

    // The warp's merge plan, fixed by the split alone: its head segment (the first one, when
    // it started before ua) and tail segment (the last one, when it goes on after ue; a single
    // segment that crosses either edge counts as the tail), their unit ranges, and for each
    // the warps of this CTA holding it (wa and their count: the warps whose ranges meet it,
    // found by all lanes at once), in the warp's row of s_winfo: [2] head, [3] tail, [5..8]
    // their ranges, [12..15] wa and count of each. Worked out before the loop (before the
    // wait for the previous kernel at early levels), so the merges start at once.
    if (active) {
        int f = 0, e = 0, sg = -1;
        if (lane < 2) sg = segment_of_unit(s_pre, B, Hkv, lane == 0 ? ua : ue - 1, f, e);
        const int sF = __shfl_sync(0xffffffffu, sg, 0), fF = __shfl_sync(0xffffffffu, f, 0),
                  eF = __shfl_sync(0xffffffffu, e, 0);
        const int sL = __shfl_sync(0xffffffffu, sg, 1), fL = __shfl_sync(0xffffffffu, f, 1),
                  eL = __shfl_sync(0xffffffffu, e, 1);
        int hs = -1, ts = -1;
        if (sF == sL) {
            if (fF < ua || eL > ue) ts = sL;
        } else {
            if (fF < ua) hs = sF;
            if (eL > ue) ts = sL;
        }
        // lane w < nw_cta: warp w's range [st, st1)
        const int st0 = lane <= nw_cta ? R0 + lane * q_w + (lane * r_w) / nw_cta : R1;
        const int st1 = __shfl_down_sync(0xffffffffu, st0, 1);
        const uint32_t mh = __ballot_sync(0xffffffffu, lane < nw_cta && st0 < eF && st1 > fF);
        const uint32_t mt = __ballot_sync(0xffffffffu, lane < nw_cta && st0 < eL && st1 > fL);
        if (lane == 0) {
            int *wi = s_winfo + warp * kWinfo;
            wi[0] = ua; wi[1] = ue; wi[2] = hs; wi[3] = ts; wi[4] = 1;
            wi[5] = fF; wi[6] = eF; wi[7] = fL; wi[8] = eL;
            wi[12] = __ffs(static_cast<int>(mh)) - 1; wi[13] = __popc(mh);
            wi[14] = __ffs(static_cast<int>(mt)) - 1; wi[15] = __popc(mt);
        }
    }

    uint8_t *wbase = smem + warp * kWarpBytes;
    const uint32_t wbase_s = smem_addr(wbase);
    // offsets of a stage's K tile, V tile and (fp8) scale rows in the warp's area
    auto k_off = [&](int st) { return KV8 ? st * kBlk8Bytes : st * kTileB; };
    auto v_off = [&](int st) { return KV8 ? st * kBlk8Bytes + kBlk8V : (kStages + st) * kTileB; };
    auto s_off = [&](int st) { return st * kBlk8Bytes + kBlk8S; };
    auto k_tile = [&](int st) { return wbase_s + k_off(st); };
    auto v_tile = [&](int st) { return wbase_s + v_off(st); };
    uint8_t *wq = qarea + warp * kStages * kQBytes;
    const uint32_t wq_s = smem_addr(wq);
    auto q_tile = [&](int st) { return wq_s + st * kQBytes; };
    int4 *wmeta = meta + warp * kStages;

    // per-lane ldmatrix offsets inside a swizzled 16 x 128 B tile
    const int lj = lane & 7, lmi = lane >> 3;
    const uint32_t k_row = ((lj + ((lmi & 1) << 3)) * 128);
    const int k_cb = lmi >> 1;
    const uint32_t v_row = ((lj + ((lmi >> 1) << 3)) * 128);
    const int v_cb = lmi & 1;

    SegState<NT> st;       // running state of the current segment
    SegState<NT> head;     // saved state of the warp's first segment when shared
    // (32 query rows: saved to global memory instead, the registers are needed in the loop)
    constexpr bool kHeadInRegs = NT < 4;
    float *const head_mem = kHeadInRegs ? nullptr
                            : p.head_scratch + (static_cast<size_t>(blockIdx.x) * kWarps + warp) * (sizeof(SegState<NT>) / 4) * 32;
    // sink logits (log2 units) of this lane's query rows: held through the loop for up to
    // DA_SINKS_REGS_MAX_NT n-tiles, read from shared memory when a segment's output is
    // written for more (their registers are needed for the n-tiles)
    constexpr bool kSinksInRegs = NT <= DA_SINKS_REGS_MAX_NT;
    float sig_r[NT][2];
    uint32_t qf[NT][4][2]; // Q as mma B operand
    int head_seg = -1, tail_seg = -1;
    bool failed = false;
    bool slots_ok = true;  // false after an expired wait: this warp's area is never read or written again

    // The segments this CTA shares with other CTAs, from the unit prefix alone (so the tickets
    // never depend on what the warps publish): the one holding its first unit (partial slot
    // 0) and the one holding its last unit (slot 1), and for each the contributing CTAs
    // (first, count) and the slot of the first one: s_flag[2..7] and s_flag[8 + 3k ..]. The
    // last warp works them out once the split is known, off the merge's path (before the
    // wait for the previous kernel when the split is worked out early); lanes 0 and 1 find
    // the two segments, lanes 0..3 the CTAs holding their first and last units, at once.
    auto find_boundary_segments = [&]() {
        int f = 0, e = 0, sg = -1;
        if (lane < 2) sg = segment_of_unit(s_pre, B, Hkv, lane == 0 ? R0 : R1 - 1, f, e);
        const int sa = __shfl_sync(0xffffffffu, sg, 0), fa = __shfl_sync(0xffffffffu, f, 0),
                  ea = __shfl_sync(0xffffffffu, e, 0);
        const int sz = __shfl_sync(0xffffffffu, sg, 1), fz = __shfl_sync(0xffffffffu, f, 1),
                  ez = __shfl_sync(0xffffffffu, e, 1);
        const bool sh0 = fa < R0 || ea > R1;   // the first unit's segment crosses a CTA edge
        const bool sh1 = sz != sa && ez > R1;  // the last unit's, when another one
        int c = 0, cs = 0;  // lane j < 4: segment j / 2, its first (j even) or last unit
        if (lane < 4 && ((lane >> 1) == 0 ? sh0 : sh1)) {
            const int x = (lane >> 1) == 0 ? ((lane & 1) ? ea - 1 : fa) : ((lane & 1) ? ez - 1 : fz);
            // the CTA whose range holds unit x: start from an estimate
            c = min(n_cta - 1, static_cast<int>(static_cast<float>(x) * (static_cast<float>(n_cta) / U)));
            while (c > 0 && cta_start(c) > x) --c;
            while (c + 1 < n_cta && cta_start(c + 1) <= x) ++c;
            cs = cta_start(c);
        }
        int cc[4], ccs[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            cc[j] = __shfl_sync(0xffffffffu, c, j);
            ccs[j] = __shfl_sync(0xffffffffu, cs, j);
        }
        if (lane == 0) {
            auto shared_seg = [&](int k, int seg, int s0, int s1) {
                s_flag[2 + k] = seg;
                s_flag[4 + 2 * k] = s0;
                s_flag[5 + 2 * k] = s1;
                s_flag[8 + 3 * k] = cc[2 * k];
                s_flag[9 + 3 * k] = cc[2 * k + 1] - cc[2 * k] + 1;
                // the first contributing CTA may have started before this segment (its slot 1)
                s_flag[10 + 3 * k] = ccs[2 * k] < s0 ? 1 : 0;
            };
            if (sh0) shared_seg(0, sa, fa, ea);
            if (sh1) shared_seg(1, sz, fz, ez);
        }
    };
    if (!active && warp == kWarps - 1) find_boundary_segments();
    if (early && !active) wait_previous();
    if (active) {
        __syncwarp();
        const uint64_t policy = evict_first_policy();

        // address batches: lane l describes unit ua + 32*k + l
        int cb = 0, cg = 0, ct = 0, cp = 0, nb = 0, ng = 0, ntl = 0, np = 0;
        auto load_batch = [&](int k, int &ob, int &og, int &ot, int &op) {
            const int x = ua + 32 * k + lane;
            ob = og = ot = op = 0;
            if (x < ue) {
                const int b = find_seq(s_pre, B, x);
                const int tiles = (s_pre[b + 1] - s_pre[b]) / Hkv;
                const int r = x - s_pre[b];
                ob = b;
                og = r / tiles;
                ot = r - og * tiles;
                if (!RING) {
                    const int L = s_len[b];
                    const int lo = MT ? ((p.window > 0) ? max(0, L - s_n[b] - p.window + 1) : 0)
                                      : ((p.window > 0 && L > p.window) ? L - p.window : 0);
                    op = __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + lo / kPage + ot);
                }
            }
        };
        load_batch(0, cb, cg, ct, cp);
        if (n_tiles > 32) load_batch(1, nb, ng, ntl, np);
        int cur_batch = 0;

        // Copies of tiles j0 .. j0 + cnt - 1 (cnt <= kStages, calls in increasing order): lane u
        // issues tile j0 + u into stage (stg0 + u) mod kStages, so several tiles go out at once.
        // prefetch_only: the cache tiles into L2, nothing else (no stage, barrier or status)
        auto issue_n = [&](int j0, int cnt, int stg0, bool prefetch_only = false) {
            if ((j0 >> 5) != cur_batch) {  // advance to the next batch, prefetch the one after
                cb = nb; cg = ng; ct = ntl; cp = np;
                ++cur_batch;
                if (n_tiles > 32 * (cur_batch + 1)) load_batch(cur_batch + 1, nb, ng, ntl, np);
            }
            const int j = j0 + (lane < cnt ? lane : 0);
            const int src = j & 31;
            int tb = __shfl_sync(0xffffffffu, cb, src);
            int tg = __shfl_sync(0xffffffffu, cg, src);
            int tt = __shfl_sync(0xffffffffu, ct, src);
            int tp = __shfl_sync(0xffffffffu, cp, src);
            const bool nxt = (j >> 5) != cur_batch;  // this lane's tile is in the prefetched batch
            if (__any_sync(0xffffffffu, nxt)) {
                const int b2 = __shfl_sync(0xffffffffu, nb, src);
                const int g2 = __shfl_sync(0xffffffffu, ng, src);
                const int t2 = __shfl_sync(0xffffffffu, ntl, src);
                const int p2 = __shfl_sync(0xffffffffu, np, src);
                if (nxt) { tb = b2; tg = g2; tt = t2; tp = p2; }
            }
            if (prefetch_only) {
                if constexpr (RING) {
                    // a (sequence, KV head) window is contiguous: one prefetch per run of the
                    // lanes' tiles in one window (the run starts where the previous lane's
                    // tile is not the one just before)
                    const int pb = __shfl_up_sync(0xffffffffu, tb, 1), pg = __shfl_up_sync(0xffffffffu, tg, 1),
                              pt = __shfl_up_sync(0xffffffffu, tt, 1);
                    const bool start = lane < cnt && (lane == 0 || pb != tb || pg != tg || pt + 1 != tt);
                    const uint32_t starts = __ballot_sync(0xffffffffu, start);
                    if (start) {
                        const uint32_t later = starts & ~((2u << lane) - 1u);
                        const int len = (later ? __ffs(static_cast<int>(later)) - 1 : cnt) - lane;
                        const size_t slice = static_cast<size_t>(tb) * Hkv + tg;
                        if constexpr (KV8) {
                            const size_t blk = slice * (p.window / kPage) + tt;
                            bulk_prefetch_l2(reinterpret_cast<const uint8_t *>(p.k_cache) + blk * kBlk8Bytes,
                                             static_cast<uint32_t>(len) * kBlk8Bytes);
                        } else {  // rows tt 16 .. up to the window's end, 128 bytes each
                            const int r0 = tt * kPage, r1 = min((tt + len) * kPage, p.window);
                            const size_t off = (slice * p.window + r0) * (kD * 2);
                            bulk_prefetch_l2(reinterpret_cast<const uint8_t *>(p.k_cache) + off, (r1 - r0) * kD * 2);
                            bulk_prefetch_l2(reinterpret_cast<const uint8_t *>(p.v_cache) + off, (r1 - r0) * kD * 2);
                        }
                    }
                } else if (lane < cnt && tp >= 0 && tp < p.num_pages) {
                    if constexpr (KV8) {
                        const size_t blk = static_cast<size_t>(tp) * Hkv + tg;
                        bulk_prefetch_l2(reinterpret_cast<const uint8_t *>(p.k_cache) + blk * kBlk8Bytes, kBlk8Bytes);
                    } else {
                        tma_prefetch_3d(&tmk, 0, 0, tp * Hkv + tg);
                        tma_prefetch_3d(&tmv, 0, 0, tp * Hkv + tg);
                    }
                }
            } else if (lane < cnt) {
                const int stg = stg0 + lane < kStages ? stg0 + lane : stg0 + lane - kStages;
                if (!RING && (tp < 0 || tp >= p.num_pages)) {
                    flag_status(DA_STATUS_BAD_PAGE);
                    tp = -1;  // TMA reads zeros out of bounds
                }
                const bool newseg = (j == 0) || (tt == 0);
                const uint32_t bar = bar0 + 8 * stg;
                const bool rows = !MT && newseg && p.k_new != nullptr;
                const bool rope = ROPE && newseg;
                // query rows this CTA stages: its row group's share of the T G (MT), or G
                const int qrows = MT ? min(GP, max(0, p.T * p.G - r0g)) : p.G;
                wmeta[stg] = make_int4(tb, tg, tt, tp);
                mbar_expect_tx(bar, Lay::kStageBytes + (newseg ? qrows * kD * 2 : 0) + (rows ? 4 * kD : 0) +
                                        (rope ? 4 * kD : 0));
                // a new segment's rows first: with several tiles issued at once, a stage's
                // barrier then does not wait for them behind every tile's copies
                if (newseg) {
                    if constexpr (MT) {  // rows r0g .. r0g + qrows - 1: for each token t the heads of
                                         // group tg whose row t G + h falls in that range
                        for (int t = r0g / p.G; t < p.T && t * p.G < r0g + qrows; ++t) {
                            const int h0 = max(0, r0g - t * p.G), h1 = min(p.G, r0g + qrows - t * p.G);
                            bulk_load(q_tile(stg) + (t * p.G + h0 - r0g) * kD * 2,
                                      p.q + ((static_cast<size_t>(tb) * p.T + t) * p.Hq + static_cast<size_t>(tg) * p.G + h0) * kD,
                                      (h1 - h0) * kD * 2, bar);
                        }
                    } else {
                        bulk_load(q_tile(stg),
                                  p.q + (static_cast<size_t>(tb) * p.Hq + static_cast<size_t>(tg) * p.G) * kD,
                                  p.G * kD * 2, bar);
                    }
                }
                if (rows) {
                    const size_t off = (static_cast<size_t>(tb) * Hkv + tg) * kD;
                    bulk_load(q_tile(stg) + GP * kD * 2, p.k_new + off, kD * 2, bar);
                    bulk_load(q_tile(stg) + GP * kD * 2 + kD * 2, p.v_new + off, kD * 2, bar);
                }
                if (rope) {  // cos/sin rows of the new token's position
                    int pos = s_len[tb] - 1;
                    if (pos >= p.max_position) {
                        flag_status(DA_STATUS_BAD_POSITION);
                        pos = 0;
                    }
                    const size_t row = static_cast<size_t>(pos) * (kD / 2);
                    bulk_load(q_tile(stg) + GP * kD * 2 + 4 * kD, p.rope_cos + row, kD * 2, bar);
                    bulk_load(q_tile(stg) + GP * kD * 2 + 6 * kD, p.rope_sin + row, kD * 2, bar);
                }
                if constexpr (KV8) {  // the whole block in one copy (a bad page reads block 0)
                    const size_t blk = RING ? (static_cast<size_t>(tb) * Hkv + tg) * (p.window / kPage) + tt
                                            : static_cast<size_t>(tp < 0 ? 0 : tp) * Hkv + tg;
                    bulk_load_hint(k_tile(stg), reinterpret_cast<const uint8_t *>(p.k_cache) + blk * kBlk8Bytes,
                                   kBlk8Bytes, bar, policy);
                } else {
                    int c1, c2;
                    if (RING) { c1 = tt * kPage; c2 = tb * Hkv + tg; }
                    else { c1 = 0; c2 = tp * Hkv + tg; }
                    tma_load_3d(k_tile(stg), &tmk, 0, c1, c2, bar, policy);
                    tma_load_3d(v_tile(stg), &tmv, 0, c1, c2, bar, policy);
                }
            }
        };

        // the first copies of every stage (with early == 2, for a warp with more tiles than
        // stages, their cache tiles are first fetched into L2 before the wait for the previous
        // kernel); one copy of this code serves every level (the short calls are sensitive to
        // the kernel's instruction footprint)
        auto first_copies = [&]() {
            if (kParIssue || DA_PAR_FILL) {
                issue_n(0, n_tiles < kStages ? n_tiles : kStages, 0);
            } else {
                for (int j = 0; j < n_tiles && j < kStages; ++j) issue_n(j, 1, j);
            }
        };
        if (p.early == 2 && n_tiles > kStages) issue_n(0, kStages, 0, true);
        if (early) {
            if (warp == kWarps - 1) find_boundary_segments();
            wait_previous();  // query rows, new tokens and cache tiles from here on
        }
        first_copies();
        if (!early && warp == kWarps - 1) find_boundary_segments();  // while the first tiles land

        // segment context
        int sb = -1, sgk = -1;  // current segment (b, g)
        int seg_first_unit = 0, seg_end_unit = 0;
        int L = 0, lo = 0, ft = 0, nvalid = 0, app_tile = -1, app_row = 0;
        // several query tokens: the segment's new-token count and first new position, the
        // tightest bounds over its rows (tiles inside [lo_max, hi_min) need no mask), the new
        // tokens' k/v (bf16 pairs of this lane), and this lane's columns' ranges [lo_c, hi_c)
        int nq_seg = 1, base = 0, lo_max = 0, hi_min = 0;
        constexpr bool kNewInRegs = NT < 4;
        uint32_t knewm[kMaxNewMT], vnewm[kMaxNewMT];
#pragma unroll
        for (int i2 = 0; i2 < kMaxNewMT; ++i2) knewm[i2] = vnewm[i2] = 0u;
        uint32_t knew = 0, vnew = 0;           // new token's k/v (bf16 pair, or 2 e4m3 codes)
        float knew_scale = 1.f, vnew_scale = 1.f;  // fp8: their scales
        const bool do_append = p.k_new != nullptr;

        // sink logits (log2 units) of this lane's query rows in the current segment
        auto sinks_of = [&](float (&sg)[NT][2]) {
            const int qrows = MT ? p.T * p.G : p.G;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int hs = r0g + n * 8 + (lane & 3) * 2 + j;
                    sg[n][j] = kSinksInRegs ? sig_r[n][j]
                                            : hs < qrows ? s_sink[sgk * p.G + (MT ? hs % p.G : hs)] : -INFINITY;
                }
        };

        int i = 0;  // first tile of the current pass
        // One pass over UT (1 or 2) consecutive tiles i .. i + UT - 1 of the current segment.
        // Two tiles give each warp two independent load / convert / MMA chains and one
        // online-softmax update per 32 tokens.
        // FAST: every tile of the pass is whole inside the attended range and none holds the
        // new token, so the append and all key-validity work are left out
        auto tiles_step = [&](auto ut_c, auto fast_c, int st0, int st1) {
            constexpr int UT = decltype(ut_c)::value;
            constexpr bool FAST = decltype(fast_c)::value;
            int stgs[UT], tts[UT], tps[UT];
#pragma unroll
            for (int u = 0; u < UT; ++u) {
                stgs[u] = u == 0 ? st0 : st1;
                if constexpr (!FAST) {
                    const int4 m = wmeta[stgs[u]];
                    tts[u] = m.z;
                    tps[u] = m.w;
                } else {
                    tts[u] = tps[u] = 0;
                }
            }
#pragma unroll
            for (int u = 0; u < UT && !FAST; ++u) {
                const int stg = stgs[u], tt = tts[u], tp = tps[u];
                uint8_t *gK = wbase + k_off(stg);
                uint8_t *gV = wbase + v_off(stg);
                if constexpr (MT) {  // fused append of the new tokens this tile holds (into the
                                     // cache by row group 0 only; every group patches its copy)
                    bool any = false;
#pragma unroll
                    for (int i2 = 0; i2 < kMaxNewMT; ++i2) {
                        const int pos = base + i2;
                        if (i2 < nq_seg && pos / kPage - ft == tt) {
                            const int row = pos % kPage;
                            const uint32_t off = row * 128 + ((((lane >> 2) ^ (row & 7))) << 4) + (lane & 3) * 4;
                            uint32_t kn, vn;
                            if constexpr (kNewInRegs) {
                                kn = knewm[i2];
                                vn = vnewm[i2];
                            } else {
                                const size_t o = ((static_cast<size_t>(sb) * p.T + i2) * Hkv + sgk) * kD;
                                kn = __ldg(reinterpret_cast<const uint32_t *>(p.k_new + o) + lane);
                                vn = __ldg(reinterpret_cast<const uint32_t *>(p.v_new + o) + lane);
                            }
                            *reinterpret_cast<uint32_t *>(gK + off) = kn;
                            *reinterpret_cast<uint32_t *>(gV + off) = vn;
                            if (tp >= 0 && rgrp == 0) {
                                const size_t c = (static_cast<size_t>(tp) * Hkv + sgk) * kPage + row;
                                reinterpret_cast<uint32_t *>(p.k_cache + c * kD)[lane] = kn;
                                reinterpret_cast<uint32_t *>(p.v_cache + c * kD)[lane] = vn;
                            }
                            any = true;
                        }
                    }
                    if (any) __syncwarp();
                }
                // fused append: this tile holds position p = L - 1
                if (!MT && do_append && tt == app_tile) {
                    size_t slice, cell;  // (KV head) slice of the cache and the token's cell in it
                    bool ok = true;
                    if (RING) {
                        slice = static_cast<size_t>(sb) * Hkv + sgk;
                        cell = tt * kPage + app_row;
                    } else {
                        ok = tp >= 0;
                        slice = static_cast<size_t>(tp < 0 ? 0 : tp) * Hkv + sgk;
                        cell = app_row;
                    }
                    if constexpr (KV8) {
                        // K row of codes, one column of the transposed V tile and both scales, in
                        // the staged block and in the cache block (the same bytes)
                        auto put = [&](uint8_t *blk) {
                            *reinterpret_cast<uint16_t *>(blk + app_row * kD + 2 * lane) = static_cast<uint16_t>(knew);
                            blk[kBlk8V + (2 * lane) * kPage + app_row] = static_cast<uint8_t>(vnew);
                            blk[kBlk8V + (2 * lane + 1) * kPage + app_row] = static_cast<uint8_t>(vnew >> 8);
                            if (lane == 0) {
                                reinterpret_cast<float *>(blk + kBlk8S)[app_row] = knew_scale;
                                reinterpret_cast<float *>(blk + kBlk8S)[kPage + app_row] = vnew_scale;
                            }
                        };
                        put(gK);
                        if (ok) {
                            const size_t blk = RING ? slice * (p.window / kPage) + tt : slice;
                            put(reinterpret_cast<uint8_t *>(p.k_cache) + blk * kBlk8Bytes);
                        }
                    } else {
                        const uint32_t off = app_row * 128 + ((((lane >> 2) ^ (app_row & 7))) << 4) + (lane & 3) * 4;
                        *reinterpret_cast<uint32_t *>(gK + off) = knew;
                        *reinterpret_cast<uint32_t *>(gV + off) = vnew;
                        if (ok) {
                            const size_t c = slice * (RING ? p.window : kPage) + cell;
                            reinterpret_cast<uint32_t *>(p.k_cache + c * kD)[lane] = knew;
                            reinterpret_cast<uint32_t *>(p.v_cache + c * kD)[lane] = vnew;
                        }
                    }
                    __syncwarp();
                }
            }

            // token validity of this lane's rows (fp8 tiles: rows are permuted tokens)
            const int lo_v = RING ? 0 : lo, hi_v = RING ? nvalid : L;
            const int row_tok = KV8 ? fp8_row_token(lane >> 2) : (lane >> 2);
            int t0[UT];
            bool partial[UT], ok_lo[UT], ok_hi[UT];
#pragma unroll
            for (int u = 0; u < UT; ++u) {
                if constexpr (FAST) {
                    t0[u] = 0;
                    partial[u] = false;
                    ok_lo[u] = ok_hi[u] = true;
                } else {
                    t0[u] = (RING ? tts[u] : ft + tts[u]) * kPage;
                    // several tokens: a tile is whole only inside every row's range
                    partial[u] = MT ? (t0[u] < lo_max) || (t0[u] + kPage > hi_min)
                                    : (t0[u] < lo_v) || (t0[u] + kPage > hi_v);
                    const int r0 = t0[u] + row_tok;
                    const int r8 = r0 + (KV8 ? 2 : 8);
                    ok_lo[u] = r0 >= lo_v && r0 < hi_v;
                    ok_hi[u] = r8 >= lo_v && r8 < hi_v;
                }
            }

            // K fragments, and the V fragments too: they do not depend on the softmax, so
            // their shared-memory latency overlaps the QK products
            uint32_t ka[UT][4][4], va[UT][4][4];
            float ks_lo[UT], ks_hi[UT], vs_lo[UT], vs_hi[UT];  // fp8 per-token scales
#pragma unroll
            for (int u = 0; u < UT; ++u) {
                ks_lo[u] = ks_hi[u] = vs_lo[u] = vs_hi[u] = 1.f;
                if constexpr (KV8) {
                    const uint8_t *gK = wbase + k_off(stgs[u]);
                    const uint8_t *gV = wbase + v_off(stgs[u]);
                    // K rows row_tok and row_tok + 2: bytes 16t..16t+15 (d), 4 per k-step
                    const uint4 klo = *reinterpret_cast<const uint4 *>(gK + row_tok * kD + 16 * (lane & 3));
                    const uint4 khi = *reinterpret_cast<const uint4 *>(gK + (row_tok + 2) * kD + 16 * (lane & 3));
                    const uint32_t wl[4] = {klo.x, klo.y, klo.z, klo.w}, wh[4] = {khi.x, khi.y, khi.z, khi.w};
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        e4m3x4_to_f16x2x2(wl[ks], ka[u][ks][0], ka[u][ks][2]);
                        e4m3x4_to_f16x2x2(wh[ks], ka[u][ks][1], ka[u][ks][3]);
                    }
                    // V^T rows d and d + 8: tokens 4t..4t+3 in one word
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        const uint32_t vl = *reinterpret_cast<const uint32_t *>(gV + (16 * mt + (lane >> 2)) * kPage + 4 * (lane & 3));
                        const uint32_t vh = *reinterpret_cast<const uint32_t *>(gV + (16 * mt + 8 + (lane >> 2)) * kPage + 4 * (lane & 3));
                        e4m3x4_to_f16x2x2(vl, va[u][mt][0], va[u][mt][2]);
                        e4m3x4_to_f16x2x2(vh, va[u][mt][1], va[u][mt][3]);
                    }
                    const float *ssr = reinterpret_cast<const float *>(wbase + s_off(stgs[u]));
                    ks_lo[u] = ssr[row_tok];
                    ks_hi[u] = ssr[row_tok + 2];
                    // V scales carry a factor 2^8 (2^4 with the lazy maximum, whose
                    // probabilities reach 2^4) so that the fp16 products stay normal; it is
                    // taken out when the segment closes
                    vs_lo[u] = ssr[kPage + row_tok] * kV8Factor;
                    vs_hi[u] = ssr[kPage + row_tok + 2] * kV8Factor;
                    if (partial[u]) {  // a row outside the attended range may hold a garbage scale
                        vs_lo[u] = ok_lo[u] ? vs_lo[u] : 0.f;
                        vs_hi[u] = ok_hi[u] ? vs_hi[u] : 0.f;
                    }
                } else {
                    const uint32_t sK = k_tile(stgs[u]), sV = v_tile(stgs[u]);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        ldsm_x4(sK + k_row + (((2 * ks + k_cb) ^ lj) << 4), ka[u][ks][0], ka[u][ks][1], ka[u][ks][2], ka[u][ks][3]);
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt)
                        ldsm_x4_t(sV + v_row + (((2 * mt + v_cb) ^ lj) << 4), va[u][mt][0], va[u][mt][1], va[u][mt][2], va[u][mt][3]);
                }
            }
            // S^T = K Q^T  (16 tokens x 8 heads per n-tile and tile), two MMA chains per tile
            uint32_t pb[UT][NT][2];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                float sv[UT][4];
#pragma unroll
                for (int u = 0; u < UT; ++u) {
                    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
                    if constexpr (KV8) {
                        mma_f16(sc, ka[u][0][0], ka[u][0][1], ka[u][0][2], ka[u][0][3], qf[n][0][0], qf[n][0][1]);
                        mma_f16(sd, ka[u][1][0], ka[u][1][1], ka[u][1][2], ka[u][1][3], qf[n][1][0], qf[n][1][1]);
                        mma_f16(sc, ka[u][2][0], ka[u][2][1], ka[u][2][2], ka[u][2][3], qf[n][2][0], qf[n][2][1]);
                        mma_f16(sd, ka[u][3][0], ka[u][3][1], ka[u][3][2], ka[u][3][3], qf[n][3][0], qf[n][3][1]);
                    } else {
                        mma_bf16(sc, ka[u][0][0], ka[u][0][1], ka[u][0][2], ka[u][0][3], qf[n][0][0], qf[n][0][1]);
                        mma_bf16(sd, ka[u][1][0], ka[u][1][1], ka[u][1][2], ka[u][1][3], qf[n][1][0], qf[n][1][1]);
                        mma_bf16(sc, ka[u][2][0], ka[u][2][1], ka[u][2][2], ka[u][2][3], qf[n][2][0], qf[n][2][1]);
                        mma_bf16(sd, ka[u][3][0], ka[u][3][1], ka[u][3][2], ka[u][3][3], qf[n][3][0], qf[n][3][1]);
                    }
                    const float sl_lo = KV8 ? p.scale_log2 * ks_lo[u] : p.scale_log2;
                    const float sl_hi = KV8 ? p.scale_log2 * ks_hi[u] : p.scale_log2;
                    sv[u][0] = (sc[0] + sd[0]) * sl_lo;
                    sv[u][1] = (sc[1] + sd[1]) * sl_lo;
                    sv[u][2] = (sc[2] + sd[2]) * sl_hi;
                    sv[u][3] = (sc[3] + sd[3]) * sl_hi;
                    if (partial[u]) {
                        if constexpr (MT) {  // key rows t0 + lane/4 and + 8 against each column's range
                            const int kl = t0[u] + (lane >> 2), kh = kl + 8;
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int r = r0g + n * 8 + (lane & 3) * 2 + j, t = r / p.G;
                                const bool ok = r < p.T * p.G && t < nq_seg;
                                const int lc = ok ? (p.window > 0 ? max(0, base + t - p.window + 1) : 0) : (1 << 30);
                                const int hc = ok ? base + t + 1 : 0;
                                if (!(kl >= lc && kl < hc)) sv[u][j] = -INFINITY;
                                if (!(kh >= lc && kh < hc)) sv[u][2 + j] = -INFINITY;
                            }
                        } else {
                            if (!ok_lo[u]) sv[u][0] = sv[u][1] = -INFINITY;
                            if (!ok_hi[u]) sv[u][2] = sv[u][3] = -INFINITY;
                        }
                    }
                }
                float mx0 = fmaxf(sv[0][0], sv[0][2]), mx1 = fmaxf(sv[0][1], sv[0][3]);
#pragma unroll
                for (int u = 1; u < UT; ++u) {
                    mx0 = fmaxf(mx0, fmaxf(sv[u][0], sv[u][2]));
                    mx1 = fmaxf(mx1, fmaxf(sv[u][1], sv[u][3]));
                }
                if constexpr (kLazy) {
                    // the reference moves (to the exact maximum) only when a score of this
                    // pass exceeds it by more than 2^kLazyLog2 in some lane
                    const bool grow = mx0 > st.m[n][0] + kLazyT || mx1 > st.m[n][1] + kLazyT;
                    if (__any_sync(0xffffffffu, grow)) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 4));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 4));
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 8));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 8));
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 16));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 16));
                        const float mn0 = fmaxf(st.m[n][0], mx0), mn1 = fmaxf(st.m[n][1], mx1);
                        const float mr0 = mn0 == -INFINITY ? 0.f : mn0, mr1 = mn1 == -INFINITY ? 0.f : mn1;
                        const float a0 = fast_exp2(st.m[n][0] - mr0), a1 = fast_exp2(st.m[n][1] - mr1);
                        st.l[n][0] *= a0;
                        st.l[n][1] *= a1;
                        st.m[n][0] = mn0;
                        st.m[n][1] = mn1;
#pragma unroll
                        for (int mt = 0; mt < 4; ++mt) {
                            st.acc[n][mt][0] *= a0;
                            st.acc[n][mt][1] *= a1;
                            st.acc[n][mt][2] *= a0;
                            st.acc[n][mt][3] *= a1;
                        }
                    }
                    // (a column that has seen no key yet, m = -inf: subtract 0, every term is 0)
                    const float mr0 = st.m[n][0] == -INFINITY ? 0.f : st.m[n][0];
                    const float mr1 = st.m[n][1] == -INFINITY ? 0.f : st.m[n][1];
                    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                    for (int u = 0; u < UT; ++u) {
                        const float p0 = fast_exp2(sv[u][0] - mr0), p1 = fast_exp2(sv[u][1] - mr1);
                        const float p2 = fast_exp2(sv[u][2] - mr0), p3 = fast_exp2(sv[u][3] - mr1);
                        ls0 += p0 + p2;
                        ls1 += p1 + p3;
                        if constexpr (KV8) {
                            pb[u][n][0] = movmatrix_t(pack_f16(p0 * vs_lo[u], p1 * vs_lo[u]));
                            pb[u][n][1] = movmatrix_t(pack_f16(p2 * vs_hi[u], p3 * vs_hi[u]));
                        } else {
                            pb[u][n][0] = movmatrix_t(pack_bf16(p0, p1));
                            pb[u][n][1] = movmatrix_t(pack_bf16(p2, p3));
                        }
                    }
                    st.l[n][0] += ls0;
                    st.l[n][1] += ls1;
                    continue;
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 4));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 4));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 8));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 8));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 16));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 16));
                const float mn0 = fmaxf(st.m[n][0], mx0), mn1 = fmaxf(st.m[n][1], mx1);
                // several tokens: a column may have seen no key yet (m = -inf); subtract 0 then
                // (every term is 0) instead of forming -inf - -inf
                const float mr0 = (MT && mn0 == -INFINITY) ? 0.f : mn0;
                const float mr1 = (MT && mn1 == -INFINITY) ? 0.f : mn1;
                const float a0 = fast_exp2(st.m[n][0] - mr0), a1 = fast_exp2(st.m[n][1] - mr1);
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int u = 0; u < UT; ++u) {
                    const float p0 = fast_exp2(sv[u][0] - mr0), p1 = fast_exp2(sv[u][1] - mr1);
                    const float p2 = fast_exp2(sv[u][2] - mr0), p3 = fast_exp2(sv[u][3] - mr1);
                    ls0 += p0 + p2;
                    ls1 += p1 + p3;
                    if constexpr (KV8) {  // probabilities times the tokens' V scales, fp16
                        pb[u][n][0] = movmatrix_t(pack_f16(p0 * vs_lo[u], p1 * vs_lo[u]));  // tokens 4t, 4t+1
                        pb[u][n][1] = movmatrix_t(pack_f16(p2 * vs_hi[u], p3 * vs_hi[u]));  // tokens 4t+2, 4t+3
                    } else {
                        pb[u][n][0] = movmatrix_t(pack_bf16(p0, p1));  // tokens 2(lane%4)+{0,1}
                        pb[u][n][1] = movmatrix_t(pack_bf16(p2, p3));  // tokens 8+2(lane%4)+{0,1}
                    }
                }
                st.l[n][0] = st.l[n][0] * a0 + ls0;
                st.l[n][1] = st.l[n][1] * a1 + ls1;
                st.m[n][0] = mn0;
                st.m[n][1] = mn1;
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    st.acc[n][mt][0] *= a0;
                    st.acc[n][mt][1] *= a1;
                    st.acc[n][mt][2] *= a0;
                    st.acc[n][mt][3] *= a1;
                }
            }

            // O^T += V^T P^T  (64 d x 8 heads per n-tile)
#pragma unroll
            for (int u = 0; u < UT; ++u) {
                if (partial[u]) {
                    // zero the V values of tokens outside the range (they may hold NaN): this
                    // lane's V^T fragment halves carry tokens 2t, 2t+1 / 2t+8, 2t+9 (bf16 tiles);
                    // 4t, 4t+1 / 4t+2, 4t+3 (fp8 tiles)
                    const int tv = t0[u] + (lane & 3) * (KV8 ? 4 : 2);
                    const int tw = tv + (KV8 ? 2 : 8);
                    const uint32_t vm0 = ((tv >= lo_v && tv < hi_v) ? 0x0000ffffu : 0u) |
                                         ((tv + 1 >= lo_v && tv + 1 < hi_v) ? 0xffff0000u : 0u);
                    const uint32_t vm1 = ((tw >= lo_v && tw < hi_v) ? 0x0000ffffu : 0u) |
                                         ((tw + 1 >= lo_v && tw + 1 < hi_v) ? 0xffff0000u : 0u);
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        va[u][mt][0] &= vm0;
                        va[u][mt][1] &= vm0;
                        va[u][mt][2] &= vm1;
                        va[u][mt][3] &= vm1;
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int u = 0; u < UT; ++u)
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        if constexpr (KV8)
                            mma_f16(st.acc[n][mt], va[u][mt][0], va[u][mt][1], va[u][mt][2], va[u][mt][3], pb[u][n][0], pb[u][n][1]);
                        else
                            mma_bf16(st.acc[n][mt], va[u][mt][0], va[u][mt][1], va[u][mt][2], va[u][mt][3], pb[u][n][0], pb[u][n][1]);
                    }

            __syncwarp();
            // refill the stages just read (tile i + u + kStages goes where tile i + u was)
            const int nref = min(UT, n_tiles - (i + kStages));
            if (nref > 0) {
                if (lane < nref) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (kParIssue) {
                    issue_n(i + kStages, nref, st0);
                } else {
#pragma unroll
                    for (int u = 0; u < UT; ++u)
                        if (u < nref) issue_n(i + kStages + u, 1, stgs[u]);
                }
            }
        };

        int stg = 0;       // stage of tile i
        uint32_t ph = 0;   // parity of its barrier phase
        const int expire_at = wid == 0 ? p.expire_at : -1;
        while (i < n_tiles) {
            // the lanes decide together: a lane whose wait expired takes the whole warp out
            const bool landed = mbar_wait_bounded(bar0 + 8 * stg, ph);
            if (__any_sync(0xffffffffu, !landed) || (expire_at >= 0 && i >= expire_at)) {
                failed = true;
                break;
            }
            const int4 md = wmeta[stg];
            const int tb = md.x, tg = md.y, tt = md.z;
            if (i == 0 || tt == 0) {
                // close the previous segment
                if (i > 0) {
                    state_reduce_l(st);
                    if constexpr (KV8) state_scale_acc(st, 1.f / kV8Factor);
                    if (seg_first_unit < ua) {  // shared with earlier workers: keep for merge
                        if constexpr (kHeadInRegs)
                            head = st;
                        else
                            state_store_lanes(st, head_mem, lane);
                        head_seg = sb * Hkv + sgk;
                    } else if constexpr (MT) {
                        float sig[NT][2];
                        sinks_of(sig);
                        state_write_out_mt(st, sig, p.out, sb, sgk, p.T, p.G, p.Hq, nq_seg, r0g, lane);
                    } else {
                        float sig[NT][2];
                        sinks_of(sig);
                        state_write_out(st, sig, p.out + (static_cast<size_t>(sb) * p.Hq + sgk * p.G) * kD,
                                        p.G, lane);
                    }
                }
                sb = tb; sgk = tg;
                L = s_len[sb];
                const int tiles = (s_pre[sb + 1] - s_pre[sb]) / Hkv;
                seg_first_unit = s_pre[sb] + sgk * tiles;
                seg_end_unit = seg_first_unit + tiles;
                if (RING) {
                    nvalid = L < p.window ? L : p.window;
                    const int cell = (L - 1) % p.window;
                    app_tile = cell / kPage;
                    app_row = cell % kPage;
                } else if constexpr (MT) {
                    nq_seg = s_n[sb];
                    base = L - nq_seg;
                    lo = p.window > 0 ? max(0, base - p.window + 1) : 0;
                    ft = lo / kPage;
                    lo_max = p.window > 0 ? max(0, L - p.window) : 0;  // the last row's window start
                    hi_min = base + 1;                                  // the first row's end
                    // the new tokens' k/v rows (this lane's bf16 pair of each): loaded now, used
                    // at the segment's last tiles, so the load latency hides behind the loop
                    // (32 rows: loaded there, the registers are needed for the four n-tiles)
#pragma unroll
                    for (int i2 = 0; i2 < kMaxNewMT; ++i2)
                        if (kNewInRegs && i2 < nq_seg) {
                            const size_t off = ((static_cast<size_t>(sb) * p.T + i2) * Hkv + sgk) * kD;
                            knewm[i2] = __ldg(reinterpret_cast<const uint32_t *>(p.k_new + off) + lane);
                            vnewm[i2] = __ldg(reinterpret_cast<const uint32_t *>(p.v_new + off) + lane);
                        }
                } else {
                    lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
                    ft = lo / kPage;
                    app_tile = (L - 1) / kPage - ft;
                    app_row = (L - 1) % kPage;
                }
                // Q fragments (B operand): q[head = lane/4][d = 16ks + 2(lane%4) (+8)]
                const uint8_t *qs = wq + stg * kQBytes;
                if (!MT && do_append) {  // the new token's k/v rows arrived with this tile
                    knew = reinterpret_cast<const uint32_t *>(qs + GP * kD * 2)[lane];
                    vnew = reinterpret_cast<const uint32_t *>(qs + GP * kD * 2 + kD * 2)[lane];
                }
                const int qrows = MT ? p.T * p.G : p.G;  // query rows (columns) of the group
                // rotary cos / sin rows of the new token's position (staged with the segment)
                const float *cr = reinterpret_cast<const float *>(qs + GP * kD * 2 + 4 * kD);
                const float *sr = cr + kD / 2;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int hq = n * 8 + (lane >> 2);  // slot row; query row r0g + hq
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        if (r0g + hq < qrows) {
                            const uint32_t *row = reinterpret_cast<const uint32_t *>(qs + hq * kD * 2);
                            if constexpr (KV8) {
                                // fp16 operands; k-step ks takes d = 16t + 4ks .. +3, the bytes
                                // one lane reads from an fp8 K row (see the QK product)
                                const int wq = 8 * (lane & 3) + 2 * ks;  // word of elements 2wq, 2wq + 1
                                uint32_t w0 = row[wq], w1 = row[wq + 1];
                                if constexpr (ROPE) {
                                    // rotated in bf16 before the conversion: the rotate-half partner
                                    // of element e is e +- 32, the word 16 away in the same row
                                    const int i0 = (2 * wq) & 31;
                                    const bool first = wq < 16;
                                    w0 = rope_half(w0, row[wq ^ 16], cr + i0, sr + i0, first);
                                    w1 = rope_half(w1, row[(wq ^ 16) + 1], cr + i0 + 2, sr + i0 + 2, first);
                                }
                                qf[n][ks][0] = bf16x2_to_f16x2(w0);
                                qf[n][ks][1] = bf16x2_to_f16x2(w1);
                            } else {
                                qf[n][ks][0] = row[ks * 8 + (lane & 3)];
                                qf[n][ks][1] = row[ks * 8 + 4 + (lane & 3)];
                            }
                        } else {
                            qf[n][ks][0] = qf[n][ks][1] = 0u;
                        }
                    }
                    if constexpr (kSinksInRegs) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int hs = r0g + n * 8 + (lane & 3) * 2 + j;
                            sig_r[n][j] = hs < qrows ? s_sink[sgk * p.G + (MT ? hs % p.G : hs)] : -INFINITY;
                        }
                    }
                }
                if constexpr (ROPE) {
                    // rotary embedding of the new token (rotate-half pairs (i, i + 32)); each
                    // product and the sum/difference rounded to fp32, then to bf16 (nearest even)
                    if constexpr (!KV8) {  // (fp8 tiles: the queries were rotated above)
                        // queries: the partner of element d (< 32) is d + 32, two k-steps further
#pragma unroll
                        for (int n = 0; n < NT; ++n)
#pragma unroll
                            for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    const int d = ks * 16 + r * 8 + (lane & 3) * 2;
                                    rope_pair(qf[n][ks][r], qf[n][ks + 2][r], cr + d, sr + d);
                                }
                    }
                    // the new key, rotated before it is stored (and, for fp8, quantised):
                    if (do_append) {  // element 2*lane pairs with lane ^ 16
                        const uint32_t other = __shfl_xor_sync(0xffffffffu, knew, 16);
                        const int d = (2 * lane) & 31;
                        knew = rope_half(knew, other, cr + d, sr + d, lane < 16);
                    }
                }
                if constexpr (KV8) {
                    if (do_append) {  // quantise the new token: per row amax / 448, e4m3 codes
                        const float2 kf = unpack_bf16(knew), vf = unpack_bf16(vnew);
                        float ka = fmaxf(fabsf(kf.x), fabsf(kf.y)), va = fmaxf(fabsf(vf.x), fabsf(vf.y));
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) {
                            ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, off));
                            va = fmaxf(va, __shfl_xor_sync(0xffffffffu, va, off));
                        }
                        knew_scale = ka > 0.f ? __fdiv_rn(ka, 448.f) : 1.f;
                        vnew_scale = va > 0.f ? __fdiv_rn(va, 448.f) : 1.f;
                        knew = f32x2_to_e4m3x2(__fdiv_rn(kf.x, knew_scale), __fdiv_rn(kf.y, knew_scale));
                        vnew = f32x2_to_e4m3x2(__fdiv_rn(vf.x, vnew_scale), __fdiv_rn(vf.y, vnew_scale));
                    }
                }
                state_reset(st);
            }
            // the next tile continues this segment: take both in one pass
            int stg1 = stg + 1;
            uint32_t ph1 = ph;
            if (stg1 == kStages) { stg1 = 0; ph1 ^= 1u; }
            if constexpr (kPair) {
                if (i + 1 < n_tiles && ua + i + 1 < seg_end_unit) {
                    if (__any_sync(0xffffffffu, !mbar_wait_bounded(bar0 + 8 * stg1, ph1))) {
                        failed = true;
                        break;
                    }
                    // both tiles whole and neither the append tile: the fast pass
                    auto whole = [&](int t) {
                        if constexpr (MT) {  // before every new token and inside every row's window
                            const int f = (ft + t) * kPage;
                            return f >= lo_max && f + kPage <= base;
                        }
                        if (do_append && t == app_tile) return false;
                        if (RING) return t * kPage + kPage <= nvalid;
                        const int f = (ft + t) * kPage;
                        return f >= lo && f + kPage <= L;
                    };
                    if ((MT || (KV8 ? DA_FAST_PASS_FP8 : DA_FAST_PASS_BF16)) && whole(tt) && whole(tt + 1))
                        tiles_step(std::integral_constant<int, 2>{}, std::true_type{}, stg, stg1);
                    else
                        tiles_step(std::integral_constant<int, 2>{}, std::false_type{}, stg, stg1);
                    i += 2;
                    stg = stg1 + 1;
                    ph = ph1;
                    if (stg == kStages) { stg = 0; ph ^= 1u; }
                    continue;
                }
            }
            if constexpr (MT) {  // several tokens: the masks only on the tiles at the rows' edges
                const int f = (ft + tt) * kPage;
                if (f >= lo_max && f + kPage <= base)
                    tiles_step(std::integral_constant<int, 1>{}, std::true_type{}, stg, stg);
                else
                    tiles_step(std::integral_constant<int, 1>{}, std::false_type{}, stg, stg);
            } else {
                tiles_step(std::integral_constant<int, 1>{}, std::false_type{}, stg, stg);
            }
            i += 1;
            stg = stg1;
            ph = ph1;
        }
        if (failed) {
            flag_status(DA_STATUS_TIMEOUT);
            // let the copies still in flight (tiles i .. i + kStages - 1) land before the CTA
            // moves on; the warp's area is then neither written nor read again (its states are
            // left out of the merges: the call's output is garbage). The tickets do not depend
            // on this warp: the CTA's boundary segments come from the unit prefix, so the
            // counters still return to zero.
            for (int j = i; j < n_tiles && j < i + kStages; ++j)
                mbar_wait_bounded(bar0 + 8 * (j % kStages), (j / kStages) & 1);
            slots_ok = false;
        }
        __syncwarp();

        // close the last segment
        state_reduce_l(st);
        if constexpr (KV8) state_scale_acc(st, 1.f / kV8Factor);
        const bool last_shared = failed || seg_first_unit < ua || seg_end_unit > ue;
        if (last_shared) {
            tail_seg = sb * Hkv + sgk;
        } else if constexpr (MT) {
            float sig[NT][2];
            sinks_of(sig);
            state_write_out_mt(st, sig, p.out, sb, sgk, p.T, p.G, p.Hq, nq_seg, r0g, lane);
        } else {
            float sig[NT][2];
            sinks_of(sig);
            state_write_out(st, sig, p.out + (static_cast<size_t>(sb) * p.Hq + sgk * p.G) * kD, p.G, lane);
        }
        // partial states -> this warp's (drained) buffer area
        Slot<NT> *slot0 = reinterpret_cast<Slot<NT> *>(wbase);
        Slot<NT> *slot1 = kSlotsInTiles ? slot0 + 1 : reinterpret_cast<Slot<NT> *>(wq);
        if (slots_ok && head_seg >= 0) {
            if constexpr (!kHeadInRegs) state_load_lanes(head, head_mem, lane);  // (own stores)
            state_to_slot(head, slot0, lane);
        }
        if (slots_ok && tail_seg >= 0) state_to_slot(st, slot1, lane);
    }
    zero_inactive();
    // (the states published in the slots are the plan's head and tail: a warp whose copies
    // never landed is left out of the merges)
    if (lane == 0) s_winfo[warp * kWinfo + 9] = slots_ok ? 1 : 0;
    __syncthreads();
    if (!early && tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the CTA's boundary segments (final before the loop) and their contributors, in registers
    const int bseg0 = s_flag[2], bseg1 = s_flag[3];
    const int bclo0 = s_flag[8], bnc0 = s_flag[9], blo0 = s_flag[10];
    const int bclo1 = s_flag[11], bnc1 = s_flag[12], blo1 = s_flag[13];

    // ---- 4. merge segments shared between warps of this CTA (all threads take part)
    // Segments shared by several warps: every warp of this CTA holding a state of one (warps
    // wa .. wb, consecutive) merges a share of it. A segment that also crosses into another
    // CTA becomes this CTA's fp32 partial; slot 0 if it holds the CTA's first unit, else 1.
    // fp32 partial slot k of the CTA with effective index c in this row group; the row
    // groups count their tickets apart
    auto part_slot = [&](int c, int k) {
        return p.part + ((static_cast<size_t>(c) * ngrp + rgrp) * 2 + k) * kSlotFloats;
    };
    int *const counters = p.counters + static_cast<size_t>(rgrp) * B * Hkv;
    if (warp < nw_cta) {
        const int *wi = s_winfo + warp * kWinfo;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
            const int seg = wi[2 + which];
            if (seg < 0) continue;
            const int s0 = wi[5 + 2 * which], s1 = wi[6 + 2 * which];
            // the warps of this CTA holding a state of seg: wa .. wa + k - 1 (the plan)
            const int wa = wi[12 + 2 * which], k = wi[13 + 2 * which], mine = warp - wa;
            const bool internal = s0 >= R0 && s1 <= R1;
            const int slot_k = s0 <= R0 ? 0 : 1;
            const int b = seg / Hkv, g = seg - b * Hkv;
            // The segment's items (a column and DPI of its dimensions, DPI 16, 8 or 4: the
            // narrowest that gives every lane of its k warps at most one item, or two when a
            // single warp holds the 16 columns of a 16-head group) are shared out over those
            // lanes; a lane loads its item from every contributor at once (contributor c is
            // warp wa + c, its slot the head or the tail one; a warp whose copies never landed
            // is skipped), four contributors per round.
            const uint32_t slots_base = smem_addr(smem), tails_base = smem_addr(qarea);
            const int qrows = MT ? p.T * p.G : p.G;  // valid query rows of the group
            auto merge_items = [&](auto dpi_c) {
                constexpr int DPI = decltype(dpi_c)::value;
                constexpr int IPC = kD / DPI;  // items per column
#pragma unroll 1
                for (int item = mine * 32 + lane; item < GP * IPC; item += k * 32) {
                    const int n = item / IPC, d0 = (item % IPC) * DPI;
                    const int rn = r0g + n;  // column n's query row
                    const float sg = (internal && rn < qrows) ? s_sink[g * p.G + (MT ? rn % p.G : rn)] : -INFINITY;
                    float M = -INFINITY, den = 0.f;
                    float acc[DPI];
#pragma unroll
                    for (int j = 0; j < DPI; ++j) acc[j] = 0.f;
#pragma unroll 1
                    for (int c0 = 0; c0 < k; c0 += 4) {
                        float mc[4], lc[4];
                        float4 a[4][DPI / 4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int c = c0 + u, w = wa + (c < k ? c : 0);
                            const bool ok = c < k && s_winfo[w * kWinfo + 9] != 0;
                            const bool tail = s_winfo[w * kWinfo + 3] == seg;
                            const uint32_t sl = !tail ? slots_base + w * kWarpBytes
                                                : kSlotsInTiles ? slots_base + w * kWarpBytes + static_cast<uint32_t>(sizeof(Slot<NT>))
                                                                : tails_base + w * kStages * kQBytes;
                            mc[u] = ok ? lds_f32(sl + 4 * n) : -INFINITY;
                            lc[u] = ok ? lds_f32(sl + 4 * (GP + n)) : 0.f;
#pragma unroll
                            for (int q = 0; q < DPI / 4; ++q)
                                a[u][q] = ok ? lds_f32x4(sl + 4 * (2 * GP + n * Slot<NT>::LD + d0 + 4 * q))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        float Mn = M;
#pragma unroll
                        for (int u = 0; u < 4; ++u) Mn = fmaxf(Mn, mc[u]);
                        const float r = M == -INFINITY ? 0.f : fast_exp2(M - Mn);  // rescale the rounds before
                        den *= r;
#pragma unroll
                        for (int j = 0; j < DPI; ++j) acc[j] *= r;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float w = mc[u] == -INFINITY ? 0.f : fast_exp2(mc[u] - Mn);  // no key: weight 0
                            den += lc[u] * w;
#pragma unroll
                            for (int q = 0; q < DPI / 4; ++q) {
                                acc[4 * q] += a[u][q].x * w;
                                acc[4 * q + 1] += a[u][q].y * w;
                                acc[4 * q + 2] += a[u][q].z * w;
                                acc[4 * q + 3] += a[u][q].w * w;
                            }
                        }
                        M = Mn;
                    }
                    if (internal) {  // sink, normalise, bf16
                        const float Mf = fmaxf(M, sg);
                        const float r = M == -INFINITY ? 0.f : fast_exp2(M - Mf);
                        den = den * r + (sg == -INFINITY ? 0.f : fast_exp2(sg - Mf));
                        if (rn < qrows) {
                            const int t = MT ? rn / p.G : 0, h = MT ? rn - t * p.G : rn;
                            const float inv = (MT && t >= s_n[b]) ? 0.f : r / den;  // no query token: zeros
                            __nv_bfloat16 *dst =
                                p.out + ((static_cast<size_t>(b) * (MT ? p.T : 1) + t) * p.Hq + g * p.G + h) * kD + d0;
                            uint32_t o[DPI / 2];
#pragma unroll
                            for (int j = 0; j < DPI / 2; ++j) o[j] = pack_bf16(acc[2 * j] * inv, acc[2 * j + 1] * inv);
                            if constexpr (DPI == 4) {
                                *reinterpret_cast<uint2 *>(dst) = make_uint2(o[0], o[1]);
                            } else {
#pragma unroll
                                for (int j = 0; j < DPI / 8; ++j)
                                    reinterpret_cast<uint4 *>(dst)[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
                            }
                        }
                    } else {  // this CTA's fp32 partial of the segment
                        float *gp = part_slot(cta, slot_k);
                        if (d0 == 0) {
                            gp[n] = M;
                            gp[GP + n] = den;
                        }
                        float4 *ga = reinterpret_cast<float4 *>(gp + 2 * GP + n * kD + d0);
#pragma unroll
                        for (int q = 0; q < DPI / 4; ++q)
                            ga[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                    }
                }
            };
            if (32 * k >= GP * 16)  // (GP * kD / 4 items of 4 dimensions)
                merge_items(std::integral_constant<int, 4>{});
            else if (32 * k >= GP * 8)
                merge_items(std::integral_constant<int, 8>{});
            else
                merge_items(std::integral_constant<int, 16>{});
        }
    }
    // (no fence here: the ticket-taking thread's fence below publishes every thread's partials)
    __syncthreads();

    // ---- 5. segments shared with other CTAs: the last CTA to arrive combines them
    if (tid == 0) {
        const int cand0 = bseg0, cand1 = bseg1;
        // the barrier above orders every thread's partial stores before this fence, which
        // orders them (cumulatively, at GPU scope) before the tickets
        if (cand0 >= 0 || cand1 >= 0) asm volatile("fence.acq_rel.gpu;" ::: "memory");
        // both tickets in flight together
        const int t0 = cand0 >= 0 ? atomicAdd(counters + cand0, 1) : 0;
        const int t1 = cand1 >= 0 ? atomicAdd(counters + cand1, 1) : 0;
        // the CTA taking the last ticket of a segment combines it
        s_flag[0] = (cand0 >= 0 && t0 == bnc0 - 1) ? cand0 : -1;
        s_flag[1] = (cand1 >= 0 && t1 == bnc1 - 1) ? cand1 : -1;
        // the other CTAs' partials, ordered before their tickets, are visible after this fence
        if (s_flag[0] >= 0 || s_flag[1] >= 0) asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    __syncthreads();
    // One pass, no barrier: every thread owns kPer outputs of one head and folds the
    // partials in batches of kCombBatch contributors whose loads are all in flight together
    // (a 131k-token sequence spread over every CTA has about 20 per KV head: one round trip).
    constexpr int kPer = GP * kD / kThreads;  // outputs per thread: 2 (8 rows), 4 (16) or 8 (32)
    constexpr int kCombBatch = (CPS > 1 || kPer == 8) ? 8 : 24;  // (the 128-register two-CTA kernel: 8)
    const int cn = tid / (kD / kPer), cd0 = (tid % (kD / kPer)) * kPer;
#pragma unroll 1
    for (int k = 0; k < 2; ++k) {
        const int seg = s_flag[k];
        if (seg < 0) continue;
        const int c_lo = k == 0 ? bclo0 : bclo1, nc = k == 0 ? bnc0 : bnc1, lo_slot = k == 0 ? blo0 : blo1;
        const int b = seg / Hkv, g = seg - b * Hkv;
        float M = -INFINITY, den = 0.f, acc[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < nc; c0 += kCombBatch) {
            float mc[kCombBatch], lc[kCombBatch], v[kCombBatch][kPer];
#pragma unroll
            for (int j = 0; j < kCombBatch; ++j) {
                mc[j] = -INFINITY;
                lc[j] = 0.f;
#pragma unroll
                for (int t = 0; t < kPer; ++t) v[j][t] = 0.f;
                if (c0 + j < nc) {
                    const int c = c0 + j;
                    const float *gp = part_slot(c_lo + c, c == 0 ? lo_slot : 0);
                    mc[j] = __ldcg(gp + cn);
                    lc[j] = __ldcg(gp + GP + cn);
                    if constexpr (kPer == 2) {
                        const float2 t2 = __ldcg(reinterpret_cast<const float2 *>(gp + 2 * GP + cn * kD + cd0));
                        v[j][0] = t2.x; v[j][1] = t2.y;
                    } else {
#pragma unroll
                        for (int q4 = 0; q4 < kPer / 4; ++q4) {
                            const float4 t4 = __ldcg(reinterpret_cast<const float4 *>(gp + 2 * GP + cn * kD + cd0) + q4);
                            v[j][4 * q4] = t4.x; v[j][4 * q4 + 1] = t4.y; v[j][4 * q4 + 2] = t4.z; v[j][4 * q4 + 3] = t4.w;
                        }
                    }
                }
            }
            float Mn = M;
#pragma unroll
            for (int j = 0; j < kCombBatch; ++j) Mn = fmaxf(Mn, mc[j]);
            const float a = M == -INFINITY ? 0.f : fast_exp2(M - Mn);  // 0 on the first batch (M = -inf)
            den *= a;
#pragma unroll
            for (int t = 0; t < kPer; ++t) acc[t] *= a;
#pragma unroll
            for (int j = 0; j < kCombBatch; ++j) {
                const float w = mc[j] == -INFINITY ? 0.f : fast_exp2(mc[j] - Mn);  // 0: padding, or no key
                den += lc[j] * w;
#pragma unroll
                for (int t = 0; t < kPer; ++t) acc[t] += v[j][t] * w;
            }
            M = Mn;
        }
        const int qrows = MT ? p.T * p.G : p.G;
        const int rc = r0g + cn;  // column cn's query row
        const float sg = rc < qrows ? s_sink[g * p.G + (MT ? rc % p.G : rc)] : -INFINITY;
        const float Mf = fmaxf(M, sg);
        const float a = M == -INFINITY ? 0.f : fast_exp2(M - Mf);
        den = den * a + (sg == -INFINITY ? 0.f : fast_exp2(sg - Mf));
        const int ct = MT ? rc / p.G : 0, ch = MT ? rc - ct * p.G : rc;
        const float f = (den > 0.f && !(MT && ct >= s_n[b])) ? a / den : 0.f;  // no query token: zeros
        if (rc < qrows) {
            __nv_bfloat16 *dst = p.out + ((static_cast<size_t>(b) * (MT ? p.T : 1) + ct) * p.Hq + g * p.G + ch) * kD + cd0;
#pragma unroll
            for (int t = 0; t < kPer; t += 2)
                *reinterpret_cast<uint32_t *>(dst + t) = pack_bf16(acc[t] * f, acc[t + 1] * f);
        }
        if (tid == 0) counters[seg] = 0;  // ready for the next call
    }
}

// ------------------------------------------------------------------ standalone append
__global__ void kv_append_kernel(const __nv_bfloat16 *__restrict__ k_new,
                                 const __nv_bfloat16 *__restrict__ v_new, __nv_bfloat16 *k_cache,
                                 __nv_bfloat16 *v_cache, const int *__restrict__ block_table,
                                 const int *__restrict__ seq_lens, int Hkv, int D, int window,
                                 int page_size, int max_pages, int num_pages) {
    const int b = blockIdx.x;
    const int L = __ldg(seq_lens + b);
    if (L <= 0) {
        if (L < 0 && threadIdx.x == 0) flag_status(DA_STATUS_BAD_SEQ_LEN);
        return;
    }
    const int pos = L - 1;
    size_t base;  // element offset of (head 0, the cell of pos) in the caches
    size_t head_stride;
    if (block_table != nullptr) {
        if (pos / page_size >= max_pages) {
            if (threadIdx.x == 0) flag_status(DA_STATUS_BAD_SEQ_LEN);
            return;
        }
        const int page = __ldg(block_table + static_cast<size_t>(b) * max_pages + pos / page_size);
        if (page < 0 || page >= num_pages) {
            if (threadIdx.x == 0) flag_status(DA_STATUS_BAD_PAGE);
            return;
        }
        base = (static_cast<size_t>(page) * Hkv * page_size + pos % page_size) * D;
        head_stride = static_cast<size_t>(page_size) * D;
    } else {
        base = (static_cast<size_t>(b) * Hkv * window + pos % window) * D;
        head_stride = static_cast<size_t>(window) * D;
    }
    const int chunks = D / 8;  // 16-byte chunks per row
    for (int i = threadIdx.x; i < Hkv * chunks; i += blockDim.x) {
        const int g = i / chunks, c = i % chunks;
        const size_t src = (static_cast<size_t>(b) * Hkv + g) * D + c * 8;
        const size_t dst = base + g * head_stride + c * 8;
        *reinterpret_cast<uint4 *>(k_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(k_new + src));
        *reinterpret_cast<uint4 *>(v_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(v_new + src));
    }
}

// ------------------------------------------------------------------ several query tokens
#include "multi_attn.cuh"
#include "multi_tc.cuh"

// ------------------------------------------------------------------ host side
thread_local char t_err[256];

int set_cuda_error(cudaError_t e) {
    snprintf(t_err, sizeof t_err, "CUDA error: %s", cudaGetErrorString(e));
    return DA_ERR_CUDA;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// The cache view a bf16 tile is copied from: [slices][rows][64], box 16 rows x 64,
// 128-byte swizzle (K and V tiles); rows = tokens per slice (16 per page, or the ring
// capacity). fp8 blocks need no map: they are contiguous.
enum MapKind { kMapBf16 = 0 };

bool encode_kv_map(CUtensorMap *map, void *base, int kind, uint64_t rows, uint64_t slices) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    if (kind == kMapBf16) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), rows, slices};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, rows * kD * 2};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kPage), 1};
        return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    return false;
}

// Encoding a map costs host time on every call; the map depends only on the
// address and the extents, so recent ones are kept.
struct MapCacheEntry {
    void *base = nullptr;
    int kind = 0;
    uint64_t rows = 0, slices = 0;
    CUtensorMap map;
};
constexpr int kMapCache = 32;
MapCacheEntry g_maps[kMapCache];
int g_map_next = 0;
std::mutex g_map_mu;

bool make_kv_map(CUtensorMap *map, void *base, uint64_t rows, uint64_t slices, int kind = kMapBf16) {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < kMapCache; ++i) {
        const MapCacheEntry &e = g_maps[i];
        if (e.base == base && e.kind == kind && e.rows == rows && e.slices == slices) {
            *map = e.map;
            return true;
        }
    }
    if (!encode_kv_map(map, base, kind, rows, slices)) return false;
    MapCacheEntry &e = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    e.base = base;
    e.kind = kind;
    e.rows = rows;
    e.slices = slices;
    e.map = *map;
    return true;
}

constexpr int kMaxDevices = 64;

// A zeroed device buffer that only grows (its arrival counters are zero at rest).
struct Workspace {
    void *p = nullptr;
    size_t bytes = 0;
};

// Per-device state. The workspace pointers change only under g_mu; the SM count and the
// "kernel attribute set" flags are caches that several host threads may fill at once (with
// the same values), so they are atomics.
struct DeviceState {
    Workspace ws;        // one-token calls: counters + CTA partials
    Workspace ws_multi;  // multi-token calls: counters + split partials
    std::atomic<int> sm_count{0};
    std::atomic<bool> attr_set[64] = {};
    std::atomic<bool> multi_attr_set[8] = {};
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// Workspaces of their own for the calls issued on one stream (decode_attn_stream_reserve),
// keyed by the stream handle, under g_mu; g_n_stream_ws lets calls skip the lookup when
// there are none.
struct StreamWorkspaces {
    int dev;
    Workspace ws, ws_multi;
};
std::unordered_map<cudaStream_t, StreamWorkspaces> g_stream_ws;
std::atomic<int> g_n_stream_ws{0};

int current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (*dev < 0 || *dev >= kMaxDevices) return DA_ERR_UNSUPPORTED;
    return DA_OK;
}

int sm_count(int dev) {
    int n = g_dev[dev].sm_count.load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        g_dev[dev].sm_count.store(n, std::memory_order_relaxed);
    }
    return n;
}

size_t slot_floats(int G) {
    const int gp = G <= 8 ? 8 : G <= 16 ? 16 : 32;
    return static_cast<size_t>(2 * gp + gp * kD);
}

// Counters and two partial slots per CTA of the largest grid a decode call of group size G
// may launch.
size_t workspace_for(int G, int sms) {
    const int ctas = sms * (G <= 8 ? kMaxCtasPerSm : 1);  // two CTAs per SM: fp8, 8-head groups
    return kCounterBytes + static_cast<size_t>(ctas) * 2 * slot_floats(G) * sizeof(float);
}

// Grow w to at least `bytes` (synchronous: the old buffer is freed, the new one zeroed).
int grow_locked(Workspace &w, size_t bytes) {
    if (w.bytes >= bytes) return DA_OK;
    if (w.p) {
        cudaError_t e = cudaFree(w.p);
        w.p = nullptr;
        w.bytes = 0;
        if (e != cudaSuccess) return set_cuda_error(e);
    }
    void *p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) return set_cuda_error(e);
    e = cudaMemset(p, 0, bytes);
    if (e != cudaSuccess) {
        cudaFree(p);
        return set_cuda_error(e);
    }
    w.p = p;
    w.bytes = bytes;
    return DA_OK;
}

// The workspace a call on `stream` uses (the stream's own if it has one, else the
// device's), grown to `need` unless the stream is capturing. Under g_mu.
int workspace_locked(int dev, cudaStream_t stream, bool multi, size_t need, void **ptr) {
    Workspace *w = multi ? &g_dev[dev].ws_multi : &g_dev[dev].ws;
    if (g_n_stream_ws.load(std::memory_order_relaxed) > 0) {
        auto it = g_stream_ws.find(stream);
        if (it != g_stream_ws.end()) {
            if (it->second.dev != dev) return DA_ERR_INVALID_ARG;  // the stream is another device's
            w = multi ? &it->second.ws_multi : &it->second.ws;
        }
    }
    if (w->bytes < need) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return set_cuda_error(e);
        if (cs != cudaStreamCaptureStatusNone) return DA_ERR_WORKSPACE;
        int rc = grow_locked(*w, need);
        if (rc != DA_OK) return rc;
    }
    *ptr = w->p;
    return DA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const da_shape &s) {
    if (s.batch < 0 || s.num_q_heads <= 0 || s.num_kv_heads <= 0 || s.head_dim <= 0) return DA_ERR_INVALID_ARG;
    if (s.num_q_heads % s.num_kv_heads != 0) return DA_ERR_INVALID_ARG;
    const int G = s.num_q_heads / s.num_kv_heads;
    if (s.head_dim != kD) return DA_ERR_UNSUPPORTED;
    if (!(G == 1 || G == 2 || G == 4 || G == 8 || G == 16)) return DA_ERR_UNSUPPORTED;
    if (s.batch > kMaxBatch || s.num_q_heads > kMaxQHeads) return DA_ERR_UNSUPPORTED;
    if (static_cast<long long>(s.batch) * s.num_kv_heads > kMaxSegments) return DA_ERR_UNSUPPORTED;
    return DA_OK;
}

template <int NT, bool RING, bool ROPE, bool KV8 = false, int CPS = 1, bool MT = false>
int launch_attn(const CUtensorMap &mk, const CUtensorMap &mv, const Params &prm, int dev, cudaStream_t stream) {
    if (sm_count(dev) > kMaxSms) return DA_ERR_UNSUPPORTED;  // the kernel keeps a boundary per CTA
    static_assert(CPS == 1 || (KV8 && NT == 1), "two CTAs per SM: fp8 kernel with 8-head groups only");
    const size_t smem = SmemLayout<NT, ROPE, KV8, CPS, MT>::bytes;
    const size_t smem_max = smem;
    auto kern = decode_attn_kernel<NT, RING, ROPE, KV8, CPS, MT>;
    const int idx = (MT ? 32 : 0) + (CPS - 1) * 16 + (NT - 1) * 8 + (RING ? 4 : 0) + (ROPE ? 2 : 0) + (KV8 ? 1 : 0);
    if (!g_dev[dev].attr_set[idx].load(std::memory_order_acquire)) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_max));
        if (e != cudaSuccess) return set_cuda_error(e);
        g_dev[dev].attr_set[idx].store(true, std::memory_order_release);
    }
    // Programmatic dependent launch: the grid may start (and run its input-free set-up)
    // while the previous kernel of the stream drains; it waits for that kernel before
    // touching memory (griddepcontrol.wait).
    cudaLaunchConfig_t cfg = {};
    // the row groups of a several-token call split the grid evenly
    cfg.gridDim = dim3(sm_count(dev) * CPS / prm.ngrp * prm.ngrp);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mk, mv, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e);
    return DA_OK;
}

int prepare_workspace(int dev, int G, cudaStream_t stream, float **part, int **counters) {
    const size_t need = workspace_for(G, sm_count(dev));
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        int rc = workspace_locked(dev, stream, false, need, &ws);
        if (rc != DA_OK) return rc;
    }
    *counters = static_cast<int *>(ws);
    *part = reinterpret_cast<float *>(static_cast<char *>(ws) + kCounterBytes);
    return DA_OK;
}

// Testing aid (decode_attn_test_expire_wait): the tile wait at which the next one-token
// call's first worker gives up; -1 = none. Taken (and cleared) by that call.
std::atomic<int> g_expire_next{-1};
// decode_attn_set_early_inputs: what is read before the wait for the previous kernel
std::atomic<int> g_early_inputs{0};

int run_attention(bool ring, const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                  const int32_t *block_table, const int32_t *seq_lens, const float *sinks, int window,
                  float scale, void *out, const da_shape &s, int page_size, int max_pages, int num_pages,
                  int max_seq_len, void *stream_v, const float *rope_cos = nullptr,
                  const float *rope_sin = nullptr, int max_position = 0, bool kv8 = false) {
    int rc = check_shape(s);
    if (rc != DA_OK) return rc;
    if (!q || !k_cache || (!kv8 && !v_cache) || !seq_lens || !out) return DA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return DA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || (!kv8 && !aligned16(v_cache)) || !aligned16(out) ||
        (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return DA_ERR_INVALID_ARG;
    if (!(scale == scale)) return DA_ERR_INVALID_ARG;
    if ((rope_cos == nullptr) != (rope_sin == nullptr)) return DA_ERR_INVALID_ARG;
    if (kv8 && ring && window % kPage != 0) return DA_ERR_UNSUPPORTED;
    if (rope_cos && (max_position <= 0 || !aligned16(rope_cos) || !aligned16(rope_sin))) return DA_ERR_INVALID_ARG;
    const int G = s.num_q_heads / s.num_kv_heads;
    if (ring) {
        if (window < kPage) return window <= 0 ? DA_ERR_INVALID_ARG : DA_ERR_UNSUPPORTED;
    } else {
        if (!block_table || window < 0 || max_pages <= 0 || num_pages <= 0 || max_seq_len < 0)
            return DA_ERR_INVALID_ARG;
        if (page_size != kPage) return DA_ERR_UNSUPPORTED;
        if (static_cast<long long>(max_pages) * kPage < max_seq_len) return DA_ERR_INVALID_ARG;
        if (static_cast<long long>(num_pages) * s.num_kv_heads > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
    }
    if (s.batch == 0) return DA_OK;
    int dev;
    rc = current_device(&dev);
    if (rc != DA_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);

    Params prm;
    prm.q = static_cast<const __nv_bfloat16 *>(q);
    prm.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    prm.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    prm.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    prm.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    prm.block_table = block_table;
    prm.seq_lens = seq_lens;
    prm.sinks = sinks;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.B = s.batch;
    prm.Hq = s.num_q_heads;
    prm.Hkv = s.num_kv_heads;
    prm.G = G;
    prm.window = window;
    prm.max_pages = ring ? 0 : max_pages;
    prm.num_pages = ring ? 0 : num_pages;
    prm.max_seq_len = ring ? 0 : max_seq_len;
    prm.scale_log2 = scale * kLog2e;
    prm.rope_cos = rope_cos;
    prm.rope_sin = rope_sin;
    prm.max_position = max_position;
    prm.T = 1;
    prm.q_lens = nullptr;
    prm.ngrp = 1;
    prm.expire_at = g_expire_next.exchange(-1);
    prm.head_scratch = nullptr;
    prm.early = g_early_inputs.load();
    rc = prepare_workspace(dev, G, stream, &prm.part, &prm.counters);
    if (rc != DA_OK) return rc;

    CUtensorMap mk, mv;
    if (kv8) {  // contiguous blocks, copied without tensor maps
        memset(&mk, 0, sizeof mk);
        memset(&mv, 0, sizeof mv);
    } else {
        const uint64_t rows = ring ? static_cast<uint64_t>(window) : static_cast<uint64_t>(kPage);
        const uint64_t slices = ring ? static_cast<uint64_t>(s.batch) * s.num_kv_heads
                                     : static_cast<uint64_t>(num_pages) * s.num_kv_heads;
        if (!make_kv_map(&mk, k_cache, rows, slices) || !make_kv_map(&mv, v_cache, rows, slices)) {
            snprintf(t_err, sizeof t_err, "CUDA error: tensor map encoding failed");
            return DA_ERR_CUDA;
        }
    }
    if (kv8) {
        if (G <= 8) {
            // an upper bound of the call's tiles, from shapes only (seq_lens stay on the device)
            long long per_seq;
            if (ring) {
                per_seq = window / kPage;
            } else {
                const int span = window > 0 ? std::min(window, max_seq_len) : max_seq_len;
                per_seq = (span + kPage - 1) / kPage + 1;
            }
            const bool two = static_cast<long long>(s.batch) * s.num_kv_heads * per_seq >= DA_FP8_2CTA_MIN_TILES;
            if (rope_cos != nullptr) {
                if (two)
                    return ring ? launch_attn<1, true, true, true, 2>(mk, mv, prm, dev, stream)
                                : launch_attn<1, false, true, true, 2>(mk, mv, prm, dev, stream);
                return ring ? launch_attn<1, true, true, true>(mk, mv, prm, dev, stream)
                            : launch_attn<1, false, true, true>(mk, mv, prm, dev, stream);
            }
            if (two)
                return ring ? launch_attn<1, true, false, true, 2>(mk, mv, prm, dev, stream)
                            : launch_attn<1, false, false, true, 2>(mk, mv, prm, dev, stream);
            return ring ? launch_attn<1, true, false, true>(mk, mv, prm, dev, stream)
                        : launch_attn<1, false, false, true>(mk, mv, prm, dev, stream);
        }
        if (rope_cos != nullptr)
            return ring ? launch_attn<2, true, true, true>(mk, mv, prm, dev, stream)
                        : launch_attn<2, false, true, true>(mk, mv, prm, dev, stream);
        return ring ? launch_attn<2, true, false, true>(mk, mv, prm, dev, stream)
                    : launch_attn<2, false, false, true>(mk, mv, prm, dev, stream);
    }
    if (rope_cos != nullptr) {
        if (G <= 8)
            return ring ? launch_attn<1, true, true>(mk, mv, prm, dev, stream)
                        : launch_attn<1, false, true>(mk, mv, prm, dev, stream);
        return ring ? launch_attn<2, true, true>(mk, mv, prm, dev, stream)
                    : launch_attn<2, false, true>(mk, mv, prm, dev, stream);
    }
    if (G <= 8)
        return ring ? launch_attn<1, true, false>(mk, mv, prm, dev, stream)
                    : launch_attn<1, false, false>(mk, mv, prm, dev, stream);
    return ring ? launch_attn<2, true, false>(mk, mv, prm, dev, stream)
                : launch_attn<2, false, false>(mk, mv, prm, dev, stream);
}

// ------------------------------------------------------------------ several query tokens: host side
// k_new / v_new [B][T][Hkv][64] bf16 seen as tiles of 16 tokens of one KV head:
// dims {64, Hkv, T, B}, box {64, 1, 16, 1}, 128-byte swizzle (the cache tiles' layout).
bool make_new_map(CUtensorMap *map, const void *base, int Hkv, int T, int B) {
    const int kind = 1000 + Hkv;  // cache key: never equal to a cache view's kind
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < kMapCache; ++i) {
        const MapCacheEntry &e = g_maps[i];
        if (e.base == base && e.kind == kind && e.rows == static_cast<uint64_t>(T) &&
            e.slices == static_cast<uint64_t>(B)) {
            *map = e.map;
            return true;
        }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(Hkv),
                                static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(Hkv) * kD * 2,
                                   static_cast<cuuint64_t>(T) * Hkv * kD * 2};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(kD), 1, static_cast<cuuint32_t>(kPage), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    MapCacheEntry &e = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    e.base = const_cast<void *>(base);
    e.kind = kind;
    e.rows = static_cast<uint64_t>(T);
    e.slices = static_cast<uint64_t>(B);
    e.map = *map;
    return true;
}

// How a multi-token call is cut: warps per CTA, query-row blocks, key splits and tiles per
// split. A function of the shape, T, the window or longest sequence and the SM count only
// (never of the lengths), so the workspace can be sized ahead and the call captured.
struct MultiPlan {
    bool dec;          // the decode kernel's several-token form (paged, T <= 4, T G <= 32)
    bool tc;           // the tcgen05 kernel (128 query rows per CTA) or the mma.sync one
    bool defer;        // many key splits: multi_combine_kernel folds the partials
    long long groups;  // (sequence, KV head, query-row block) triples, one counter each
    int nw, rows, row_blocks, splits, chunk;
    size_t counter_bytes, part_bytes;
};

// Paged calls with at least this many query rows per (sequence, KV head) run on tcgen05
// (measured: from 64 rows on it beats the mma.sync kernel; the ring's few keys per row block
// do not fill its pipeline, so ring calls stay on mma.sync).
#ifndef DA_MULTI_TC_MIN_ROWS
#define DA_MULTI_TC_MIN_ROWS 64
#endif
#ifndef DA_MULTI_DECODE_ROUTE  // 0: every multi-token call on the row-block kernels
#define DA_MULTI_DECODE_ROUTE 1
#endif
#ifndef DA_MULTI_DECODE_MAX_ROWS  // query rows per KV head the decode kernel takes (16 or 32)
#define DA_MULTI_DECODE_MAX_ROWS 32
#endif
// 17 to 32 rows per KV head: 1 = one warp takes all of them (four n-tiles), 0 = two row
// groups of 16 on pairs of CTAs that cover the same units
#ifndef DA_MULTI_DECODE_NT4
#define DA_MULTI_DECODE_NT4 1
#endif
// Key splits from which the partials are folded by a kernel of their own (spread over many
// SMs) rather than by the last CTA of each row block
#ifndef DA_MULTI_DEFER_SPLITS
#define DA_MULTI_DEFER_SPLITS 8
#endif
#ifndef DA_MULTI_TC_CTAS_PER_SM  // tcgen05 calls: key splits aim at this many CTAs per SM
#define DA_MULTI_TC_CTAS_PER_SM 2
#endif
// Key tiles per CTA of the mma.sync kernel at most: a long sequence is split however many
// groups there are (the host knows only the longest possible length; CTAs past a shorter
// sequence's end exit at once). Not for tcgen05 CTAs, whose set-up (TMEM, staged queries)
// makes more, shorter CTAs slower (measured).
#ifndef DA_MULTI_MAX_CHUNK
#define DA_MULTI_MAX_CHUNK 128
#endif
#ifndef DA_MULTI_TC_MAX_CHUNK  // the same cap for tcgen05 CTAs, whose set-up is heavier
#define DA_MULTI_TC_MAX_CHUNK 1024
#endif
// Key tiles per split at least, where the SM target alone would cut finer: a split of fewer
// keys saves less than its partial and the combine cost (a 128-token window is never split)
#ifndef DA_MULTI_MIN_CHUNK
#define DA_MULTI_MIN_CHUNK 16
#endif

MultiPlan multi_plan(const da_shape &s, int T, bool ring, int window, int max_seq_len, int sms) {
    MultiPlan m;
    const int G = s.num_q_heads / s.num_kv_heads;
    const long long TG = static_cast<long long>(T) * G;
    // Up to kMaxNewMT query tokens of at most 32 rows per KV head on a paged cache take the
    // decode kernel's device-balanced split (measured faster than the row-block kernel; the
    // ring keeps the row-block kernel, whose separate append leaves the cells the earlier
    // tokens read). Over 16 rows, one warp takes all 32 (four n-tiles), or (switch off) two
    // row groups of 16 on pairs of CTAs that cover the same units.
    m.dec = !ring && T <= kMaxNewMT && TG <= DA_MULTI_DECODE_MAX_ROWS && DA_MULTI_DECODE_ROUTE;
    if (m.dec) {  // counters (one set per row group) in the fixed region, then one pair of
                  // partial slots per CTA
        m.tc = false;
        m.defer = false;
        m.nw = kWarps;
        const bool nt4 = DA_MULTI_DECODE_NT4 && TG > 16;
        m.rows = TG <= 8 ? 8 : nt4 ? 32 : 16;
        m.row_blocks = nt4 ? 1 : static_cast<int>((TG + 15) / 16);
        m.splits = 1;
        m.chunk = 0;
        m.groups = static_cast<long long>(s.batch) * s.num_kv_heads * m.row_blocks;
        m.counter_bytes = static_cast<size_t>(kMMaxGroups) * sizeof(int);
        // the CTAs' partial slots; with 32 rows also every warp's saved first-segment state
        m.part_bytes = static_cast<size_t>(sms) * 2 * slot_floats(m.rows) * sizeof(float) +
                       (m.rows == 32 ? static_cast<size_t>(sms) * kWarps * 32 * (4 * 16 + 4 * 4) * sizeof(float) : 0);
        return m;
    }
    m.tc = !ring && TG >= DA_MULTI_TC_MIN_ROWS;
    if (m.tc) {
        m.nw = kTcWarps;
        m.rows = kTcRows;
    } else {
        m.nw = static_cast<int>(std::min<long long>(kMWarps, (TG + kMRowsPerWarp - 1) / kMRowsPerWarp));
        m.rows = kMRowsPerWarp * m.nw;
    }
    m.row_blocks = static_cast<int>((TG + m.rows - 1) / m.rows);
    const long long cached = ring ? (window + kPage - 1) / kPage : (max_seq_len + kPage - 1) / kPage;
    const long long max_tiles = cached + (T + kPage - 1) / kPage + 1;
    const long long groups = static_cast<long long>(s.batch) * s.num_kv_heads * m.row_blocks;
    const long long target = static_cast<long long>(m.tc ? DA_MULTI_TC_CTAS_PER_SM : DA_MULTI_CTAS_PER_SM) * sms;
    long long sp = std::max<long long>(1, (target + groups - 1) / std::max<long long>(1, groups));
    sp = std::min(sp, std::max<long long>(1, max_tiles / DA_MULTI_MIN_CHUNK));
    sp = std::max(sp, (max_tiles + kMMaxChunk - 1) / kMMaxChunk);  // a CTA's pages fit its smem
    const long long cap = m.tc ? DA_MULTI_TC_MAX_CHUNK : DA_MULTI_MAX_CHUNK;
    sp = std::max(sp, (max_tiles + cap - 1) / cap);
    sp = std::min(sp, max_tiles);
    m.chunk = static_cast<int>((max_tiles + sp - 1) / sp);
    m.splits = static_cast<int>((max_tiles + m.chunk - 1) / m.chunk);
    m.defer = m.splits >= DA_MULTI_DEFER_SPLITS;
    // the counters sit in a fixed region: a later call with more groups must find zeros
    // there, not the partials of an earlier call with fewer
    m.groups = groups;
    m.counter_bytes = static_cast<size_t>(kMMaxGroups) * sizeof(int);
    m.part_bytes =
        m.splits > 1 ? static_cast<size_t>(groups) * m.splits * m.rows * kMSlotFloats * sizeof(float) : 0;
    return m;
}

// Bytes of the rotated q and k_new of a several-token call with the rotary embedding (they
// follow the counters and partials in the multi-token workspace, 256-byte aligned).
size_t rope_scratch_bytes(const da_shape &s, int T) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t rows = static_cast<size_t>(s.batch) * T;
    return up(rows * s.num_q_heads * kD * 2) + up(rows * s.num_kv_heads * kD * 2);
}

int run_multi(bool ring, const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
              const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens, const float *sinks,
              int window, float scale, void *out, const da_shape &s, int T, int page_size, int max_pages,
              int num_pages, int max_seq_len, void *stream_v, const float *rope_cos = nullptr,
              const float *rope_sin = nullptr, int max_position = 0) {
    int rc = check_shape(s);
    if (rc != DA_OK) return rc;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !seq_lens || !out) return DA_ERR_INVALID_ARG;
    const bool rope = rope_cos != nullptr || rope_sin != nullptr;
    if (rope && (!rope_cos || !rope_sin || !aligned16(rope_cos) || !aligned16(rope_sin) || max_position <= 0))
        return DA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(out))
        return DA_ERR_INVALID_ARG;
    if (!(scale == scale) || T <= 0) return DA_ERR_INVALID_ARG;
    if (T > kMMaxTokens) return DA_ERR_UNSUPPORTED;
    if (ring) {
        if (window < kPage) return window <= 0 ? DA_ERR_INVALID_ARG : DA_ERR_UNSUPPORTED;
    } else {
        if (!block_table || window < 0 || max_pages <= 0 || num_pages <= 0 || max_seq_len < 0)
            return DA_ERR_INVALID_ARG;
        if (page_size != kPage) return DA_ERR_UNSUPPORTED;
        if (static_cast<long long>(max_pages) * kPage < max_seq_len) return DA_ERR_INVALID_ARG;
        if (static_cast<long long>(num_pages) * s.num_kv_heads > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
    }
    if (s.batch == 0) return DA_OK;
    int dev;
    rc = current_device(&dev);
    if (rc != DA_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const MultiPlan m = multi_plan(s, T, ring, window, max_seq_len, sm_count(dev));
    if (static_cast<long long>(m.splits) * m.row_blocks > 0x7fffffffLL || m.groups > kMMaxGroups)
        return DA_ERR_UNSUPPORTED;
    void *ws = nullptr;
    const size_t rope_off = (m.counter_bytes + m.part_bytes + 255) & ~static_cast<size_t>(255);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        rc = workspace_locked(dev, stream, true, rope ? rope_off + rope_scratch_bytes(s, T) : m.counter_bytes + m.part_bytes,
                              &ws);
        if (rc != DA_OK) return rc;
    }
    if (rope) {  // rotate q and k_new into the workspace; the attention reads them from there
        __nv_bfloat16 *q_rot = reinterpret_cast<__nv_bfloat16 *>(static_cast<char *>(ws) + rope_off);
        __nv_bfloat16 *k_rot = q_rot + ((static_cast<size_t>(s.batch) * T * s.num_q_heads * kD + 127) & ~static_cast<size_t>(127));
        rope_multi_kernel<<<dim3(static_cast<unsigned>(T), static_cast<unsigned>(s.batch)), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k_new), seq_lens, q_lens,
            rope_cos, rope_sin, max_position, T, s.num_q_heads, s.num_kv_heads, q_rot, k_rot);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_cuda_error(e);
        q = q_rot;
        k_new = k_rot;
    }
    if (m.dec) {  // the decode kernel's several-token form, on this workspace
        Params dp;
        dp.q = static_cast<const __nv_bfloat16 *>(q);
        dp.k_new = static_cast<const __nv_bfloat16 *>(k_new);
        dp.v_new = static_cast<const __nv_bfloat16 *>(v_new);
        dp.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
        dp.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
        dp.block_table = block_table;
        dp.seq_lens = seq_lens;
        dp.sinks = sinks;
        dp.out = static_cast<__nv_bfloat16 *>(out);
        dp.counters = static_cast<int *>(ws);
        dp.part = reinterpret_cast<float *>(static_cast<char *>(ws) + m.counter_bytes);
        dp.B = s.batch;
        dp.Hq = s.num_q_heads;
        dp.Hkv = s.num_kv_heads;
        dp.G = s.num_q_heads / s.num_kv_heads;
        dp.window = window;
        dp.max_pages = max_pages;
        dp.num_pages = num_pages;
        dp.max_seq_len = max_seq_len;
        dp.scale_log2 = scale * kLog2e;
        dp.rope_cos = nullptr;
        dp.rope_sin = nullptr;
        dp.max_position = 0;
        dp.T = T;
        dp.q_lens = q_lens;
        dp.ngrp = m.row_blocks;
        dp.expire_at = -1;
        dp.head_scratch = m.rows == 32 ? dp.part + static_cast<size_t>(sm_count(dev)) * 2 * slot_floats(m.rows) : nullptr;
        dp.early = g_early_inputs.load();
        CUtensorMap mk, mv;
        const uint64_t slices = static_cast<uint64_t>(num_pages) * s.num_kv_heads;
        if (!make_kv_map(&mk, k_cache, kPage, slices) || !make_kv_map(&mv, v_cache, kPage, slices)) {
            snprintf(t_err, sizeof t_err, "CUDA error: tensor map encoding failed");
            return DA_ERR_CUDA;
        }
        return m.rows == 8    ? launch_attn<1, false, false, false, 1, true>(mk, mv, dp, dev, stream)
               : m.rows == 16 ? launch_attn<2, false, false, false, 1, true>(mk, mv, dp, dev, stream)
                              : launch_attn<4, false, false, false, 1, true>(mk, mv, dp, dev, stream);
    }
    MultiParams prm;
    prm.q = static_cast<const __nv_bfloat16 *>(q);
    prm.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    prm.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.block_table = block_table;
    prm.seq_lens = seq_lens;
    prm.q_lens = q_lens;
    prm.sinks = sinks;
    prm.scale_log2 = scale * kLog2e;
    prm.B = s.batch;
    prm.Hq = s.num_q_heads;
    prm.Hkv = s.num_kv_heads;
    prm.G = s.num_q_heads / s.num_kv_heads;
    prm.T = T;
    prm.window = window;
    prm.max_pages = ring ? 0 : max_pages;
    prm.num_pages = ring ? 0 : num_pages;
    prm.max_seq_len = ring ? 0 : max_seq_len;
    prm.row_blocks = m.row_blocks;
    prm.splits = m.splits;
    prm.chunk = m.chunk;
    prm.counters = static_cast<int *>(ws);
    prm.part = reinterpret_cast<float *>(static_cast<char *>(ws) + m.counter_bytes);
    prm.defer = m.defer ? 1 : 0;

    CUtensorMap mk, mv, nk, nv;
    const uint64_t rows = ring ? static_cast<uint64_t>(window) : static_cast<uint64_t>(kPage);
    const uint64_t slices = ring ? static_cast<uint64_t>(s.batch) * s.num_kv_heads
                                 : static_cast<uint64_t>(num_pages) * s.num_kv_heads;
    if (!make_kv_map(&mk, k_cache, rows, slices) || !make_kv_map(&mv, v_cache, rows, slices) ||
        !make_new_map(&nk, k_new, s.num_kv_heads, T, s.batch) ||
        !make_new_map(&nv, v_new, s.num_kv_heads, T, s.batch)) {
        snprintf(t_err, sizeof t_err, "CUDA error: tensor map encoding failed");
        return DA_ERR_CUDA;
    }
    const bool small = !m.tc && m.nw <= 2;
    auto kern = m.tc ? (ring ? multi_tc_kernel<true> : multi_tc_kernel<false>)
                     : small ? (ring ? multi_attn_kernel<true, 2> : multi_attn_kernel<false, 2>)
                             : (ring ? multi_attn_kernel<true, kMWarps> : multi_attn_kernel<false, kMWarps>);
    const int smem = m.tc ? kTcSmem : small ? MultiShape<2>::kSmem : MultiShape<kMWarps>::kSmem;
    const int aidx = (ring ? 1 : 0) + (m.tc ? 2 : 0) + (small ? 4 : 0);
    if (!g_dev[dev].multi_attr_set[aidx].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)  // room for as many resident CTAs as the registers allow
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return set_cuda_error(e);
        g_dev[dev].multi_attr_set[aidx].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(m.splits * m.row_blocks), static_cast<unsigned>(s.num_kv_heads),
                       static_cast<unsigned>(s.batch));
    cfg.blockDim = dim3(32 * m.nw);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mk, mv, nk, nv, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e);
    if (m.defer) {  // the fold of the split partials: one warp per query row
        cudaLaunchConfig_t cc = {};
        cc.gridDim = dim3(static_cast<unsigned>(m.row_blocks * ((m.rows + kCombWarps - 1) / kCombWarps)),
                          static_cast<unsigned>(s.num_kv_heads), static_cast<unsigned>(s.batch));
        cc.blockDim = dim3(kCombWarps * 32);
        cc.dynamicSmemBytes = 0;
        cc.stream = stream;
        cc.attrs = attr;
        cc.numAttrs = 1;
        e = cudaLaunchKernelEx(&cc, multi_combine_kernel, prm, m.rows, ring ? 1 : 0);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return set_cuda_error(e);
    }
    // the append, after every read of the cache (an ordinary launch: it waits for the kernel)
    kv_append_multi_kernel<<<s.batch, 256, 0, stream>>>(
        prm.k_new, prm.v_new, static_cast<__nv_bfloat16 *>(k_cache), static_cast<__nv_bfloat16 *>(v_cache),
        ring ? nullptr : block_table, seq_lens, q_lens, T, s.num_kv_heads, ring ? window : 0, prm.max_pages,
        prm.num_pages, prm.max_seq_len);
    e = cudaGetLastError();
    return e == cudaSuccess ? DA_OK : set_cuda_error(e);
}

// ------------------------------------------------------------------ allocation-free variant
// Some callers cannot allocate device memory at the point where they run decode
// attention: a runtime whose memory is handed out up front by its own pool, a plugin
// that is not allowed to call cudaMalloc, or code that must not synchronise the device
// (cudaMalloc/cudaFree may). For them, decode_attn_paged_noalloc keeps its scratch (the
// split partials and the arrival counters) in the fixed array below instead of the
// library workspace. The array is part of the module image: every GPU that loads this
// library holds its 1.3 MiB until the process exits.
constexpr int kNoAllocMaxCtas = 160;        // one CTA per SM; GB300 has 152 SMs
constexpr int kNoAllocMaxSegments = 4096;   // batch * KV heads
constexpr size_t kNoAllocCounterBytes = static_cast<size_t>(kNoAllocMaxSegments) * sizeof(int);
constexpr size_t kNoAllocPartialFloats = 2 * 16 + 16 * kD;  // one partial slot at 16 heads per group
constexpr size_t kNoAllocScratchBytes =
    kNoAllocCounterBytes + static_cast<size_t>(kNoAllocMaxCtas) * 2 * kNoAllocPartialFloats * sizeof(float);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void *g_noalloc_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device
std::mutex g_noalloc_mu;

// The array's name means nothing to host code; its device address is looked up once
// per device, with that device current. The lookup may load the module on the device, so
// a first call made while `stream` is capturing a graph is refused (DA_ERR_WORKSPACE).
int noalloc_scratch(int dev, cudaStream_t stream, void **addr) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t ce = cudaStreamIsCapturing(stream, &cs);
        if (ce != cudaSuccess) return set_cuda_error(ce);
        if (cs != cudaStreamCaptureStatusNone) return DA_ERR_WORKSPACE;
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return set_cuda_error(e);
        g_noalloc_addr[dev] = ptr;
    }
    *addr = g_noalloc_addr[dev];
    return DA_OK;
}

int run_paged_noalloc(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                      const int32_t *block_table, const int32_t *seq_lens, const float *sinks, int window,
                      float scale, void *out, const da_shape &s, int page_size, int max_pages, int num_pages,
                      int max_seq_len, void *stream_v) {
    int rc = check_shape(s);
    if (rc != DA_OK) return rc;
    if (!q || !k_cache || !v_cache || !seq_lens || !out || !block_table) return DA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return DA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return DA_ERR_INVALID_ARG;
    if (!(scale == scale)) return DA_ERR_INVALID_ARG;
    if (window < 0 || max_pages <= 0 || num_pages <= 0 || max_seq_len < 0) return DA_ERR_INVALID_ARG;
    if (page_size != kPage) return DA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_pages) * kPage < max_seq_len) return DA_ERR_INVALID_ARG;
    if (static_cast<long long>(num_pages) * s.num_kv_heads > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
    if (static_cast<long long>(s.batch) * s.num_kv_heads > kNoAllocMaxSegments) return DA_ERR_SCRATCH_LIMIT;
    if (s.batch == 0) return DA_OK;
    int dev;
    rc = current_device(&dev);
    if (rc != DA_OK) return rc;
    if (sm_count(dev) > kNoAllocMaxCtas) return DA_ERR_SCRATCH_LIMIT;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    void *scratch = nullptr;
    rc = noalloc_scratch(dev, stream, &scratch);
    if (rc != DA_OK) return rc;

    Params prm;
    prm.q = static_cast<const __nv_bfloat16 *>(q);
    prm.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    prm.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    prm.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    prm.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    prm.block_table = block_table;
    prm.seq_lens = seq_lens;
    prm.sinks = sinks;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.B = s.batch;
    prm.Hq = s.num_q_heads;
    prm.Hkv = s.num_kv_heads;
    prm.G = s.num_q_heads / s.num_kv_heads;
    prm.window = window;
    prm.max_pages = max_pages;
    prm.num_pages = num_pages;
    prm.max_seq_len = max_seq_len;
    prm.scale_log2 = scale * kLog2e;
    prm.rope_cos = nullptr;
    prm.rope_sin = nullptr;
    prm.max_position = 0;
    prm.T = 1;
    prm.q_lens = nullptr;
    prm.ngrp = 1;
    prm.expire_at = -1;
    prm.head_scratch = nullptr;
    prm.early = g_early_inputs.load();
    prm.counters = static_cast<int *>(scratch);
    prm.part = reinterpret_cast<float *>(static_cast<char *>(scratch) + kNoAllocCounterBytes);
    // The array keeps whatever the previous call left: the arrival counters this call
    // uses must start at zero. (The partials need no clearing; each is written before
    // it is read.)
    cudaError_t e = cudaMemsetAsync(prm.counters, 0, static_cast<size_t>(s.batch) * s.num_kv_heads * sizeof(int),
                                    stream);
    if (e != cudaSuccess) return set_cuda_error(e);

    CUtensorMap mk, mv;
    const uint64_t slices = static_cast<uint64_t>(num_pages) * s.num_kv_heads;
    if (!make_kv_map(&mk, k_cache, kPage, slices) || !make_kv_map(&mv, v_cache, kPage, slices)) {
        snprintf(t_err, sizeof t_err, "CUDA error: tensor map encoding failed");
        return DA_ERR_CUDA;
    }
    return prm.G <= 8 ? launch_attn<1, false, false>(mk, mv, prm, dev, stream)
                      : launch_attn<2, false, false>(mk, mv, prm, dev, stream);
}

}  // namespace

// ------------------------------------------------------------------ C ABI
extern "C" {

int decode_attn_paged(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                      const int32_t *block_table, const int32_t *seq_lens, const float *sinks, int window,
                      float scale, void *out, da_shape s, int page_size, int max_pages_per_seq, int num_pages,
                      int max_seq_len, void *stream) {
    return run_attention(false, q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks, window, scale,
                         out, s, page_size, max_pages_per_seq, num_pages, max_seq_len, stream);
}

int decode_attn_ring(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                     const int32_t *seq_lens, const float *sinks, int window, float scale, void *out, da_shape s,
                     void *stream) {
    return run_attention(true, q, k_new, v_new, k_cache, v_cache, nullptr, seq_lens, sinks, window, scale, out, s,
                         kPage, 0, 0, 0, stream);
}

int decode_attn_paged_rope(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens, const float *sinks,
                           const float *rope_cos, const float *rope_sin, int max_position, int window,
                           float scale, void *out, da_shape s, int page_size, int max_pages_per_seq,
                           int num_pages, int max_seq_len, void *stream) {
    if (!rope_cos || !rope_sin) return DA_ERR_INVALID_ARG;
    return run_attention(false, q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks, window, scale,
                         out, s, page_size, max_pages_per_seq, num_pages, max_seq_len, stream, rope_cos, rope_sin,
                         max_position);
}

int decode_attn_ring_rope(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          const int32_t *seq_lens, const float *sinks, const float *rope_cos,
                          const float *rope_sin, int max_position, int window, float scale, void *out,
                          da_shape s, void *stream) {
    if (!rope_cos || !rope_sin) return DA_ERR_INVALID_ARG;
    return run_attention(true, q, k_new, v_new, k_cache, v_cache, nullptr, seq_lens, sinks, window, scale, out, s,
                         kPage, 0, 0, 0, stream, rope_cos, rope_sin, max_position);
}

int decode_attn_paged_fp8(const void *q, const void *k_new, const void *v_new, void *kv_cache,
                          const int32_t *block_table, const int32_t *seq_lens, const float *sinks, int window,
                          float scale, void *out, da_shape s, int page_size, int max_pages_per_seq, int num_pages,
                          int max_seq_len, void *stream) {
    return run_attention(false, q, k_new, v_new, kv_cache, nullptr, block_table, seq_lens, sinks, window, scale,
                         out, s, page_size, max_pages_per_seq, num_pages, max_seq_len, stream, nullptr, nullptr, 0,
                         true);
}

int decode_attn_ring_fp8(const void *q, const void *k_new, const void *v_new, void *kv_cache,
                         const int32_t *seq_lens, const float *sinks, int window, float scale, void *out,
                         da_shape s, void *stream) {
    return run_attention(true, q, k_new, v_new, kv_cache, nullptr, nullptr, seq_lens, sinks, window, scale, out,
                         s, kPage, 0, 0, 0, stream, nullptr, nullptr, 0, true);
}

int decode_attn_paged_fp8_rope(const void *q, const void *k_new, const void *v_new, void *kv_cache,
                               const int32_t *block_table, const int32_t *seq_lens, const float *sinks,
                               const float *rope_cos, const float *rope_sin, int max_position, int window,
                               float scale, void *out, da_shape s, int page_size, int max_pages_per_seq,
                               int num_pages, int max_seq_len, void *stream) {
    if (!rope_cos || !rope_sin) return DA_ERR_INVALID_ARG;
    return run_attention(false, q, k_new, v_new, kv_cache, nullptr, block_table, seq_lens, sinks, window, scale,
                         out, s, page_size, max_pages_per_seq, num_pages, max_seq_len, stream, rope_cos, rope_sin,
                         max_position, true);
}

int decode_attn_ring_fp8_rope(const void *q, const void *k_new, const void *v_new, void *kv_cache,
                              const int32_t *seq_lens, const float *sinks, const float *rope_cos,
                              const float *rope_sin, int max_position, int window, float scale, void *out,
                              da_shape s, void *stream) {
    if (!rope_cos || !rope_sin) return DA_ERR_INVALID_ARG;
    return run_attention(true, q, k_new, v_new, kv_cache, nullptr, nullptr, seq_lens, sinks, window, scale, out,
                         s, kPage, 0, 0, 0, stream, rope_cos, rope_sin, max_position, true);
}

int kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache, const int32_t *block_table,
              const int32_t *seq_lens, int window, da_shape s, int page_size, int max_pages_per_seq, int num_pages,
              void *stream) {
    if (s.batch < 0 || s.num_kv_heads <= 0 || s.head_dim <= 0) return DA_ERR_INVALID_ARG;
    if (s.head_dim % 8 != 0) return DA_ERR_UNSUPPORTED;
    if (!k_new || !v_new || !k_cache || !v_cache || !seq_lens) return DA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return DA_ERR_INVALID_ARG;
    if (block_table) {
        if (page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0) return DA_ERR_INVALID_ARG;
    } else if (window <= 0) {
        return DA_ERR_INVALID_ARG;
    }
    if (s.batch == 0) return DA_OK;
    kv_append_kernel<<<s.batch, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(k_new), static_cast<const __nv_bfloat16 *>(v_new),
        static_cast<__nv_bfloat16 *>(k_cache), static_cast<__nv_bfloat16 *>(v_cache), block_table, seq_lens,
        s.num_kv_heads, s.head_dim, window, page_size, max_pages_per_seq, num_pages);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DA_OK : set_cuda_error(e);
}

int decode_attn_paged_noalloc(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                              const int32_t *block_table, const int32_t *seq_lens, const float *sinks, int window,
                              float scale, void *out, da_shape s, int page_size, int max_pages_per_seq,
                              int num_pages, int max_seq_len, void *stream) {
    return run_paged_noalloc(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, sinks, window, scale, out,
                             s, page_size, max_pages_per_seq, num_pages, max_seq_len, stream);
}

int decode_attn_paged_multi(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                            const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens,
                            const float *sinks, int window, float scale, void *out, da_shape s, int q_tokens,
                            int page_size, int max_pages_per_seq, int num_pages, int max_seq_len, void *stream) {
    return run_multi(false, q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, q_lens, sinks, window, scale,
                     out, s, q_tokens, page_size, max_pages_per_seq, num_pages, max_seq_len, stream);
}

int decode_attn_ring_multi(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                           const int32_t *seq_lens, const int32_t *q_lens, const float *sinks, int window,
                           float scale, void *out, da_shape s, int q_tokens, void *stream) {
    return run_multi(true, q, k_new, v_new, k_cache, v_cache, nullptr, seq_lens, q_lens, sinks, window, scale, out,
                     s, q_tokens, kPage, 0, 0, 0, stream);
}

int decode_attn_paged_multi_rope(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                 void *v_cache, const int32_t *block_table, const int32_t *seq_lens,
                                 const int32_t *q_lens, const float *sinks, const float *rope_cos,
                                 const float *rope_sin, int max_position, int window, float scale, void *out,
                                 da_shape s, int q_tokens, int page_size, int max_pages_per_seq, int num_pages,
                                 int max_seq_len, void *stream) {
    if (!rope_cos || !rope_sin) return DA_ERR_INVALID_ARG;
    return run_multi(false, q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, q_lens, sinks, window, scale,
                     out, s, q_tokens, page_size, max_pages_per_seq, num_pages, max_seq_len, stream, rope_cos,
                     rope_sin, max_position);
}

int decode_attn_ring_multi_rope(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                void *v_cache, const int32_t *seq_lens, const int32_t *q_lens,
                                const float *sinks, const float *rope_cos, const float *rope_sin,
                                int max_position, int window, float scale, void *out, da_shape s, int q_tokens,
                                void *stream) {
    if (!rope_cos || !rope_sin) return DA_ERR_INVALID_ARG;
    return run_multi(true, q, k_new, v_new, k_cache, v_cache, nullptr, seq_lens, q_lens, sinks, window, scale, out,
                     s, q_tokens, kPage, 0, 0, 0, stream, rope_cos, rope_sin, max_position);
}

size_t decode_attn_multi_workspace_bytes(da_shape s, int q_tokens, int ring_window, int max_seq_len) {
    if (check_shape(s) != DA_OK || q_tokens <= 0 || q_tokens > kMMaxTokens || max_seq_len < 0 || ring_window < 0)
        return 0;
    int dev;
    if (current_device(&dev) != DA_OK) return 0;
    const MultiPlan m = multi_plan(s, q_tokens, ring_window > 0, ring_window, max_seq_len, sm_count(dev));
    // with room for the rotated q and k_new of the calls with the rotary embedding
    return ((m.counter_bytes + m.part_bytes + 255) & ~static_cast<size_t>(255)) + rope_scratch_bytes(s, q_tokens);
}

int decode_attn_multi_launches(da_shape s, int q_tokens, int ring_window, int max_seq_len) {
    if (check_shape(s) != DA_OK || q_tokens <= 0 || q_tokens > kMMaxTokens || max_seq_len < 0 || ring_window < 0)
        return 0;
    int dev;
    if (current_device(&dev) != DA_OK) return 0;
    const MultiPlan m = multi_plan(s, q_tokens, ring_window > 0, ring_window, max_seq_len, sm_count(dev));
    return m.dec ? 1 : 2 + (m.defer ? 1 : 0);
}

int decode_attn_multi_reserve(size_t bytes) {
    int dev;
    int rc = current_device(&dev);
    if (rc != DA_OK) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    return grow_locked(g_dev[dev].ws_multi, bytes);
}

size_t decode_attn_workspace_bytes(da_shape s, int max_seq_len) {
    (void)max_seq_len;
    if (check_shape(s) != DA_OK) return 0;
    int dev;
    if (current_device(&dev) != DA_OK) return 0;
    return workspace_for(s.num_q_heads / s.num_kv_heads, sm_count(dev));
}

int decode_attn_reserve(size_t bytes) {
    int dev;
    int rc = current_device(&dev);
    if (rc != DA_OK) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    return grow_locked(g_dev[dev].ws, bytes);
}

int decode_attn_stream_reserve(void *stream_v, size_t bytes, size_t multi_bytes) {
    int dev;
    int rc = current_device(&dev);
    if (rc != DA_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (cs != cudaStreamCaptureStatusNone) return DA_ERR_WORKSPACE;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_stream_ws.find(stream);
    if (it == g_stream_ws.end()) {
        it = g_stream_ws.emplace(stream, StreamWorkspaces{dev, {}, {}}).first;
        g_n_stream_ws.fetch_add(1, std::memory_order_relaxed);
    } else if (it->second.dev != dev) {
        return DA_ERR_INVALID_ARG;
    }
    rc = grow_locked(it->second.ws, bytes);
    if (rc == DA_OK) rc = grow_locked(it->second.ws_multi, multi_bytes);
    return rc;
}

int decode_attn_stream_release(void *stream_v) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_stream_ws.find(stream);
    if (it == g_stream_ws.end()) return DA_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (cs != cudaStreamCaptureStatusNone) return DA_ERR_WORKSPACE;
    int prev = -1;
    e = cudaGetDevice(&prev);
    if (e == cudaSuccess && prev != it->second.dev) e = cudaSetDevice(it->second.dev);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);  // its calls are done with them
    for (Workspace *w : {&it->second.ws, &it->second.ws_multi}) {
        if (e == cudaSuccess && w->p) {
            e = cudaFree(w->p);
            w->p = nullptr;
            w->bytes = 0;
        }
    }
    if (prev >= 0 && prev != it->second.dev) cudaSetDevice(prev);
    if (e != cudaSuccess) return set_cuda_error(e);
    g_stream_ws.erase(it);
    g_n_stream_ws.fetch_sub(1, std::memory_order_relaxed);
    return DA_OK;
}

int decode_attn_test_expire_wait(int tile) {
    g_expire_next.store(tile < 0 ? -1 : tile);
    return DA_OK;
}

int decode_attn_set_early_inputs(int level) {
    if (level < 0 || level > 2) return DA_ERR_INVALID_ARG;
    return g_early_inputs.exchange(level);
}

int decode_attn_device_status(void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int h = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_status, sizeof h, 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return set_cuda_error(e);
    return static_cast<int>(h & 0x7fffffffu);
}

const char *decode_attn_error_string(int code) {
    switch (code) {
        case DA_OK: return "ok";
        case DA_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size, Hq % Hkv != 0)";
        case DA_ERR_UNSUPPORTED: return "unsupported shape (needs head_dim 64, page 16, G in {1,2,4,8,16}, batch <= 1024, ring window >= 16)";
        case DA_ERR_WORKSPACE: return "workspace too small during stream capture: call decode_attn_reserve() first";
        case DA_ERR_CUDA: return t_err[0] ? t_err : "CUDA error";
        case DA_ERR_SCRATCH_LIMIT:
            return "beyond the fixed scratch of the allocation-free call (batch * kv_heads <= 4096, at most 160 SMs)";
        default: return "unknown error code";
    }
}

}  // extern "C"
