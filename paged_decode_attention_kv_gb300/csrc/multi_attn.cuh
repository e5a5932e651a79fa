// Several query tokens per sequence in one call: speculative verification (the draft
// tokens and the bonus token checked in one step) and chunked prefill appending a run of
// tokens into pages (the teaching repo's chapters "Speculative Decoding" and "Chunked
// Prefill", table "The files" on the page "Run it locally", name both; the plain causal
// reading is used).
//
//   n = q_lens[b] (T when q_lens is null) new tokens at positions base = L - n .. L - 1,
//   L = seq_lens[b]. Query row (t, h), t < n, at position p = base + t attends the
//   positions lo .. p (causal), lo = max(0, p - W + 1) under a window W, else 0.
//   Positions >= base are the new tokens, read from k_new / v_new [B][T][Hkv][64]; the
//   rest come from the cache, which holds the history before the step. Rows t >= n and
//   inactive slots are zero. The new tokens are appended by a second kernel after the
//   attention: in a W-cell ring the early query tokens still read the cells that the later
//   new tokens overwrite. (Paged calls of up to four tokens with T G <= 32 run in the
//   decode kernel instead, append fused: see decode_attn_kernel's MT form.)
//
// Included into decode_attn.cu (inside its anonymous namespace): one translation unit,
// sharing the PTX helpers, the status word and the online-softmax state.
//
// Work split: one CTA per (sequence b, KV head g, block of 8 * warps query rows, key
// split). Query rows of (b, g) are ordered (t, head): row r = t * G + (h - g * G). Each warp
// owns 8 rows (one 8-row n-tile of the same mma.sync shapes as the decode kernel). The
// CTA streams the key tiles of its split through one TMA pipeline that every warp reads:
// cached tiles first (pages, or 16-cell groups of the ring), then tiles of 16 new tokens
// copied straight out of k_new / v_new by a 4-D tensor map. Splits of the same rows leave
// fp32 partials; the CTA with the last ticket (many splits: multi_combine_kernel) folds them with the sink.

#ifndef DA_MULTI_NT
#define DA_MULTI_NT 1
#endif
#ifndef DA_MULTI_WARPS
#define DA_MULTI_WARPS 4
#endif
// Two CTA shapes, by the warps a call needs: up to 2 (at most 16 query rows per sequence and
// KV head: ring calls of one or two tokens at 8 heads per group) and up to 4. Small CTAs gain most from
// residency (many CTAs per SM with 4 stages each), 4-warp CTAs from deep pipelines (8 stages
// at 4 CTAs per SM): measured on both shapes.
#ifndef DA_MULTI_MIN_BLOCKS  // resident 4-warp CTAs per SM the register budget is cut for
#define DA_MULTI_MIN_BLOCKS 4
#endif
#ifndef DA_MULTI_MIN_BLOCKS_SMALL  // the same for 1- and 2-warp CTAs
#define DA_MULTI_MIN_BLOCKS_SMALL 10
#endif
#ifndef DA_MULTI_STAGES
#define DA_MULTI_STAGES 8
#endif
#ifndef DA_MULTI_STAGES_SMALL
#define DA_MULTI_STAGES_SMALL 4
#endif
constexpr int kMNT = DA_MULTI_NT;                 // 8-row n-tiles per warp (8 query rows each)
constexpr int kMRowsPerWarp = 8 * kMNT;
constexpr int kMWarps = DA_MULTI_WARPS;           // query-row warps per CTA at most
constexpr int kMStageBytes = 2 * kTileBytes;      // K tile, then V tile
// the shape of a CTA of at most NW warps: K/V tile pairs in flight, dynamic shared memory,
// resident CTAs per SM for the register budget
template <int NW>
struct MultiShape {
    static constexpr int kStages = NW <= 2 ? DA_MULTI_STAGES_SMALL : DA_MULTI_STAGES;
    static constexpr int kSmem = 1024 + kStages * kMStageBytes + 2 * kStages * 8;
    static constexpr int kMinBlocks = NW <= 2 ? DA_MULTI_MIN_BLOCKS_SMALL : DA_MULTI_MIN_BLOCKS;
};
constexpr int kMSlotFloats = 4 + kD;              // per query row: m, l (log2 units), 2 pad, acc[64]
constexpr int kMAccOff = 4;                       // acc starts 16-byte aligned
constexpr int kMMaxTokens = 4096;                 // query tokens per sequence per call
constexpr int kMMaxGroups = 1 << 18;              // (b, g, row block) counters: a fixed 1 MiB
constexpr int kMMaxChunk = 1024;                  // key tiles per CTA at most (page indices in smem)

struct MultiParams {
    const __nv_bfloat16 *q, *k_new, *v_new;  // [B][T][Hq][64], [B][T][Hkv][64]
    __nv_bfloat16 *out;                      // [B][T][Hq][64]
    const int32_t *block_table, *seq_lens, *q_lens;
    const float *sinks;
    float scale_log2;
    int B, Hq, Hkv, G, T, window, max_pages, num_pages, max_seq_len;
    int row_blocks, splits, chunk;  // query-row blocks per (b, g); key splits; tiles per split
    float *part;                    // [B * Hkv * row_blocks][splits][rows per CTA][kMSlotFloats]
    int *counters;                  // [B * Hkv * row_blocks], zero at rest
    int defer;                      // 1: the split partials are left for multi_combine_kernel
};

// The key tiles of the block of query rows r0 .. r_end - 1 of sequence b: the cached tiles
// (pages pt_lo .. pt_lo + ncache - 1, or the ring's 16-cell groups) come first, then tiles of
// 16 new tokens from nt_base on.
struct MultiKeys {
    int L, n, base;  // length, new tokens (rows t >= n are empty), first new position L - n
    int ncache, pt_lo, nvalid, nt_base, ntiles;
    int ring_off;    // ring: position of cell c = c + ring_off, less W past the newest cell
    bool bad;        // counts out of range: the slot is treated as inactive
};
__device__ __forceinline__ MultiKeys multi_keys(const MultiParams &p, bool ring, int b, int r0, int r_end) {
    MultiKeys k;
    k.L = __ldg(p.seq_lens + b);
    k.n = p.q_lens != nullptr ? __ldg(p.q_lens + b) : p.T;
    k.bad = k.L < 0 || k.n < 0 || k.n > p.T || (k.L > 0 && k.n > k.L);
    if (!ring) k.bad = k.bad || k.L > p.max_seq_len || k.L > p.max_pages * kPage;
    if (k.bad) k.L = 0;
    if (k.L == 0) k.n = 0;
    k.base = k.L - k.n;
    const int W = p.window;
    const int t0 = r0 / p.G;                        // first query token of the block
    const int t1 = min(k.n - 1, (r_end - 1) / p.G);  // last valid one (< t0: none)
    k.ncache = k.pt_lo = k.nvalid = k.nt_base = k.ntiles = k.ring_off = 0;
    if (t1 >= t0) {
        const int lo_min = W > 0 ? max(0, k.base + t0 - W + 1) : 0;
        if (k.base > lo_min) {  // cached keys
            if (ring) {
                k.nvalid = min(k.base, W);
                k.ncache = (k.nvalid + kPage - 1) / kPage;
                k.ring_off = k.base - 1 - (k.base - 1) % W;
            } else {
                k.pt_lo = lo_min / kPage;
                k.ncache = (k.base - 1) / kPage - k.pt_lo + 1;
            }
        }
        k.nt_base = max(0, lo_min - k.base) / kPage;  // first tile of new tokens (16 per tile)
        k.ntiles = k.ncache + t1 / kPage - k.nt_base + 1;
    }
    return k;
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The last split of a row block (or multi_combine_kernel) folds every split's partial (m, l,
// acc per row) of the block's rows rl_lo .. rl_hi - 1 into the output, with the sink. A warp takes kCombRows of the block's rows at a time, so that their
// loads are in flight together (rows one after another left a chain of dependent L2 round
// trips in the CTA that finishes last). First pass: lanes stride over the splits and merge
// (m, l) online, then across the warp. Second pass: lane = (split phase s = lane / 8, output
// octet q = lane % 8) sums the weighted acc[8 q .. 8 q + 7] of splits s, s + 4, ..., and the four
// phases are added across the warp.
constexpr int kCombRows = 4;
__device__ __noinline__ void multi_combine_rows(const MultiParams &p, const float *all, int RB, int r0, int r_end,
                                                int n, int b, int g, int nsplit, int rl_lo, int rl_hi, int warp,
                                                int nw, int lane) {
    auto slot = [&](int sp, int rl) { return all + (static_cast<size_t>(sp) * RB + rl) * kMSlotFloats; };
    const int phase = lane >> 3, q = lane & 7;
    for (int rl0 = rl_lo + warp; rl0 < rl_hi; rl0 += kCombRows * nw) {
        int rl[kCombRows];
        bool row[kCombRows];   // an output row of this block
        bool live[kCombRows];  // a query row (t < n); the other output rows are zeros
        float sg[kCombRows], M[kCombRows], den[kCombRows];
#pragma unroll
        for (int i = 0; i < kCombRows; ++i) {
            rl[i] = rl0 + i * nw;
            const int r = r0 + rl[i];
            const int t = r / p.G;
            row[i] = rl[i] < rl_hi && r < r_end;
            live[i] = row[i] && t < n;
            sg[i] = live[i] && p.sinks != nullptr ? __ldg(p.sinks + g * p.G + (r - t * p.G)) * kLog2e : -INFINITY;
            M[i] = -INFINITY;
            den[i] = 0.f;
        }
        for (int sp = lane; sp < nsplit; sp += 32) {
            float2 ml[kCombRows];
#pragma unroll
            for (int i = 0; i < kCombRows; ++i)
                ml[i] = live[i] ? __ldcg(reinterpret_cast<const float2 *>(slot(sp, rl[i]))) : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int i = 0; i < kCombRows; ++i) {
                if (ml[i].x == -INFINITY) continue;  // a split that saw no key of the row
                const float Mn = fmaxf(M[i], ml[i].x);
                den[i] = den[i] * exp2f(M[i] - Mn) + ml[i].y * exp2f(ml[i].x - Mn);
                M[i] = Mn;
            }
        }
        float Mf[kCombRows], inv[kCombRows];
#pragma unroll
        for (int i = 0; i < kCombRows; ++i) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float Mo = __shfl_xor_sync(0xffffffffu, M[i], off);
                const float Do = __shfl_xor_sync(0xffffffffu, den[i], off);
                const float Mn = fmaxf(M[i], Mo);
                den[i] = Mn == -INFINITY ? 0.f : den[i] * exp2f(M[i] - Mn) + Do * exp2f(Mo - Mn);
                M[i] = Mn;
            }
            // the sink joins the denominator; no key and no sink: a zero row
            Mf[i] = fmaxf(M[i], sg[i]);
            inv[i] = 0.f;
            if (Mf[i] != -INFINITY) {
                const float d = den[i] * exp2f(M[i] - Mf[i]) + (sg[i] == -INFINITY ? 0.f : exp2f(sg[i] - Mf[i]));
                inv[i] = d > 0.f ? 1.f / d : 0.f;
            }
        }
        float o[kCombRows][8];
#pragma unroll
        for (int i = 0; i < kCombRows; ++i)
#pragma unroll
            for (int k = 0; k < 8; ++k) o[i][k] = 0.f;
        for (int sp = phase; sp < nsplit; sp += 4) {
#pragma unroll
            for (int i = 0; i < kCombRows; ++i) {
                if (Mf[i] == -INFINITY) continue;  // the same on every lane: M is an exact maximum
                const float *s = slot(sp, rl[i]);
                const float m = __ldcg(s);
                const float4 a = __ldcg(reinterpret_cast<const float4 *>(s + kMAccOff) + 2 * q);
                const float4 c = __ldcg(reinterpret_cast<const float4 *>(s + kMAccOff) + 2 * q + 1);
                const float w = m == -INFINITY ? 0.f : exp2f(m - Mf[i]);
                o[i][0] += a.x * w;
                o[i][1] += a.y * w;
                o[i][2] += a.z * w;
                o[i][3] += a.w * w;
                o[i][4] += c.x * w;
                o[i][5] += c.y * w;
                o[i][6] += c.z * w;
                o[i][7] += c.w * w;
            }
        }
#pragma unroll
        for (int i = 0; i < kCombRows; ++i)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                o[i][k] += __shfl_xor_sync(0xffffffffu, o[i][k], 8);
                o[i][k] += __shfl_xor_sync(0xffffffffu, o[i][k], 16);
            }
        if (phase == 0) {
#pragma unroll
            for (int i = 0; i < kCombRows; ++i) {
                if (!row[i]) continue;
                const int r = r0 + rl[i], t = r / p.G, hl = r - t * p.G;
                const float f = inv[i];
                const uint4 v = make_uint4(pack_bf16(o[i][0] * f, o[i][1] * f), pack_bf16(o[i][2] * f, o[i][3] * f),
                                           pack_bf16(o[i][4] * f, o[i][5] * f), pack_bf16(o[i][6] * f, o[i][7] * f));
                *reinterpret_cast<uint4 *>(p.out + ((static_cast<size_t>(b) * p.T + t) * p.Hq + g * p.G + hl) * kD +
                                           8 * q) = v;
            }
        }
    }
}

template <bool RING, int NW>
__global__ void __launch_bounds__(NW * 32, MultiShape<NW>::kMinBlocks)
    multi_attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ CUtensorMap tnk, const __grid_constant__ CUtensorMap tnv,
                      const MultiParams p) {
    constexpr int kMStages = MultiShape<NW>::kStages;
    extern __shared__ uint8_t smem_raw[];
    // the 1024-byte aligned base, derived from the shared array itself so that every access
    // through it compiles to a shared-memory instruction (not a generic one)
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t tiles_s = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kMStages * kMStageBytes);
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kMStages);
    __shared__ int s_ticket;
    __shared__ int s_failed;
    __shared__ int s_page[kMMaxChunk];  // this CTA's page indices (paged cache), -1 = bad

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int nw = blockDim.x >> 5;
    const int RB = nw * kMRowsPerWarp;  // query rows per CTA
    const int split = blockIdx.x % p.splits, rb = blockIdx.x / p.splits;
    const int g = blockIdx.y, b = blockIdx.z;

    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tnk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tnv)) : "memory");
        for (int s = 0; s < kMStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, nw);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_failed = 0;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- this sequence's counts and the block's key tiles
    const int W = p.window;
    const int TG = p.T * p.G;
    const int r0 = rb * RB;
    const int r_end = min(r0 + RB, TG);
    const MultiKeys keys = multi_keys(p, RING, b, r0, r_end);
    if (keys.bad && tid == 0 && g == 0 && blockIdx.x == 0) flag_status(DA_STATUS_BAD_SEQ_LEN);
    const int n = keys.n, base = keys.base;
    const int ncache = keys.ncache, pt_lo = keys.pt_lo, nvalid = keys.nvalid, nt_base = keys.nt_base;
    const int ntiles = keys.ntiles, ring_off = keys.ring_off;
    const int kb = split * p.chunk;
    const int ke = min(kb + p.chunk, ntiles);
    const int nsplit = (ntiles + p.chunk - 1) / p.chunk;
    const size_t bg = static_cast<size_t>(b) * p.Hkv + g;
    auto row_off = [&](int r) {  // element offset of query row r of (b, g) in q and out
        const int t = r / p.G, hl = r - t * p.G;
        return ((static_cast<size_t>(b) * p.T + t) * p.Hq + g * p.G + hl) * kD;
    };
    auto out_row = [&](int r) { return p.out + row_off(r); };
    if (kb >= ke) {
        if (ntiles == 0 && split == 0)  // no valid query row here: zeros
            for (int i = tid; i < (r_end - r0) * (kD / 8); i += blockDim.x)
                *reinterpret_cast<uint4 *>(out_row(r0 + i / (kD / 8)) + (i % (kD / 8)) * 8) = make_uint4(0, 0, 0, 0);
        return;
    }
    const int cnt = ke - kb;
    if (!RING) {  // the pages of the CTA's cached tiles, read once
        for (int i2 = tid; i2 < cnt && kb + i2 < ncache; i2 += blockDim.x) {
            int page = __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + pt_lo + kb + i2);
            if (page < 0 || page >= p.num_pages) {
                flag_status(DA_STATUS_BAD_PAGE);
                page = -1;  // out of the map: the copy reads zeros
            }
            s_page[i2] = page;
        }
        __syncthreads();
    }

    // ---- producer (thread 0): tile k into stage s
    const uint64_t policy = evict_first_policy();
    auto issue = [&](int k, int s) {
        const uint32_t fb = full0 + 8 * s;
        const uint32_t dk = tiles_s + s * kMStageBytes, dv = dk + kTileBytes;
        mbar_expect_tx(fb, kMStageBytes);
        if (k < ncache) {
            if (RING) {
                tma_load_3d(dk, &tmk, 0, k * kPage, static_cast<int>(bg), fb, policy);
                tma_load_3d(dv, &tmv, 0, k * kPage, static_cast<int>(bg), fb, policy);
            } else {
                const int page = s_page[k - kb];
                tma_load_3d(dk, &tmk, 0, 0, page * p.Hkv + g, fb, policy);
                tma_load_3d(dv, &tmv, 0, 0, page * p.Hkv + g, fb, policy);
            }
        } else {
            const int tt = (nt_base + k - ncache) * kPage;  // first new token of the tile
            tma_load_4d(dk, &tnk, 0, g, tt, b, fb, policy);
            tma_load_4d(dv, &tnv, 0, g, tt, b, fb, policy);
        }
    };
    int issued = 0;  // tiles issued so far (thread 0)
    if (tid == 0) {
        for (; issued < cnt && issued < kMStages; ++issued) issue(kb + issued, issued);
    }

    // ---- this lane's query rows: n-tile j, column c -> row r0 + RW warp + 8 j + 2 (lane % 4) + c
    int rp[kMNT][2], rlo[kMNT][2];  // position and window start of the row (invalid: no key passes)
    float sig[kMNT][2];
#pragma unroll
    for (int j = 0; j < kMNT; ++j)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int r = r0 + kMRowsPerWarp * warp + 8 * j + 2 * (lane & 3) + c;
            const int t = r / p.G;
            const bool ok = r < r_end && t < n;
            rp[j][c] = ok ? base + t : -1;
            rlo[j][c] = ok && W > 0 ? max(0, base + t - W + 1) : 0;
            const int h = g * p.G + (r - t * p.G);
            sig[j][c] = ok && p.sinks != nullptr ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
        }
    // query fragments (B operand): row r0 + RW warp + 8 j + lane / 4, d = 16 ks + 2 (lane % 4) (+ 8)
    uint32_t qf[kMNT][4][2];
#pragma unroll
    for (int j = 0; j < kMNT; ++j) {
        const int r = r0 + kMRowsPerWarp * warp + 8 * j + (lane >> 2);
        const int t = r / p.G;
        const bool ok = r < r_end && t < n;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) qf[j][ks][0] = qf[j][ks][1] = 0u;
        if (ok) {
            const uint32_t *row = reinterpret_cast<const uint32_t *>(p.q + row_off(r));
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                qf[j][ks][0] = __ldg(row + ks * 8 + (lane & 3));
                qf[j][ks][1] = __ldg(row + ks * 8 + 4 + (lane & 3));
            }
        }
    }

    // per-lane ldmatrix offsets inside a swizzled 16 x 128 B tile (as in the decode kernel)
    const int lj = lane & 7, lmi = lane >> 3;
    const uint32_t k_row = ((lj + ((lmi & 1) << 3)) * 128);
    const int k_cb = lmi >> 1;
    const uint32_t v_row = ((lj + ((lmi >> 1) << 3)) * 128);
    const int v_cb = lmi & 1;

    // position of key row kr of tile k, and whether it is a real key
    auto key_at = [&](int k, int kr, int &j) -> bool {
        if (k < ncache) {
            if (RING) {
                const int c = k * kPage + kr;
                if (c >= nvalid) return false;
                j = c + ring_off;  // the newest cached position in cell c
                if (j >= base) j -= W;
                return true;
            }
            j = (pt_lo + k) * kPage + kr;
            return j < base;
        }
        const int tn = (nt_base + k - ncache) * kPage + kr;
        j = base + tn;
        return tn < n;
    };

    SegState<kMNT> st;
    state_reset(st);
    bool failed = false;
    int s = 0;
    uint32_t ph = 0;
    int i = 0;
    for (; i < cnt; ++i) {
        // producer: refill the stage of tile i - 1 (its readers are most likely done)
        if (tid == 0 && i >= 1 && issued < cnt) {
            const int sp = s == 0 ? kMStages - 1 : s - 1;
            const uint32_t pp = s == 0 ? ph ^ 1u : ph;
            if (!mbar_wait_bounded(empty0 + 8 * sp, pp)) {
                failed = true;
                break;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(kb + issued, sp);
            ++issued;
        }
        if (!mbar_wait_bounded(full0 + 8 * s, ph)) {
            failed = true;
            break;
        }
        const int k = kb + i;
        int jS[2];
        bool okS[2];
        okS[0] = key_at(k, lane >> 2, jS[0]);
        okS[1] = key_at(k, (lane >> 2) + 8, jS[1]);
        int jlast;
        const bool full_tile = key_at(k, kPage - 1, jlast);  // keys only end at a tile's top

        const uint32_t sK = tiles_s + s * kMStageBytes, sV = sK + kTileBytes;
        uint32_t ka[4][4], va[4][4];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            ldsm_x4(sK + k_row + (((2 * ks + k_cb) ^ lj) << 4), ka[ks][0], ka[ks][1], ka[ks][2], ka[ks][3]);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
            ldsm_x4_t(sV + v_row + (((2 * mt + v_cb) ^ lj) << 4), va[mt][0], va[mt][1], va[mt][2], va[mt][3]);
        if (!full_tile) {  // zero the V values of keys that do not exist (they may hold NaN)
            int jj;
            const int kv = 2 * (lane & 3);
            const uint32_t vm0 = (key_at(k, kv, jj) ? 0x0000ffffu : 0u) | (key_at(k, kv + 1, jj) ? 0xffff0000u : 0u);
            const uint32_t vm1 = (key_at(k, kv + 8, jj) ? 0x0000ffffu : 0u) | (key_at(k, kv + 9, jj) ? 0xffff0000u : 0u);
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                va[mt][0] &= vm0;
                va[mt][1] &= vm0;
                va[mt][2] &= vm1;
                va[mt][3] &= vm1;
            }
        }
        uint32_t pb[kMNT][2];
#pragma unroll
        for (int j = 0; j < kMNT; ++j) {
            float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16(sc, ka[0][0], ka[0][1], ka[0][2], ka[0][3], qf[j][0][0], qf[j][0][1]);
            mma_bf16(sd, ka[1][0], ka[1][1], ka[1][2], ka[1][3], qf[j][1][0], qf[j][1][1]);
            mma_bf16(sc, ka[2][0], ka[2][1], ka[2][2], ka[2][3], qf[j][2][0], qf[j][2][1]);
            mma_bf16(sd, ka[3][0], ka[3][1], ka[3][2], ka[3][3], qf[j][3][0], qf[j][3][1]);
            // [key lane/4 | lane/4 + 8][row 2(lane%4) | + 1], causal and window masks per row
            auto keep = [&](int kk, int c) { return okS[kk] && jS[kk] >= rlo[j][c] && jS[kk] <= rp[j][c]; };
            const float s00 = keep(0, 0) ? (sc[0] + sd[0]) * p.scale_log2 : -INFINITY;
            const float s01 = keep(0, 1) ? (sc[1] + sd[1]) * p.scale_log2 : -INFINITY;
            const float s10 = keep(1, 0) ? (sc[2] + sd[2]) * p.scale_log2 : -INFINITY;
            const float s11 = keep(1, 1) ? (sc[3] + sd[3]) * p.scale_log2 : -INFINITY;
            float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 4));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 4));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 8));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 8));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 16));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 16));
            const float mn0 = fmaxf(st.m[j][0], mx0), mn1 = fmaxf(st.m[j][1], mx1);
            // a row with no key so far keeps m = -inf: subtract 0 instead (every term is 0)
            const float mr0 = mn0 == -INFINITY ? 0.f : mn0, mr1 = mn1 == -INFINITY ? 0.f : mn1;
            const float a0 = fast_exp2(st.m[j][0] - mr0), a1 = fast_exp2(st.m[j][1] - mr1);
            const float p00 = fast_exp2(s00 - mr0), p01 = fast_exp2(s01 - mr1);
            const float p10 = fast_exp2(s10 - mr0), p11 = fast_exp2(s11 - mr1);
            st.l[j][0] = st.l[j][0] * a0 + (p00 + p10);
            st.l[j][1] = st.l[j][1] * a1 + (p01 + p11);
            st.m[j][0] = mn0;
            st.m[j][1] = mn1;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                st.acc[j][mt][0] *= a0;
                st.acc[j][mt][1] *= a1;
                st.acc[j][mt][2] *= a0;
                st.acc[j][mt][3] *= a1;
            }
            pb[j][0] = movmatrix_t(pack_bf16(p00, p01));  // keys 2(lane%4), +1
            pb[j][1] = movmatrix_t(pack_bf16(p10, p11));  // keys 2(lane%4) + 8, + 9
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int j = 0; j < kMNT; ++j)
                mma_bf16(st.acc[j][mt], va[mt][0], va[mt][1], va[mt][2], va[mt][3], pb[j][0], pb[j][1]);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (++s == kMStages) {
            s = 0;
            ph ^= 1u;
        }
    }
    if (failed) {
        flag_status(DA_STATUS_TIMEOUT);
        s_failed = 1;
    }
    __syncthreads();
    if (tid == 0 && s_failed) {  // let the copies still in flight land before the CTA leaves
        for (int j = i; j < issued; ++j) mbar_wait_bounded(full0 + 8 * (j % kMStages), (j / kMStages) & 1);
    }
    state_reduce_l(st);

    // ---- finish: one split writes the rows, several leave partials for the last to combine
    auto finish_row = [&](float m, float l, float sg, float &f) {  // f: factor on acc; false: zero row
        const float M = fmaxf(m, sg);
        if (M == -INFINITY) {
            f = 0.f;
            return;
        }
        const float den = l * exp2f(m - M) + (sg == -INFINITY ? 0.f : exp2f(sg - M));
        f = den > 0.f ? exp2f(m - M) / den : 0.f;
    };
    if (nsplit == 1) {
#pragma unroll
        for (int j = 0; j < kMNT; ++j)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int r = r0 + kMRowsPerWarp * warp + 8 * j + 2 * (lane & 3) + c;
                if (r >= r_end) continue;
                float f = 0.f;
                if (rp[j][c] >= 0) finish_row(st.m[j][c], st.l[j][c], sig[j][c], f);
                __nv_bfloat16 *o = out_row(r);
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    o[mt * 16 + (lane >> 2)] = __float2bfloat16_rn(st.acc[j][mt][c] * f);
                    o[mt * 16 + (lane >> 2) + 8] = __float2bfloat16_rn(st.acc[j][mt][c + 2] * f);
                }
            }
        return;
    }
    const size_t slot0 = ((bg * p.row_blocks + rb) * p.splits) * static_cast<size_t>(RB);
    float *mine = p.part + (slot0 + static_cast<size_t>(split) * RB) * kMSlotFloats;
#pragma unroll
    for (int j = 0; j < kMNT; ++j)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int rl = kMRowsPerWarp * warp + 8 * j + 2 * (lane & 3) + c;
            float *o = mine + static_cast<size_t>(rl) * kMSlotFloats;
            if (lane < 4) {
                o[0] = st.m[j][c];
                o[1] = st.l[j][c];
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                o[kMAccOff + mt * 16 + (lane >> 2)] = st.acc[j][mt][c];
                o[kMAccOff + mt * 16 + (lane >> 2) + 8] = st.acc[j][mt][c + 2];
            }
        }
    if (p.defer) return;  // multi_combine_kernel follows
    __threadfence();
    __syncthreads();
    int *ctr = p.counters + bg * p.row_blocks + rb;
    if (tid == 0) s_ticket = atomicAdd(ctr, 1);
    __syncthreads();
    if (s_ticket != nsplit - 1) return;
    __threadfence();
    multi_combine_rows(p, p.part + slot0 * kMSlotFloats, RB, r0, r_end, n, b, g, nsplit, 0, RB, warp, nw, lane);
    __syncthreads();
    if (tid == 0) *ctr = 0;  // ready for the next call
}

// Calls whose row blocks are split over many CTAs fold the partials in a kernel of their own,
// after the attention kernel, so the fold runs on many SMs at once instead of in the one CTA
// per row block that arrives last. One warp per query row, one lane per split (lanes take
// splits l, l + 32, ...): each lane merges its splits' (m, l) online, the warp merges the
// lanes' maxima and sums, then each lane adds up its splits' weighted accumulators (64
// values) and the warp sums them over the lanes through shared memory (a padded 32 x 64
// transpose), so a row costs about three dependent L2 round trips however many splits.
constexpr int kCombWarps = 4;  // query rows per CTA
__global__ void __launch_bounds__(kCombWarps * 32) multi_combine_kernel(const MultiParams p, int RB, int ring) {
    __shared__ float s_sum[kCombWarps][32][kD + 1];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the partials of the attention kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slices = (RB + kCombWarps - 1) / kCombWarps;
    const int rb = blockIdx.x / slices, sl = blockIdx.x - rb * slices;
    const int g = blockIdx.y, b = blockIdx.z;
    const int r0 = rb * RB, r_end = min(r0 + RB, p.T * p.G);
    if (r0 + sl * kCombWarps >= r_end) return;
    const MultiKeys k = multi_keys(p, ring != 0, b, r0, r_end);
    const int nsplit = (k.ntiles + p.chunk - 1) / p.chunk;
    if (nsplit <= 1) return;  // the attention kernel wrote these rows (or their zeros)
    const int rl = sl * kCombWarps + warp;  // this warp's row of the block
    const int r = r0 + rl;
    if (rl >= RB || r >= r_end) return;  // no barrier follows: warps leave on their own
    const int t = r / p.G, hl = r - t * p.G;
    __nv_bfloat16 *out = p.out + ((static_cast<size_t>(b) * p.T + t) * p.Hq + g * p.G + hl) * kD;
    if (t >= k.n) {  // not a query row: zeros
        reinterpret_cast<uint32_t *>(out)[lane] = 0u;
        return;
    }
    const size_t bg = static_cast<size_t>(b) * p.Hkv + g;
    const float *all = p.part + ((bg * p.row_blocks + rb) * p.splits) * static_cast<size_t>(RB) * kMSlotFloats;
    auto slot = [&](int sp) { return all + (static_cast<size_t>(sp) * RB + rl) * kMSlotFloats; };
    // (m, l) of this lane's splits, merged online
    float M = -INFINITY, den = 0.f;
    for (int sp = lane; sp < nsplit; sp += 32) {
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(slot(sp)));
        if (ml.x == -INFINITY) continue;  // a split that saw no key of the row
        const float Mn = fmaxf(M, ml.x);
        den = den * exp2f(M - Mn) + ml.y * exp2f(ml.x - Mn);
        M = Mn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, off);
        const float Do = __shfl_xor_sync(0xffffffffu, den, off);
        const float Mn = fmaxf(M, Mo);
        den = Mn == -INFINITY ? 0.f : den * exp2f(M - Mn) + Do * exp2f(Mo - Mn);
        M = Mn;
    }
    const float sg = p.sinks != nullptr ? __ldg(p.sinks + g * p.G + hl) * kLog2e : -INFINITY;
    const float Mf = fmaxf(M, sg);  // the same on every lane: an exact maximum
    float inv = 0.f;
    if (Mf != -INFINITY) {
        const float d = den * exp2f(M - Mf) + (sg == -INFINITY ? 0.f : exp2f(sg - Mf));
        inv = d > 0.f ? 1.f / d : 0.f;
    }
    // this lane's splits' weighted accumulators
    float o[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) o[d] = 0.f;
    if (Mf != -INFINITY) {
        for (int sp = lane; sp < nsplit; sp += 32) {
            const float *s = slot(sp);
            const float m = __ldcg(s);
            const float w = m == -INFINITY ? 0.f : exp2f(m - Mf);
            const float4 *a4 = reinterpret_cast<const float4 *>(s + kMAccOff);
#pragma unroll
            for (int c = 0; c < kD / 4; ++c) {
                const float4 a = __ldcg(a4 + c);
                o[4 * c] += a.x * w;
                o[4 * c + 1] += a.y * w;
                o[4 * c + 2] += a.z * w;
                o[4 * c + 3] += a.w * w;
            }
        }
    }
    // the sum over the lanes: lane l writes its 64 values as row l, then sums columns 2l, 2l + 1
#pragma unroll
    for (int d = 0; d < kD; ++d) s_sum[warp][lane][d] = o[d];
    __syncwarp();
    float x0 = 0.f, x1 = 0.f;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
        x0 += s_sum[warp][j][2 * lane];
        x1 += s_sum[warp][j][2 * lane + 1];
    }
    reinterpret_cast<uint32_t *>(out)[lane] = pack_bf16(x0 * inv, x1 * inv);
}

// The append of a multi-token step: new token t < n of b goes to position L - n + t. In a
// ring only the last W of them survive (one write per cell).
__global__ void kv_append_multi_kernel(const __nv_bfloat16 *__restrict__ k_new,
                                       const __nv_bfloat16 *__restrict__ v_new, __nv_bfloat16 *k_cache,
                                       __nv_bfloat16 *v_cache, const int *__restrict__ block_table,
                                       const int *__restrict__ seq_lens, const int *__restrict__ q_lens, int T,
                                       int Hkv, int window, int max_pages, int num_pages, int max_seq_len) {
    const int b = blockIdx.x;
    const int L = __ldg(seq_lens + b);
    const int n = q_lens != nullptr ? __ldg(q_lens + b) : T;
    bool bad = L < 0 || n < 0 || n > T || (L > 0 && n > L);
    if (block_table != nullptr) bad = bad || L > max_seq_len || L > max_pages * kPage;
    if (bad) {
        if (threadIdx.x == 0) flag_status(DA_STATUS_BAD_SEQ_LEN);
        return;
    }
    if (L == 0 || n == 0) return;
    const int base = L - n;
    const int first = block_table == nullptr && n > window ? n - window : 0;  // ring: last W only
    constexpr int kChunks = kD / 8;  // 16-byte pieces per row
    for (int i = threadIdx.x; i < (n - first) * Hkv * kChunks; i += blockDim.x) {
        const int t = first + i / (Hkv * kChunks);
        const int g = (i / kChunks) % Hkv, c = i % kChunks;
        const int pos = base + t;
        size_t dst;
        if (block_table != nullptr) {
            const int page = __ldg(block_table + static_cast<size_t>(b) * max_pages + pos / kPage);
            if (page < 0 || page >= num_pages) {
                flag_status(DA_STATUS_BAD_PAGE);
                continue;
            }
            dst = ((static_cast<size_t>(page) * Hkv + g) * kPage + pos % kPage) * kD + c * 8;
        } else {
            dst = ((static_cast<size_t>(b) * Hkv + g) * window + pos % window) * kD + c * 8;
        }
        const size_t src = ((static_cast<size_t>(b) * T + t) * Hkv + g) * kD + c * 8;
        *reinterpret_cast<uint4 *>(k_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(k_new + src));
        *reinterpret_cast<uint4 *>(v_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(v_new + src));
    }
}

// The rotary embedding of a several-token step, ahead of its attention: query row (t, h) and
// new key (t, g) of every new token t < n are rotated to their own position p = L - n + t
// (rotate-half pairs (i, i + D/2); each product and the sum or difference rounded to fp32,
// then to bf16 nearest even, as the one-token steps' fused rotation does) into q_rot / k_rot;
// the rows of tokens t >= n and of inactive slots are copied as they are. One block per
// (t, b). A position beyond the tables raises DA_STATUS_BAD_POSITION and uses row 0.
__global__ void rope_multi_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k_new,
                                  const int *__restrict__ seq_lens, const int *__restrict__ q_lens,
                                  const float *__restrict__ rope_cos, const float *__restrict__ rope_sin,
                                  int max_position, int T, int Hq, int Hkv, __nv_bfloat16 *__restrict__ q_rot,
                                  __nv_bfloat16 *__restrict__ k_rot) {
    const int t = blockIdx.x, b = blockIdx.y;
    const int L = __ldg(seq_lens + b);
    const int n = q_lens != nullptr ? __ldg(q_lens + b) : T;
    const bool active = L > 0 && t < n && n <= L;
    int pos = L - n + t;
    if (active && pos >= max_position) {
        if (threadIdx.x == 0) flag_status(DA_STATUS_BAD_POSITION);
        pos = 0;
    }
    constexpr int kHalf = kD / 2;
    const size_t qrow0 = (static_cast<size_t>(b) * T + t) * Hq, krow0 = (static_cast<size_t>(b) * T + t) * Hkv;
    const int pairs = (Hq + Hkv) * kHalf;
    for (int i = threadIdx.x; i < pairs; i += blockDim.x) {
        const int r = i / kHalf, d = i % kHalf;  // rows 0 .. Hq - 1: queries, then keys
        const __nv_bfloat16 *src = r < Hq ? q + (qrow0 + r) * kD : k_new + (krow0 + r - Hq) * kD;
        __nv_bfloat16 *dst = r < Hq ? q_rot + (qrow0 + r) * kD : k_rot + (krow0 + r - Hq) * kD;
        const __nv_bfloat16 x1 = src[d], x2 = src[d + kHalf];
        if (!active) {
            dst[d] = x1;
            dst[d + kHalf] = x2;
            continue;
        }
        const float c = __ldg(rope_cos + static_cast<size_t>(pos) * kHalf + d);
        const float sn = __ldg(rope_sin + static_cast<size_t>(pos) * kHalf + d);
        const float f1 = __bfloat162float(x1), f2 = __bfloat162float(x2);
        dst[d] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(f1, c), __fmul_rn(f2, sn)));
        dst[d + kHalf] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(f2, c), __fmul_rn(f1, sn)));
    }
}
