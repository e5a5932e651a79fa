// Several query tokens per sequence on the 5th-generation tensor cores: the step of
// multi_attn_kernel (same definition, masks, key tiles, splits, partials and combine) with
// the contraction on tcgen05 and the query rows on the TMEM lanes.
//
// One CTA per (sequence, KV head, block of 128 query rows, key split); 6 warps:
//   warps 0-3  one query row per thread (TMEM lane = row): the online softmax of S and the
//              finish; warp 0 also zeroes the V rows of keys that do not exist
//   warp 4     lane 0 issues the TMA copies of 64-key blocks (4 tiles of K and of V)
//   warp 5     lane 0 issues the MMAs:  S_j = Q K_j^T  (M 128, N 64, K 64; A = Q, B = K, both
//              K-major in shared memory, 128-byte swizzle)  and  O += P_j V_j  (M 128, N 64,
//              K 64; A = P_j in TMEM as bf16, B = V_j with d contiguous)
// TMEM: S buffers b = 0 .. kTcSBufs - 1 at columns [64 b, 64 b + 64), O after them. Block j
// uses buffer j % kTcSBufs; P_j overwrites S_j there as two bf16 parts, P = hi + lo (hi = P rounded to bf16 in columns [0, 32), lo = the rest in [32, 64)),
// and the PV product runs on both: about 16 significant bits on every probability, so a
// sharply peaked softmax loses nothing to the bf16 operand. The softmax keeps a per-row
// reference maximum and
// rescales O (in TMEM) only when a block's maximum exceeds it by more than 2^8, so the
// probabilities stay below 256 and O is rarely touched; O and l share the reference, so the
// final O / l is exact.
// Barriers: kv_full / kv_empty per stage (TMA <-> MMA); s_full / p_full / o_done per S buffer
// (S_j written, P_j written, PV_j done: one phase per use of the buffer, so every parity wait
// below is at most one phase behind its barrier); drain (all MMAs before TMEM is freed).

constexpr int kTcRows = 128;                               // query rows per CTA (MMA M)
constexpr int kTcKeys = 64;                                // keys per block (MMA N of S)
constexpr int kTcTilesPerBlock = kTcKeys / kPage;          // 4
#ifndef DA_TC_STAGES
#define DA_TC_STAGES 5
#endif
constexpr int kTcStages = DA_TC_STAGES;                    // key blocks in flight
constexpr int kTcBlockBytes = kTcTilesPerBlock * kTileBytes;  // 8 KiB of K (or V)
constexpr int kTcStageBytes = 2 * kTcBlockBytes;           // K block, then V block
constexpr int kTcQBytes = kTcRows * kD * 2;                // 16 KiB
// S / P buffers in TMEM: S_j waits for PV_{j-kTcSBufs}. A third buffer (TMEM has the room)
// measured no faster: the row warps' softmax, not the MMA hand-off, sets the pace.
#ifndef DA_TC_SBUFS
#define DA_TC_SBUFS 2
#endif
constexpr int kTcSBufs = DA_TC_SBUFS;
constexpr int kTcBars = 2 * kTcStages + 3 * kTcSBufs + 1;
constexpr int kTcSmem = 1024 + kTcQBytes + kTcStages * kTcStageBytes + kTcBars * 8;
constexpr int kTcWarps = 6;
constexpr int kTcThreads = kTcWarps * 32;
constexpr uint32_t kTcTmemCols = 256;
constexpr uint32_t kTcColS = 0, kTcColO = 64 * kTcSBufs;  // S_b at kTcColS + 64 b
static_assert(kTcColO + 64 <= kTcTmemCols, "S buffers and O fit the TMEM allocation");
constexpr float kTcRescale = 8.f;                          // log2 of the largest probability

// Shared-memory matrix descriptor (tcgen05): start, leading / stride byte offsets (16-byte
// units), descriptor version 1, 128-byte swizzle. K-major operands: the stride offset is the
// distance between 8-row groups (1024 bytes). The V operand (d contiguous): the stride offset
// is the distance between groups of 8 keys along the contraction (1024 bytes), the leading
// offset the distance between 64-wide groups along d (unused at d = 64).
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A K-major, B K-major
// or (b_mn) contiguous along N, N and M.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive TMEM columns of this warp's 32 lanes (one row per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
        "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
        "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <bool RING>
__global__ void __launch_bounds__(kTcThreads, 2)
    multi_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ CUtensorMap tnk, const __grid_constant__ CUtensorMap tnv,
                    const MultiParams p) {
    extern __shared__ uint8_t smem_raw[];
    // the 1024-byte aligned base, derived from the shared array itself so that every access
    // through it compiles to a shared-memory instruction (not a generic one)
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem;                                  // [128 rows][128 B], 128-byte swizzle
    uint8_t *sKV = smem + kTcQBytes;                     // [stage][K block | V block]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sKV + kTcStages * kTcStageBytes);
    const uint32_t kv_full = smem_addr(bars), kv_empty = kv_full + 8 * kTcStages;
    const uint32_t s_full = kv_empty + 8 * kTcStages, p_full = s_full + 8 * kTcSBufs;
    const uint32_t o_done = p_full + 8 * kTcSBufs, drain = o_done + 8 * kTcSBufs;
    __shared__ int s_page[kMMaxChunk];
    __shared__ uint32_t s_tmem;
    __shared__ int s_ticket, s_failed;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int split = blockIdx.x % p.splits, rb = blockIdx.x / p.splits;
    const int g = blockIdx.y, b = blockIdx.z;

    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tnk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tnv)) : "memory");
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(kv_full + 8 * s, 1);
            mbar_init(kv_empty + 8 * s, 1);
        }
        for (int s = 0; s < kTcSBufs; ++s) {
            mbar_init(s_full + 8 * s, 1);
            mbar_init(p_full + 8 * s, 4);  // the four row warps
            mbar_init(o_done + 8 * s, 1);
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_failed = 0;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- counts and the key tiles of this row block (as in multi_attn_kernel)
    const int W = p.window;
    const int TG = p.T * p.G;
    const int r0 = rb * kTcRows;
    const int r_end = min(r0 + kTcRows, TG);
    const MultiKeys keys = multi_keys(p, RING, b, r0, r_end);
    if (keys.bad && tid == 0 && g == 0 && blockIdx.x == 0) flag_status(DA_STATUS_BAD_SEQ_LEN);
    const int n = keys.n, base = keys.base;
    const int ncache = keys.ncache, pt_lo = keys.pt_lo, nvalid = keys.nvalid, nt_base = keys.nt_base;
    const int ntiles = keys.ntiles, ring_off = keys.ring_off;
    const int kb = split * p.chunk;
    const int ke = min(kb + p.chunk, ntiles);
    const int nsplit = (ntiles + p.chunk - 1) / p.chunk;
    const size_t bg = static_cast<size_t>(b) * p.Hkv + g;
    auto row_off = [&](int r) {
        const int t = r / p.G, hl = r - t * p.G;
        return ((static_cast<size_t>(b) * p.T + t) * p.Hq + g * p.G + hl) * kD;
    };
    if (kb >= ke) {
        if (ntiles == 0 && split == 0)
            for (int i = tid; i < (r_end - r0) * (kD / 8); i += blockDim.x)
                *reinterpret_cast<uint4 *>(p.out + row_off(r0 + i / (kD / 8)) + (i % (kD / 8)) * 8) =
                    make_uint4(0, 0, 0, 0);
        return;
    }
    const int cnt = ke - kb;
    const int nblk = (cnt + kTcTilesPerBlock - 1) / kTcTilesPerBlock;
    const int r_valid = min(r_end, r0 + max(0, n * p.G - r0));  // rows r0 .. r_valid-1 are queries

    // ---- page indices, query rows (zero past the valid ones), TMEM
    if (!RING)
        for (int i = tid; i < cnt && kb + i < ncache; i += blockDim.x) {
            int page = __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + pt_lo + kb + i);
            if (page < 0 || page >= p.num_pages) {
                flag_status(DA_STATUS_BAD_PAGE);
                page = -1;  // out of the map: the copy reads zeros
            }
            s_page[i] = page;
        }
    if (warp < 4) {
        const int r = r0 + tid;
        uint4 qv[8];
        const bool ok = r < r_valid;
        const uint4 *src = ok ? reinterpret_cast<const uint4 *>(p.q + row_off(r)) : nullptr;
#pragma unroll
        for (int c = 0; c < 8; ++c) qv[c] = ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(sQ + tid * 128 + ((c ^ (tid & 7)) << 4)) = qv[c];
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q is read by the tensor cores
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                     "r"(kTcTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s_tmem;

    // position of key row kr of tile k, and whether it exists (as in multi_attn_kernel)
    auto key_at = [&](int k, int kr, int &j) -> bool {
        if (k < ncache) {
            if (RING) {
                const int c = k * kPage + kr;
                if (c >= nvalid) return false;
                j = c + ring_off;
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

    bool failed = false;
    if (warp == 4) {
        // ---- TMA producer
        if (lane == 0) {
            const uint64_t policy = evict_first_policy();
            for (int j = 0; j < nblk && !failed; ++j) {
                const int s = j % kTcStages;
                if (j >= kTcStages && !mbar_wait_bounded(kv_empty + 8 * s, ((j / kTcStages) - 1) & 1)) {
                    failed = true;
                    break;
                }
                const int k0 = kb + j * kTcTilesPerBlock;
                const int nt = min(kTcTilesPerBlock, ke - k0);
                const uint32_t fb = kv_full + 8 * s;
                const uint32_t dK = smem_addr(sKV + s * kTcStageBytes), dV = dK + kTcBlockBytes;
                mbar_expect_tx(fb, nt * 2 * kTileBytes);
                for (int u = 0; u < nt; ++u) {
                    const int k = k0 + u;
                    const uint32_t dk = dK + u * kTileBytes, dv = dV + u * kTileBytes;
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
                        const int tt = (nt_base + k - ncache) * kPage;
                        tma_load_4d(dk, &tnk, 0, g, tt, b, fb, policy);
                        tma_load_4d(dv, &tnv, 0, g, tt, b, fb, policy);
                    }
                }
            }
            // nothing may still be landing when the CTA leaves: the last copy of every stage
            for (int j = max(0, nblk - kTcStages); j < nblk; ++j)
                mbar_wait_bounded(kv_full + 8 * (j % kTcStages), (j / kTcStages) & 1);
        }
    } else if (warp == 5) {
        // ---- MMA issuer: S_j = Q K_j^T, then O += P_{j-1} V_{j-1}
        if (lane == 0) {
            const uint32_t id_qk = umma_idesc_bf16(kTcRows, kTcKeys, false);
            const uint32_t id_pv = umma_idesc_bf16(kTcRows, kD, true);
            const uint32_t q_s = smem_addr(sQ);
            for (int j = 0; j <= nblk && !failed; ++j) {
                if (j < nblk) {
                    const int s = j % kTcStages;
                    if (!mbar_wait_bounded(kv_full + 8 * s, (j / kTcStages) & 1)) {
                        failed = true;
                        break;
                    }
                    // buffer j % kTcSBufs last held P_{j-kTcSBufs}: its PV must be done
                    const int sb = j % kTcSBufs;
                    if (j >= kTcSBufs && !mbar_wait_bounded(o_done + 8 * sb, ((j / kTcSBufs) - 1) & 1)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k_s = smem_addr(sKV + s * kTcStageBytes);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)
                        umma_bf16_ss(tm + kTcColS + 64 * sb, umma_sdesc(q_s + 32 * kk, 16, 1024),
                                     umma_sdesc(k_s + 32 * kk, 16, 1024), id_qk, kk > 0);
                    umma_commit(s_full + 8 * sb);
                }
                if (j >= 1) {
                    const int jj = j - 1, s = jj % kTcStages, pb = jj % kTcSBufs;
                    if (!mbar_wait_bounded(p_full + 8 * pb, (jj / kTcSBufs) & 1)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t v_s = smem_addr(sKV + s * kTcStageBytes + kTcBlockBytes);
#pragma unroll
                    for (int part = 0; part < 2; ++part)  // P = hi + lo
#pragma unroll
                        for (int kk = 0; kk < kTcKeys / 16; ++kk)
                            umma_bf16_ts(tm + kTcColO, tm + kTcColS + 64 * pb + 32 * part + 8 * kk,
                                         umma_sdesc(v_s + 2048 * kk, 2048, 1024), id_pv,
                                         (jj > 0 || part > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(o_done + 8 * pb);
                    umma_commit(kv_empty + 8 * s);
                }
            }
            umma_commit(drain);  // completes when every MMA issued above has
        }
    } else {
        // ---- query rows: one per thread
        const int r = r0 + tid;
        const bool valid = r < r_valid;
        const bool warp_active = r0 + 32 * warp < r_valid;
        const int t = r / p.G;
        const int pr = valid ? base + t : -1;
        const int lor = valid && W > 0 ? max(0, base + t - W + 1) : 0;
        const uint32_t lanes = static_cast<uint32_t>(32 * warp) << 16;
        float m_ref = -INFINITY, l = 0.f;
        for (int j = 0; j < nblk; ++j) {
            const int k0 = kb + j * kTcTilesPerBlock;
            // every row warp waits for S_j, rows or not, so that no warp's arrival on p_full
            // can run ahead into a later phase (a give-up is taken by the whole warp: the TMEM
            // accesses below are warp-wide)
            const int sb = j % kTcSBufs;
            if (__any_sync(0xffffffffu, !mbar_wait_bounded(s_full + 8 * sb, (j / kTcSBufs) & 1))) {
                failed = true;
                break;
            }
            if (warp_active) {
                tc_fence_after();
                const uint32_t sc = tm + lanes + kTcColS + 64 * sb;
                uint32_t raw[2][32];
                tmem_ld32(sc, raw[0]);
                tmem_ld32(sc + 32, raw[1]);
                tmem_wait_ld();
                // raw dot products; a key this row must not see becomes -inf
                float x[64];
#pragma unroll
                for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(raw[c >> 5][c & 31]);
                // a block whose 64 keys are consecutive positions, all present and all inside
                // the row's window [lor, pr] needs no per-key mask (most blocks of a long sequence)
                int jf = 0, jl = 0;
                const bool okf = key_at(k0, 0, jf);
                const bool okl = k0 + kTcTilesPerBlock - 1 < ke && key_at(k0 + kTcTilesPerBlock - 1, kPage - 1, jl);
                const bool interior = valid && okf && okl && jl - jf == kTcKeys - 1 && jf >= lor && jl <= pr;
                if (!interior) {
#pragma unroll
                    for (int u = 0; u < kTcTilesPerBlock; ++u) {
                        const int k = k0 + u;
                        // keys of tile u this row sees: kr in [a, e)
                        int a = 0, e = 0;
                        if (k < ke && (!RING || k >= ncache)) {
                            int j0;
                            key_at(k, 0, j0);  // first position of the tile (consecutive positions)
                            const int cntk = k < ncache ? min(kPage, base - j0) : min(kPage, n - (j0 - base));
                            a = max(0, lor - j0);
                            e = min(cntk, pr - j0 + 1);
                        }
#pragma unroll
                        for (int kr = 0; kr < kPage; ++kr) {
                            bool keep;
                            if (RING && k < ncache && k < ke) {
                                int jp;
                                keep = key_at(k, kr, jp) && jp >= lor && jp <= pr;
                            } else {
                                keep = kr >= a && kr < e;
                            }
                            if (!keep) x[u * kPage + kr] = -INFINITY;
                        }
                    }
                }
                // maximum as a pairwise tree (6 dependent steps instead of 64)
                float mx[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) mx[c] = fmaxf(x[c], x[c + 32]);
#pragma unroll
                for (int w = 16; w > 0; w >>= 1)
#pragma unroll
                    for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
                const float mraw = mx[0];
                const float mb = mraw * p.scale_log2;  // the scale is positive
                const bool need = valid && mb > m_ref + kTcRescale;
                const float m_new = need ? mb : m_ref;
                // P_j goes over S_j, whose buffer PV_{j-kTcSBufs} read: the MMA warp waited for
                // that PV before it wrote S_j. Only a rescale of O needs PV_{j-1} done. Its
                // buffer's o_done is exact for that wait: the buffer's previous PV
                // (PV_{j-1-kTcSBufs}) is complete since S_{j-1} exists, and its next one
                // cannot be issued before P_{j-1+kTcSBufs}.
                const bool resc = j > 0 && __any_sync(0xffffffffu, need);
                if (resc) {
                    const int jb = (j - 1) % kTcSBufs;
                    if (__any_sync(0xffffffffu, !mbar_wait_bounded(o_done + 8 * jb, ((j - 1) / kTcSBufs) & 1))) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    // O holds PV_0 .. PV_{j-1}: rescale the rows that need it
                    const float f = need ? exp2f(m_ref - m_new) : 1.f;  // m_ref = -inf: 0 (O and l are 0)
                    uint32_t o[32];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {  // the store must finish before o is reloaded
                        tmem_ld32(tm + lanes + kTcColO + 32 * h, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
                        tmem_st32(tm + lanes + kTcColO + 32 * h, o);
                        tmem_wait_st();
                    }
                }
                if (need) {
                    l *= exp2f(m_ref - m_new);
                    m_ref = m_new;
                }
                const float mr = m_ref == -INFINITY ? 0.f : m_ref;
                float ls4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent partial sums
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // keys 32h .. 32h + 31: hi and lo, 16 columns each
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float p0 = fast_exp2(fmaf(x[32 * h + 2 * c], p.scale_log2, -mr));
                        const float p1 = fast_exp2(fmaf(x[32 * h + 2 * c + 1], p.scale_log2, -mr));
                        ls4[c & 3] += p0 + p1;
                        hi[c] = pack_bf16(p0, p1);
                        const float2 r2 = unpack_bf16(hi[c]);
                        lo[c] = pack_bf16(p0 - r2.x, p1 - r2.y);
                    }
                    tmem_st16(tm + lanes + kTcColS + 64 * sb + 16 * h, hi);
                    tmem_st16(tm + lanes + kTcColS + 64 * sb + 32 + 16 * h, lo);
                    tmem_wait_st();
                }
                l += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
            }
            if (warp == 0) {  // V rows of keys that do not exist may hold anything: zero them
                uint8_t *vb = sKV + (j % kTcStages) * kTcStageBytes + kTcBlockBytes;
                bool touched = false;
                for (int u = 0; u < kTcTilesPerBlock; ++u) {
                    const int k = k0 + u;
                    int jj;
                    const bool full = k < ke && key_at(k, kPage - 1, jj);
                    if (full) continue;  // keys only end at a tile's top
                    for (int i = lane; i < kPage * 8; i += 32) {
                        const int kr = i >> 3;
                        if (k >= ke || !key_at(k, kr, jj))
                            *reinterpret_cast<uint4 *>(vb + (u * kPage + kr) * 128 + (i & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    touched = true;
                }
                if (touched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + 8 * sb);
        }
        // ---- finish this thread's row: O (after the last PV) -> output or partial
        float o[64];
        bool have = false;
        // the last PV (its buffer's previous PV is complete: S_{nblk-1} exists); the PVs
        // complete in issue order, so O then holds all of them
        const int lb = (nblk - 1) % kTcSBufs;
        if (!failed && warp_active &&
            !__any_sync(0xffffffffu, !mbar_wait_bounded(o_done + 8 * lb, ((nblk - 1) / kTcSBufs) & 1))) {
            tc_fence_after();
            uint32_t raw[2][32];
            tmem_ld32(tm + lanes + kTcColO, raw[0]);
            tmem_ld32(tm + lanes + kTcColO + 32, raw[1]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 64; ++c) o[c] = __uint_as_float(raw[c >> 5][c & 31]);
            have = true;
        } else if (warp_active) {
            failed = true;
        }
        if (!have)
#pragma unroll
            for (int c = 0; c < 64; ++c) o[c] = 0.f;
        if (!valid)
#pragma unroll
            for (int c = 0; c < 64; ++c) o[c] = 0.f;  // not a query row: zeros
        if (nsplit == 1) {
            if (r < r_end) {
                float f = 0.f;
                if (valid) {
                    const int h = g * p.G + (r - t * p.G);
                    const float sg = p.sinks != nullptr ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
                    const float M = fmaxf(m_ref, sg);
                    if (M != -INFINITY) {
                        const float den = l * exp2f(m_ref - M) + (sg == -INFINITY ? 0.f : exp2f(sg - M));
                        f = den > 0.f ? exp2f(m_ref - M) / den : 0.f;
                    }
                }
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + row_off(r));
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16(o[8 * c] * f, o[8 * c + 1] * f);
                    w.y = pack_bf16(o[8 * c + 2] * f, o[8 * c + 3] * f);
                    w.z = pack_bf16(o[8 * c + 4] * f, o[8 * c + 5] * f);
                    w.w = pack_bf16(o[8 * c + 6] * f, o[8 * c + 7] * f);
                    dst[c] = w;
                }
            }
        } else if (r < r_valid) {
            float *slot = p.part + ((((bg * p.row_blocks + rb) * p.splits + split) * kTcRows) + tid) * kMSlotFloats;
            slot[0] = m_ref;
            slot[1] = l;
            float4 *acc = reinterpret_cast<float4 *>(slot + kMAccOff);
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        }
    }
    if (failed) {
        flag_status(DA_STATUS_TIMEOUT);
        s_failed = 1;
    }

    // ---- teardown: every MMA done before TMEM is released
    if (tid == 5 * 32) mbar_wait_bounded(drain, 0);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(kTcTmemCols));
    }
    if (nsplit == 1 || p.defer) return;  // p.defer: multi_combine_kernel follows
    __threadfence();
    __syncthreads();
    int *ctr = p.counters + bg * p.row_blocks + rb;
    if (tid == 0) s_ticket = atomicAdd(ctr, 1);
    __syncthreads();
    if (s_ticket != nsplit - 1) return;
    __threadfence();
    const size_t slot0 = ((bg * p.row_blocks + rb) * p.splits) * static_cast<size_t>(kTcRows);
    multi_combine_rows(p, p.part + slot0 * kMSlotFloats, kTcRows, r0, r_end, n, b, g, nsplit, 0, kTcRows, warp,
                       kTcWarps, lane);
    __syncthreads();
    if (tid == 0) *ctr = 0;  // ready for the next call
}
