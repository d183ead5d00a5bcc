// Deterministic dQ pass of the attention backward for sm_103a.
//
// The main backward kernel (bwd.cu) adds each key tile's dQ contribution into
// an fp32 accumulator with reductions whose order varies from run to run.
// When bitwise reproducible gradients are asked for, that kernel skips its
// dQ product and this kernel computes dQ instead, query-stationary: one CTA
// per 128-row query tile walks the key tiles its rows can see, recomputes
//   S   = Q K_j^T,  P = exp2(S * scale*log2e - LSE*log2e)   (LSE from the forward)
//   dP  = dO V_j^T,  dS' = P o (dP - D)
//   dQ += dS' K_j                      (TMEM accumulator, dS' from TMEM)
// and writes dQ = scale * dQ once, in a fixed order.  cudnn-frontend PR #554
// names the two ways to a deterministic backward (an ordered semaphore relay
// or a separate dQ pass); this is the separate pass, chosen because it needs
// no CTA to wait on another.
//
// The per-row terms come from the preprocess kernel's row-term array (the
// pairs that sum to -LSE/scale and -D); each thread owns one query row (TMEM
// lane), so they are plain registers here.
//
// Roles (192 threads): warp 0 TMA (Q and dO once, then K_j and V_j, into
// rings of three and two stages, on one barrier), warp 1 MMA issuer, warps
// 2-5 compute (thread = row).
// TMEM: S_j in buffer j & 1 (columns 0 and 128), dP at 256, dQ at 384.
// dS'_j goes back packed into the first 64 columns of its S buffer and feeds
// dQ += dS'_j K_j straight from TMEM; S_{j+1} is issued into the other buffer
// meanwhile, so the tensor core has S_{j+1}, dP_{j+1} and dQ_j to run while
// the compute warps work on tile j.
#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {
namespace {

template <int D>
struct DqLayout {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = kTileM * 128;
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    // K_j is read by S_j and, one tile later, by dQ += dS'_j K_j, so the K
    // ring has a third stage for the load of K_{j+2} to overlap dQ_j; V_j is
    // read by dP_j alone.  K_j and V_j land on one barrier (K_j's full
    // barrier).  A V stage is released once dP has read it, and that release
    // also frees the K ring: the pair K_j, V_j takes the stages of
    // K_{j-kKStages} and V_{j-kVStages}, and V_{j-kVStages}'s release is
    // committed behind dP_{j-kVStages}, which is issued after dQ_{j-kKStages},
    // the last reader of K_{j-kKStages}, when the K ring is one stage deeper.
    static constexpr int kKStages = 3;
    static constexpr int kVStages = 2;
    static_assert(kKStages == kVStages + 1, "the V releases must cover the K ring");
    static constexpr int kQ = 0;
    static constexpr int kDO = kQ + kTileBytes;
    static constexpr int kK = kDO + kTileBytes;
    static constexpr int kV = kK + kKStages * kTileBytes;
    static constexpr int kBar = kV + kVStages * kTileBytes;
    static constexpr int bQFull = 0;                 // Q and dO
    static constexpr int bKFull = 1;                 // K_j and V_j
    static constexpr int bVEmpty = bKFull + kKStages;
    static constexpr int bSFull = bVEmpty + kVStages;  // two: S buffer
    static constexpr int bDPFull = bSFull + 2;
    static constexpr int bDSReady = bDPFull + 1;      // two: S buffer holds dS'
    static constexpr int bDQDone = bDSReady + 2;      // two: dQ += dS' K read the buffer
    static constexpr int bDQFinal = bDQDone + 2;
    static constexpr int kNumBars = bDQFinal + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kSmemAlloc = kBytes + 1024;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColDP = 256;
    static constexpr uint32_t kColDQ = 384;
};

constexpr int kDqThreads = 192;

SDPA_DEV bool warp_wait_d(uint32_t bar, uint32_t parity, const WaitCtx &w, uint32_t site) {
    bool ok = mbar_wait(bar, parity, w, site);
    return __all_sync(0xffffffffu, ok);
}

// The query tile of CTA u (latest tiles first, so the heaviest start first
// under a causal mask), its slice, lengths, layout bases and key tiles.
struct DqUnit {
    int slice, head, kv_slice, kv_head, Lq, Lkv, tok_q0, tok_kv0, row0, kt0, n_kv, delta;
    int64_t io_row0, io_rs, st_row0, st_rs;  // I/O rows (elements), row-term rows
};

template <int D, bool kPacked>
SDPA_DEV DqUnit decode_dq(const BwdParams &p, int u, int q_tiles) {
    DqUnit U;
    const int qt = q_tiles - 1 - u / p.bh;
    U.slice = u % p.bh;
    if constexpr (!kPacked) {
        U.head = U.kv_head = 0;
        U.kv_slice = (U.slice / p.h) * p.h_kv + (U.slice % p.h) / p.group;
        U.tok_q0 = U.tok_kv0 = 0;
        U.Lq = p.s_q;
        U.Lkv = p.s_kv;
        U.io_row0 = (int64_t)U.slice * p.s_q * D;
        U.io_rs = D;
        U.st_row0 = (int64_t)U.slice * p.s_q;
        U.st_rs = 1;
    } else {
        const int n = U.slice / p.h;
        U.head = U.slice % p.h;
        U.kv_head = U.head / p.group;
        U.kv_slice = 0;
        U.tok_q0 = p.cu_q[n];
        U.tok_kv0 = p.cu_kv[n];
        U.Lq = p.cu_q[n + 1] - U.tok_q0;
        U.Lkv = p.cu_kv[n + 1] - U.tok_kv0;
        U.io_row0 = ((int64_t)U.tok_q0 * p.h + U.head) * D;
        U.io_rs = (int64_t)p.h * D;
        U.st_row0 = (int64_t)U.tok_q0 * p.h + U.head;
        U.st_rs = p.h;
    }
    U.row0 = qt * kTileM;
    U.delta = mask_delta(p.mask, U.Lq, U.Lkv);
    const bool live = U.row0 < U.Lq;
    const int lo = max(0, key_range(p.mask, p.window, U.row0, U.delta, U.Lkv).lo);
    const int hi = key_range(p.mask, p.window, min(U.row0 + kTileM, U.Lq) - 1, U.delta, U.Lkv).hi;
    U.kt0 = lo / kTileN;
    U.n_kv = (live && hi > lo) ? (hi + kTileN - 1) / kTileN - U.kt0 : 0;
    return U;
}

template <int D, bool kBf16, bool kPacked>
__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p, int q_tiles) {
    using L = DqLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    const DqUnit U = decode_dq<D, kPacked>(p, blockIdx.x, q_tiles);
    if (U.row0 >= U.Lq) return;  // packed: the sequence has fewer query tiles
    uint16_t *dq = static_cast<uint16_t *>(p.dq);
    if (U.n_kv == 0) {
        // No row of the tile sees a key: dQ = 0.
        for (int r = threadIdx.x; r < kTileM; r += blockDim.x) {
            if (U.row0 + r >= U.Lq) break;
            uint4 *dst = reinterpret_cast<uint4 *>(dq + U.io_row0 + (int64_t)(U.row0 + r) * U.io_rs);
#pragma unroll
            for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
        }
        return;
    }

    if (threadIdx.x == 0) {
        mbar_init(bar(L::bQFull), 1);
        for (int s = 0; s < L::kKStages; ++s) mbar_init(bar(L::bKFull + s), 1);
        for (int s = 0; s < L::kVStages; ++s) mbar_init(bar(L::bVEmpty + s), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::bSFull + b), 1);
            mbar_init(bar(L::bDSReady + b), kTileM);
            mbar_init(bar(L::bDQDone + b), 1);
        }
        mbar_init(bar(L::bDPFull), 1);
        mbar_init(bar(L::bDQFinal), 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kMisc, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const WaitCtx wc{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.err, kTagBwdDq};
    const int n = U.n_kv;

    if (warp == 0) {
        // ============================================================ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
            const int qy = kPacked ? U.head : U.row0;
            const int qz = kPacked ? U.tok_q0 + U.row0 : U.slice;
            mbar_arrive_expect_tx(bar(L::bQFull), 2 * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
                tma_load_3d(sbase + L::kQ + c * L::kChunkBytes, &tm_q, bar(L::bQFull), c * 64, qy, qz);
                tma_load_3d(sbase + L::kDO + c * L::kChunkBytes, &tm_do, bar(L::bQFull), c * 64, qy, qz);
            }
            int issued = 0;
            for (int j = 0; j < n; ++j) {
                const int k0 = (U.kt0 + j) * kTileN;
                const int ky = kPacked ? U.kv_head : k0;
                const int kz = kPacked ? U.tok_kv0 + k0 : U.kv_slice;
                // the V stage's release also frees the K stage (see DqLayout)
                const int ks = j % L::kKStages, vs = j % L::kVStages, vuse = j / L::kVStages;
                if (vuse > 0 && !mbar_wait(bar(L::bVEmpty + vs), (vuse - 1) & 1, wc, 2)) break;
                const uint32_t full = bar(L::bKFull + ks);
                mbar_arrive_expect_tx(full, 2 * L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c) {
                    tma_load_3d(sbase + L::kK + ks * L::kTileBytes + c * L::kChunkBytes, &tm_k, full, c * 64,
                                ky, kz);
                    tma_load_3d(sbase + L::kV + vs * L::kTileBytes + c * L::kChunkBytes, &tm_v, full, c * 64,
                                ky, kz);
                }
                issued = j + 1;
            }
            // every load issued must land before the CTA may exit
            mbar_wait_drain(bar(L::bQFull), 0);
            for (int j = max(0, issued - L::kKStages); j < issued; ++j)
                mbar_wait_drain(bar(L::bKFull + j % L::kKStages), (j / L::kKStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = make_idesc_f16(kTileM, kTileN, kBf16, false, false);
            constexpr uint32_t id_q = make_idesc_f16(kTileM, D, kBf16, false, true);
            constexpr uint32_t kChunk16 = L::kChunkBytes >> 4, kTile16 = L::kTileBytes >> 4;
            auto kstep = [](int k) -> uint32_t { return (uint32_t)((k >> 2) * kChunk16 + (k & 3) * 2); };
            const uint64_t dQ_k = smem_desc_sw128(sbase + L::kQ, 16, 1024);
            const uint64_t dDO_k = smem_desc_sw128(sbase + L::kDO, 16, 1024);
            const uint64_t dK_k = smem_desc_sw128(sbase + L::kK, 16, 1024);
            const uint64_t dK_mn = smem_desc_sw128(sbase + L::kK, L::kChunkBytes, 1024);
            const uint64_t dV_k = smem_desc_sw128(sbase + L::kV, 16, 1024);
            // X = A B^T over the head dim, both K-major, 128 x 128 into TMEM col
            auto issue_nt = [&](uint64_t a, uint64_t b, uint32_t col) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) mma_ss(tmem + col, a + kstep(k), b + kstep(k), id_s, k > 0);
            };
            auto issue_s = [&](int j) -> bool {  // S_j into buffer j & 1
                const int st = j % L::kKStages;
                if (!mbar_wait(bar(L::bKFull + st), (j / L::kKStages) & 1, wc, 3)) return false;
                if (j >= 2 && !mbar_wait(bar(L::bDQDone + (j & 1)), ((j - 2) >> 1) & 1, wc, 4)) return false;
                tc_fence_after();
                issue_nt(dQ_k, dK_k + st * kTile16, (j & 1) * 128);
                mma_commit(bar(L::bSFull + (j & 1)));
                return true;
            };
            auto issue_dp = [&](int j) -> bool {  // dP_j: V_j landed with K_j, waited for by S_j
                const int st = j % L::kVStages;
                tc_fence_after();
                issue_nt(dDO_k, dV_k + st * kTile16, L::kColDP);
                mma_commit(bar(L::bDPFull));
                mma_commit(bar(L::bVEmpty + st));
                return true;
            };
            bool ok = mbar_wait(bar(L::bQFull), 0, wc, 6) && issue_s(0) && issue_dp(0);
            for (int j = 0; ok && j < n; ++j) {
                if (j + 1 < n && !(ok = issue_s(j + 1))) break;
                // dQ += dS'_j K_j: A = dS'_j packed in buffer j & 1 (8 columns
                // per 16 keys), B = K_j MN-major (head dim contiguous)
                if (!(ok = mbar_wait(bar(L::bDSReady + (j & 1)), (j >> 1) & 1, wc, 7))) break;
                tc_fence_after();
                {
                    const uint64_t b = dK_mn + (j % L::kKStages) * kTile16;
#pragma unroll
                    for (int k = 0; k < kTileN / 16; ++k)
                        mma_ts(tmem + L::kColDQ, tmem + (j & 1) * 128 + k * 8, b + k * 128, id_q,
                               (j > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(L::bDQDone + (j & 1)));
                // dP_{j+1} overwrites dP_j, which the compute warps have read
                // (they wrote dS'_j after loading it)
                if (j + 1 < n && !(ok = issue_dp(j + 1))) break;
            }
            mma_commit(bar(L::bDQFinal));
            mbar_wait_drain(bar(L::bDQFinal), 0);
        }
        __syncwarp();
    } else {
        // ============================================================ compute
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const int q_idx = U.row0 + r;
        const bool row_ok = q_idx < U.Lq;
        const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
        // row terms: -LSE/scale and -D (zero-filled for rows past the sequence)
        float nlse = 0.f, nd = 0.f;
        if (row_ok) {
            const float4 t = p.rowx[U.st_row0 + (int64_t)q_idx * U.st_rs];
            nlse = t.x + t.y;
            nd = t.z + t.w;
        }
        const float sl2 = p.scale_log2;
        const KeyRange kr = key_range(p.mask, p.window, q_idx, U.delta, U.Lkv);
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const uint32_t sb = (j & 1) * 128;
            ok = warp_wait_d(bar(L::bSFull + (j & 1)), (j >> 1) & 1, wc, 8) &&
                 warp_wait_d(bar(L::bDPFull), j & 1, wc, 9);
            if (!ok) break;
            tc_fence_after();
            const int k0 = (U.kt0 + j) * kTileN;
            const int c_lo = kr.lo - k0, c_hi = kr.hi - k0;  // visible: c_lo <= c < c_hi
            uint32_t ds[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t s[32], dp[32];
                tmem_ld32(t_lane + sb + c * 32, s);
                tmem_ld32(t_lane + L::kColDP + c * 32, dp);
                tmem_ld_wait_regs<32>(s);
                tmem_ld_wait_regs<32>(dp);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int col = c * 32 + e;
                    float pr[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float x = (__uint_as_float(s[e + u]) + nlse) * sl2;
                        const bool vis = row_ok && col + u >= c_lo && col + u < c_hi;
                        pr[u] = vis ? ex2_approx(x) : 0.f;
                    }
                    const float g0 = pr[0] * (__uint_as_float(dp[e]) + nd);
                    const float g1 = pr[1] * (__uint_as_float(dp[e + 1]) + nd);
                    ds[col / 2] = pack2<kBf16>(g0, g1);
                }
            }
            tmem_st32(t_lane + sb, ds);
            tmem_st32(t_lane + sb + 32, ds + 32);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(L::bDSReady + (j & 1)));
        }
        // epilogue: dQ = scale * accumulated dS' K, in the I/O dtype
        if (ok) ok = warp_wait_d(bar(L::bDQFinal), 0, wc, 10);
        if (ok) {
            tc_fence_after();
            uint16_t *dst_row = dq + U.io_row0 + (int64_t)q_idx * U.io_rs;
            const float sc = p.scale;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(t_lane + L::kColDQ + c * 32, v);
                tmem_ld_wait_regs<32>(v);
                if (row_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(dst_row + c * 32);
                    auto g = [&](int e) { return __uint_as_float(v[e]) * sc; };
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        dst[w] = make_uint4(pack2<kBf16>(g(8 * w), g(8 * w + 1)),
                                            pack2<kBf16>(g(8 * w + 2), g(8 * w + 3)),
                                            pack2<kBf16>(g(8 * w + 4), g(8 * w + 5)),
                                            pack2<kBf16>(g(8 * w + 6), g(8 * w + 7)));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int D, bool kBf16, bool kPacked>
cudaError_t launch_dq_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &tdo, const BwdParams &p, int q_tiles, bool overlap,
                        cudaStream_t stream) {
    using L = DqLayout<D>;
    auto kern = bwd_dq_kernel<D, kBf16, kPacked>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
    if (e != cudaSuccess) return e;
    const int grid = q_tiles * p.bh;
    // overlap: start as the main kernel's last CTAs start (they signal once
    // the row terms this pass reads are complete); it shares no data with
    // the main kernel
    if (overlap)
        return launch_overlapped(kern, dim3(grid), dim3(kDqThreads), L::kSmemAlloc, stream, tq, tk, tv,
                                 tdo, p, q_tiles);
    kern<<<grid, kDqThreads, L::kSmemAlloc, stream>>>(tq, tk, tv, tdo, p, q_tiles);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tdo, const BwdParams &p, int q_tiles, int d, bool bf16,
                          bool packed, bool overlap, cudaStream_t stream) {
#define SDPA_DQ_CASE(D_, BF_, PK_)                                             \
    if (d == D_ && bf16 == BF_ && packed == PK_)                               \
        return launch_dq_t<D_, BF_, PK_>(tq, tk, tv, tdo, p, q_tiles, overlap, stream);
    SDPA_DQ_CASE(64, true, false)
    SDPA_DQ_CASE(64, true, true)
    SDPA_DQ_CASE(64, false, false)
    SDPA_DQ_CASE(64, false, true)
    SDPA_DQ_CASE(128, true, false)
    SDPA_DQ_CASE(128, true, true)
    SDPA_DQ_CASE(128, false, false)
    SDPA_DQ_CASE(128, false, true)
#undef SDPA_DQ_CASE
    return cudaErrorInvalidValue;
}

}  // namespace sdpa
