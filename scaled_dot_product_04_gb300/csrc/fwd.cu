// Fused attention forward for sm_103a: O = softmax(scale * Q K^T + mask) V and
// the per-row log-sum-exp, dense BHSD or packed THD.
//
// Operation: "Inside NVIDIA's cuDNN Graph API" (tradepoint.io), section 5
// "SDPA (Flash Attention) with causal masking" -- top-left causal alignment,
// fp32 intermediate and compute type.  Softmax runs in the base-2 domain with
// scale*log2(e) folded into one multiplier (cudnn-frontend PR #554, SM100
// FP8 d512 notes: scale_softmax_log2); LSE is converted back to the natural
// log on write-out.  Tiles wholly above the causal diagonal are never loaded
// or multiplied; only diagonal and ragged-tail tiles pay for masking
// (cudnn-frontend PR #554, SM80 backward notes on PARTIAL/GATE tile bounds).
//
// One CTA owns one 128-row query tile of one (batch, head) or (sequence,
// head) and streams the key/value tiles it may see:
//   warp 0      TMA producer: Q once, then K_j / V_j into a ring of stages;
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into TMEM (two S
//               buffers so S_{j+1} overlaps the softmax of S_j), then
//               O += P_j V_j with P_j read straight from TMEM;
//   warps 2..5  softmax: thread r owns query row r (= TMEM lane r); it reads
//               S_j, applies the mask, keeps the fp32 running max/sum,
//               writes P_j (bf16/fp16) back into the S_j columns, rescales O
//               in TMEM when the running max grows by more than 2^8, and
//               finally normalises O and writes O and LSE to global memory.
// TMEM columns: S buffers at 0 and 128, O at 256 (d columns).
//
// Packed layout: the Q/K/V tensor maps span exactly total_q / total_kv
// tokens, so a tile that steps past the packed total reads TMA zero fill and
// never the caller's capacity tail (cudnn-frontend PR #554, "clamp the f16
// THD K/V descriptors to the packed total"); keys of the next sequence that
// share a tile are masked to -inf before the exponent.
#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {
namespace {

template <int D>
struct FwdLayout {
    static constexpr int kChunks = D / 64;                // 128-byte swizzle columns per row
    static constexpr int kChunkBytes = kTileM * 128;      // 16 KiB: 128 rows x 64 elements
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    // K and V have rings of their own: a K stage is released once S = Q K^T
    // has read it, a V stage once O += P V has, so the next loads start early.
    static constexpr int kStages = (D == 128) ? 3 : 5;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTileBytes;
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kBar = kV + kStages * kTileBytes;
    static constexpr int bQFull = 0;
    static constexpr int bKFull = 1;
    static constexpr int bVFull = bKFull + kStages;
    static constexpr int bKEmpty = bVFull + kStages;
    static constexpr int bVEmpty = bKEmpty + kStages;
    static constexpr int bSFull = bVEmpty + kStages;  // two
    static constexpr int bPReady = bSFull + 2;
    static constexpr int bPVDone = bPReady + 1;
    static constexpr int bMmaIdle = bPVDone + 1;
    static constexpr int kNumBars = bMmaIdle + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;  // u32[0] TMEM base, u32[1] abort flag
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kSmemAlloc = kBytes + 1024;  // slack to align the base to 1024 B
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 256;
};

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only if the max grows by 2^8

// Each lane waits; the warp proceeds only if every lane saw the phase, so the
// warp-collective tcgen05.ld/st that follow stay convergent.
SDPA_DEV bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx &w, uint32_t site) {
    bool ok = mbar_wait(bar, parity, w, site);
    return __all_sync(0xffffffffu, ok);
}

template <int D, bool kBf16, bool kPacked>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);

    // ---------------------------------------------------------------- work unit
    // Units are ordered by query tile, latest (heaviest under the causal mask)
    // first, so the longest tiles start in the first wave.
    const int unit = blockIdx.x;
    const int qt = p.q_tiles - 1 - unit / p.bh;
    const int slice = unit % p.bh;  // dense: b*h index.  packed: seq*h + head
    int Lq, Lkv, tok_q0 = 0, tok_kv0 = 0, head = 0;
    int64_t o_row0, o_rs, lse_row0, lse_rs;
    if constexpr (!kPacked) {
        Lq = p.s_q;
        Lkv = p.s_kv;
        o_row0 = (int64_t)slice * p.s_q * D;
        o_rs = D;
        lse_row0 = (int64_t)slice * p.s_q;
        lse_rs = 1;
    } else {
        const int n = slice / p.h;
        head = slice % p.h;
        tok_q0 = p.cu_q[n];
        tok_kv0 = p.cu_kv[n];
        Lq = p.cu_q[n + 1] - tok_q0;
        Lkv = p.cu_kv[n + 1] - tok_kv0;
        o_row0 = ((int64_t)tok_q0 * p.h + head) * D;
        o_rs = (int64_t)p.h * D;
        lse_row0 = (int64_t)tok_q0 * p.h + head;
        lse_rs = p.h;
    }
    const int row0 = qt * kTileM;
    if (row0 >= Lq) return;  // packed: this sequence has fewer query tiles

    int n_kv = (Lkv + kTileN - 1) / kTileN;
    if (p.causal) {
        const int q_last = min(row0 + kTileM - 1, Lq - 1);
        n_kv = min(n_kv, q_last / kTileN + 1);
    }

    using io_t = uint16_t;
    io_t *const o_base = reinterpret_cast<io_t *>(p.o) + o_row0;

    if (n_kv == 0) {
        // No key is visible to any row of this tile: O = 0, LSE = -inf.
        if (threadIdx.x < kTileM) {
            const int r = row0 + threadIdx.x;
            if (r < Lq) {
                uint4 *dst = reinterpret_cast<uint4 *>(o_base + (int64_t)r * o_rs);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                if (p.lse) p.lse[lse_row0 + (int64_t)r * lse_rs] = -INFINITY;
            }
        }
        return;
    }

    auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(bar(L::bQFull), 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(bar(L::bKFull + s), 1);
            mbar_init(bar(L::bVFull + s), 1);
            mbar_init(bar(L::bKEmpty + s), 1);
            mbar_init(bar(L::bVEmpty + s), 1);
        }
        mbar_init(bar(L::bSFull + 0), 1);
        mbar_init(bar(L::bSFull + 1), 1);
        mbar_init(bar(L::bPReady), kTileM);
        mbar_init(bar(L::bPVDone), 1);
        mbar_init(bar(L::bMmaIdle), 1);
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
    const WaitCtx wc{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.err, kTagFwd};

    if (warp == 0) {
        // ============================================================ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const int qy = kPacked ? head : row0;
            const int qz = kPacked ? tok_q0 + row0 : slice;
            mbar_arrive_expect_tx(bar(L::bQFull), L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c)
                tma_load_3d(sbase + L::kQ + c * L::kChunkBytes, &tm_q, bar(L::bQFull), c * 64, qy,
                            qz);
            int issued = 0, issued_k = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % L::kStages, use = j / L::kStages;
                if (use > 0 && !mbar_wait(bar(L::bKEmpty + st), (use - 1) & 1, wc, 1)) break;
                const int ky = kPacked ? head : j * kTileN;
                const int kz = kPacked ? tok_kv0 + j * kTileN : slice;
                const uint32_t ks = sbase + L::kK + st * L::kTileBytes;
                const uint32_t vs = sbase + L::kV + st * L::kTileBytes;
                mbar_arrive_expect_tx(bar(L::bKFull + st), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(ks + c * L::kChunkBytes, &tm_k, bar(L::bKFull + st), c * 64, ky, kz);
                if (use > 0 && !mbar_wait(bar(L::bVEmpty + st), (use - 1) & 1, wc, 11)) {
                    issued_k = j + 1;
                    break;
                }
                mbar_arrive_expect_tx(bar(L::bVFull + st), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(vs + c * L::kChunkBytes, &tm_v, bar(L::bVFull + st), c * 64, ky, kz);
                issued = issued_k = j + 1;
            }
            // Every load issued must land before the CTA may exit.
            mbar_wait_drain(bar(L::bQFull), 0);
            for (int j = max(0, issued_k - L::kStages); j < issued_k; ++j)
                mbar_wait_drain(bar(L::bKFull + j % L::kStages), (j / L::kStages) & 1);
            for (int j = max(0, issued - L::kStages); j < issued; ++j)
                mbar_wait_drain(bar(L::bVFull + j % L::kStages), (j / L::kStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = make_idesc_f16(kTileM, kTileN, kBf16, false, false);
            constexpr uint32_t idesc_o = make_idesc_f16(kTileM, D, kBf16, false, true);
            // S = Q K^T: both operands K-major (head dim contiguous), 16 per step.
            auto issue_s = [&](int st, uint32_t col) {
                const uint32_t qs = sbase + L::kQ;
                const uint32_t ks = sbase + L::kK + st * L::kTileBytes;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k / 4) * L::kChunkBytes + (k % 4) * 32;
                    mma_ss(tmem + col, smem_desc_sw128(qs + off, 16, 1024),
                           smem_desc_sw128(ks + off, 16, 1024), idesc_s, k > 0);
                }
            };
            // O += P V: P from TMEM (two bf16 per column, 8 columns per 16 keys),
            // V MN-major (head dim contiguous); 64-wide head-dim halves are
            // 16 KiB apart (leading offset), 8-key groups 1 KiB apart.
            auto issue_pv = [&](int st, uint32_t pcol, bool acc) {
                const uint32_t vs = sbase + L::kV + st * L::kTileBytes;
#pragma unroll
                for (int k = 0; k < kTileN / 16; ++k) {
                    mma_ts(tmem + L::kColO, tmem + pcol + k * 8,
                           smem_desc_sw128(vs + k * 2048, L::kChunkBytes, 1024), idesc_o,
                           (acc || k > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(bar(L::bQFull), 0, wc, 2) && mbar_wait(bar(L::bKFull), 0, wc, 3);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                mma_commit(bar(L::bSFull + 0));
                mma_commit(bar(L::bKEmpty + 0));
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) {
                    const int st1 = (j + 1) % L::kStages, use1 = (j + 1) / L::kStages;
                    ok = mbar_wait(bar(L::bKFull + st1), use1 & 1, wc, 4);
                    // S_{j+1} reuses the columns that held P_{j-1}: wait until the
                    // P_{j-1} V_{j-1} product that reads them has retired.
                    if (ok && j >= 1) ok = mbar_wait(bar(L::bPVDone), (j - 1) & 1, wc, 5);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(st1, ((j + 1) & 1) * 128);
                    mma_commit(bar(L::bSFull + ((j + 1) & 1)));
                    mma_commit(bar(L::bKEmpty + st1));
                }
                ok = mbar_wait(bar(L::bPReady), j & 1, wc, 6) &&
                     mbar_wait(bar(L::bVFull + j % L::kStages), (j / L::kStages) & 1, wc, 7);
                if (!ok) break;
                tc_fence_after();
                issue_pv(j % L::kStages, (j & 1) * 128, j > 0);
                mma_commit(bar(L::bPVDone));
                mma_commit(bar(L::bVEmpty + j % L::kStages));
            }
            // Let every MMA issued above retire before TMEM is released.
            mma_commit(bar(L::bMmaIdle));
            mbar_wait_drain(bar(L::bMmaIdle), 0);
        }
        __syncwarp();
    } else {
        // ============================================================ softmax
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // row of the tile == TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
        const int q_idx = row0 + r;
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY;  // running max actually used as exponent base (log2 units)
        float l = 0.f;             // running sum of P
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const uint32_t cs = (j & 1) * 128;
            ok = warp_wait(bar(L::bSFull + (j & 1)), (j >> 1) & 1, wc, 8);
            if (!ok) break;
            tc_fence_after();
            uint32_t s[kTileN];
#pragma unroll
            for (int c = 0; c < kTileN / 32; ++c) tmem_ld32(t_lane + cs + c * 32, s + c * 32);
            tmem_ld_wait_regs<kTileN>(s);

            const int k0 = j * kTileN;
            if ((k0 + kTileN > Lkv) || (p.causal && k0 + kTileN - 1 > row0)) {
                int lim = Lkv - k0;  // columns c < lim are visible
                if (p.causal) lim = min(lim, q_idx - k0 + 1);
#pragma unroll
                for (int c = 0; c < kTileN; ++c)
                    if (c >= lim) s[c] = __float_as_uint(-INFINITY);
            }
            // row max: four independent chains of 3-input max
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kTileN; c += 8) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    mx4[u] = fmax3(mx4[u], __uint_as_float(s[c + 2 * u]),
                                   __uint_as_float(s[c + 2 * u + 1]));
            }
            const float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
            const float m_tile = mx * sl2;
            float alpha = 1.f;
            bool rescale = false;
            if (m_tile > m_used + kRescaleThreshold) {
                rescale = true;
                alpha = ex2_approx(m_used - m_tile);
                m_used = m_tile;
                l *= alpha;
            }
            const float base = (m_used == -INFINITY) ? 0.f : m_used;
            const uint64_t sl2_2 = f2_pack(sl2, sl2), nbase_2 = f2_pack(-base, -base);
            // P = exp2(s * scale*log2e - base), pairs packed in place into s[0..64)
            uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
            for (int i = 0; i < kTileN / 2; ++i) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                                 sl2_2, nbase_2),
                          x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                sum2[i & 3] = f2_add(sum2[i & 3], f2_pack(p0, p1));
                s[i] = pack2<kBf16>(p0, p1);  // i <= 2i: packs in place
            }
            {
                float a0, a1;
                f2_unpack(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), a0, a1);
                l += a0 + a1;
            }
            tmem_st32(t_lane + cs, s);
            tmem_st32(t_lane + cs + 32, s + 32);

            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                // O holds P_0..P_{j-1} V products; it may be rescaled only once
                // the last of them has retired.
                ok = warp_wait(bar(L::bPVDone), (j - 1) & 1, wc, 9);
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + L::kColO + c * 32, o);
                    tmem_ld_wait_regs<32>(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(t_lane + L::kColO + c * 32, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(L::bPReady));
        }
        if (ok) ok = warp_wait(bar(L::bPVDone), (n_kv - 1) & 1, wc, 10);
        if (ok) {
            tc_fence_after();
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            const bool row_ok = q_idx < Lq;
            io_t *orow = o_base + (int64_t)q_idx * o_rs;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(t_lane + L::kColO + c * 32, o);
                tmem_ld_wait_regs<32>(o);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack2<kBf16>(__uint_as_float(o[2 * i]) * inv_l,
                                         __uint_as_float(o[2 * i + 1]) * inv_l);
                if (row_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            if (row_ok && p.lse)
                p.lse[lse_row0 + (int64_t)q_idx * lse_rs] =
                    (l > 0.f) ? (m_used + lg2_approx(l)) * kLn2 : -INFINITY;
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
cudaError_t launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const FwdParams &p, int grid, cudaStream_t stream,
                         const KernelTimer &timer) {
    using L = FwdLayout<D>;
    auto kern = fwd_kernel<D, kBf16, kPacked>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmemAlloc);
    if (e != cudaSuccess) return e;
    if (timer.start) cudaEventRecord(timer.start, stream);
    kern<<<grid, 192, L::kSmemAlloc, stream>>>(tq, tk, tv, p);
    e = cudaGetLastError();
    if (timer.stop) cudaEventRecord(timer.stop, stream);
    return e;
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdParams &p, int d, bool bf16, bool packed, int grid,
                       cudaStream_t stream, const KernelTimer &timer) {
#define SDPA_FWD_CASE(D_, BF_, PK_)                                            \
    if (d == D_ && bf16 == BF_ && packed == PK_)                               \
        return launch_fwd_t<D_, BF_, PK_>(tq, tk, tv, p, grid, stream, timer);
    SDPA_FWD_CASE(64, true, false)
    SDPA_FWD_CASE(64, true, true)
    SDPA_FWD_CASE(64, false, false)
    SDPA_FWD_CASE(64, false, true)
    SDPA_FWD_CASE(128, true, false)
    SDPA_FWD_CASE(128, true, true)
    SDPA_FWD_CASE(128, false, false)
    SDPA_FWD_CASE(128, false, true)
#undef SDPA_FWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace sdpa
