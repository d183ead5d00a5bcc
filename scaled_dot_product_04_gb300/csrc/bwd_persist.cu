// Attention backward main kernel, persistent form: one CTA per SM, each
// walking many (key/value slice, key tile) units instead of one.
//
// Same products, layouts, warp roles and per-tile protocol as bwd_main_kernel
// (bwd.cu), whose header gives the math (S'^T = K Q^T - LSE/scale with the
// row terms as a tf32 K-step, P^T = exp2(...), dV += P^T dO, dS'^T = P^T o
// dP'^T, dQ = dS' K added into the fp32 accumulator, dK += dS'^T Q).  What
// the one-CTA-per-unit form pays per unit -- barrier set-up, TMEM allocation,
// the first K/V/Q loads with nothing to overlap them, the dK/dV write-out and
// the CTA's exit before the next CTA starts on the SM -- weighs heavily when
// units are short (a few query tiles each: short packed sequences, d = 64,
// short dense problems).  Here the set-up happens once per CTA, the next
// unit's Q and dO load while the current unit ends, its K and V come from L2
// (prefetched when the unit is taken), and its first S^T and dP^T products and
// softmax run while the dQ warps write the previous unit's dK and dV.
//
// Units are taken dynamically: the producer warp takes the next index of the
// unit list from a counter in global memory (zeroed by the preprocess kernel)
// when it has issued the current unit's loads, and hands it to the other roles
// through a ring of kRing slots in shared memory (bUFull / bUEmpty); -1 ends
// the list.  The list is the one-CTA-per-unit kernel's (dense: slice groups,
// key tile major; packed: sequences longest first, from a table each CTA
// builds in shared memory, at most kPersistSeqMax sequences), so the heaviest
// units start first and the resident CTAs share a few slices in L2.
//
// Across units every per-tile barrier keeps counting (phase parities follow
// the CTA's running tile count), and these join consecutive units:
//   bVFree     committed after a unit's last dP'^T (the last reader of V):
//              the next unit's V loads (bVFull) a tile before the unit ends;
//   bKFree     committed after its last dQ (or, without dQ, its last S'^T):
//              the next unit's K loads (bKVFull) ahead of that tile's dQ
//              boxes in the SM's copy queue;
//   bUnitDone  committed after its last product: the dK, dV accumulators may
//              be read out;
//   bAccFree   the dQ warps have read dK and dV out of TMEM: the next unit's
//              first dV and dK products may overwrite them.
#include "bwd_layout.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {
namespace {

template <int D>
struct PersistLayout {
    using L = BwdLayout<D>;
    static constexpr int kRing = 4;
    static constexpr int kRingReaders = 1 + 8 + 4;  // MMA thread, compute warps, dQ warps
    static constexpr int kPBar = (L::kBytes + 15) & ~15;
    static constexpr int bUFull = 0;  // kRing
    static constexpr int bUEmpty = kRing;  // kRing
    static constexpr int bUnitDone = 2 * kRing;
    static constexpr int bAccFree = 2 * kRing + 1;
    static constexpr int bVFull = 2 * kRing + 2;  // K is the layout's bKVFull
    static constexpr int bKFree = 2 * kRing + 3;
    static constexpr int bVFree = 2 * kRing + 4;
    static constexpr int kNumPBars = 2 * kRing + 5;
    static constexpr int kRingSlots = kPBar + kNumPBars * 8;
    static constexpr int kTable = kRingSlots + 4 * kRing;
    // packed: cu_q, cu_kv (ns + 1 each), order (ns), first unit (ns + 1)
    static constexpr int kTableBytes = 4 * (4 * kPersistSeqMax + 3);
    static constexpr int kBytes = kTable + kTableBytes;
};
static_assert(PersistLayout<128>::kBytes <= 232448, "persistent backward exceeds shared memory");

struct PUnit {
    int slice, hk, Lq, Lkv, tok_q0, tok_kv0, q_slice0, k0, delta, qt_begin, n_q, n_it;
    RowMap km;
};

// Unit u of the list.  cq, ckv, order, first: the packed table.
template <int D, bool kPacked>
SDPA_DEV PUnit decode_punit(const BwdParams &p, int u, const int *cq, const int *ckv, const int *order,
                            const int *first) {
    PUnit U;
    int kt;
    if constexpr (kPacked) {
        int lo = 0, hi = p.num_seqs;  // first[lo] <= u < first[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (first[mid] <= u) lo = mid;
            else hi = mid;
        }
        const int n = order[lo], local = u - first[lo];
        U.tok_q0 = cq[n];
        U.tok_kv0 = ckv[n];
        U.Lq = cq[n + 1] - U.tok_q0;
        U.Lkv = ckv[n + 1] - U.tok_kv0;
        // within the sequence: key/value heads in groups of p.slice_group, key
        // tile major within a group
        const int n_kt = (U.Lkv + kTileN - 1) / kTileN;
        const int per_group = p.slice_group * n_kt;
        const int group_i = local / per_group;
        const int in_group = local - group_i * per_group;
        const int group_n = min(p.slice_group, p.h_kv - group_i * p.slice_group);
        kt = in_group / group_n;
        U.slice = n * p.h_kv + group_i * p.slice_group + in_group % group_n;
    } else {
        const int per_group = p.slice_group * p.kv_tiles;
        const int group_i = u / per_group;
        const int in_group = u - group_i * per_group;
        const int group_n = min(p.slice_group, p.kv_slices - group_i * p.slice_group);
        U.slice = group_i * p.slice_group + in_group % group_n;
        kt = in_group / group_n;
        U.tok_q0 = U.tok_kv0 = 0;
        U.Lq = p.s_q;
        U.Lkv = p.s_kv;
    }
    U.hk = U.slice % p.h_kv;
    if constexpr (!kPacked) {
        U.q_slice0 = (U.slice / p.h_kv) * p.h + U.hk * p.group;
        U.km = {(int64_t)U.slice * p.s_kv * D, D, 0};
    } else {
        U.q_slice0 = 0;
        U.km = {((int64_t)U.tok_kv0 * p.h_kv + U.hk) * D, (int64_t)p.h_kv * D, 0};
    }
    U.k0 = kt * kTileN;
    // query rows that see at least one key of the tile: a causal mask needs
    // i + delta >= k0, a window i + delta - window <= k_last
    U.delta = mask_delta(p.mask, U.Lq, U.Lkv);
    const int k_last = min(U.k0 + kTileN, U.Lkv) - 1;
    const int row_lo = p.mask != kMaskNone ? max(0, U.k0 - U.delta) : 0;
    const int row_hi = p.window >= 0 ? min(U.Lq, k_last - U.delta + p.window + 1) : U.Lq;
    U.qt_begin = row_lo / kTileM;
    U.n_q = row_hi > row_lo ? (row_hi + kTileM - 1) / kTileM - U.qt_begin : 0;
    U.n_it = U.n_q * p.group;  // (query head, query tile) pairs, head-major
    return U;
}

template <int D, bool kBf16, bool kPacked>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_rx,
                       const BwdParams p) {
    using L = BwdLayout<D>;
    using PL = PersistLayout<D>;
    constexpr int R = PL::kRing;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();
    auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
    auto pbar = [&](int i) -> uint32_t { return sbase + PL::kPBar + 8u * i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *ring = reinterpret_cast<volatile int *>(smem + PL::kRingSlots);

    // ---------------------------------------------------------------- unit list
    int *cq = reinterpret_cast<int *>(smem + PL::kTable);
    int *ckv = cq + (kPersistSeqMax + 1);
    int *order = ckv + (kPersistSeqMax + 1);
    int *first_u = order + kPersistSeqMax;  // kPersistSeqMax + 1 entries
    int n_units;
    if constexpr (kPacked) {
        const int ns = p.num_seqs;  // <= kPersistSeqMax (the host checks)
        for (int i = threadIdx.x; i <= ns; i += blockDim.x) {
            cq[i] = p.cu_q[i];
            ckv[i] = p.cu_kv[i];
        }
        __syncthreads();
        // sequences by query tiles, most first (ties in sequence order)
        for (int n = threadIdx.x; n < ns; n += blockDim.x) {
            const int tn = (cq[n + 1] - cq[n] + kTileM - 1) / kTileM;
            int rank = 0;
            for (int m = 0; m < ns; ++m) {
                const int tm = (cq[m + 1] - cq[m] + kTileM - 1) / kTileM;
                rank += (tm > tn || (tm == tn && m < n)) ? 1 : 0;
            }
            order[rank] = n;
        }
        __syncthreads();
        if (threadIdx.x == 0) {  // first unit of each sequence in table order
            int run = 0;
            for (int i = 0; i < ns; ++i) {
                first_u[i] = run;
                const int n = order[i];
                run += (ckv[n + 1] - ckv[n] + kTileN - 1) / kTileN * p.h_kv;
            }
            first_u[ns] = run;
        }
        __syncthreads();
        n_units = first_u[ns];
    } else {
        n_units = p.kv_tiles * p.kv_slices;
    }
    if ((int)blockIdx.x >= n_units || (sbase & 1023u) != 0) {
        // No unit for this CTA (the host sizes packed grids by an upper
        // bound), or a misaligned base (reported).  The CTA still waits for
        // the preprocess grid: the kernel behind this one (the deterministic
        // dQ pass, which reads the row terms without a wait of its own) may
        // start once every CTA has signalled or exited.
        if ((sbase & 1023u) != 0 && threadIdx.x == 0) atomicCAS(p.err, 0u, (kTagBwdMain << 16) | 0xfffu);
        griddep_wait();
        return;
    }
    auto unit = [&](int u) { return decode_punit<D, kPacked>(p, u, cq, ckv, order, first_u); };

    // ---------------------------------------------------------------- set-up
    if (threadIdx.x == 0) {
        mbar_init(bar(L::bKVFull), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(L::bQFull + s), 1);
            mbar_init(bar(L::bDOFull + s), 1);
            mbar_init(bar(L::bQEmpty + s), 1);
            if (s < L::kDOStages) mbar_init(bar(L::bDOEmpty + s), 1);
        }
        mbar_init(bar(L::bSFull), 1);
        mbar_init(bar(L::bDPFull), 1);
        mbar_init(bar(L::bPReady), 256);
        mbar_init(bar(L::bDSReady), 256);
        mbar_init(bar(L::bDQFull), 1);
        mbar_init(bar(L::bDQFree), 128);
        mbar_init(bar(L::bMmaIdle), 1);
        for (int r = 0; r < R; ++r) {
            mbar_init(pbar(PL::bUFull + r), 1);
            mbar_init(pbar(PL::bUEmpty + r), PL::kRingReaders);
        }
        mbar_init(pbar(PL::bUnitDone), 1);
        mbar_init(pbar(PL::bAccFree), 128);
        mbar_init(pbar(PL::bVFull), 1);
        mbar_init(pbar(PL::bKFree), 1);
        mbar_init(pbar(PL::bVFree), 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kMisc, L::kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x >= 128 && threadIdx.x < 256) {
        // the constant A operands of the row-term K-steps (as bwd_main_kernel)
        const int r = threadIdx.x - 128;
        reinterpret_cast<float4 *>(smem + L::kAexS)[r] = make_float4(0.5f, 0.5f, 0.f, 0.f);
        reinterpret_cast<float4 *>(smem + L::kAexD)[r] = make_float4(0.f, 0.f, 0.5f, 0.5f);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const WaitCtx wc{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.err, kTagBwdMain};

    if (warp == 0) {
        // ============================================================ producer
        // Per unit: take it, hand it on, then load Q, row terms and dO of its
        // first query tile, V and K (each once the previous unit's products
        // are done with it), and the rest of its query tiles.  The Q and dO
        // rings count tiles across units.
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
            tma_prefetch_desc(&tm_rx);
        }
        // The row terms, the zeroed unit counter and dQ accumulator come from
        // the preprocess grid; once it is done, the kernel behind this one may
        // start filling freed SMs.
        bool pre_done = false;
        auto after_preprocess = [&]() {
            if (pre_done) return;
            griddep_wait();
            if (lane == 0) griddep_launch_dependents();
            pre_done = true;
        };
        int gq = 0, gdo = 0, kv = 0, nv = 0;  // Q tiles, dO tiles, K and V tiles issued
        bool ok = true;
        // Q_G (freed by dK_{G-2}) is needed first, by S^T_G; dO_G (freed by
        // dV_{G-kDOStages}) only by dP^T_G.  i: the tile's index in unit U.
        auto q_coords = [&](const PUnit &U, int i, int &qy, int &qz) {
            const int q0 = (U.qt_begin + i % U.n_q) * kTileM;
            qy = kPacked ? U.hk * p.group + i / U.n_q : q0;
            qz = kPacked ? U.tok_q0 + q0 : U.q_slice0 + i / U.n_q;
        };
        auto load_q = [&](const PUnit &U, int i) -> bool {
            const int G = gq, st = G & 1, use = G >> 1;
            int qy, qz;
            q_coords(U, i, qy, qz);
            if (use > 0 && !warp_wait_b(bar(L::bQEmpty + st), (use - 1) & 1, wc, 18)) return false;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(L::bQFull + st), L::kTileBytes + L::kRowXBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kQ + st * L::kTileBytes + c * L::kChunkBytes, &tm_q,
                                bar(L::bQFull + st), c * 64, qy, qz);
                tma_load_3d(sbase + L::kRowX + st * L::kRowXBytes, &tm_rx, bar(L::bQFull + st), 0, qy, qz);
            }
            gq = G + 1;
            return true;
        };
        auto load_do = [&](const PUnit &U, int i) -> bool {
            const int G = gdo, dst = G % L::kDOStages, duse = G / L::kDOStages;
            int qy, qz;
            q_coords(U, i, qy, qz);
            if (duse > 0 && !warp_wait_b(bar(L::bDOEmpty + dst), (duse - 1) & 1, wc, 1)) return false;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(L::bDOFull + dst), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kDO + dst * L::kTileBytes + c * L::kChunkBytes, &tm_do,
                                bar(L::bDOFull + dst), c * 64, qy, qz);
            }
            gdo = G + 1;
            return true;
        };
        auto kv_coords = [&](const PUnit &U, int &ky, int &kz) {
            ky = kPacked ? U.hk : U.k0;
            kz = kPacked ? U.tok_kv0 + U.k0 : U.slice;
        };
        auto load_k = [&](const PUnit &U) {
            int ky, kz;
            kv_coords(U, ky, kz);
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(L::bKVFull), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kK + c * L::kChunkBytes, &tm_k, bar(L::bKVFull), c * 64, ky, kz);
            }
        };
        auto load_v = [&](const PUnit &U) {
            int ky, kz;
            kv_coords(U, ky, kz);
            if (lane == 0) {
                mbar_arrive_expect_tx(pbar(PL::bVFull), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kV + c * L::kChunkBytes, &tm_v, pbar(PL::bVFull), c * 64, ky, kz);
            }
        };
        for (int k = 0; ok; ++k) {
            const int slot = k % R;
            if (k >= R && !(ok = warp_wait_b(pbar(PL::bUEmpty + slot), ((k / R) - 1) & 1, wc, 21))) break;
            int u = blockIdx.x;  // the first unit needs no counter
            if (k > 0) {
                after_preprocess();
                int t = 0;
                if (lane == 0) t = (int)atomicAdd(p.unit_ctr, 1u);
                u = (int)gridDim.x + __shfl_sync(0xffffffffu, t, 0);
                if (u >= n_units) u = -1;
            }
            if (lane == 0) {
                ring[slot] = u;
                mbar_arrive(pbar(PL::bUFull + slot));
            }
            if (u < 0) break;
            const PUnit U = unit(u);
            if (U.n_q == 0) continue;  // the dQ warps write zeros
            if (kv == 0) {
                load_k(U);  // inputs only: no wait for the preprocess grid
                load_v(U);
                ++kv;
                ++nv;
                after_preprocess();
                ok = load_q(U, 0) && load_do(U, 0);
            } else {
                if (lane == 0) {
                    int ky, kz;
                    kv_coords(U, ky, kz);
                    for (int c = 0; c < L::kChunks; ++c) {
                        tma_prefetch_l2_3d(&tm_k, c * 64, ky, kz);
                        tma_prefetch_l2_3d(&tm_v, c * 64, ky, kz);
                    }
                }
                // the first dO waits for the previous unit's last dV, which
                // comes after its last readers of V and K
                ok = load_q(U, 0) && warp_wait_b(pbar(PL::bVFree), (kv - 1) & 1, wc, 19);
                if (!ok) break;
                load_v(U);
                ++nv;
                if (!(ok = warp_wait_b(pbar(PL::bKFree), (kv - 1) & 1, wc, 25))) break;
                load_k(U);
                ++kv;
                ok = load_do(U, 0);
            }
            for (int i = 1; ok && i < U.n_it; ++i) ok = load_q(U, i) && load_do(U, i);
        }
        after_preprocess();
        if (lane == 0) {
            // every load issued lands before the CTA may exit
            if (kv > 0) mbar_wait_drain(bar(L::bKVFull), (kv - 1) & 1);
            if (nv > 0) mbar_wait_drain(pbar(PL::bVFull), (nv - 1) & 1);
            for (int i = max(0, gq - 2); i < gq; ++i) mbar_wait_drain(bar(L::bQFull + (i & 1)), (i >> 1) & 1);
            for (int i = max(0, gdo - L::kDOStages); i < gdo; ++i)
                mbar_wait_drain(bar(L::bDOFull + i % L::kDOStages), (i / L::kDOStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_sq = make_idesc_f16(128, 128, kBf16, false, false);
            constexpr uint32_t id_mn = make_idesc_f16(128, D, kBf16, false, true);
            constexpr uint32_t id_dq = make_idesc_f16(128, D, kBf16, true, true);
            constexpr uint32_t id_rx = make_idesc_tf32(128, 128);
            // operand descriptors as in bwd_main_kernel
            constexpr uint32_t kChunk16 = L::kChunkBytes >> 4, kTile16 = L::kTileBytes >> 4;
            auto kstep = [](int k) -> uint32_t { return (uint32_t)((k >> 2) * kChunk16 + (k & 3) * 2); };
            const uint64_t dK_k = smem_desc_sw128(sbase + L::kK, 16, 1024);
            const uint64_t dK_mn = smem_desc_sw128(sbase + L::kK, L::kChunkBytes, 1024);
            const uint64_t dV_k = smem_desc_sw128(sbase + L::kV, 16, 1024);
            const uint64_t dQ_k = smem_desc_sw128(sbase + L::kQ, 16, 1024);
            const uint64_t dQ_mn = smem_desc_sw128(sbase + L::kQ, L::kChunkBytes, 1024);
            const uint64_t dDO_k = smem_desc_sw128(sbase + L::kDO, 16, 1024);
            const uint64_t dDO_mn = smem_desc_sw128(sbase + L::kDO, L::kChunkBytes, 1024);
            const uint64_t dDS_k = smem_desc_sw128(sbase + L::kDS, 16, 1024);
            const uint64_t dDS_mn = smem_desc_sw128(sbase + L::kDS, L::kChunkBytes, 1024);
            const uint64_t dAS = smem_desc_plain(sbase + L::kAexS, 0, 128);
            const uint64_t dAD = smem_desc_plain(sbase + L::kAexD, 0, 128);
            const uint64_t dRX = smem_desc_plain(sbase + L::kRowX, 0, 128);
            constexpr uint32_t kRowX16 = L::kRowXBytes >> 4;
            auto issue_kmajor = [&](uint64_t a, uint64_t b, uint64_t a_ex, int st, uint32_t col) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss(tmem + col, a + kstep(k), b + kstep(k), id_sq, k > 0);
                mma_ss_tf32(tmem + col, a_ex, dRX + st * kRowX16, id_rx, 1u);
            };
            const bool do_dq = !p.deterministic;
            int g = 0, kv = 0;  // tiles and live units before the current unit
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int slot = k % R;
                if (!(ok = mbar_wait_lean(pbar(PL::bUFull + slot), (k / R) & 1, wc, 22))) break;
                const int u = ring[slot];
                mbar_arrive(pbar(PL::bUEmpty + slot));
                if (u < 0) break;
                const PUnit U = unit(u);
                if (U.n_q == 0) continue;
                // The unit's first S'^T and dP'^T.  The previous unit's last
                // dV, which reads P^T from the S^T columns, is complete: K is
                // loaded only after its last dQ (or S'^T), issued after that
                // dV.  At d = 128 its last dQ shares the dP^T columns and must
                // have been read out.  A one-tile unit's first products are
                // its last readers of K (without dQ) and of V.
                {
                    const int st = g & 1, dst = g % L::kDOStages;
                    ok = mbar_wait_lean(bar(L::bKVFull), kv & 1, wc, 2) &&
                         mbar_wait_lean(bar(L::bQFull + st), (g >> 1) & 1, wc, 3);
                    if (!ok) break;
                    tc_fence_after();
                    issue_kmajor(dK_k, dQ_k + st * kTile16, dAS, st, L::kColS);
                    mma_commit(bar(L::bSFull));
                    if (U.n_it == 1 && !do_dq) mma_commit(pbar(PL::bKFree));
                    ok = mbar_wait_lean(pbar(PL::bVFull), kv & 1, wc, 26) &&
                         mbar_wait_lean(bar(L::bDOFull + dst), (g / L::kDOStages) & 1, wc, 4);
                    if (ok && do_dq && L::kDQAliasDP && g > 0)
                        ok = mbar_wait_lean(bar(L::bDQFree), (g - 1) & 1, wc, 11);
                    if (!ok) break;
                    tc_fence_after();
                    issue_kmajor(dV_k, dDO_k + dst * kTile16, dAD, st, L::kColDP);
                    mma_commit(bar(L::bDPFull));
                    if (U.n_it == 1) mma_commit(pbar(PL::bVFree));
                }
                for (int i = 0; ok && i < U.n_it; ++i) {
                    const int G = g + i;
                    const int st = G & 1;
                    const int dst = G % L::kDOStages;
                    ok = mbar_wait_lean(bar(L::bPReady), G & 1, wc, 5);
                    // the unit's first dV and dK overwrite the accumulators
                    // that the previous unit's epilogue reads out
                    if (ok && i == 0 && kv > 0) ok = mbar_wait_lean(pbar(PL::bAccFree), (kv - 1) & 1, wc, 20);
                    if (!ok) break;
                    tc_fence_after();
                    {  // dV += P^T dO
                        const uint64_t b = dDO_mn + dst * kTile16;
#pragma unroll
                        for (int k = 0; k < 128 / 16; ++k)
                            mma_ts(tmem + L::kColDV, tmem + L::kColS + (k >> 2) * 64 + (k & 3) * 8,
                                   b + k * 128, id_mn, (i > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(L::bDOEmpty + dst));  // also: dV has read P^T
                    if (i + 1 < U.n_it) {  // S'^T_{G+1}, once dV has read P^T_G
                        const int st1 = (G + 1) & 1;
                        ok = mbar_wait_lean(bar(L::bQFull + st1), ((G + 1) >> 1) & 1, wc, 6) &&
                             mbar_wait_lean(bar(L::bDOEmpty + dst), (G / L::kDOStages) & 1, wc, 7);
                        if (!ok) break;
                        tc_fence_after();
                        issue_kmajor(dK_k, dQ_k + st1 * kTile16, dAS, st1, L::kColS);
                        mma_commit(bar(L::bSFull));
                        if (i + 2 == U.n_it && !do_dq) mma_commit(pbar(PL::bKFree));
                    }
                    ok = mbar_wait_lean(bar(L::bDSReady), G & 1, wc, 8);
                    if (ok && do_dq && !L::kDQAliasDP && G > 0)
                        ok = mbar_wait_lean(bar(L::bDQFree), (G - 1) & 1, wc, 9);
                    if (!ok) break;
                    tc_fence_after();
                    if (do_dq) {  // dQ_G = dS' K
#pragma unroll
                        for (int k = 0; k < 128 / 16; ++k)
                            mma_ss(tmem + L::kColDQ, dDS_mn + k * 128, dK_mn + k * 128, id_dq, k > 0);
                        mma_commit(bar(L::bDQFull));
                        if (i + 1 == U.n_it) mma_commit(pbar(PL::bKFree));
                    }
                    {  // dK += dS'^T Q
                        const uint64_t b = dQ_mn + st * kTile16;
#pragma unroll
                        for (int k = 0; k < 128 / 16; ++k)
                            mma_ss(tmem + L::kColDK, dDS_k + kstep(k), b + k * 128, id_mn,
                                   (i > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(L::bQEmpty + st));  // also: dK and dQ have read dS'
                    if (i + 1 < U.n_it) {  // dP'^T_{G+1}
                        const int dst1 = (G + 1) % L::kDOStages;
                        ok = mbar_wait_lean(bar(L::bDOFull + dst1), ((G + 1) / L::kDOStages) & 1, wc, 10);
                        if (ok && do_dq && L::kDQAliasDP) ok = mbar_wait_lean(bar(L::bDQFree), G & 1, wc, 11);
                        if (!ok) break;
                        tc_fence_after();
                        issue_kmajor(dV_k, dDO_k + dst1 * kTile16, dAD, (G + 1) & 1, L::kColDP);
                        mma_commit(bar(L::bDPFull));
                        if (i + 2 == U.n_it) mma_commit(pbar(PL::bVFree));
                    }
                }
                if (!ok) break;
                mma_commit(pbar(PL::bUnitDone));  // dK, dV complete
                g += U.n_it;
                ++kv;
            }
            mma_commit(bar(L::bMmaIdle));
            mbar_wait_drain(bar(L::bMmaIdle), 0);
        }
        __syncwarp();
    } else if (warp < 10) {
        // ============================================================ compute
        // As in bwd_main_kernel: group grp owns queries [64 grp, 64 grp + 64)
        // of every tile for all 128 key rows (thread = key row = TMEM lane).
        // The dQ warps write the unit's dK and dV, so these warps go on to the
        // next unit's first tile at once.
        const int grp = (int)(warp - 2) >> 2;
        const int quad = warp & 3;
        const int j = quad * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t col_s = t_lane + L::kColS + grp * 64;
        const uint32_t col_dp = t_lane + L::kColDP + grp * 64;
        const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
        uint8_t *ds_row = smem + L::kDS + grp * L::kChunkBytes + j * 128;
        int g = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int slot = k % R;
            if (!(ok = warp_wait_b(pbar(PL::bUFull + slot), (k / R) & 1, wc, 23))) break;
            const int u = ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(pbar(PL::bUEmpty + slot));
            if (u < 0) break;
            const PUnit U = unit(u);
            const int key = U.k0 + j;
            const bool key_ok = key < U.Lkv;
            for (int i = 0; i < U.n_it; ++i) {
                const int G = g + i;
                const int q0 = (U.qt_begin + i % U.n_q) * kTileM + grp * 64;  // query of local column 0
                if (!(ok = warp_wait_b(bar(L::bSFull), G & 1, wc, 12))) break;
                tc_fence_after();
                uint32_t s[64];
                tmem_ld32(col_s, s);
                tmem_ld32(col_s + 32, s + 32);
                tmem_ld_wait_regs<64>(s);
                // local column c (query q0 + c) is visible iff lo <= c < hi
                int lo = p.mask != kMaskNone ? key - U.delta - q0 : 0;
                int hi = U.Lq - q0;
                if (p.window >= 0) hi = min(hi, key - U.delta + p.window + 1 - q0);
                if (!key_ok) lo = 64;
                uint32_t pk[32];
                if (__all_sync(0xffffffffu, lo <= 0 && hi >= 64)) {
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        float x0, x1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2), x0, x1);
                        pk[c / 2] = pack2<kBf16>(ex2_approx(x0), ex2_approx(x1));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        float x0, x1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2), x0, x1);
                        const float p0 = (c >= lo && c < hi) ? ex2_approx(x0) : 0.f;
                        const float p1 = (c + 1 >= lo && c + 1 < hi) ? ex2_approx(x1) : 0.f;
                        pk[c / 2] = pack2<kBf16>(p0, p1);
                    }
                }
                tmem_st32(col_s, pk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(L::bPReady));

                ok = warp_wait_b(bar(L::bDPFull), G & 1, wc, 14);
                if (ok && G > 0) ok = warp_wait_b(bar(L::bQEmpty + ((G - 1) & 1)), ((G - 1) >> 1) & 1, wc, 15);
                if (!ok) break;
                tc_fence_after();
                uint32_t dp[64];
                tmem_ld32(col_dp, dp);
                tmem_ld32(col_dp + 32, dp + 32);
                tmem_ld_wait_regs<64>(dp);
#pragma unroll
                for (int v8 = 0; v8 < 8; ++v8) {  // 16-byte unit v8: queries 8 v8 .. 8 v8 + 7
                    uint32_t w[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int e = v8 * 8 + v * 2;
                        const float2 pp = unpack2<kBf16>(pk[e / 2]);
                        float g0, g1;
                        f2_unpack(f2_mul(f2_pack(pp.x, pp.y),
                                         f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1]))),
                                  g0, g1);
                        w[v] = pack2<kBf16>(g0, g1);
                    }
                    *reinterpret_cast<uint4 *>(ds_row + ((v8 ^ (j & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(L::bDSReady));
            }
            g += U.n_it;
        }
    } else {
        // ============================================================ dQ, dK, dV
        // As in bwd_main_kernel: each warp owns 32 query rows of a tile and
        // adds its dQ into the fp32 accumulator through staged 32 x 16 boxes.
        // At the end of a unit each warp also writes dV and dK of its 32 key
        // rows (its TMEM lane quarter), staged in its 6 KB of dQ boxes, and a
        // unit that no query sees gets zeros.
        const int quad = warp & 3;
        const uint32_t t_dq = tmem + ((uint32_t)(quad * 32) << 16) + L::kColDQ;
        const uint32_t stage = sbase + L::kDQStage + quad * (L::kDQSlots * L::kDQBoxBytes);
        uint8_t *stage_ptr = smem + L::kDQStage + quad * (L::kDQSlots * L::kDQBoxBytes) + lane * 64;
        int boxes = 0, slot_box = 0;
        griddep_wait();  // the preprocess grid has zeroed the accumulator
        auto send = [&](const uint32_t *r, int col, int arow) {
            if (boxes >= L::kDQSlots) {
                if (lane == 0) bulk_wait_read<L::kDQSlots - 1>();
                __syncwarp();
            }
            uint8_t *row = stage_ptr + slot_box * L::kDQBoxBytes;
#pragma unroll
            for (int uu = 0; uu < 4; ++uu)
                *reinterpret_cast<uint4 *>(row + ((uu ^ ((lane >> 1) & 3)) << 4)) =
                    make_uint4(r[4 * uu], r[4 * uu + 1], r[4 * uu + 2], r[4 * uu + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_reduce_add_2d(&tm_dq, stage + slot_box * L::kDQBoxBytes, col, arow);
                bulk_commit();
            }
            ++boxes;
            slot_box = slot_box + 1 == L::kDQSlots ? 0 : slot_box + 1;
        };
        int g = 0, kv = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int slot = k % R;
            if (!(ok = warp_wait_b(pbar(PL::bUFull + slot), (k / R) & 1, wc, 24))) break;
            const int u = ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(pbar(PL::bUEmpty + slot));
            if (u < 0) break;
            const PUnit U = unit(u);
            // the warp's key rows of dV and dK (decoded again after the tile
            // loop, which then holds no more of the unit than it uses)
            auto rows = [&](const PUnit &W, uint16_t *&dv0, uint16_t *&dk0, int &n_valid) {
                const int key0 = W.k0 + quad * 32;
                n_valid = min(32, W.Lkv - key0);
                dv0 = static_cast<uint16_t *>(p.dv) + W.km.io0 + (int64_t)key0 * W.km.io_rs;
                dk0 = static_cast<uint16_t *>(p.dk) + W.km.io0 + (int64_t)key0 * W.km.io_rs;
            };
            if (U.n_q == 0) {
                uint16_t *dv0, *dk0;
                int n_valid;
                rows(U, dv0, dk0, n_valid);
                const int64_t rs = U.km.io_rs;
                // no query sees these keys: dK = dV = 0, whole rows per store
                for (int e = lane; e < 32 * (D / 8); e += 32) {
                    const int r = e / (D / 8), c = e % (D / 8);
                    if (r < n_valid) {
                        *reinterpret_cast<uint4 *>(dv0 + r * rs + c * 8) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(dk0 + r * rs + c * 8) = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            for (int i = 0; i < (p.deterministic ? 0 : U.n_it); ++i) {
                const int G = g + i;
                if (!(ok = warp_wait_b(bar(L::bDQFull), G & 1, wc, 17))) break;
                tc_fence_after();
                const int qrow0 = (U.qt_begin + i % U.n_q) * kTileM + quad * 32;
                const int arow = (kPacked ? (U.hk * p.group + i / U.n_q) * p.total_q + U.tok_q0
                                          : (U.q_slice0 + i / U.n_q) * p.s_q) +
                                 qrow0;
                const bool live = qrow0 < U.Lq;  // any live row in this warp's quarter
                if constexpr (D == 128) {
                    uint32_t r[96];
                    tmem_ld32(t_dq, r);
                    tmem_ld32(t_dq + 32, r + 32);
                    tmem_ld32(t_dq + 64, r + 64);
                    tmem_ld_wait_regs<96>(r);
                    if (live) {
                        send(r, 0, arow);
                        send(r + 16, 16, arow);
                    }
                    tmem_ld32(t_dq + 96, r);
                    tmem_ld_wait_regs<32>(r);
                    tc_fence_before();
                    mbar_arrive(bar(L::bDQFree));
                    if (live) {
#pragma unroll
                        for (int c = 32; c < 96; c += 16) send(r + c, c, arow);
                        send(r, 96, arow);
                        send(r + 16, 112, arow);
                    }
                } else {
                    uint32_t r[D];
#pragma unroll
                    for (int c = 0; c < D; c += 32) tmem_ld32(t_dq + c, r + c);
                    tmem_ld_wait_regs<D>(r);
                    tc_fence_before();
                    mbar_arrive(bar(L::bDQFree));
                    if (live) {
#pragma unroll
                        for (int c = 0; c < D; c += 16) send(r + c, c, arow);
                    }
                }
            }
            if (!ok) break;
            g += U.n_it;
            // dV and dK of the unit's keys: the staging boxes are free once
            // the reduce-adds issued from them have read them
            if (!(ok = warp_wait_b(pbar(PL::bUnitDone), kv & 1, wc, 16))) break;
            tc_fence_after();
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            const PUnit W = unit(u);
            uint16_t *dv0, *dk0;
            int n_valid;
            rows(W, dv0, dk0, n_valid);
            const int64_t rs = W.km.io_rs;
            uint8_t *box0 = stage_ptr - lane * 64;  // this warp's kDQSlots boxes
            const uint32_t t_rows = tmem + ((uint32_t)(quad * 32) << 16);
            store_tile_rows<D, kBf16>(t_rows + L::kColDV, box0, lane, dv0, rs, n_valid, 1.f, [] {});
            store_tile_rows<D, kBf16>(t_rows + L::kColDK, box0, lane, dk0, rs, n_valid, p.scale, [&] {
                tc_fence_before();
                mbar_arrive(pbar(PL::bAccFree));  // the accumulators are read out
            });
            ++kv;
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace

cudaError_t launch_bwd_persist(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                               const CUtensorMap &tdo, const CUtensorMap &tdq, const CUtensorMap &trx,
                               const BwdParams &p, int d, bool bf16, bool packed, cudaStream_t stream) {
#define SDPA_BWDP_CASE(D_, BF_, PK_)                                                               \
    if (d == D_ && bf16 == BF_ && packed == PK_) {                                                 \
        auto kern = bwd_persist_kernel<D_, BF_, PK_>;                                              \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                                             PersistLayout<D_>::kBytes);                           \
        if (e != cudaSuccess) return e;                                                            \
        return launch_overlapped(kern, dim3(p.grid), dim3(kBwdThreads), PersistLayout<D_>::kBytes, \
                                 stream, tq, tk, tv, tdo, tdq, trx, p);                            \
    }
    SDPA_BWDP_CASE(64, true, false)
    SDPA_BWDP_CASE(64, true, true)
    SDPA_BWDP_CASE(64, false, false)
    SDPA_BWDP_CASE(64, false, true)
    SDPA_BWDP_CASE(128, true, false)
    SDPA_BWDP_CASE(128, true, true)
    SDPA_BWDP_CASE(128, false, false)
    SDPA_BWDP_CASE(128, false, true)
#undef SDPA_BWDP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace sdpa
