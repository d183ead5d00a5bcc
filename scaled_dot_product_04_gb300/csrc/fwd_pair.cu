// Fused attention forward, two-tile variant: each work unit is 256 query rows
// held as two 128-row tiles A and B that share every K/V tile, so the MMA
// warp can run one tile's products while the other tile's softmax works.
// Same operation, masks, grouped key/value heads, statistics and layouts as
// fwd.cu ("Inside NVIDIA's cuDNN Graph API" (tradepoint.io), section 5;
// cudnn-frontend PR #554 notes on scale_softmax_log2, LSE layouts, the `sdpa`
// op's masks and GQA, persistent scheduling and the packed total clamp); the
// host picks this kernel for long d = 128 problems, where every unit visits
// many key tiles.  Without a left window both tiles walk the key tiles from 0
// (tile A leaves one key tile before B under a causal mask).  The kWin
// instantiations, for left windows, walk from the first key tile tile A can
// see (kt0); tile X takes part in steps [first[X], n_kv[X]) of that walk, so
// tile B joins one key tile after A.  They are separate instantiations so
// that the unwindowed loop compiles exactly as it would without them.
//
// Roles inside a CTA (12 warps):
//   warp 0       TMA producer: Q_A, Q_B and the first K tile of each unit,
//                then per key tile j the pair V_j, K_{j+1} on one barrier
//                (K and V keep rings of their own);
//   warp 1       MMA issuer (one thread).  Per key tile j it issues
//                O_A += P_A(j) V_j, S_A(j+1) = Q_A K_{j+1}^T,
//                O_B += P_B(j) V_j, S_B(j+1) = Q_B K_{j+1}^T.
//                Each S follows its own tile's P V, so the two chains run half
//                a period apart and each softmax is covered by two products
//                of the other tile (and the two softmaxes do not contend for
//                the exponent unit at the same time);
//   warps 4..7   softmax of tile A, warps 8..11 softmax of tile B (thread r
//                owns row r = TMEM lane r), as in fwd.cu.
// Warps 0..3 (TMA, MMA and two idle warps) form warpgroup 0, which gives up
// registers with setmaxnreg to the two softmax warpgroups, whose row of S
// (128 fp32 values) and running state then fit without spilling.
// TMEM columns: S_A 0, S_B 128, O_A 256, O_B 256 + d.  S_X(j+1) is issued right
// behind O_X += P_X(j) V_j although P_X lives in the S_X columns: tcgen05.mma
// instructions of one thread execute in issue order, so the earlier product
// has read P_X before the later one writes S_X (the same ordering every
// chained accumulation relies on).  When the softmax sees S_X(j+1) complete,
// O_X therefore holds every earlier product and may be rescaled at once.
#include <atomic>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int kPairThreads = 384;
constexpr int kPairRows = 2 * kTileM;  // query rows per work unit
// registers per thread the kernel is launched with (the most 384 threads may
// have); the setmaxnreg split below hands out exactly kPairThreads x this
constexpr int kPairLaunchRegs = 168;

// kEb: bytes per input element (2 for bf16/fp16, 1 for E4M3).  kPk: packed
// inputs, whose cu_seqlens cache also holds the sequence table of the unit
// list (order, first unit) and a scan scratch.
template <int D, int kEb = 2, bool kPk = false>
struct PairLayout {
    static constexpr int kChunks = D * kEb / 128;     // 128-byte swizzle columns per row
    static constexpr int kChunkBytes = kTileM * 128;  // 16 KiB: 128 rows x 128 bytes
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kKStages = (kTileBytes >= 32768) ? 3 : 5;
    static constexpr int kVStages = (kTileBytes >= 32768) ? 2 : 4;
    // cu_seqlens entries cached (packed: with the unit list's sequence table)
    static constexpr int kCuCap = kPk ? ((kTileBytes >= 32768) ? 96 : 1024) : ((kTileBytes >= 32768) ? 192 : 2048);
    static constexpr int kCuArrays = kPk ? 4 : 2;
    static constexpr int kQ = 0;                             // Q_A, Q_B
    static constexpr int kK = kQ + 2 * kTileBytes;
    static constexpr int kV = kK + kKStages * kTileBytes;
    // int32 cu_q[kCuCap], cu_kv[kCuCap] (packed: then order[kCuCap], first_unit[kCuCap])
    static constexpr int kCu = kV + kVStages * kTileBytes;
    static constexpr int kScan = kCu + kCuArrays * kCuCap * 4;  // packed: 16 int32, per-warp sums
    static constexpr int kBar = kScan + (kPk ? 64 : 0);
    static constexpr int bQFull = 0;
    static constexpr int bQEmpty = 1;
    static constexpr int bKFull = 2;
    // K stages have no release barrier of their own: K_i's stage is refilled
    // only after the release of V_{i-1-kVStages} has been seen, which the MMA
    // thread commits behind every product that reads K_{i-kKStages} as long as
    // the K ring is at least one stage deeper than the V ring.
    static_assert(kKStages >= kVStages + 1, "the V releases must cover the K ring");
    static constexpr int bVFull = bKFull + kKStages;
    static constexpr int bVEmpty = bVFull + kVStages;
    // per tile X in {A, B}: index + X
    static constexpr int bSFull = bVEmpty + kVStages;
    static constexpr int bPReady = bSFull + 2;
    static constexpr int bOFull = bPReady + 2;
    static constexpr int bOFree = bOFull + 2;
    static constexpr int bMmaIdle = bOFree + 2;
    static constexpr int kNumBars = bMmaIdle + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;  // u32[0] TMEM base, u32[1] abort flag
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kSmemAlloc = kBytes + 1024;  // slack to align the base to 1024 B
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;    // S_X at kColS + X * 128
    static constexpr uint32_t kColO = 256;  // O_X at kColO + X * D
};

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only if the max grows by 2^8

// Units taken dynamically (kDyn, packed lists with a sequence table): the
// list runs sequence by sequence, longest first, and within a sequence from
// its heaviest 256-row block to its lightest, a sawtooth that a fixed deal
// spreads unevenly over the CTAs.  The kDyn instantiations take units from a
// counter instead, in the same order: the producer thread takes the next unit
// once it has issued the current one's loads and hands it to the MMA thread
// and the softmax warps through a ring of kUnitRing slots placed after the
// layout.  The counter is a slot of g_pair_unit_counters, zeroed by the host
// before the launch; packed launches carry that slot + 1 in FwdParams::s_q,
// which no packed kernel reads otherwise.
constexpr int kUnitRing = 4;
constexpr int kPairCounterSlots = 1024;
__device__ uint32_t g_pair_unit_counters[kPairCounterSlots];
template <int D, int kEb>
struct PairDynLayout {
    using L = PairLayout<D, kEb, true>;
    static constexpr int kRing = L::kBytes;                  // kUnitRing ints
    static constexpr int kRingBar = kRing + 4 * kUnitRing;  // full, empty: kUnitRing each
    static constexpr int kBytes = kRingBar + 2 * kUnitRing * 8;
    static constexpr int kSmemAlloc = kBytes + 1024;
};
static_assert(PairDynLayout<128, 2>::kSmemAlloc <= 232448, "dynamic two-tile forward exceeds shared memory");

SDPA_DEV bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx &w, uint32_t site) {
    bool ok = mbar_wait(bar, parity, w, site);
    return __all_sync(0xffffffffu, ok);
}

// k-th unit of CTA `first` out of `step`: boustrophedon walk over the
// heaviest-first list (c, 2G-1-c, 2G+c, 4G-1-c, ...).
SDPA_DEV int unit_of(int k, int first, int step) {
    return k * step + ((k & 1) ? step - 1 - first : first);
}

// One work unit: rows [row0, row0 + 256) of one slice; tile A is the first
// 128 rows, tile B the next 128.
struct PairUnit {
    int slice, head, kv_slice, kv_head, Lq, Lkv, tok_q0, tok_kv0, row0, delta;
    int n_kv[2];   // walk steps tile A / tile B takes part in, up to (0: no row or key)
    int kt0;       // kWin: first key tile of the walk (else 0)
    int first[2];  // kWin: first walk step of tile A / B (else 0)
    bool live;    // tile A holds at least one query row
    bool single;  // a 128-row unit: tile B takes no part
    int64_t o_row0, o_rs, lse_row0, lse_rs;
};

// Unit u: latest (heaviest) rows first over all slices; packed units with a
// cached sequence table (order != nullptr) run sequence by sequence instead,
// longest first: sequence order[i] owns units [first_unit[i], first_unit[i+1]),
// its 256-row blocks latest first with the heads innermost, so the CTAs in
// flight share one or two sequences' K and V in L2.
//
// Dense lists of equal units whose count leaves a partial last wave end with
// n_split = p.n_units - p.q_tiles * p.bh of their 256-row blocks cut in two:
// the host sizes the list so that the blocks before them fill whole waves of
// the grid and the 2 n_split 128-row units of the cut blocks take at most one
// more wave, each about half a block's time, where the uncut blocks would
// have taken a whole one.  Only the kSplit instantiations decode such a list,
// so the others compile as they did without it.
template <int D, bool kPacked, bool kWin, bool kSplit = false>
SDPA_DEV PairUnit decode_pair(const FwdParams &p, int u, const int *cu_q, const int *cu_kv,
                              const int *order, const int *first_unit) {
    PairUnit U;
    int qp;
    if constexpr (kPacked) {
        if (order) {
            int lo = 0, hi = p.num_seqs;  // first_unit[lo] <= u < first_unit[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (first_unit[mid] <= u) lo = mid;
                else hi = mid;
            }
            const int n = order[lo], local = u - first_unit[lo];
            qp = (cu_q[n + 1] - cu_q[n] + kPairRows - 1) / kPairRows - 1 - local / p.h;
            U.slice = n * p.h + local % p.h;
        } else {
            qp = p.q_tiles - 1 - u / p.bh;
            U.slice = u % p.bh;
        }
    } else {
        int half = -1;  // a cut block: which 128-row half
        if constexpr (kSplit) {
            const int split_from = 2 * p.q_tiles * p.bh - p.n_units;  // blocks - cut blocks
            if (u >= split_from) {
                half = (u - split_from) & 1;
                u = split_from + ((u - split_from) >> 1);
            }
        }
        qp = p.q_tiles - 1 - u / p.bh;  // latest (heaviest) rows first
        U.slice = u % p.bh;
        U.single = half >= 0;
        U.row0 = qp * kPairRows + (half > 0 ? kTileM : 0);
    }
    if constexpr (!kPacked) {
        U.head = 0;
        U.kv_head = 0;
        U.kv_slice = (U.slice / p.h) * p.h_kv + (U.slice % p.h) / p.group;
        U.tok_q0 = U.tok_kv0 = 0;
        U.Lq = p.s_q;
        U.Lkv = p.s_kv;
        U.o_row0 = (int64_t)U.slice * p.s_q * D;
        U.o_rs = D;
        U.lse_row0 = (int64_t)U.slice * p.s_q;
        U.lse_rs = 1;
    } else {
        const int n = U.slice / p.h;
        U.head = U.slice % p.h;
        U.kv_head = U.head / p.group;
        U.kv_slice = 0;
        U.tok_q0 = cu_q[n];
        U.tok_kv0 = cu_kv[n];
        U.Lq = cu_q[n + 1] - U.tok_q0;
        U.Lkv = cu_kv[n + 1] - U.tok_kv0;
        U.o_row0 = ((int64_t)U.tok_q0 * p.h + U.head) * D;
        U.o_rs = (int64_t)p.h * D;
        U.lse_row0 = (int64_t)U.tok_q0 * p.h + U.head;
        U.lse_rs = p.h;
    }
    if constexpr (kPacked) {
        U.single = false;
        U.row0 = qp * kPairRows;
    }
    U.live = U.row0 < U.Lq;
    U.delta = mask_delta(p.mask, U.Lq, U.Lkv);
    U.kt0 = 0;
    U.first[0] = U.first[1] = 0;
    if constexpr (!kWin) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int r0 = U.row0 + x * kTileM;
            int n = 0;
            if (r0 < U.Lq && !(kSplit && x == 1 && U.single)) {
                const int hi = key_range(p.mask, p.window, min(r0 + kTileM, U.Lq) - 1, U.delta, U.Lkv).hi;
                n = hi > 0 ? (hi + kTileN - 1) / kTileN : 0;
            }
            U.n_kv[x] = n;
        }
    } else {
        // absolute key-tile range [f, e) of each tile: from its first row's
        // window start to its last row's causal end
        int f[2], e[2];
        U.kt0 = 1 << 30;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int r0 = U.row0 + x * kTileM;
            f[x] = e[x] = 0;
            if (r0 < U.Lq && !(kSplit && x == 1 && U.single)) {
                const int lo = max(0, key_range(p.mask, p.window, r0, U.delta, U.Lkv).lo);
                const int hi = key_range(p.mask, p.window, min(r0 + kTileM, U.Lq) - 1, U.delta, U.Lkv).hi;
                if (hi > lo) {
                    f[x] = lo / kTileN;
                    e[x] = (hi + kTileN - 1) / kTileN;
                    U.kt0 = min(U.kt0, f[x]);
                }
            }
        }
        if (U.kt0 == (1 << 30)) U.kt0 = 0;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            U.first[x] = e[x] > f[x] ? f[x] - U.kt0 : 0;
            U.n_kv[x] = e[x] > f[x] ? e[x] - U.kt0 : 0;
        }
    }
    return U;
}

// kEl / kOut: input and output element kinds as in fwd.cu (E4M3 inputs with
// device descales, P as E4M3 quads, kind::f8f6f4 products; amax of O).
template <int D, int kEl, bool kPacked, int kOut, bool kWin, bool kSplit = false, bool kDyn = false>
__global__ void __launch_bounds__(kPairThreads, 1)
    fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    constexpr bool kFp8 = kEl == kElE4m3;
    constexpr bool kBf16 = kEl == kElBf16;
    constexpr int kEb = kFp8 ? 1 : 2;
    constexpr int kOb = kOut == kElE4m3 ? 1 : 2;
    using L = PairLayout<D, kEb, kPacked>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    // cu_seqlens of packed inputs, cached when they fit, and then the
    // sequence table of the unit list (see decode_pair)
    int *cu_q_s = reinterpret_cast<int *>(smem + L::kCu);
    int *cu_kv_s = cu_q_s + L::kCuCap;
    int *order_s = cu_kv_s + L::kCuCap;  // packed layout only
    int *first_s = order_s + L::kCuCap;
    const int *cu_q = p.cu_q, *cu_kv = p.cu_kv;
    const int *order = nullptr;
    int n_units = p.n_units;
    if constexpr (kPacked) {
        if (p.num_seqs + 1 <= L::kCuCap) {
            const int ns = p.num_seqs;
            for (int i = threadIdx.x; i <= ns; i += blockDim.x) {
                cu_q_s[i] = p.cu_q[i];
                cu_kv_s[i] = p.cu_kv[i];
            }
            cu_q = cu_q_s;
            cu_kv = cu_kv_s;
            __syncthreads();
            auto blocks = [&](int n) { return (cu_q_s[n + 1] - cu_q_s[n] + kPairRows - 1) / kPairRows; };
            // most 256-row blocks first, ties in sequence order (a rank count;
            // long lists keep their own order)
            for (int n = threadIdx.x; n < ns; n += blockDim.x) {
                int rank = n;
                if (ns <= 256) {
                    const int bn = blocks(n);
                    rank = 0;
                    for (int m = 0; m < ns; ++m) {
                        const int bm = blocks(m);
                        rank += (bm > bn || (bm == bn && m < n)) ? 1 : 0;
                    }
                }
                order_s[rank] = n;
            }
            __syncthreads();
            // first_unit = exclusive prefix sum of blocks(order[i]) * h: chunk
            // sums per thread, scanned in the warp and across the warps
            int *scan = reinterpret_cast<int *>(smem + L::kScan);
            const int per = (ns + blockDim.x - 1) / blockDim.x;
            const int b0 = min(ns, (int)threadIdx.x * per), b1 = min(ns, b0 + per);
            int csum = 0;
            for (int i = b0; i < b1; ++i) csum += blocks(order_s[i]) * p.h;
            int incl = csum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if ((int)lane >= off) incl += y;
            }
            if (lane == 31) scan[warp] = incl;
            __syncthreads();
            int run = incl - csum;
            for (int w = 0; w < (int)warp; ++w) run += scan[w];
            for (int i = b0; i < b1; ++i) {
                first_s[i] = run;
                run += blocks(order_s[i]) * p.h;
            }
            if (threadIdx.x == blockDim.x - 1) first_s[ns] = run;  // the last chunk ends the list
            __syncthreads();
            order = order_s;
            n_units = first_s[ns];
        }
    }

    if (threadIdx.x == 0) {
        mbar_init(bar(L::bQFull), 1);
        mbar_init(bar(L::bQEmpty), 1);
        for (int s = 0; s < L::kKStages; ++s) mbar_init(bar(L::bKFull + s), 1);
        for (int s = 0; s < L::kVStages; ++s) {
            mbar_init(bar(L::bVFull + s), 1);
            mbar_init(bar(L::bVEmpty + s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(L::bSFull + x), 1);
            mbar_init(bar(L::bPReady + x), kTileM);
            mbar_init(bar(L::bOFull + x), 1);
            mbar_init(bar(L::bOFree + x), kTileM);
        }
        mbar_init(bar(L::bMmaIdle), 1);
        if constexpr (kDyn) {
            const uint32_t rb = sbase + PairDynLayout<D, kEb>::kRingBar;  // the unit ring's barriers
            for (int b = 0; b < kUnitRing; ++b) {
                mbar_init(rb + 8u * b, 1);                // full: the producer
                mbar_init(rb + 8u * (kUnitRing + b), 9);  // empty: the MMA thread and 8 softmax warps
            }
        }
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
    const int first = blockIdx.x, step = gridDim.x;
    // Registers: warpgroup 0 (TMA, MMA, two idle warps) hands 64 per thread
    // to the two softmax warpgroups: 128 x 104 + 256 x 200 = 384 x 168 (the
    // kWin walk's bookkeeping takes 48: 128 x 120 + 256 x 192).
    constexpr uint32_t kRegsWg0 = kWin ? 120 : 104, kRegsSoftmax = kWin ? 192 : 200;
    static_assert(128 * kRegsWg0 + 256 * kRegsSoftmax == kPairThreads * kPairLaunchRegs,
                  "register split must hand out exactly the launch's registers");
    if (warp < 4) {
        setmaxnreg_dec<kRegsWg0>();
        if (warp == 0) {
            // ============================================================ producer
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                // Per unit: Q_A, Q_B, the unit's first K tile (on its K stage's
                // full barrier), then per key step j the pair V_j, K_{j+1}: both
                // land on V_j's full barrier, so the MMA thread waits once per
                // step.  A K tile that rides on a V barrier still completes a
                // phase of its own stage's full barrier (a plain arrive), so the
                // K barriers keep one phase per K tile; the MMA thread waits on
                // them only for a unit's first K, whose stage cannot be refilled
                // before that wait (the refill waits for a V release that the MMA
                // thread commits only after it).
                int k_it = 0, v_it = 0, units = 0;
                bool ok = true;
                // K_{j+1} of a pair, landing on `full` (V_j's barrier); its own
                // stage's full barrier gets a plain arrive.  The stage is free:
                // the V stage wait just before it covers the K ring (see
                // PairLayout).
                auto k_stage = [&](uint32_t full, int ky, int kz) {
                    const int ks = k_it % L::kKStages;
                    mbar_arrive(bar(L::bKFull + ks));
    #pragma unroll
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_3d(sbase + L::kK + ks * L::kTileBytes + c * L::kChunkBytes, &tm_k, full,
                                    c * (128 / kEb), ky, kz);
                    ++k_it;
                };
                for (int k = 0; ok; ++k) {
                    int u;
                    if constexpr (kDyn) {
                        // take the next unit (the first by the CTA's index) and hand it on
                        using DL = PairDynLayout<D, kEb>;
                        const uint32_t rb = sbase + DL::kRingBar;
                        const int slot = k % kUnitRing;
                        if (k >= kUnitRing &&
                            !mbar_wait(rb + 8u * (kUnitRing + slot), ((k / kUnitRing) - 1) & 1, wc, 20))
                            break;
                        u = k == 0 ? (int)blockIdx.x
                                   : (int)gridDim.x + (int)atomicAdd(g_pair_unit_counters + (p.s_q - 1), 1u);
                        if (u >= n_units) u = -1;
                        reinterpret_cast<volatile int *>(smem + DL::kRing)[slot] = u;
                        mbar_arrive(rb + 8u * slot);
                        if (u < 0) break;
                    } else {
                        u = unit_of(k, first, step);
                        if (u >= n_units) break;
                    }
                    const PairUnit U = decode_pair<D, kPacked, kWin, kSplit>(p, u, cu_q, cu_kv, order, first_s);
                    const int nmax = max(U.n_kv[0], U.n_kv[1]);
                    if (nmax == 0) continue;
                    if (units > 0 && !mbar_wait(bar(L::bQEmpty), (units - 1) & 1, wc, 1)) break;
                    mbar_arrive_expect_tx(bar(L::bQFull), 2 * L::kTileBytes);
    #pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const int qy = kPacked ? U.head : U.row0 + x * kTileM;
                        const int qz = kPacked ? U.tok_q0 + U.row0 + x * kTileM : U.slice;
    #pragma unroll
                        for (int c = 0; c < L::kChunks; ++c)
                            tma_load_3d(sbase + L::kQ + x * L::kTileBytes + c * L::kChunkBytes, &tm_q,
                                        bar(L::bQFull), c * (128 / kEb), qy, qz);
                    }
                    ++units;
                    // key tile j of the unit's walk: (y, z) coordinates of K_j and V_j
                    auto kv_yz = [&](int j, int &y, int &z) {
                        const int kj = kWin ? U.kt0 + j : j;  // absolute key tile
                        y = kPacked ? U.kv_head : kj * kTileN;
                        z = kPacked ? U.tok_kv0 + kj * kTileN : U.kv_slice;
                    };
                    {
                        int ky, kz;
                        kv_yz(0, ky, kz);
                        const uint32_t full = bar(L::bKFull + k_it % L::kKStages);
                        const int ks = k_it % L::kKStages;
                        mbar_arrive_expect_tx(full, L::kTileBytes);
    #pragma unroll
                        for (int c = 0; c < L::kChunks; ++c)
                            tma_load_3d(sbase + L::kK + ks * L::kTileBytes + c * L::kChunkBytes, &tm_k, full,
                                        c * (128 / kEb), ky, kz);
                        ++k_it;
                    }
                    for (int j = 0; j < nmax; ++j) {
                        const int vs = v_it % L::kVStages, vuse = v_it / L::kVStages;
                        if (vuse > 0 && !mbar_wait(bar(L::bVEmpty + vs), (vuse - 1) & 1, wc, 3)) {
                            ok = false;
                            break;
                        }
                        const bool pair_k = j + 1 < nmax;
                        const uint32_t vfull = bar(L::bVFull + vs);
                        int vy, vz;
                        kv_yz(j, vy, vz);
                        mbar_arrive_expect_tx(vfull, pair_k ? 2 * L::kTileBytes : L::kTileBytes);
    #pragma unroll
                        for (int c = 0; c < L::kChunks; ++c)
                            tma_load_3d(sbase + L::kV + vs * L::kTileBytes + c * L::kChunkBytes, &tm_v, vfull,
                                        c * (128 / kEb), vy, vz);
                        ++v_it;
                        if (pair_k) {
                            int ky, kz;
                            kv_yz(j + 1, ky, kz);
                            k_stage(vfull, ky, kz);
                        }
                    }
                }
                // Every load issued must land before the CTA may exit (a K tile
                // that rode on a V barrier lands with that V tile).
                if (units > 0) mbar_wait_drain(bar(L::bQFull), (units - 1) & 1);
                for (int i = max(0, k_it - L::kKStages); i < k_it; ++i)
                    mbar_wait_drain(bar(L::bKFull + i % L::kKStages), (i / L::kKStages) & 1);
                for (int i = max(0, v_it - L::kVStages); i < v_it; ++i)
                    mbar_wait_drain(bar(L::bVFull + i % L::kVStages), (i / L::kVStages) & 1);
            }
            __syncwarp();
        } else if (warp == 1) {
            // ============================================================ MMA issuer
            if (lane == 0) {
                constexpr uint32_t idesc_s = kFp8 ? make_idesc_e4m3(kTileM, kTileN, false, false)
                                                  : make_idesc_f16(kTileM, kTileN, kBf16, false, false);
                constexpr uint32_t idesc_o = kFp8 ? make_idesc_e4m3(kTileM, D, false, true)
                                                  : make_idesc_f16(kTileM, D, kBf16, false, true);
                // Operand descriptors, built once and advanced by constant offsets
                // (a descriptor's low 14 bits are the address / 16).
                constexpr uint32_t kChunk16 = L::kChunkBytes >> 4, kTile16 = L::kTileBytes >> 4;
                const uint64_t dQ_k = smem_desc_sw128(sbase + L::kQ, 16, 1024);
                const uint64_t dK_k = smem_desc_sw128(sbase + L::kK, 16, 1024);
                const uint64_t dV_mn = smem_desc_sw128(sbase + L::kV, L::kChunkBytes, 1024);
                // S_X = Q_X K^T: both operands K-major (head dim contiguous), 32
                // bytes (16 bf16 or 32 E4M3 elements) per step.
                auto issue_s = [&](int x, int ks) {
                    const uint64_t a = dQ_k + x * kTile16, b = dK_k + ks * kTile16;
    #pragma unroll
                    for (int k = 0; k < D * kEb / 32; ++k) {
                        const uint32_t off = (k / 4) * kChunk16 + (k % 4) * 2;
                        if constexpr (kFp8)
                            mma_ss_f8(tmem + L::kColS + x * 128, a + off, b + off, idesc_s, k > 0);
                        else
                            mma_ss(tmem + L::kColS + x * 128, a + off, b + off, idesc_s, k > 0);
                    }
                };
                // O_X += P_X V: P from TMEM (8 columns per step: 16 keys as bf16
                // pairs or 32 keys as E4M3 quads), V MN-major (head dim
                // contiguous); 128-byte head-dim chunks are 16 KiB apart (leading
                // offset), 8-key groups 1 KiB apart, so a step advances 2 or 4 KiB.
                auto issue_pv = [&](int x, int vs, bool acc) {
                    const uint64_t b = dV_mn + vs * kTile16;
    #pragma unroll
                    for (int k = 0; k < kTileN * kEb / 32; ++k) {
                        const uint64_t vdesc = b + k * ((4096 / kEb) >> 4);
                        if constexpr (kFp8)
                            mma_ts_f8(tmem + L::kColO + x * D, tmem + L::kColS + x * 128 + k * 8, vdesc,
                                      idesc_o, (acc || k > 0) ? 1u : 0u);
                        else
                            mma_ts(tmem + L::kColO + x * D, tmem + L::kColS + x * 128 + k * 8, vdesc,
                                   idesc_o, (acc || k > 0) ? 1u : 0u);
                    }
                };
                // cnt[x]: products P_X V issued so far (one per tile of X); uo[x]:
                // units in which tile X took part.
                int t = 0, units = 0, cnt[2] = {0, 0}, uo[2] = {0, 0};
                bool ok = true;
                for (int k = 0; ok; ++k) {
                    int u;
                    if constexpr (kDyn) {
                        using DL = PairDynLayout<D, kEb>;
                        const uint32_t rb = sbase + DL::kRingBar;
                        const int slot = k % kUnitRing;
                        if (!(ok = mbar_wait(rb + 8u * slot, (k / kUnitRing) & 1, wc, 21))) break;
                        u = reinterpret_cast<volatile int *>(smem + DL::kRing)[slot];
                        mbar_arrive(rb + 8u * (kUnitRing + slot));
                        if (u < 0) break;
                    } else {
                        u = unit_of(k, first, step);
                        if (u >= n_units) break;
                    }
                    const PairUnit U = decode_pair<D, kPacked, kWin, kSplit>(p, u, cu_q, cu_kv, order, first_s);
                    const int nmax = max(U.n_kv[0], U.n_kv[1]);
                    if (nmax == 0) continue;
                    ok = mbar_wait(bar(L::bQFull), units & 1, wc, 4) &&
                         mbar_wait(bar(L::bKFull + t % L::kKStages), (t / L::kKStages) & 1, wc, 5);
    #pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (!ok || U.n_kv[x] == 0) continue;
                        if constexpr (kWin) {
                            if (U.first[x] != 0) continue;  // joins the walk later
                        }
                        tc_fence_after();
                        issue_s(x, t % L::kKStages);
                        mma_commit(bar(L::bSFull + x));
                    }
                    if (!ok) break;
                    if (nmax == 1) mma_commit(bar(L::bQEmpty));
                    // Per key tile j: O_A += P_A V_j, S_A(j+1), O_B += P_B V_j, S_B(j+1).
                    for (int j = 0; j < nmax; ++j, ++t) {
                        const int t1 = t + 1;
                        ok = mbar_wait(bar(L::bVFull + t % L::kVStages), (t / L::kVStages) & 1, wc, 7);
    #pragma unroll
                        for (int x = 0; x < 2; ++x) {
                            if constexpr (!kWin) {
                                if (!ok || j >= U.n_kv[x]) continue;
                            } else {
                                if (!ok) continue;
                            }
                            // kWin: tile X takes part in steps [first, n_kv); S_X(j+1)
                            // below also opens its walk when it joins at step j + 1
                            if (!kWin || (j >= U.first[x] && j < U.n_kv[x])) {
                                ok = mbar_wait(bar(L::bPReady + x), cnt[x] & 1, wc, 8);
                                // the unit's first P V overwrites O_X: its previous
                                // epilogue must have read it out
                                if (ok && j == U.first[x] && uo[x] > 0)
                                    ok = mbar_wait(bar(L::bOFree + x), (uo[x] - 1) & 1, wc, 9);
                                if (!ok) continue;
                                tc_fence_after();
                                issue_pv(x, t % L::kVStages, j > U.first[x]);
                                ++cnt[x];
                            }
                            if (j + 1 >= U.n_kv[x]) continue;
                            if constexpr (kWin) {
                                if (j + 1 < U.first[x]) continue;
                            }
                            // K_{j+1} landed with V_j (see the producer).  S_X(j+1)
                            // overwrites the P_X(j) that O_X += P_X V reads; issue
                            // order keeps them apart (see the header)
                            tc_fence_after();
                            issue_s(x, t1 % L::kKStages);
                            mma_commit(bar(L::bSFull + x));
                        }
                        if (!ok) break;
                        // releases V_j, and with it the K stages (see PairLayout)
                        mma_commit(bar(L::bVEmpty + t % L::kVStages));
                        if (j + 2 == nmax) mma_commit(bar(L::bQEmpty));  // last reader of Q
                    }
                    if (!ok) break;
    #pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (U.n_kv[x] == U.first[x]) continue;
                        mma_commit(bar(L::bOFull + x));
                        ++uo[x];
                    }
                    ++units;
                }
                // Let every MMA issued above retire before TMEM is released.
                mma_commit(bar(L::bMmaIdle));
                mbar_wait_drain(bar(L::bMmaIdle), 0);
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ============================================================ softmax
        const int x = (warp - 4) >> 2;  // 0: tile A (warps 4-7), 1: tile B (warps 8-11)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // row of the tile == TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t scol = L::kColS + x * 128, ocol = L::kColO + x * D;
        float sl2 = p.scale_log2;
        float o_factor = 1.f;  // descale_v (E4M3 inputs)
        if constexpr (kFp8) {
            sl2 *= *p.descale_q * *p.descale_k;
            o_factor = *p.descale_v;
        }
        float amax = 0.f;  // max |O| over this thread's rows (E4M3 inputs)
        int cnt = 0, uo = 0;  // tiles and units of this tile's chain
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int u;
            if constexpr (kDyn) {
                using DL = PairDynLayout<D, kEb>;
                const uint32_t rb = sbase + DL::kRingBar;
                const int slot = k % kUnitRing;
                if (!(ok = warp_wait(rb + 8u * slot, (k / kUnitRing) & 1, wc, 22))) break;
                u = reinterpret_cast<volatile int *>(smem + DL::kRing)[slot];
                __syncwarp();
                if (lane == 0) mbar_arrive(rb + 8u * (kUnitRing + slot));
                if (u < 0) break;
            } else {
                u = unit_of(k, first, step);
                if (u >= n_units) break;
            }
            const PairUnit U = decode_pair<D, kPacked, kWin, kSplit>(p, u, cu_q, cu_kv, order, first_s);
            const int row0 = U.row0 + x * kTileM;
            if (!U.live || row0 >= U.Lq || (kSplit && x == 1 && U.single)) continue;  // no row of this tile
            const int q_idx = row0 + r;
            const bool row_ok = q_idx < U.Lq;
            uint8_t *orow = static_cast<uint8_t *>(p.o) + (U.o_row0 + (int64_t)q_idx * U.o_rs) * kOb;
            float *lse_ptr = p.lse ? p.lse + U.lse_row0 + (int64_t)q_idx * U.lse_rs : nullptr;
            const int n_kv = U.n_kv[x] - U.first[x];  // key tiles of this tile's walk
            const int kt_x = U.kt0 + U.first[x];       // its first key tile
            if (n_kv == 0) {
                // No key is visible to any row of this tile: O = 0, LSE = -inf.
                if (row_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
                    for (int i = 0; i < D * kOb / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                    if (lse_ptr) *lse_ptr = -INFINITY;
                }
                continue;
            }
            float m_used = -INFINITY;  // running max used as exponent base (log2 units)
            float l = 0.f;             // running sum of P
            for (int j = 0; j < n_kv; ++j, ++cnt) {
                ok = warp_wait(bar(L::bSFull + x), cnt & 1, wc, 12);
                if (!ok) break;
                tc_fence_after();
                uint32_t s[kTileN];
#pragma unroll
                for (int c = 0; c < kTileN / 32; ++c) tmem_ld32(t_lane + scol + c * 32, s + c * 32);
                tmem_ld_wait_regs<kTileN>(s);

                const int k0 = (kt_x + j) * kTileN;
                // the tile needs a mask unless every row sees all of its keys
                if ((k0 + kTileN > U.Lkv) ||
                    (p.mask != kMaskNone && k0 + kTileN - 1 > row0 + U.delta) ||
                    (p.window >= 0 && k0 < row0 + kTileM - 1 + U.delta - p.window)) {
                    const KeyRange kr = key_range(p.mask, p.window, q_idx, U.delta, U.Lkv);
                    const int c_lo = kr.lo - k0, c_hi = kr.hi - k0;  // visible: c_lo <= c < c_hi
#pragma unroll
                    for (int c = 0; c < kTileN; ++c)
                        if (c < c_lo || c >= c_hi) s[c] = __float_as_uint(-INFINITY);
                }
                // row max: four independent chains of 3-input max
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < kTileN; c += 8) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        mx4[v] = fmax3(mx4[v], __uint_as_float(s[c + 2 * v]),
                                       __uint_as_float(s[c + 2 * v + 1]));
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
                // P = exp2(s * scale*log2e - base), packed in place into s[0..64)
                // as bf16/fp16 pairs, or into s[0..32) as E4M3 quads
                uint64_t sum2[4] = {0, 0, 0, 0};
                if constexpr (kFp8) {
#pragma unroll
                    for (int i = 0; i < kTileN / 4; ++i) {
                        float x0, x1, x2, x3;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1])),
                                         sl2_2, nbase_2),
                                  x0, x1);
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3])),
                                         sl2_2, nbase_2),
                                  x2, x3);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
                        sum2[(2 * i) & 3] = f2_add(sum2[(2 * i) & 3], f2_pack(p0, p1));
                        sum2[(2 * i + 1) & 3] = f2_add(sum2[(2 * i + 1) & 3], f2_pack(p2, p3));
                        s[i] = pack_e4m3x4(p0, p1, p2, p3);  // i <= 4i: packs in place
                    }
                } else {
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
                }
                {
                    float a0, a1;
                    f2_unpack(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), a0, a1);
                    l += a0 + a1;
                }
                tmem_st32(t_lane + scol, s);
                if constexpr (!kFp8) tmem_st32(t_lane + scol + 32, s + 32);

                if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                    // The commit behind S_X(j) completed only once every earlier
                    // product had, O_X += P_X(j-1) V included, so O_X holds all
                    // of them and nothing writes it now.
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + ocol + c * 32, o);
                        tmem_ld_wait_regs<32>(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(t_lane + ocol + c * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(L::bPReady + x));
            }
            if (!ok) break;
            // epilogue: O / l and LSE; then O_X is free for the next unit
            ok = warp_wait(bar(L::bOFull + x), uo & 1, wc, 14);
            if (!ok) break;
            tc_fence_after();
            const float inv_l = (l > 0.f) ? o_factor / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(t_lane + ocol + c * 32, o);
                tmem_ld_wait_regs<32>(o);
                if (c == D / 32 - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(L::bOFree + x));
                }
                if constexpr (kFp8) {
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            amax = fmaxf(amax, fabsf(__uint_as_float(o[i]) * inv_l));
                    }
                }
                if constexpr (kOut == kElE4m3) {
                    const float so = inv_l * *p.scale_o;
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[i] = pack_e4m3x4(__uint_as_float(o[4 * i]) * so, __uint_as_float(o[4 * i + 1]) * so,
                                            __uint_as_float(o[4 * i + 2]) * so, __uint_as_float(o[4 * i + 3]) * so);
                    if (row_ok) st_global_32b(orow + c * 32 * kOb, pk);
                } else {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack2<kOut == kElBf16>(__uint_as_float(o[2 * i]) * inv_l,
                                                       __uint_as_float(o[2 * i + 1]) * inv_l);
                    if (row_ok) {  // whole 32-byte sectors
                        st_global_32b(orow + c * 32 * kOb, pk);
                        st_global_32b(orow + c * 32 * kOb + 32, pk + 8);
                    }
                }
            }
            if (row_ok && lse_ptr) *lse_ptr = (l > 0.f) ? (m_used + lg2_approx(l)) * kLn2 : -INFINITY;
            ++uo;
        }
        if constexpr (kFp8) {
            // max |O| of the tile chain's rows into the caller's amax
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            if (p.amax_o && lane == 0 && amax > 0.f)
                atomicMax(reinterpret_cast<int *>(p.amax_o), __float_as_int(amax));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// launch register count of the last build launch_pair_t refused on this thread
thread_local int t_refused_regs = 0;

std::atomic<uint32_t> g_pair_counter_next{0};

template <int D, int kEl, bool kPacked, int kOut, bool kWin = false, bool kSplit = false, bool kDyn = false>
cudaError_t launch_pair_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const FwdParams &p, int grid, cudaStream_t stream,
                          const KernelTimer &timer) {
    using L = PairLayout<D, kEl == kElE4m3 ? 1 : 2, kPacked>;
    auto kern = fwd_pair_kernel<D, kEl, kPacked, kOut, kWin, kSplit, kDyn>;
    // The softmax warpgroups' setmaxnreg.inc waits for the registers warpgroup
    // 0 releases; a build launched with any other per-thread count than the
    // split assumes would leave it waiting, so such a build is not launched.
    // The count is read once per instantiation; a failed query is passed on
    // (a missing kernel image stays "unsupported") and asked again next time.
    static std::atomic<int> launch_regs{0};  // 0: not read yet
    t_refused_regs = 0;
    int regs = launch_regs.load(std::memory_order_relaxed);
    if (regs == 0) {
        cudaFuncAttributes fa{};
        const cudaError_t q = cudaFuncGetAttributes(&fa, kern);
        if (q != cudaSuccess) return q;
        regs = fa.numRegs;
        launch_regs.store(regs, std::memory_order_relaxed);
    }
    if (regs != kPairLaunchRegs) {
        t_refused_regs = regs;
        return cudaErrorInvalidConfiguration;
    }
    if constexpr (kDyn) {
        // a zeroed counter slot for this launch, carried in s_q (see PairDynLayout)
        using DL = PairDynLayout<D, kEl == kElE4m3 ? 1 : 2>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DL::kSmemAlloc);
        if (e != cudaSuccess) return e;
        const int slot = (int)(g_pair_counter_next.fetch_add(1) % kPairCounterSlots);
        void *ctr = nullptr;
        e = cudaGetSymbolAddress(&ctr, g_pair_unit_counters);
        if (e != cudaSuccess) return e;
        e = cudaMemsetAsync(static_cast<uint32_t *>(ctr) + slot, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
        FwdParams pd = p;
        pd.s_q = slot + 1;
        if (timer.start) cudaEventRecord(timer.start, stream);
        kern<<<grid, kPairThreads, DL::kSmemAlloc, stream>>>(tq, tk, tv, pd);
        e = cudaGetLastError();
        if (timer.stop) cudaEventRecord(timer.stop, stream);
        return e;
    } else {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             L::kSmemAlloc);
        if (e != cudaSuccess) return e;
        if (timer.start) cudaEventRecord(timer.start, stream);
        kern<<<grid, kPairThreads, L::kSmemAlloc, stream>>>(tq, tk, tv, p);
        e = cudaGetLastError();
        if (timer.stop) cudaEventRecord(timer.stop, stream);
        return e;
    }
}

// Packed lists: those that fit the kernel's sequence table take their units
// dynamically (PairDynLayout), longer ones keep the fixed deal.
template <int D, int kEl, int kOut>
cudaError_t launch_pair_packed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                               const FwdParams &p, int grid, cudaStream_t stream, const KernelTimer &timer) {
    using L = PairLayout<D, kEl == kElE4m3 ? 1 : 2, true>;
    if (p.num_seqs + 1 <= L::kCuCap)
        return launch_pair_t<D, kEl, true, kOut, false, false, true>(tq, tk, tv, p, grid, stream, timer);
    return launch_pair_t<D, kEl, true, kOut>(tq, tk, tv, p, grid, stream, timer);
}

}  // namespace

int fwd_pair_rows() { return kPairRows; }
int fwd_pair_table_cap(int d, bool fp8) {
    if (fp8) return PairLayout<128, 1, true>::kCuCap;
    return d == 64 ? PairLayout<64, 2, true>::kCuCap : PairLayout<128, 2, true>::kCuCap;
}
int fwd_pair_split_regs() { return kPairLaunchRegs; }
int fwd_pair_refused_regs() { return t_refused_regs; }

cudaError_t launch_fwd_pair(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const FwdParams &p, int d, bool bf16, bool packed, int grid,
                            cudaStream_t stream, const KernelTimer &timer) {
    // left windows: the walking instantiations, bf16 / fp16 at d = 128 only
    // (the host sends every other windowed problem to the one-tile kernel)
    if (p.window >= 0) {
        if (d != 128) return cudaErrorInvalidValue;
        if (bf16)
            return packed ? launch_pair_t<128, kElBf16, true, kElBf16, true>(tq, tk, tv, p, grid, stream, timer)
                          : launch_pair_t<128, kElBf16, false, kElBf16, true>(tq, tk, tv, p, grid, stream, timer);
        return packed ? launch_pair_t<128, kElFp16, true, kElFp16, true>(tq, tk, tv, p, grid, stream, timer)
                      : launch_pair_t<128, kElFp16, false, kElFp16, true>(tq, tk, tv, p, grid, stream, timer);
    }
    // dense lists with a cut tail (more units than blocks)
    if (!packed && p.n_units > p.q_tiles * p.bh) {
        if (d == 64)
            return bf16 ? launch_pair_t<64, kElBf16, false, kElBf16, false, true>(tq, tk, tv, p, grid, stream, timer)
                        : launch_pair_t<64, kElFp16, false, kElFp16, false, true>(tq, tk, tv, p, grid, stream, timer);
        if (d == 128)
            return bf16 ? launch_pair_t<128, kElBf16, false, kElBf16, false, true>(tq, tk, tv, p, grid, stream, timer)
                        : launch_pair_t<128, kElFp16, false, kElFp16, false, true>(tq, tk, tv, p, grid, stream, timer);
        return cudaErrorInvalidValue;
    }
#define SDPA_PAIR_CASE(D_, EL_)                                                \
    if (d == D_ && (bf16 ? kElBf16 : kElFp16) == EL_)                          \
        return packed ? launch_pair_packed<D_, EL_, EL_>(tq, tk, tv, p, grid, stream, timer) \
                      : launch_pair_t<D_, EL_, false, EL_>(tq, tk, tv, p, grid, stream, timer);
    SDPA_PAIR_CASE(64, kElBf16)
    SDPA_PAIR_CASE(64, kElFp16)
    SDPA_PAIR_CASE(128, kElBf16)
    SDPA_PAIR_CASE(128, kElFp16)
#undef SDPA_PAIR_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_pair_fp8(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                const FwdParams &p, int out, bool packed, int grid,
                                cudaStream_t stream, const KernelTimer &timer) {
    if (p.window >= 0) return cudaErrorInvalidValue;  // the host keeps windows on the one-tile kernel
    if (!packed && p.n_units > p.q_tiles * p.bh) {  // dense lists with a cut tail
        if (out == kElBf16) return launch_pair_t<128, kElE4m3, false, kElBf16, false, true>(tq, tk, tv, p, grid, stream, timer);
        if (out == kElFp16) return launch_pair_t<128, kElE4m3, false, kElFp16, false, true>(tq, tk, tv, p, grid, stream, timer);
        if (out == kElE4m3) return launch_pair_t<128, kElE4m3, false, kElE4m3, false, true>(tq, tk, tv, p, grid, stream, timer);
        return cudaErrorInvalidValue;
    }
#define SDPA_PAIR_FP8_CASE(OUT_)                                               \
    if (out == OUT_)                                                           \
        return packed ? launch_pair_packed<128, kElE4m3, OUT_>(tq, tk, tv, p, grid, stream, timer) \
                      : launch_pair_t<128, kElE4m3, false, OUT_>(tq, tk, tv, p, grid, stream, timer);
    SDPA_PAIR_FP8_CASE(kElBf16)
    SDPA_PAIR_FP8_CASE(kElFp16)
    SDPA_PAIR_FP8_CASE(kElE4m3)
#undef SDPA_PAIR_FP8_CASE
    return cudaErrorInvalidValue;
}

}  // namespace sdpa
