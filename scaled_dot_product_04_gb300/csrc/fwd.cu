// Fused attention forward for sm_103a: O = softmax(scale * Q K^T + mask) V and
// the per-row log-sum-exp, dense BHSD or packed THD.
//
// Operation: "Inside NVIDIA's cuDNN Graph API" (tradepoint.io), section 5
// "SDPA (Flash Attention) with causal masking" -- top-left causal alignment,
// fp32 intermediate and compute type -- widened to the masks and grouped
// key/value heads of the cudnn-frontend PR #554 `sdpa` op (causal_bottom_right,
// window_left; GQA): a unit visits only the key tiles its rows can see, and
// query head hq reads key/value head hq / (h / h_kv).  Softmax runs in the base-2 domain with
// scale*log2(e) folded into one multiplier (cudnn-frontend PR #554, SM100
// FP8 d512 notes: scale_softmax_log2); LSE is converted back to the natural
// log on write-out.  Tiles wholly above the causal diagonal are never loaded
// or multiplied; only diagonal and ragged-tail tiles pay for masking
// (cudnn-frontend PR #554, SM80 backward notes on PARTIAL/GATE tile bounds).
//
// Persistent schedule (cudnn-frontend PR #554, "Thd persistent grid" and the
// LPT scheduler notes): the grid is capped at one CTA per SM; CTA c walks
// the units c, c + grid, c + 2*grid, ... of a list ordered latest query tile
// first, which under the causal mask is heaviest first.  A unit is one
// 128-row query tile of one (batch, head) or (sequence, head).  When K and V
// outgrow L2 the list runs slice group by slice group instead (dense: the
// heads of one batch; packed: one sequence, longest first), latest tile
// first within a group, so the units in flight share a few slices' K and V
// in L2 rather than streaming a different slice each from HBM.  Packed
// sequences are found from cu_seqlens on the device (cached in shared
// memory); a unit past its sequence's end costs a few instructions.
//
// Roles inside a CTA:
//   warp 0      TMA producer: Q and the first K tile of each unit, then per
//               key tile j the pair V_j, K_{j+1} on one barrier (K and V keep
//               rings of their own);
//   warp 1      MMA issuer (one thread): S_t = Q K_t^T into TMEM (two S
//               buffers, alternating over the CTA's running tile count t),
//               then O += P_t V_t with P_t read straight from TMEM;
//   warps 2..5  softmax: thread r owns query row r (= TMEM lane r); it reads
//               S_t, applies the mask, keeps the fp32 running max/sum, writes
//               P_t (bf16/fp16) back into the S_t columns, rescales O in TMEM
//               when the running max grows by more than 2^8, and finally
//               normalises O and writes O and LSE -- while the MMA warp
//               already runs the next unit's first products.
// TMEM columns: S buffers at 0 and 128, O at 256 (d columns).
//
// Packed layout: the Q/K/V tensor maps span exactly total_q / total_kv
// tokens, so a tile that steps past the packed total reads TMA zero fill and
// never the caller's capacity tail (cudnn-frontend PR #554, "clamp the f16
// THD K/V descriptors to the packed total"); keys of the next sequence that
// share a tile are masked to -inf before the exponent.
#include <atomic>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {
namespace {

// kEb: bytes per input element (2 for bf16/fp16, 1 for E4M3).
template <int D, int kEb = 2>
struct FwdLayout {
    static constexpr int kChunks = D * kEb / 128;          // 128-byte swizzle columns per row
    static constexpr int kChunkBytes = kTileM * 128;      // 16 KiB: 128 rows x 128 bytes
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    // K and V have rings of their own.  Per key tile t the producer issues
    // V_t and K_{t+1} as a pair on V_t's full barrier, and a V stage is
    // released once O += P V has read it (the P V retired barrier below).  That release also frees the K ring:
    // K_{i-kKStages} is read by S products issued before the release of
    // V_{i-1-kVStages}, which the producer waits for before it loads K_i, as
    // long as the K ring is at least one stage deeper than the V ring.
    static constexpr int kKStages = (kTileBytes >= 32768) ? 3 : 5;
    static constexpr int kVStages = (kTileBytes >= 32768) ? 2 : 4;
    static_assert(kKStages >= kVStages + 1, "the V releases must cover the K ring");
    // Q is double-buffered by unit parity so the next unit's Q arrives while
    // the current unit still runs.
    static constexpr int kQStages = 2;
    // cu_seqlens entries cached in shared memory, with the packed unit list's
    // sequence order and unit offsets (longer lists are read from global
    // memory in the envelope order); at d = 128 only the room left by the
    // rings is used.
    static constexpr int kCuCap = (kTileBytes >= 32768) ? 96 : 1024;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kQStages * kTileBytes;
    static constexpr int kV = kK + kKStages * kTileBytes;
    // int32 cu_q[kCuCap], cu_kv[kCuCap], order[kCuCap], first_unit[kCuCap]
    static constexpr int kCu = kV + kVStages * kTileBytes;
    static constexpr int kScan = kCu + 4 * kCuCap * 4;  // 8 int32: per-warp sums
    static constexpr int kBar = kScan + 32;
    static constexpr int bQFull = 0;   // two
    static constexpr int bQEmpty = 2;  // two
    static constexpr int bKFull = 4;
    static constexpr int bVFull = bKFull + kKStages;
    static constexpr int bSFull = bVFull + kVStages;  // two
    // P_t ready: two barriers, indexed by t & 1; P_t V_t retired: one per V
    // stage, indexed by t % kVStages, which is also V_t's release (and with it
    // the K stages', see above).  No waiter can be two phases away from the
    // barrier it polls.
    static constexpr int bPReady = bSFull + 2;   // two
    static constexpr int bPVDone = bPReady + 2;  // kVStages
    // O is double-buffered by unit parity: the epilogue of unit k overlaps
    // the products of unit k+1.
    static constexpr int bOFull = bPVDone + kVStages;  // two: a unit's last P V retired
    static constexpr int bOFree = bOFull + 2;    // two: the epilogue has read O
    static constexpr int bMmaIdle = bOFree + 2;
    static constexpr int kNumBars = bMmaIdle + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;  // u32[0] TMEM base, u32[1] abort flag
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kSmemAlloc = kBytes + 1024;  // slack to align the base to 1024 B
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 256;  // O buffer b at kColO + b * D
};

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only if the max grows by 2^8

// Each lane waits; the warp proceeds only if every lane saw the phase, so the
// warp-collective tcgen05.ld/st that follow stay convergent.
SDPA_DEV bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx &w, uint32_t site) {
    bool ok = mbar_wait(bar, parity, w, site);
    return __all_sync(0xffffffffu, ok);
}

// k-th unit of CTA `first` out of `step`: a boustrophedon walk over the
// heaviest-first list (c, 2G-1-c, 2G+c, 4G-1-c, ...), which evens out the
// per-CTA sums of a decreasing cost list better than plain striding.
SDPA_DEV int unit_of(int k, int first, int step) {
    return k * step + ((k & 1) ? step - 1 - first : first);
}

// One work unit: a 128-row query tile of one slice.  It visits key tiles
// kt0 .. kt0 + n_kv - 1; K/V come from slice kv_slice (dense) or head
// kv_head (packed).
struct Unit {
    int slice, head, kv_slice, kv_head, Lq, Lkv, tok_q0, tok_kv0, row0, kt0, n_kv, delta;
    bool live;  // the tile holds at least one query row
    int64_t o_row0, o_rs, lse_row0, lse_rs;
};

// Packed units in sequence-major order: `order` lists the sequences by
// query-tile count, most first, and sequence order[i] owns units
// [first_unit[i], first_unit[i + 1]), its query tiles latest first with the
// heads innermost.  The CTAs running at any time then share one or two
// sequences, whose K and V stay in L2 while every head's units stream them.
SDPA_DEV void packed_slot(const FwdParams &p, int u, const int *cu_q, const int *order,
                          const int *first_unit, int &qt, int &slice) {
    int lo = 0, hi = p.num_seqs;  // first_unit[lo] <= u < first_unit[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (first_unit[mid] <= u) lo = mid;
        else hi = mid;
    }
    const int n = order[lo], local = u - first_unit[lo];
    const int tiles = (cu_q[n + 1] - cu_q[n] + kTileM - 1) / kTileM;
    qt = tiles - 1 - local / p.h;
    slice = n * p.h + local % p.h;
}

// Unit u.  With slice_major, dense units run batch by batch (the h
// slices of one batch, latest query tile first, heads innermost) and packed
// ones sequence by sequence (order != nullptr, see packed_slot); otherwise,
// and for packed lists too long for the shared table, latest query tile
// first over all slices (heaviest first, which balances small problems best).
template <int D, bool kPacked>
SDPA_DEV Unit decode_unit(const FwdParams &p, int u, const int *cu_q, const int *cu_kv,
                          bool slice_major, const int *order, const int *first_unit) {
    Unit U;
    int qt;
    if (kPacked && order) {
        packed_slot(p, u, cu_q, order, first_unit, qt, U.slice);
    } else {
        // slice groups of gs slices (all of them unless slice-major dense)
        const int gs = (!kPacked && slice_major) ? p.h : p.bh;
        const int per_group = gs * p.q_tiles;
        const int g = u / per_group, local = u - g * per_group;
        qt = p.q_tiles - 1 - local / gs;
        U.slice = g * gs + local % gs;
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
    U.row0 = qt * kTileM;
    U.live = U.row0 < U.Lq;
    // keys seen by any row: from the first row's window start to the last
    // row's causal end
    U.delta = mask_delta(p.mask, U.Lq, U.Lkv);
    const int lo = max(0, key_range(p.mask, p.window, U.row0, U.delta, U.Lkv).lo);
    const int hi = key_range(p.mask, p.window, min(U.row0 + kTileM, U.Lq) - 1, U.delta, U.Lkv).hi;
    U.kt0 = lo / kTileN;
    U.n_kv = (U.live && hi > lo) ? (hi + kTileN - 1) / kTileN - U.kt0 : 0;
    return U;
}

// Element kinds: kEl is the input type (kElBf16, kElFp16 or kElE4m3), kOut
// the output type (the input type for 16-bit inputs; bf16, fp16 or E4M3 for
// E4M3 inputs).  E4M3 inputs (cudnn-frontend PR #554, per-tensor FP8
// forward) carry per-tensor descales read from device memory:
// descale_q * descale_k folds into the softmax multiplier and descale_v
// (times scale_o for an E4M3 output) into the output factor; amax_o, if
// given, receives max |O| of the real-valued output.  P enters P V as E4M3,
// four per TMEM column; every product is a kind::f8f6f4 MMA of K = 32.
// Units taken dynamically (kDyn): packed lists ordered sequence by sequence
// (see packed_slot) are sawtooth-shaped -- each sequence's units go from
// heaviest to lightest -- so a fixed deal of the list leaves some CTAs with
// more work than others (a dispatch simulation of the 16-sequence workload:
// makespan 370 tile steps against 352 dealt on demand).  The kDyn
// instantiations take units from a counter instead, in the same list order
// (which keeps each sequence's K and V in L2): the producer thread takes the
// next unit when it has issued the current one's loads and hands it to the
// MMA thread and the softmax warps through a ring of kUnitRing slots placed
// after the layout.  `sched`: bit 0 selects the slice-major order; kDyn
// launches carry their counter's slot (in g_fwd_unit_counters) + 1 above it.
// The other instantiations read `sched` as the plain slice-major flag and
// compile as before.
constexpr int kUnitRing = 4;
constexpr int kFwdCounterSlots = 1024;
__device__ uint32_t g_fwd_unit_counters[kFwdCounterSlots];
template <int D, int kEb>
struct FwdDynLayout {
    using L = FwdLayout<D, kEb>;
    static constexpr int kRing = L::kBytes;                  // kUnitRing ints
    static constexpr int kRingBar = kRing + 4 * kUnitRing;  // full, empty: kUnitRing each
    static constexpr int kBytes = kRingBar + 2 * kUnitRing * 8;
    static constexpr int kSmemAlloc = kBytes + 1024;
};
static_assert(FwdDynLayout<128, 2>::kSmemAlloc <= 232448, "dynamic one-tile forward exceeds shared memory");

template <int D, int kEl, bool kPacked, int kOut, bool kDyn = false>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p, const int sched) {
    const int slice_major = kDyn ? (sched & 1) : sched;
    constexpr bool kFp8 = kEl == kElE4m3;
    constexpr bool kBf16 = kEl == kElBf16;
    constexpr int kEb = kFp8 ? 1 : 2;
    using L = FwdLayout<D, kEb>;
    using io_t = uint16_t;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();
    // kDyn: the unit ring, its barriers and this launch's counter
    using DL = FwdDynLayout<D, kEb>;
    auto dbar = [&](int i) -> uint32_t { return sbase + DL::kRingBar + 8u * i; };
    volatile int *ring = reinterpret_cast<volatile int *>(smem + DL::kRing);
    uint32_t *unit_ctr = kDyn ? g_fwd_unit_counters + ((sched >> 1) - 1) : nullptr;

    // cu_seqlens of packed inputs, cached when they fit, and then the
    // sequence-major unit list (see packed_slot)
    int *cu_q_s = reinterpret_cast<int *>(smem + L::kCu);
    int *cu_kv_s = cu_q_s + L::kCuCap;
    int *order_s = cu_kv_s + L::kCuCap;
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
        }
        if (p.num_seqs + 1 <= L::kCuCap && slice_major) {
            const int ns = p.num_seqs;
            __syncthreads();
            auto tiles = [&](int n) { return (cu_q_s[n + 1] - cu_q_s[n] + kTileM - 1) / kTileM; };
            // most query tiles first, ties in sequence order (a rank count;
            // long lists keep their own order)
            for (int n = threadIdx.x; n < ns; n += blockDim.x) {
                int rank = n;
                if (ns <= 256) {
                    const int tn = tiles(n);
                    rank = 0;
                    for (int m = 0; m < ns; ++m) {
                        const int tm = tiles(m);
                        rank += (tm > tn || (tm == tn && m < n)) ? 1 : 0;
                    }
                }
                order_s[rank] = n;
            }
            __syncthreads();
            // first_unit = exclusive prefix sum of tiles(order[i]) * h: each
            // thread sums a chunk, the chunk sums are scanned in the warp and
            // across the warps
            int *scan = reinterpret_cast<int *>(smem + L::kScan);
            const int per = (ns + blockDim.x - 1) / blockDim.x;
            const int b0 = min(ns, (int)threadIdx.x * per), b1 = min(ns, b0 + per);
            int csum = 0;
            for (int i = b0; i < b1; ++i) csum += tiles(order_s[i]) * p.h;
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
                run += tiles(order_s[i]) * p.h;
            }
            if (threadIdx.x == blockDim.x - 1) first_s[ns] = run;  // the last chunk ends the list
            __syncthreads();
            order = order_s;
            n_units = first_s[ns];
        }
    }

    if (threadIdx.x == 0) {
        for (int b = 0; b < L::kQStages; ++b) {
            mbar_init(bar(L::bQFull + b), 1);
            mbar_init(bar(L::bQEmpty + b), 1);
        }
        for (int s = 0; s < L::kKStages; ++s) mbar_init(bar(L::bKFull + s), 1);
        for (int s = 0; s < L::kVStages; ++s) {
            mbar_init(bar(L::bVFull + s), 1);
            mbar_init(bar(L::bPVDone + s), 1);
        }
        mbar_init(bar(L::bSFull + 0), 1);
        mbar_init(bar(L::bSFull + 1), 1);
        for (int b = 0; b < 2; ++b) mbar_init(bar(L::bPReady + b), kTileM);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::bOFull + b), 1);
            mbar_init(bar(L::bOFree + b), kTileM);
        }
        mbar_init(bar(L::bMmaIdle), 1);
        if constexpr (kDyn) {
            for (int b = 0; b < kUnitRing; ++b) {
                mbar_init(dbar(b), 1);              // full: the producer
                mbar_init(dbar(kUnitRing + b), 5);  // empty: the MMA thread and 4 softmax warps
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

    if (warp == 0) {
        // ============================================================ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            // Per unit: Q, the unit's first K tile (on its K stage's full
            // barrier), then per key tile j the pair V_j, K_{j+1}, both on V_j's
            // full barrier, so the MMA thread waits once per key tile.  A K tile
            // that rides on a V barrier gives its own stage's full barrier a
            // plain arrive, so the K barriers keep one phase per K tile; the
            // MMA thread waits on them only for a unit's first K, whose stage
            // cannot be refilled before that wait (the refill waits for a V
            // release that the MMA thread commits only after it).
            int k_it = 0, v_it = 0, units = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                int u;
                if constexpr (kDyn) {
                    // take the next unit (the first by the CTA's index) and hand it on
                    const int slot = k % kUnitRing;
                    if (k >= kUnitRing && !mbar_wait(dbar(kUnitRing + slot), ((k / kUnitRing) - 1) & 1, wc, 20))
                        break;
                    u = k == 0 ? (int)blockIdx.x : (int)gridDim.x + (int)atomicAdd(unit_ctr, 1u);
                    if (u >= n_units) u = -1;
                    ring[slot] = u;
                    mbar_arrive(dbar(slot));
                    if (u < 0) break;
                } else {
                    u = unit_of(k, first, step);
                    if (u >= n_units) break;
                }
                const Unit U = decode_unit<D, kPacked>(p, u, cu_q, cu_kv, slice_major, order, first_s);
                if (U.n_kv == 0) continue;
                const int qs = units & 1;
                if (units > 1 && !mbar_wait(bar(L::bQEmpty + qs), ((units - 2) >> 1) & 1, wc, 1)) break;
                const int qy = kPacked ? U.head : U.row0;
                const int qz = kPacked ? U.tok_q0 + U.row0 : U.slice;
                mbar_arrive_expect_tx(bar(L::bQFull + qs), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kQ + qs * L::kTileBytes + c * L::kChunkBytes, &tm_q,
                                bar(L::bQFull + qs), c * (128 / kEb), qy, qz);
                ++units;
                // key tile j of the unit: (y, z) coordinates of K_j and V_j
                auto kv_yz = [&](int j, int &y, int &z) {
                    const int k0 = (U.kt0 + j) * kTileN;
                    y = kPacked ? U.kv_head : k0;
                    z = kPacked ? U.tok_kv0 + k0 : U.kv_slice;
                };
                // K tile number k_it into its stage (free: see FwdLayout), on `full`
                auto load_k = [&](uint32_t full, int j) {
                    int ky, kz;
                    kv_yz(j, ky, kz);
                    const int ks = k_it % L::kKStages;
#pragma unroll
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_3d(sbase + L::kK + ks * L::kTileBytes + c * L::kChunkBytes, &tm_k, full,
                                    c * (128 / kEb), ky, kz);
                    ++k_it;
                };
                {
                    const uint32_t kfull = bar(L::bKFull + k_it % L::kKStages);
                    mbar_arrive_expect_tx(kfull, L::kTileBytes);
                    load_k(kfull, 0);
                }
                for (int j = 0; j < U.n_kv; ++j) {
                    const int vs = v_it % L::kVStages, vuse = v_it / L::kVStages;
                    if (vuse > 0 && !mbar_wait(bar(L::bPVDone + vs), (vuse - 1) & 1, wc, 3)) {
                        ok = false;
                        break;
                    }
                    const bool pair_k = j + 1 < U.n_kv;
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
                        mbar_arrive(bar(L::bKFull + k_it % L::kKStages));
                        load_k(vfull, j + 1);
                    }
                }
            }
            // Every load issued must land before the CTA may exit.
            for (int i = max(0, units - 2); i < units; ++i)
                mbar_wait_drain(bar(L::bQFull + (i & 1)), (i >> 1) & 1);
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
            // S = Q K^T: both operands K-major (head dim contiguous), 32 bytes
            // (16 bf16 or 32 E4M3 elements) per step.
            int units = 0;  // live units processed by this CTA (selects the Q buffer)
            auto issue_s = [&](int ks, uint32_t col) {
                const uint64_t a = dQ_k + (units & 1) * kTile16, b = dK_k + ks * kTile16;
#pragma unroll
                for (int k = 0; k < D * kEb / 32; ++k) {
                    const uint32_t off = (k / 4) * kChunk16 + (k % 4) * 2;
                    if constexpr (kFp8)
                        mma_ss_f8(tmem + col, a + off, b + off, idesc_s, k > 0);
                    else
                        mma_ss(tmem + col, a + off, b + off, idesc_s, k > 0);
                }
            };
            // O += P V: P from TMEM (8 columns per step: 16 keys as bf16 pairs
            // or 32 keys as E4M3 quads), V MN-major (head dim contiguous);
            // 128-byte head-dim chunks are 16 KiB apart (leading offset),
            // 8-key groups 1 KiB apart, so a step advances 2 or 4 KiB.
            auto issue_pv = [&](int vs, uint32_t pcol, uint32_t ocol, bool acc) {
                const uint64_t vb = dV_mn + vs * kTile16;
#pragma unroll
                for (int k = 0; k < kTileN * kEb / 32; ++k) {
                    const uint64_t vdesc = vb + k * ((4096 / kEb) >> 4);
                    if constexpr (kFp8)
                        mma_ts_f8(tmem + ocol, tmem + pcol + k * 8, vdesc, idesc_o, (acc || k > 0) ? 1u : 0u);
                    else
                        mma_ts(tmem + ocol, tmem + pcol + k * 8, vdesc, idesc_o, (acc || k > 0) ? 1u : 0u);
                }
            };
            // S_x goes to S buffer x&1, which held P_{x-2}: it waits for that
            // P V product (barrier (x-2) % kVStages, phase (x-2) / kVStages).
            // Every P V phase is waited here in order, so the waits stay within
            // one phase.
            // K_x has landed when this is called: a unit's first K tile is
            // waited for on its own barrier, every other one with V_{x-1}.
            auto issue_s_tile = [&](int x) -> bool {
                if (x >= 2 &&
                    !mbar_wait(bar(L::bPVDone + (x - 2) % L::kVStages), ((x - 2) / L::kVStages) & 1, wc, 6))
                    return false;
                tc_fence_after();
                issue_s(x % L::kKStages, (x & 1) * 128);
                mma_commit(bar(L::bSFull + (x & 1)));
                return true;
            };
            int t = 0;  // tiles processed by this CTA
            bool ok = true;
            for (int k = 0; ok; ++k) {
                int u;
                if constexpr (kDyn) {
                    const int slot = k % kUnitRing;
                    if (!(ok = mbar_wait(dbar(slot), (k / kUnitRing) & 1, wc, 21))) break;
                    u = ring[slot];
                    mbar_arrive(dbar(kUnitRing + slot));
                    if (u < 0) break;
                } else {
                    u = unit_of(k, first, step);
                    if (u >= n_units) break;
                }
                const Unit U = decode_unit<D, kPacked>(p, u, cu_q, cu_kv, slice_major, order, first_s);
                if (U.n_kv == 0) continue;
                ok = mbar_wait(bar(L::bQFull + (units & 1)), (units >> 1) & 1, wc, 4) &&
                     mbar_wait(bar(L::bKFull + t % L::kKStages), (t / L::kKStages) & 1, wc, 5) &&
                     issue_s_tile(t);
                if (!ok) break;
                if (U.n_kv == 1) mma_commit(bar(L::bQEmpty + (units & 1)));
                for (int j = 0; j < U.n_kv; ++j, ++t) {
                    // V_t and, within the unit, K_{t+1} (see the producer)
                    if (!(ok = mbar_wait(bar(L::bVFull + t % L::kVStages), (t / L::kVStages) & 1, wc, 10)))
                        break;
                    if (j + 1 < U.n_kv) {
                        if (!(ok = issue_s_tile(t + 1))) break;
                        if (j + 2 == U.n_kv) mma_commit(bar(L::bQEmpty + (units & 1)));  // last reader of Q
                    }
                    ok = mbar_wait(bar(L::bPReady + (t & 1)), (t >> 1) & 1, wc, 9);
                    // The unit's first P V overwrites O buffer units&1: the epilogue
                    // of the unit two back must have read it out.
                    if (ok && j == 0 && units > 1)
                        ok = mbar_wait(bar(L::bOFree + (units & 1)), ((units - 2) >> 1) & 1, wc, 11);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(t % L::kVStages, (t & 1) * 128, L::kColO + (units & 1) * D, j > 0);
                    mma_commit(bar(L::bPVDone + t % L::kVStages));  // also V_t's release
                }
                if (!ok) break;
                mma_commit(bar(L::bOFull + (units & 1)));
                ++units;
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
        float sl2 = p.scale_log2;
        float o_factor = 1.f;  // descale_v (times scale_o for an E4M3 output)
        if constexpr (kFp8) {
            sl2 *= *p.descale_q * *p.descale_k;
            o_factor = *p.descale_v;
        }
        constexpr int kOb = kOut == kElE4m3 ? 1 : 2;  // output bytes per element
        float amax = 0.f;  // max |O| over this thread's rows (E4M3 inputs)
        // A unit's epilogue (O / l, LSE) is deferred until the next unit's
        // first P is out, so the MMA warp has work while O is written.
        struct Pending {
            bool on;
            bool row_ok;
            int unit;
            float l, m;
            uint8_t *orow;
            float *lse;
        } pend{false, false, 0, 0.f, 0.f, nullptr, nullptr};
        auto epilogue = [&]() -> bool {
            const int ob = pend.unit & 1;
            if (!warp_wait(bar(L::bOFull + ob), (pend.unit >> 1) & 1, wc, 14)) return false;
            tc_fence_after();
            const float inv_l = (pend.l > 0.f) ? o_factor / pend.l : 0.f;
            const uint32_t ocol = L::kColO + ob * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(t_lane + ocol + c * 32, o);
                tmem_ld_wait_regs<32>(o);
                if (c == D / 32 - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(L::bOFree + ob));
                }
                if constexpr (kFp8) {
                    if (pend.row_ok) {
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
                    if (pend.row_ok) st_global_32b(pend.orow + c * 32 * kOb, pk);
                } else {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack2<kOut == kElBf16>(__uint_as_float(o[2 * i]) * inv_l,
                                                       __uint_as_float(o[2 * i + 1]) * inv_l);
                    if (pend.row_ok) {  // whole 32-byte sectors
                        st_global_32b(pend.orow + c * 32 * kOb, pk);
                        st_global_32b(pend.orow + c * 32 * kOb + 32, pk + 8);
                    }
                }
            }
            if (pend.row_ok && pend.lse)
                *pend.lse = (pend.l > 0.f) ? (pend.m + lg2_approx(pend.l)) * kLn2 : -INFINITY;
            pend.on = false;
            return true;
        };
        int t = 0, units = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int u;
            if constexpr (kDyn) {
                const int slot = k % kUnitRing;
                if (!(ok = warp_wait(dbar(slot), (k / kUnitRing) & 1, wc, 22))) break;
                u = ring[slot];
                __syncwarp();
                if (lane == 0) mbar_arrive(dbar(kUnitRing + slot));
                if (u < 0) break;
            } else {
                u = unit_of(k, first, step);
                if (u >= n_units) break;
            }
            const Unit U = decode_unit<D, kPacked>(p, u, cu_q, cu_kv, slice_major, order, first_s);
            if (!U.live) continue;
            const int q_idx = U.row0 + r;
            const bool row_ok = q_idx < U.Lq;
            uint8_t *orow = static_cast<uint8_t *>(p.o) + (U.o_row0 + (int64_t)q_idx * U.o_rs) * kOb;
            float *lse_ptr = p.lse ? p.lse + U.lse_row0 + (int64_t)q_idx * U.lse_rs : nullptr;
            if (U.n_kv == 0) {
                // No key is visible to any row of this tile: O = 0, LSE = -inf.
                if (row_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
                    for (int i = 0; i < D * kOb / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                    if (lse_ptr) *lse_ptr = -INFINITY;
                }
                continue;
            }
            const uint32_t ocol = L::kColO + (units & 1) * D;
            float m_used = -INFINITY;  // running max used as exponent base (log2 units)
            float l = 0.f;             // running sum of P
            for (int j = 0; j < U.n_kv; ++j, ++t) {
                const uint32_t cs = (t & 1) * 128;
                ok = warp_wait(bar(L::bSFull + (t & 1)), (t >> 1) & 1, wc, 12);
                if (!ok) break;
                tc_fence_after();
                uint32_t s[kTileN];
#pragma unroll
                for (int c = 0; c < kTileN / 32; ++c) tmem_ld32(t_lane + cs + c * 32, s + c * 32);
                tmem_ld_wait_regs<kTileN>(s);

                const int k0 = (U.kt0 + j) * kTileN;
                // the tile needs a mask unless every row sees all of its keys
                if ((k0 + kTileN > U.Lkv) ||
                    (p.mask != kMaskNone && k0 + kTileN - 1 > U.row0 + U.delta) ||
                    (p.window >= 0 && k0 < U.row0 + kTileM - 1 + U.delta - p.window)) {
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
                tmem_st32(t_lane + cs, s);
                if constexpr (!kFp8) tmem_st32(t_lane + cs + 32, s + 32);

                if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                    // O holds the unit's earlier P V products; it may be rescaled
                    // only once the last of them has retired.
                    ok = warp_wait(bar(L::bPVDone + (t - 1) % L::kVStages), ((t - 1) / L::kVStages) & 1, wc, 13);
                    if (!ok) break;
                    tc_fence_after();
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
                mbar_arrive(bar(L::bPReady + (t & 1)));
                // the previous unit's epilogue, now that this unit's first P is out
                if (j == 0 && pend.on && !(ok = epilogue())) break;
            }
            if (!ok) break;
            pend = Pending{true, row_ok, units, l, m_used, orow, lse_ptr};
            ++units;
        }
        if (ok && pend.on) epilogue();
        if constexpr (kFp8) {
            // max |O| of the CTA's rows into the caller's amax (non-negative
            // floats order as their bit patterns)
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

std::atomic<uint32_t> g_fwd_counter_next{0};

template <int D, int kEl, bool kPacked, int kOut>
cudaError_t launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const FwdParams &p, int grid, bool slice_major, cudaStream_t stream,
                         const KernelTimer &timer) {
    constexpr int kEb = kEl == kElE4m3 ? 1 : 2;
    using L = FwdLayout<D, kEb>;
    // packed lists in the sequence-major order (the kernel's sequence table)
    // take their units dynamically
    if constexpr (kPacked) {
      if (slice_major && p.num_seqs + 1 <= L::kCuCap) {
        using DL = FwdDynLayout<D, kEb>;
        auto kern = fwd_kernel<D, kEl, kPacked, kOut, true>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DL::kSmemAlloc);
        if (e != cudaSuccess) return e;
        const int slot = (int)(g_fwd_counter_next.fetch_add(1) % kFwdCounterSlots);
        void *ctr = nullptr;
        e = cudaGetSymbolAddress(&ctr, g_fwd_unit_counters);
        if (e != cudaSuccess) return e;
        e = cudaMemsetAsync(static_cast<uint32_t *>(ctr) + slot, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
        if (timer.start) cudaEventRecord(timer.start, stream);
        kern<<<grid, 192, DL::kSmemAlloc, stream>>>(tq, tk, tv, p, 1 | ((slot + 1) << 1));
        e = cudaGetLastError();
        if (timer.stop) cudaEventRecord(timer.stop, stream);
        return e;
      }
    }
    auto kern = fwd_kernel<D, kEl, kPacked, kOut>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmemAlloc);
    if (e != cudaSuccess) return e;
    if (timer.start) cudaEventRecord(timer.start, stream);
    kern<<<grid, 192, L::kSmemAlloc, stream>>>(tq, tk, tv, p, slice_major ? 1 : 0);
    e = cudaGetLastError();
    if (timer.stop) cudaEventRecord(timer.stop, stream);
    return e;
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdParams &p, int d, bool bf16, bool packed, int grid,
                       bool slice_major, cudaStream_t stream, const KernelTimer &timer) {
#define SDPA_FWD_CASE(D_, EL_, PK_)                                            \
    if (d == D_ && (bf16 ? kElBf16 : kElFp16) == EL_ && packed == PK_)         \
        return launch_fwd_t<D_, EL_, PK_, EL_>(tq, tk, tv, p, grid, slice_major, stream, timer);
    SDPA_FWD_CASE(64, kElBf16, false)
    SDPA_FWD_CASE(64, kElBf16, true)
    SDPA_FWD_CASE(64, kElFp16, false)
    SDPA_FWD_CASE(64, kElFp16, true)
    SDPA_FWD_CASE(128, kElBf16, false)
    SDPA_FWD_CASE(128, kElBf16, true)
    SDPA_FWD_CASE(128, kElFp16, false)
    SDPA_FWD_CASE(128, kElFp16, true)
#undef SDPA_FWD_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_fp8(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const FwdParams &p, int out, bool packed, int grid, bool slice_major,
                           cudaStream_t stream, const KernelTimer &timer) {
#define SDPA_FP8_CASE(OUT_, PK_)                                               \
    if (out == OUT_ && packed == PK_)                                          \
        return launch_fwd_t<128, kElE4m3, PK_, OUT_>(tq, tk, tv, p, grid, slice_major, stream, timer);
    SDPA_FP8_CASE(kElBf16, false)
    SDPA_FP8_CASE(kElBf16, true)
    SDPA_FP8_CASE(kElFp16, false)
    SDPA_FP8_CASE(kElFp16, true)
    SDPA_FP8_CASE(kElE4m3, false)
    SDPA_FP8_CASE(kElE4m3, true)
#undef SDPA_FP8_CASE
    return cudaErrorInvalidValue;
}

}  // namespace sdpa
