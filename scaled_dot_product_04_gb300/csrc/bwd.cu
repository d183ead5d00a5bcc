// Attention backward for sm_103a: dQ, dK, dV from dO, O and the forward's
// LSE, recomputing P instead of storing it.
//
// The chain follows the backward structure cudnn-frontend PR #554 describes
// for its SM80 kernels ("do_dot", main kernel, "dQ cast"), rebuilt for
// tcgen05/TMEM:
//   bwd_preprocess   D_i = sum_k dO_ik O_ik (fp32), the row terms below and
//                    zeroing of the fp32 dQ accumulator (the PR's fp32 dq
//                    accumulator);
//   bwd_main         one CTA per (slice, 128-key tile), walking the query
//                    tiles that can see those keys;
//   bwd_dq_convert   fp32 accumulator -> dQ in the I/O dtype and Q's layout.
//
// Math per (key tile, query tile), all in the transposed orientation so the
// key tile's rows are TMEM lanes:
//   S'^T = K Q^T - LSE/scale             (tcgen05, K-major operands)
//   P^T  = exp2(S'^T * scale*log2e), masked                   (registers)
//   dP'^T = V dO^T - D
//   dV  += P^T dO                        (A = P^T straight from TMEM)
//   dS'^T = P^T o dP'^T                  (bf16, written once to shared memory)
//   dQ_t = dS' K                         (A = dS'^T's bytes, M-major view)
//   dK  += dS'^T Q                       (A = dS'^T, K-major view)
//   dQacc[rows of the query tile] += dQ_t  (fp32 reductions into global memory)
// dS = scale * dS', so dK and dQ take the factor once, when they are written.
// The row terms -LSE/scale and -D enter the two products as one more K-step
// each (kind::tf32, K = 8): the preprocess kernel stores them per query row as
// tf32 pairs (hi, lo) that sum to the fp32 value within 2^-21 relative, the
// producer loads the 128 rows of a query tile with the tile's Q, and a
// constant operand of 0.5s selects the pair (LSE or D) and adds it into every
// key row of the accumulator.  The compute warps then need no per-query
// statistics at all: those broadcast reads from shared memory had cost as
// many shared-memory cycles as the dS stores and the dQ staging together.
//
// Two compute warpgroups split every tile's 128 query columns in halves, so
// each SM sub-partition has two warps on the exponentials and dS (whose
// latencies one warp alone leaves exposed).  The MMA warp issues dQ before dK:
// dQ shares its TMEM columns with dP at d = 128, and the dQ epilogue's read-out
// then overlaps dK, so dP of the next tile follows without a gap.
#include "bwd_layout.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {
namespace {

// x rounded to the 11 significant bits a tf32 operand keeps (x - result is
// then exact in fp32 and is the low part of the pair).
SDPA_DEV float tf32_hi(float x) { return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u); }



// ------------------------------------------------------------------ preprocess
// One warp handles 32/(d/8) rows at a time; each lane reads 8 elements of O
// and dO with 16-byte loads.
template <int D, bool kBf16, bool kPacked>
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const BwdParams p, int64_t rows, int64_t acc_elems) {
    // the main kernel may set up (barriers, TMEM, its K and V loads) meanwhile;
    // it waits for this grid before it reads a row term or adds into dQ
    griddep_launch_dependents();
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    const int64_t warp_global = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t warps_total = (gridDim.x * (int64_t)blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane / kLanesPerRow, part = lane % kLanesPerRow;
    const uint16_t *o = static_cast<const uint16_t *>(p.o);
    const uint16_t *dout = static_cast<const uint16_t *>(p.dout);
    for (int64_t r0 = warp_global * kRowsPerWarp; r0 < rows; r0 += warps_total * kRowsPerWarp) {
        const int64_t r = r0 + sub;  // row in the I/O order (dense: slice*S+i, packed: t*h+head)
        float acc = 0.f;
        if (r < rows) {
            const uint4 a = *reinterpret_cast<const uint4 *>(o + r * D + part * 8);
            const uint4 b = *reinterpret_cast<const uint4 *>(dout + r * D + part * 8);
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 fa = unpack2<kBf16>(av[i]), fb = unpack2<kBf16>(bv[i]);
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
        }
#pragma unroll
        for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (r < rows && part == 0) {  // row-term layout == I/O row order
            // A row with no visible key (LSE = -inf: a sequence without keys)
            // is masked wherever it appears, also as a tail row of another
            // sequence's tile; its term is made finite so that the 0 * inf of
            // the other row-term K-step cannot turn that tile's dP' into NaN.
            float cl = -p.lse[r] / p.scale;
            if (!isfinite(cl)) cl = 0.f;
            const float cd = -acc;
            float4 t;
            t.x = tf32_hi(cl);
            t.y = cl - t.x;
            t.z = tf32_hi(cd);
            t.w = cd - t.z;
            p.rowx[r] = t;
        }
    }
    if (p.unit_ctr && blockIdx.x == 0 && threadIdx.x == 0) *p.unit_ctr = 0u;
    // zero the fp32 dQ accumulator
    float4 *acc4 = reinterpret_cast<float4 *>(p.dq_acc);
    const int64_t n4 = acc_elems / 4;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
         i += gridDim.x * (int64_t)blockDim.x)
        acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ dq convert
template <int D, bool kBf16, bool kPacked>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const BwdParams p, int64_t rows) {
    griddep_wait();  // the main kernel's dQ accumulator is complete
    // thread handles 8 consecutive elements of one row of dQ (I/O order)
    constexpr int kPerRow = D / 8;
    const int64_t total = rows * kPerRow;
    uint16_t *dq = static_cast<uint16_t *>(p.dq);
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += gridDim.x * (int64_t)blockDim.x) {
        const int64_t r = idx / kPerRow;
        const int part = (int)(idx % kPerRow);
        int64_t acc_row;
        if constexpr (kPacked) {
            const int64_t t = r / p.h, head = r % p.h;
            acc_row = head * (int64_t)p.total_q + t;
        } else {
            acc_row = r;
        }
        const float4 *src = reinterpret_cast<const float4 *>(p.dq_acc + acc_row * D + part * 8);
        const float4 a = src[0], b = src[1];
        uint4 out;
        const float sc = p.scale;  // the accumulator holds dS' K
        out.x = pack2<kBf16>(a.x * sc, a.y * sc);
        out.y = pack2<kBf16>(a.z * sc, a.w * sc);
        out.z = pack2<kBf16>(b.x * sc, b.y * sc);
        out.w = pack2<kBf16>(b.z * sc, b.w * sc);
        *reinterpret_cast<uint4 *>(dq + r * D + part * 8) = out;
    }
}

// ------------------------------------------------------------------ main

template <int D, bool kBf16, bool kPacked>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_rx,
                    const BwdParams p) {
    using L = BwdLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);

    // ---------------------------------------------------------------- work unit
    // A CTA owns one key tile of one key/value slice ((batch, kv head) or
    // (sequence, kv head)) and walks every query tile that can see it, for
    // each of the group's h / h_kv query heads in turn, so dK and dV sum over
    // the group in TMEM.  Order: slices in groups of p.slice_group, key tile
    // major within a group (under a causal mask the first key tiles see the
    // most query tiles, so the heaviest units of a group start first).  For
    // large problems the groups hold four slices: the CTAs resident at
    // any time then share a few slices, whose fp32 dQ accumulator, Q and dO
    // stay in L2 instead of every head's at once, and the heaviest unit of
    // the last group starts early enough not to run alone at the end, as the
    // last slice's first key tile would in plain slice-major order.  When the
    // whole problem fits in L2 anyway, one group holds every slice, which
    // starts the heaviest units of all slices first.
    //
    // Packed inputs with a sequence table (p.seq_table) use a compact grid:
    // the units are the sequences' own key tiles, sequences longest first
    // (most query tiles) and, within a sequence, its key/value heads in groups
    // of p.slice_group with the key tiles major within a group, so no CTA
    // lands past its sequence's last key tile, the resident CTAs share a few
    // heads' Q, dO and dQ accumulator in L2, and the last units to start are
    // the shortest sequence's.
    int slice, kt;
    int Lq, Lkv, tok_q0 = 0, tok_kv0 = 0;
    if constexpr (kPacked) {
        if (p.seq_table) {
            // The table: sequences ordered by query tiles, most first (ties in
            // sequence order); first unit of each = exclusive prefix sum of
            // key tiles x key/value heads in that order.  Lists of up to 32
            // sequences are tabulated by warp 0 in registers (lane = sequence);
            // longer ones in the dS tile's shared memory (unused until the
            // compute warps' first dS), sorted only up to 256 sequences.
            static_assert(4 * (4 * kBwdSeqTableMax + 7) <= 2 * L::kChunkBytes,
                          "the sequence table must fit in the dS tile");
            const int ns = p.num_seqs;
            const int u = blockIdx.x;
            int *pick = reinterpret_cast<int *>(smem + L::kDS);  // [n, first unit, total units]
            if (ns <= 32) {
                if (threadIdx.x < 32) {
                    const int ln = threadIdx.x;
                    int tq = -1, tk = 0;
                    if (ln < ns) {
                        tq = (p.cu_q[ln + 1] - p.cu_q[ln] + kTileM - 1) / kTileM;
                        tk = (p.cu_kv[ln + 1] - p.cu_kv[ln] + kTileN - 1) / kTileN;
                    }
                    const int units = tk * p.h_kv;
                    int first = 0, total = 0;
                    for (int m = 0; m < ns; ++m) {
                        const int tm = __shfl_sync(0xffffffffu, tq, m);
                        const int um = __shfl_sync(0xffffffffu, units, m);
                        // m comes before this lane's sequence in the table
                        if (tm > tq || (tm == tq && m < ln)) first += um;
                        total += um;
                    }
                    const bool mine = ln < ns && u >= first && u < first + units;
                    const unsigned who = __ballot_sync(0xffffffffu, mine);
                    if (mine) {
                        pick[0] = ln;
                        pick[1] = first;
                    }
                    if (ln == 0) pick[2] = total;
                    if (who == 0 && ln == 0) pick[0] = -1;
                }
            } else {
                int *cq = pick + 4;
                int *ckv = cq + (ns + 1);
                int *order = ckv + (ns + 1);
                int *first = order + ns;  // ns + 1 entries
                for (int i = threadIdx.x; i <= ns; i += blockDim.x) {
                    cq[i] = p.cu_q[i];
                    ckv[i] = p.cu_kv[i];
                }
                __syncthreads();
                auto q_tiles_of = [&](int n) { return (cq[n + 1] - cq[n] + kTileM - 1) / kTileM; };
                for (int n = threadIdx.x; n < ns; n += blockDim.x) {
                    int rank = n;  // long lists keep their own order
                    if (ns <= 256) {
                        const int tn = q_tiles_of(n);
                        rank = 0;
                        for (int m = 0; m < ns; ++m) {
                            const int tm = q_tiles_of(m);
                            rank += (tm > tn || (tm == tn && m < n)) ? 1 : 0;
                        }
                    }
                    order[rank] = n;
                }
                __syncthreads();
                if (threadIdx.x == 0) {
                    int run = 0;
                    for (int i = 0; i < ns; ++i) {
                        first[i] = run;
                        const int n = order[i];
                        run += (ckv[n + 1] - ckv[n] + kTileN - 1) / kTileN * p.h_kv;
                    }
                    first[ns] = run;
                    pick[2] = run;
                    pick[0] = -1;
                    if (u < run) {
                        int lo = 0, hi = ns;  // first[lo] <= u < first[hi]
                        while (hi - lo > 1) {
                            const int mid = (lo + hi) >> 1;
                            if (first[mid] <= u) lo = mid;
                            else hi = mid;
                        }
                        pick[0] = order[lo];
                        pick[1] = first[lo];
                    }
                }
            }
            __syncthreads();
            const int n = pick[0], first_u = pick[1];
            __syncthreads();  // every thread has read the pick before the region is reused
            if (n < 0) {  // the host sizes the grid by an upper bound
                griddep_wait();  // see the early exits below
                return;
            }
            tok_q0 = p.cu_q[n];
            tok_kv0 = p.cu_kv[n];
            Lq = p.cu_q[n + 1] - tok_q0;
            Lkv = p.cu_kv[n + 1] - tok_kv0;
            // within the sequence: its key/value heads in groups of
            // p.slice_group, key tile major within a group (as the dense order)
            const int local = u - first_u;
            const int n_kt = (Lkv + kTileN - 1) / kTileN;
            const int per_group = p.slice_group * n_kt;
            const int group_i = local / per_group;
            const int in_group = local - group_i * per_group;
            const int group_n = min(p.slice_group, p.h_kv - group_i * p.slice_group);
            kt = in_group / group_n;
            slice = n * p.h_kv + group_i * p.slice_group + in_group % group_n;
        }
    }
    if (!kPacked || !p.seq_table) {
        const int per_group = p.slice_group * p.kv_tiles;
        const int group_i = blockIdx.x / per_group;
        const int in_group = blockIdx.x - group_i * per_group;
        const int group_n = min(p.slice_group, p.kv_slices - group_i * p.slice_group);
        slice = group_i * p.slice_group + in_group % group_n;  // key/value slice
        kt = in_group / group_n;
        if constexpr (kPacked) {
            const int n = slice / p.h_kv;
            tok_q0 = p.cu_q[n];
            tok_kv0 = p.cu_kv[n];
            Lq = p.cu_q[n + 1] - tok_q0;
            Lkv = p.cu_kv[n + 1] - tok_kv0;
        } else {
            Lq = p.s_q;
            Lkv = p.s_kv;
        }
    }
    const int hk = slice % p.h_kv;              // key/value head
    int q_slice0;                               // dense: query slice of the group's first head
    RowMap km;
    if constexpr (!kPacked) {
        q_slice0 = (slice / p.h_kv) * p.h + hk * p.group;
        km = {(int64_t)slice * p.s_kv * D, D, 0};
    } else {
        q_slice0 = 0;
        km = {((int64_t)tok_kv0 * p.h_kv + hk) * D, (int64_t)p.h_kv * D, 0};
    }
    const int k0 = kt * kTileN;
    // Every early exit waits for the preprocess grid first: the kernel behind
    // this one (the deterministic dQ pass, which reads the row terms without a
    // wait of its own) may start once every CTA has signalled or exited, so no
    // CTA may exit before the row terms are complete.
    if (k0 >= Lkv) {  // packed: this sequence has fewer key tiles
        griddep_wait();
        return;
    }
    // Query rows that see at least one key of [k0, k_last]: a causal mask
    // needs i + delta >= k0, a window i + delta - window <= k_last.
    const int delta = mask_delta(p.mask, Lq, Lkv);
    const int k_last = min(k0 + kTileN, Lkv) - 1;
    const int row_lo = p.mask != kMaskNone ? max(0, k0 - delta) : 0;
    const int row_hi = p.window >= 0 ? min(Lq, k_last - delta + p.window + 1) : Lq;
    const int qt_begin = row_lo / kTileM;
    const int n_q = row_hi > row_lo ? (row_hi + kTileM - 1) / kTileM - qt_begin : 0;
    const int n_it = n_q * p.group;  // (query head, query tile) pairs, head-major
    // Iteration i: query head hk * group + i / n_q, query tile qt_begin + i % n_q;
    // the dQ accumulator row of that head's query row r is acc_base(i) + r.
    auto q_head = [&](int i) { return hk * p.group + i / n_q; };
    auto q_tile_row0 = [&](int i) { return (qt_begin + i % n_q) * kTileM; };
    auto acc_base = [&](int i) -> int {
        return kPacked ? q_head(i) * p.total_q + tok_q0 : (q_slice0 + i / n_q) * p.s_q;
    };

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    if (n_q == 0) {
        // No query sees these keys: dK = dV = 0.
        if (threadIdx.x < kTileN) {
            const int j = k0 + threadIdx.x;
            if (j < Lkv) {
                uint4 *a = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.dk) + km.io0 + j * km.io_rs);
                uint4 *b = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.dv) + km.io0 + j * km.io_rs);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) a[i] = b[i] = make_uint4(0, 0, 0, 0);
            }
        }
        griddep_wait();
        return;
    }

    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    if ((sbase & 1023u) != 0) {
        // The swizzled operand tiles need a 1024-byte aligned base.
        if (threadIdx.x == 0) atomicCAS(p.err, 0u, (kTagBwdMain << 16) | 0xfffu);
        griddep_wait();
        return;
    }
    auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };

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
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kMisc, L::kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x >= 128 && threadIdx.x < 256) {
        // The constant A operands of the row-term K-steps, one 16-byte row
        // per key (unswizzled core matrices, rows 16 bytes apart).
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
        const int ky = kPacked ? hk : k0;
        const int kz = kPacked ? tok_kv0 + k0 : slice;
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
            tma_prefetch_desc(&tm_rx);
            mbar_arrive_expect_tx(bar(L::bKVFull), 2 * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
                tma_load_3d(sbase + L::kK + c * L::kChunkBytes, &tm_k, bar(L::bKVFull), c * 64, ky, kz);
                tma_load_3d(sbase + L::kV + c * L::kChunkBytes, &tm_v, bar(L::bKVFull), c * 64, ky, kz);
            }
        }
        // The row terms come from the preprocess grid; once it is done, the
        // kernel behind this one (dQ convert, or the deterministic dQ pass,
        // which needs only the row terms) may start filling freed SMs.
        griddep_wait();
        if (lane == 0) griddep_launch_dependents();
        int issued = 0, issued_do = 0;
        for (int i = 0; i < n_it; ++i) {
            const int st = i & 1, use = i >> 1;
            const int dst = i % L::kDOStages, duse = i / L::kDOStages;
            const int q0 = q_tile_row0(i);
            const int qy = kPacked ? q_head(i) : q0;
            const int qz = kPacked ? tok_q0 + q0 : q_slice0 + i / n_q;
            // Q_i (freed by dK_{i-2}) is needed first, by S^T_i; dO_i (freed by
            // dV_{i-kDOStages}) only by dP^T_i.
            if (use > 0 && !warp_wait_b(bar(L::bQEmpty + st), (use - 1) & 1, wc, 18)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(L::bQFull + st), L::kTileBytes + L::kRowXBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kQ + st * L::kTileBytes + c * L::kChunkBytes, &tm_q,
                                bar(L::bQFull + st), c * 64, qy, qz);
                tma_load_3d(sbase + L::kRowX + st * L::kRowXBytes, &tm_rx, bar(L::bQFull + st), 0,
                            qy, qz);
            }
            issued = i + 1;
            if (duse > 0 && !warp_wait_b(bar(L::bDOEmpty + dst), (duse - 1) & 1, wc, 1)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(L::bDOFull + dst), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sbase + L::kDO + dst * L::kTileBytes + c * L::kChunkBytes, &tm_do,
                                bar(L::bDOFull + dst), c * 64, qy, qz);
            }
            issued_do = i + 1;
        }
        if (lane == 0) {
            mbar_wait_drain(bar(L::bKVFull), 0);
            for (int i = max(0, issued - 2); i < issued; ++i)
                mbar_wait_drain(bar(L::bQFull + (i & 1)), (i >> 1) & 1);
            for (int i = max(0, issued_do - L::kDOStages); i < issued_do; ++i)
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
            // Operand descriptors, built once: a descriptor's low 14 bits are
            // the address / 16, so a tile offset is added to it directly
            // (every address stays below 256 KiB).  K-major views step 32
            // bytes per K-step within a 128-byte row and a 16 KiB chunk per
            // 64 elements; MN-major views step 16 rows (2 KiB) per K-step.
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
            // Row terms: A rows (0.5, 0.5, 0, 0) or (0, 0, 0.5, 0.5), B rows
            // (hi_l, lo_l, hi_d, lo_d) of query stage st; both operands name
            // their first 16-byte core matrix twice (K-direction offset 0), so
            // the K = 8 sum is 2 * 0.5 * (hi + lo).
            const uint64_t dAS = smem_desc_plain(sbase + L::kAexS, 0, 128);
            const uint64_t dAD = smem_desc_plain(sbase + L::kAexD, 0, 128);
            const uint64_t dRX = smem_desc_plain(sbase + L::kRowX, 0, 128);
            constexpr uint32_t kRowX16 = L::kRowXBytes >> 4;
            // X'^T = A B^T over the head dim (both K-major) + row term, 128 x 128
            auto issue_kmajor = [&](uint64_t a, uint64_t b, uint64_t a_ex, int st, uint32_t col) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss(tmem + col, a + kstep(k), b + kstep(k), id_sq, k > 0);
                mma_ss_tf32(tmem + col, a_ex, dRX + st * kRowX16, id_rx, 1u);
            };
            bool ok = mbar_wait_lean(bar(L::bKVFull), 0, wc, 2) && mbar_wait_lean(bar(L::bQFull), 0, wc, 3);
            if (ok) {
                tc_fence_after();
                issue_kmajor(dK_k, dQ_k, dAS, 0, L::kColS);  // S'^T_0
                mma_commit(bar(L::bSFull));
                ok = mbar_wait_lean(bar(L::bDOFull), 0, wc, 4);
            }
            if (ok) {
                tc_fence_after();
                issue_kmajor(dV_k, dDO_k, dAD, 0, L::kColDP);  // dP'^T_0
                mma_commit(bar(L::bDPFull));
            }
            for (int i = 0; ok && i < n_it; ++i) {
                const int st = i & 1;
                const int dst = L::kDOStages == 1 ? 0 : (i & 1);
                // dV += P^T dO.  P^T is packed two per column into the first 32
                // columns of each compute group's 64 S^T columns.
                ok = mbar_wait_lean(bar(L::bPReady), i & 1, wc, 5);
                if (!ok) break;
                tc_fence_after();
                {
                    const uint64_t b = dDO_mn + dst * kTile16;
#pragma unroll
                    for (int k = 0; k < 128 / 16; ++k)
                        mma_ts(tmem + L::kColDV, tmem + L::kColS + (k >> 2) * 64 + (k & 3) * 8,
                               b + k * 128, id_mn, (i > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(L::bDOEmpty + dst));  // also: dV_i has read P^T_i
                // S'^T_{i+1}, once the dV product has finished reading P^T_i
                if (i + 1 < n_it) {
                    const int st1 = (i + 1) & 1, use1 = (i + 1) >> 1;
                    ok = mbar_wait_lean(bar(L::bQFull + st1), use1 & 1, wc, 6) &&
                         mbar_wait_lean(bar(L::bDOEmpty + dst), (i / L::kDOStages) & 1, wc, 7);
                    if (!ok) break;
                    tc_fence_after();
                    issue_kmajor(dK_k, dQ_k + st1 * kTile16, dAS, st1, L::kColS);
                    mma_commit(bar(L::bSFull));
                }
                // dQ_i = dS' K (unless the deterministic dQ pass computes dQ),
                // then dK += dS'^T Q (last reader of Q_i)
                const bool do_dq = !p.deterministic;
                ok = mbar_wait_lean(bar(L::bDSReady), i & 1, wc, 8);
                if (ok && do_dq && !L::kDQAliasDP && i > 0)
                    ok = mbar_wait_lean(bar(L::bDQFree), (i - 1) & 1, wc, 9);
                if (!ok) break;
                tc_fence_after();
                if (do_dq) {
#pragma unroll
                    for (int k = 0; k < 128 / 16; ++k)
                        mma_ss(tmem + L::kColDQ, dDS_mn + k * 128, dK_mn + k * 128, id_dq, k > 0);
                    mma_commit(bar(L::bDQFull));
                }
                {
                    const uint64_t b = dQ_mn + st * kTile16;
#pragma unroll
                    for (int k = 0; k < 128 / 16; ++k)
                        mma_ss(tmem + L::kColDK, dDS_k + kstep(k), b + k * 128, id_mn,
                               (i > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(L::bQEmpty + st));  // also: dK and dQ have read dS'_i
                // dP'^T_{i+1}
                if (i + 1 < n_it) {
                    const int dst1 = L::kDOStages == 1 ? 0 : ((i + 1) & 1);
                    const int duse1 = (i + 1) / L::kDOStages;
                    ok = mbar_wait_lean(bar(L::bDOFull + dst1), duse1 & 1, wc, 10);
                    if (ok && do_dq && L::kDQAliasDP) ok = mbar_wait_lean(bar(L::bDQFree), i & 1, wc, 11);
                    if (!ok) break;
                    tc_fence_after();
                    issue_kmajor(dV_k, dDO_k + dst1 * kTile16, dAD, (i + 1) & 1, L::kColDP);
                    mma_commit(bar(L::bDPFull));
                }
            }
            mma_commit(bar(L::bMmaIdle));
            mbar_wait_drain(bar(L::bMmaIdle), 0);
        }
        __syncwarp();
    } else if (warp < 10) {
        // ============================================================ compute
        // Group g (warps 2-5 or 6-9) owns queries [64g, 64g+64) of every
        // tile for all 128 key rows: its S^T and dP^T columns are
        // [64g, 64g+64) of those regions, P^T goes back packed into the first
        // 32 of its S^T columns, and dS^T into the g-th 128-byte chunk.
        const int grp = (int)(warp - 2) >> 2;
        const int quad = warp & 3;
        const int j = quad * 32 + lane;  // key row of the tile == TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t col_s = t_lane + L::kColS + grp * 64;
        const uint32_t col_dp = t_lane + L::kColDP + grp * 64;
        const int key = k0 + j;
        const bool key_ok = key < Lkv;
        const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
        uint8_t *ds_row = smem + L::kDS + grp * L::kChunkBytes + j * 128;
        bool ok = true;
        for (int i = 0; i < n_it; ++i) {
            const int q0 = q_tile_row0(i) + grp * 64;  // query of local column 0
            ok = warp_wait_b(bar(L::bSFull), i & 1, wc, 12);
            if (!ok) break;
            tc_fence_after();
            uint32_t s[64];
            tmem_ld32(col_s, s);
            tmem_ld32(col_s + 32, s + 32);
            tmem_ld_wait_regs<64>(s);
            // Local column c (query q0 + c) is visible iff lo <= c < hi: key <
            // Lkv, query < Lq (rows past it carry no row terms), under a causal
            // mask query + delta >= key, under a window query + delta -
            // window <= key.
            int lo = p.mask != kMaskNone ? key - delta - q0 : 0;
            int hi = Lq - q0;
            if (p.window >= 0) hi = min(hi, key - delta + p.window + 1 - q0);
            if (!key_ok) lo = 64;
            uint32_t pk[32];  // P^T, packed pairs: feeds the dV product (via TMEM) and dS
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

            // dS'^T = P^T o dP'^T  ->  shared memory (SW128)
            ok = warp_wait_b(bar(L::bDPFull), i & 1, wc, 14);
            if (ok && i > 0) ok = warp_wait_b(bar(L::bQEmpty + ((i - 1) & 1)), ((i - 1) >> 1) & 1, wc, 15);
            if (!ok) break;
            tc_fence_after();
            uint32_t dp[64];
            tmem_ld32(col_dp, dp);
            tmem_ld32(col_dp + 32, dp + 32);
            tmem_ld_wait_regs<64>(dp);
#pragma unroll
            for (int u = 0; u < 8; ++u) {  // 16-byte unit u of the row: queries 8u .. 8u+7
                uint32_t w[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int e = u * 8 + v * 2;
                    const float2 pp = unpack2<kBf16>(pk[e / 2]);
                    float g0, g1;
                    f2_unpack(f2_mul(f2_pack(pp.x, pp.y),
                                     f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1]))),
                              g0, g1);
                    w[v] = pack2<kBf16>(g0, g1);
                }
                *reinterpret_cast<uint4 *>(ds_row + ((u ^ (j & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(L::bDSReady));
        }
        // dK, dV epilogue: group 0 writes dV, group 1 dK, each warp its 32
        // key rows, staged in its rows of the dS tile (every product is done)
        if (ok) ok = warp_wait_b(bar(L::bMmaIdle), 0, wc, 16);
        if (ok) {
            tc_fence_after();
            const uint32_t col = grp == 0 ? L::kColDV : L::kColDK;
            const int key0 = k0 + quad * 32;  // the warp's first key
            uint16_t *row0 = static_cast<uint16_t *>(grp == 0 ? p.dv : p.dk) + km.io0 + (int64_t)key0 * km.io_rs;
            const float f = grp == 0 ? 1.f : p.scale;  // dK = scale * sum dS'^T Q
            store_tile_rows<D, kBf16>(t_lane + col, ds_row - lane * 128, lane, row0, km.io_rs,
                                      min(32, Lkv - key0), f, [] {});
        }
    } else {
        // ============================================================ dQ epilogue
        // Each warp owns 32 query rows (its TMEM lane quadrant).  dQ_i goes
        // out in 32 x 16 fp32 boxes, staged in shared memory with the 64-byte
        // swizzle and added into the fp32 accumulator by TMA reduce-add
        // through tm_dq, kDQSlots boxes in flight per warp.  At d = 128 the
        // first 96 columns are read from TMEM at once, the first two boxes go
        // out, the last 32 columns take their registers and the columns are
        // freed before the remaining six boxes are staged.  Rows past the
        // sequence carry exact zeros (their P is 0); rows past the
        // accumulator are dropped by the map.
        const int quad = warp & 3;
        const uint32_t t_dq = tmem + ((uint32_t)(quad * 32) << 16) + L::kColDQ;
        const uint32_t stage = sbase + L::kDQStage + quad * (L::kDQSlots * L::kDQBoxBytes);
        uint8_t *stage_ptr = smem + L::kDQStage + quad * (L::kDQSlots * L::kDQBoxBytes) + lane * 64;
        int boxes = 0, slot = 0;  // boxes sent by this warp; slot of the next one
        griddep_wait();  // the preprocess grid has zeroed the accumulator
        // one 32 x 16 box: registers r[0..16) -> staging slot -> reduce-add
        // into accumulator rows [arow, arow + 32), columns [col, col + 16)
        auto send = [&](const uint32_t *r, int col, int arow) {
            if (boxes >= L::kDQSlots) {
                if (lane == 0) bulk_wait_read<L::kDQSlots - 1>();  // the slot's last box was read
                __syncwarp();
            }
            uint8_t *row = stage_ptr + slot * L::kDQBoxBytes;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4 *>(row + ((u ^ ((lane >> 1) & 3)) << 4)) =
                    make_uint4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_reduce_add_2d(&tm_dq, stage + slot * L::kDQBoxBytes, col, arow);
                bulk_commit();
            }
            ++boxes;
            slot = slot + 1 == L::kDQSlots ? 0 : slot + 1;
        };
        for (int i = 0; i < (p.deterministic ? 0 : n_it); ++i) {
            if (!warp_wait_b(bar(L::bDQFull), i & 1, wc, 17)) break;
            tc_fence_after();
            const int qrow0 = q_tile_row0(i) + quad * 32;
            const int arow = acc_base(i) + qrow0;
            const bool live = qrow0 < Lq;  // any live row in this warp's quarter
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

template <int D, bool kBf16, bool kPacked>
cudaError_t launch_bwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const CUtensorMap &tdo, const CUtensorMap &tdq, const CUtensorMap &trx,
                         const BwdParams &p, cudaStream_t stream, const KernelTimer &timer) {
    using L = BwdLayout<D>;
    const int64_t rows = kPacked ? (int64_t)p.total_q * p.h : (int64_t)p.bh * p.s_q;
    const int64_t acc_elems = rows * D;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int small_grid = sms * 8;
    bwd_preprocess_kernel<D, kBf16, kPacked><<<small_grid, 256, 0, stream>>>(
        p, rows, p.deterministic ? 0 : acc_elems);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kern = bwd_main_kernel<D, kBf16, kPacked>;
    if (!p.persist) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
    }
    const int grid = p.grid;  // 0 when no sequence has a key: dK, dV are empty then
    if (timer.start) cudaEventRecord(timer.start, stream);
    if (grid > 0 && p.persist)
        e = launch_bwd_persist(tq, tk, tv, tdo, tdq, trx, p, D, kBf16, kPacked, stream);
    else if (grid > 0)
        e = launch_overlapped(kern, dim3(grid), dim3(kBwdThreads), L::kBytes, stream, tq, tk, tv, tdo,
                              tdq, trx, p);
    if (p.deterministic) {
        // the timed span covers the main kernel and the dQ pass
        // it overlaps the main kernel's last wave; with no main kernel it
        // follows the preprocess kernel in plain stream order
        if (e == cudaSuccess)
            e = launch_bwd_dq(tq, tk, tv, tdo, p, p.q_tiles, D, kBf16, kPacked, grid > 0, stream);
        if (timer.stop) cudaEventRecord(timer.stop, stream);
        return e;
    }
    if (timer.stop) cudaEventRecord(timer.stop, stream);
    if (e != cudaSuccess) return e;
    return launch_overlapped(bwd_dq_convert_kernel<D, kBf16, kPacked>, dim3(small_grid), dim3(256), 0,
                             stream, p, rows);
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const CUtensorMap &tdq, const CUtensorMap &trx,
                       const BwdParams &p, int d, bool bf16, bool packed, cudaStream_t stream,
                       const KernelTimer &timer) {
#define SDPA_BWD_CASE(D_, BF_, PK_)                                            \
    if (d == D_ && bf16 == BF_ && packed == PK_)                               \
        return launch_bwd_t<D_, BF_, PK_>(tq, tk, tv, tdo, tdq, trx, p, stream, timer);
    SDPA_BWD_CASE(64, true, false)
    SDPA_BWD_CASE(64, true, true)
    SDPA_BWD_CASE(64, false, false)
    SDPA_BWD_CASE(64, false, true)
    SDPA_BWD_CASE(128, true, false)
    SDPA_BWD_CASE(128, true, true)
    SDPA_BWD_CASE(128, false, false)
    SDPA_BWD_CASE(128, false, true)
#undef SDPA_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace sdpa
