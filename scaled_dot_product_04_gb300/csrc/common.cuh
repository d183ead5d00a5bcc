// Shared definitions of the attention kernels and their host launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sdpa {

constexpr int kTileM = 128;  // query rows per tile (MMA M, TMEM lanes)
constexpr int kTileN = 128;  // keys per tile

// Kernel tags written into the high half of the device error word.
enum KernelTag : uint32_t {
    kTagFwd = 1,
    kTagBwdPre = 2,
    kTagBwdMain = 3,
    kTagBwdConvert = 4,
    kTagBwdDq = 5,
    kTagSelftest = 6,
};

// Where a tile lives: dense tensors are [b*h, s, d] (row stride d), packed
// tensors are [T, h, d] (row stride h*d).  The TMA maps use the same two
// shapes, so a tile of 128 rows is addressed by (y, z) = (row0, bh) when
// dense and (h, tok0) when packed.
// Masks (cudnn-frontend PR #554 `sdpa` op: is_causal, causal_bottom_right,
// window_left).  In a sequence of Lq queries and Lkv keys, query i sees keys
// j with lo_i <= j < hi_i, where delta = Lkv - Lq for kMaskBottomRight and 0
// otherwise, hi_i = min(Lkv, i + delta + 1) under a causal mask (Lkv without
// one) and lo_i = max(0, i + delta - window) for window >= 0 (0 without).
enum MaskKind : int { kMaskNone = 0, kMaskTopLeft = 1, kMaskBottomRight = 2 };

// Element kinds of inputs and outputs (the values of the ABI's sdpa_dtype).
enum ElemKind : int { kElBf16 = 0, kElFp16 = 1, kElE4m3 = 2 };

struct FwdParams {
    void *o;                     // output [.. , d] in the I/O dtype
    float *lse;                  // may be null
    const int32_t *cu_q;         // packed only
    const int32_t *cu_kv;        // packed only
    uint32_t *err;               // device error word
    int bh;                      // query slices: dense b*h, packed num_seqs*h
    int h;                       // query heads
    int h_kv;                    // key/value heads (h is a multiple)
    int group;                   // h / h_kv: query head hq reads key/value head hq / group
    int s_q, s_kv;               // dense lengths (packed two-tile launches that take their
                                 // units dynamically carry their counter slot + 1 in s_q)
    int num_seqs;                // packed
    int q_tiles;                 // row blocks per slice (128 rows, or 256 for the
                                 // two-tile kernel): dense from s_q, packed from max_seqlen_q
    int n_units;                 // units a persistent CTA may visit: q_tiles * bh (dense two-tile
                                 // lists with a cut tail: plus the number of cut 256-row units)
    int mask;                    // MaskKind
    int window;                  // window_left, -1 for none
    float scale_log2;            // attn_scale * log2(e)
    // E4M3 inputs only: per-tensor factors in device memory (fp32 scalars)
    const float *descale_q, *descale_k, *descale_v;
    const float *scale_o;        // E4M3 output: O is stored as O * scale_o
    float *amax_o;               // may be null: receives max |O| (atomic max)
};

// Key range [lo, hi) of query row i (see MaskKind), for the row order of one
// sequence; lo may come out negative and hi above Lkv only where the callers
// clamp them.
struct KeyRange {
    int lo, hi;
};
__host__ __device__ inline int mask_delta(int mask, int Lq, int Lkv) {
    return mask == kMaskBottomRight ? Lkv - Lq : 0;
}
__host__ __device__ inline KeyRange key_range(int mask, int window, int i, int delta, int Lkv) {
    KeyRange r;
    r.hi = mask != kMaskNone ? (i + delta + 1 < Lkv ? i + delta + 1 : Lkv) : Lkv;
    r.lo = window >= 0 ? i + delta - window : -(1 << 30);
    return r;
}

struct BwdParams {
    const void *o, *dout;        // [.., d] I/O dtype
    const float *lse;            // [b,h,s_q] or [T,h]
    void *dq, *dk, *dv;          // outputs, I/O dtype
    float *dq_acc;               // fp32 [rows, h?, d] accumulator (Q layout, fp32)
    float4 *rowx;                // per query row, same layout as lse: the row terms
                                 // -LSE/scale and -D, each split into a tf32 pair (hi, lo)
    const int32_t *cu_q, *cu_kv;
    uint32_t *err;
    int bh;                      // query slices: dense b*h, packed num_seqs*h
    int h, h_kv, group;          // query heads, key/value heads, h / h_kv
    int kv_slices;               // key/value slices: dense b*h_kv, packed num_seqs*h_kv
    int s_q, s_kv;
    int num_seqs;
    int kv_tiles;                // dense: ceil(s_kv/128); packed: ceil(max_seqlen_kv/128)
    int total_q;                 // packed: number of query tokens; dense: b*h*s_q rows
    int mask;                    // MaskKind
    int window;                  // window_left, -1 for none
    float scale;                 // attn_scale
    float scale_log2;            // attn_scale * log2(e)
    int deterministic;           // 1: the main kernel skips dQ (bwd_dq.cu computes it)
    int q_tiles;                 // query tiles per slice: dense ceil(s_q/128), packed
                                 // ceil(max_seqlen_q/128) (the dQ pass's grid)
    int slice_group;             // key/value slices interleaved in the main kernel's CTA order
    int seq_table;               // packed: 1 = compact grid over a per-CTA table of the
                                 // sequences (longest first), 0 = envelope grid
    int grid;                    // main kernel CTAs
    int persist;                 // 1: persistent main kernel (bwd_persist.cu), units taken
                                 // from *unit_ctr, which the preprocess kernel zeroes
    uint32_t *unit_ctr;
};
// Largest sequence count of the packed backward's per-CTA sequence table (it
// is built in the dS tile's shared memory before that is used).
constexpr int kBwdSeqTableMax = 1024;
// Largest sequence count of the persistent backward's packed unit table (in
// shared memory beside the kernel's operand tiles).
constexpr int kPersistSeqMax = 128;

// Failure-detection self-test (selftest.cu): one CTA waits, with the bounded
// wait of every kernel and the given limit, on a barrier phase that nothing
// completes, and so records a timeout in the error word.
cudaError_t launch_wait_selftest(uint32_t *err, uint64_t limit_ns, cudaStream_t stream);

// Host launchers (one translation unit each).
// Optional measurement events recorded on `stream` right before and right
// after the main kernel of a call (both null = none).
struct KernelTimer {
    cudaEvent_t start = nullptr, stop = nullptr;
};

// Launch with programmatic stream serialization (see griddep_wait in
// ptx.cuh): the kernel may start while the previous kernel on `stream`
// finishes, and waits for it only where it reads that kernel's results.
template <class... KArgs, class... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Two-tile forward (fwd_pair.cu): 256 query rows per unit; q_tiles / n_units
// then count 256-row blocks.
int fwd_pair_rows();
// Entries of the two-tile kernel's packed sequence table (num_seqs + 1 must
// fit for its sequence-by-sequence, dynamically taken unit list).
int fwd_pair_table_cap(int d, bool fp8);
// The two-tile kernel's setmaxnreg split hands out exactly fwd_pair_split_regs()
// registers per launched thread.  A build whose launch register count differs
// is not launched: launch_fwd_pair* then return cudaErrorInvalidConfiguration
// and fwd_pair_refused_regs() gives that build's count (0 after any launch
// attempt that was not refused for this reason, on this host thread).
int fwd_pair_split_regs();
int fwd_pair_refused_regs();
cudaError_t launch_fwd_pair(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const FwdParams &p, int d, bool bf16, bool packed, int grid,
                            cudaStream_t stream, const KernelTimer &timer);
// slice_major: order the units slice group by slice group (K and V too large
// for L2), else latest query tile first over all slices.
cudaError_t launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdParams &p, int d, bool bf16, bool packed, int grid,
                       bool slice_major, cudaStream_t stream, const KernelTimer &timer);
// E4M3 inputs, d = 128, output kind `out` (ElemKind): one-tile and two-tile kernels.
cudaError_t launch_fwd_pair_fp8(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                const FwdParams &p, int out, bool packed, int grid,
                                cudaStream_t stream, const KernelTimer &timer);
cudaError_t launch_fwd_fp8(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const FwdParams &p, int out, bool packed, int grid, bool slice_major,
                           cudaStream_t stream, const KernelTimer &timer);
// Deterministic dQ pass (bwd_dq.cu): one CTA per (query slice, query tile);
// q_tiles = query tiles per slice.  Writes p.dq from the row terms in p.rowx.
// overlap: launched to overlap the main kernel just ahead of it on `stream`
// (which must wait for the preprocess kernel before signalling), else in plain
// stream order.
cudaError_t launch_bwd_dq(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tdo, const BwdParams &p, int q_tiles, int d, bool bf16,
                          bool packed, bool overlap, cudaStream_t stream);
// tdq: 2-D fp32 map over the dQ accumulator [rows][d], box 16 x 32, 64-byte swizzle.
// trx: map over the row terms (dense [b*h][s_q][4], packed [T][h][4] fp32), 128-row boxes.
// Persistent main kernel alone (p.grid CTAs, p.unit_ctr zeroed by the kernel
// ahead of it on `stream`, which must signal its dependents).
cudaError_t launch_bwd_persist(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                               const CUtensorMap &tdo, const CUtensorMap &tdq, const CUtensorMap &trx,
                               const BwdParams &p, int d, bool bf16, bool packed, cudaStream_t stream);
cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const CUtensorMap &tdq, const CUtensorMap &trx,
                       const BwdParams &p, int d, bool bf16, bool packed, cudaStream_t stream,
                       const KernelTimer &timer);

}  // namespace sdpa
