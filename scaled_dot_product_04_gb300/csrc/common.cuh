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
};

// Where a tile lives: dense tensors are [b*h, s, d] (row stride d), packed
// tensors are [T, h, d] (row stride h*d).  The TMA maps use the same two
// shapes, so a tile of 128 rows is addressed by (y, z) = (row0, bh) when
// dense and (h, tok0) when packed.
struct FwdParams {
    void *o;                     // output [.. , d] in the I/O dtype
    float *lse;                  // may be null
    const int32_t *cu_q;         // packed only
    const int32_t *cu_kv;        // packed only
    uint32_t *err;               // device error word
    int bh;                      // dense: b*h.  packed: num_seqs*h
    int h;
    int s_q, s_kv;               // dense lengths
    int num_seqs;                // packed
    int q_tiles;                 // row blocks per slice (128 rows, or 256 for the
                                 // two-tile kernel): dense from s_q, packed from max_seqlen_q
    int n_units;                 // q_tiles * bh (units a persistent CTA may visit)
    int causal;
    float scale_log2;            // attn_scale * log2(e)
};

struct BwdParams {
    const void *o, *dout;        // [.., d] I/O dtype
    const float *lse;            // [b,h,s_q] or [T,h]
    void *dq, *dk, *dv;          // outputs, I/O dtype
    float *dq_acc;               // fp32 [rows, h?, d] accumulator (Q layout, fp32)
    float4 *rowx;                // per query row, same layout as lse: the row terms
                                 // -LSE/scale and -D, each split into a tf32 pair (hi, lo)
    const int32_t *cu_q, *cu_kv;
    uint32_t *err;
    int bh, h;
    int s_q, s_kv;
    int num_seqs;
    int kv_tiles;                // dense: ceil(s_kv/128); packed: ceil(max_seqlen_kv/128)
    int total_q;                 // packed: number of query tokens; dense: b*h*s_q rows
    int causal;
    float scale;                 // attn_scale
    float scale_log2;            // attn_scale * log2(e)
};

// Host launchers (one translation unit each).
// Optional measurement events recorded on `stream` right before and right
// after the main kernel of a call (both null = none).
struct KernelTimer {
    cudaEvent_t start = nullptr, stop = nullptr;
};

// Two-tile forward (fwd_pair.cu): 256 query rows per unit; q_tiles / n_units
// then count 256-row blocks.
int fwd_pair_rows();
cudaError_t launch_fwd_pair(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const FwdParams &p, int d, bool bf16, bool packed, int grid,
                            cudaStream_t stream, const KernelTimer &timer);
cudaError_t launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdParams &p, int d, bool bf16, bool packed, int grid,
                       cudaStream_t stream, const KernelTimer &timer);
// tdq: 2-D fp32 map over the dQ accumulator [rows][d], box 16 x 32, 64-byte swizzle.
// trx: map over the row terms (dense [b*h][s_q][4], packed [T][h][4] fp32), 128-row boxes.
cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const CUtensorMap &tdq, const CUtensorMap &trx,
                       const BwdParams &p, int d, bool bf16, bool packed, cudaStream_t stream,
                       const KernelTimer &timer);

}  // namespace sdpa
