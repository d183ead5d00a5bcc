// Shared-memory, TMEM and barrier layout of the backward main kernels
// (bwd.cu: one CTA per key tile; bwd_persist.cu: persistent CTAs walking
// many key tiles) and their small helpers.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {

SDPA_DEV bool warp_wait_b(uint32_t bar, uint32_t parity, const WaitCtx &w, uint32_t site) {
    bool ok = mbar_wait_lean(bar, parity, w, site);
    return __all_sync(0xffffffffu, ok);
}

// -------------------------------------------------------------------- layouts
// Row r of a problem slice in the I/O tensors and in the fp32 buffers:
//   dense  : I/O element offset (slice*S + r)*d, row-term index slice*S + r
//   packed : I/O element offset ((tok0 + r)*h + head)*d, row terms (tok0 + r)*h + head
// The dQ accumulator is head-major in both cases: [slices or heads][rows][d],
// so a query tile of one head is contiguous.
struct RowMap {
    int64_t io0, io_rs;      // I/O tensors (elements)
    int64_t acc0;            // dQ accumulator row 0 (elements, row stride d)
};

template <int D>
struct BwdLayout {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = 128 * 128;          // 128 rows x 128 bytes
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kK = 0;
    static constexpr int kV = kK + kTileBytes;
    // dO is read by dP^T_i and dV_i only, and dO_{i+1} is not needed before
    // dP^T_{i+1}, so one buffer suffices at d = 128 and frees room for the
    // dQ staging boxes.
    static constexpr int kDOStages = (D == 128) ? 1 : 2;
    static constexpr int kQ = kV + kTileBytes;               // 2 stages
    static constexpr int kDO = kQ + 2 * kTileBytes;          // kDOStages stages
    static constexpr int kDS = kDO + kDOStages * kTileBytes; // 128 keys x 128 queries bf16
    static constexpr int kDQBoxBytes = 32 * 16 * 4;           // 32 rows x 16 fp32
    static constexpr int kDQSlots = 3;                        // staging boxes per warp
    static constexpr int kDQStage = kDS + 2 * kChunkBytes;   // 4 warps x kDQSlots boxes
    static constexpr int kRowXBytes = 128 * 16;               // 128 query rows x 4 fp32
    static constexpr int kRowX = kDQStage + 4 * kDQSlots * kDQBoxBytes;  // 2 stages, with Q
    static constexpr int kAexS = kRowX + 2 * kRowXBytes;      // 128 rows (0.5, 0.5, 0, 0)
    static constexpr int kAexD = kAexS + kRowXBytes;          // 128 rows (0, 0, 0.5, 0.5)
    static constexpr int kBar = kAexD + kRowXBytes;
    // barriers
    static constexpr int bKVFull = 0;
    static constexpr int bQFull = 1;       // 2: Q and its row terms
    static constexpr int bDOFull = 3;      // 2
    static constexpr int bQEmpty = 7;      // 2: Q (and row terms) stage, freed after dK;
                                           // it also tells the compute warps that dS' is read
    static constexpr int bDOEmpty = 18;    // kDOStages: dO stage, freed after dV; it also
                                           // tells the MMA thread that P^T is read
    static constexpr int bSFull = 9;
    static constexpr int bDPFull = 10;
    static constexpr int bPReady = 11;
    static constexpr int bDSReady = 12;
    static constexpr int bDQFull = 14;
    static constexpr int bDQFree = 15;
    static constexpr int bMmaIdle = 17;
    static constexpr int kNumBars = 20;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColDV = 0;
    static constexpr uint32_t kColDK = D;
    static constexpr uint32_t kColS = 2 * D;
    static constexpr uint32_t kColDP = 2 * D + 128;
    static constexpr bool kDQAliasDP = (D == 128);  // no spare columns at d = 128
    static constexpr uint32_t kColDQ = kDQAliasDP ? kColDP : 2 * D + 256;
};

// warps: 0 TMA, 1 MMA, 2-5 compute (queries 0-63 of a tile), 6-9 compute
// (queries 64-127), 10-13 dQ epilogue
constexpr int kBwdThreads = 448;

// dV or dK of a key tile, from TMEM to global memory.  The calling warp's 32
// key rows (its TMEM lane quarter; this thread: row `lane`) hold fp32 sums in
// columns [0, D) from t_col.  Each 64-column half is scaled by f, converted,
// staged in the warp's own 32 rows (128 bytes each) of `stage`, and stored 4
// rows x 128 bytes per instruction: whole lines, where storing straight from
// the registers would write one 16-byte piece of each of 32 rows per
// instruction.  Staged rows keep the dS tile's 16-byte swizzle (unit u of row
// r at u ^ (r & 7)), so both the staging and the read-back run at the
// shared-memory minimum of 4 wavefronts per 512 bytes.  last_read() runs right
// after the final TMEM read; rows at or past n_valid are not written; row0 is
// row 0 of the warp's rows, row_stride in elements.
template <int D, bool kBf16, class LastRead>
SDPA_DEV void store_tile_rows(uint32_t t_col, uint8_t *stage, uint32_t lane, uint16_t *row0, int64_t row_stride,
                              int n_valid, float f, LastRead &&last_read) {
#pragma unroll 1
    for (int h = 0; h < D / 64; ++h) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t r[32];
            tmem_ld32(t_col + h * 64 + q * 32, r);
            tmem_ld_wait_regs<32>(r);
            if (h == D / 64 - 1 && q == 1) last_read();
            auto g = [&](int e) { return __uint_as_float(r[e]) * f; };
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int unit = q * 4 + v;
                *reinterpret_cast<uint4 *>(stage + lane * 128 + ((unit ^ (lane & 7)) << 4)) =
                    make_uint4(pack2<kBf16>(g(8 * v), g(8 * v + 1)), pack2<kBf16>(g(8 * v + 2), g(8 * v + 3)),
                               pack2<kBf16>(g(8 * v + 4), g(8 * v + 5)), pack2<kBf16>(g(8 * v + 6), g(8 * v + 7)));
            }
        }
        __syncwarp();
        const int c = lane & 7;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int r = 4 * t + (int)(lane >> 3);
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + r * 128 + ((c ^ (r & 7)) << 4));
            if (r < n_valid) *reinterpret_cast<uint4 *>(row0 + r * row_stride + h * 64 + c * 8) = v;
        }
        __syncwarp();
    }
}

}  // namespace sdpa
