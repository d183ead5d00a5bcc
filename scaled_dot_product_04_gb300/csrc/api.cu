// C ABI of the attention library: argument validation, TMA descriptor
// construction and kernel launch.  Nothing here allocates device memory or
// synchronises the host (except sdpa_check_device_error, which exists to do
// exactly that).  Declarations and the contract live in include/sdpa.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "../../include/sdpa.h"

namespace sdpa {
namespace {

// First bounded-wait failure of any kernel launched by this library on the
// device: (kernel tag << 16) | wait site.  Read and cleared by
// sdpa_check_device_error.
__device__ uint32_t g_error_word;
// Unit counters of the persistent backward kernel, one per call in flight: a
// call takes the next slot, its preprocess kernel zeroes it and its main
// kernel's CTAs take units from it.
constexpr int kUnitCounterSlots = 1024;
__device__ uint32_t g_unit_counters[kUnitCounterSlots];
std::atomic<uint32_t> g_unit_counter_next{0};

thread_local std::string t_last_error;
thread_local KernelTimer t_timer;
thread_local int t_fwd_variant = 0;  // 0 auto, 1 one-tile, 2 two-tile
thread_local int t_bwd_variant = 0;  // 0 auto, 1 one CTA per key tile, 2 persistent

// K + V bytes above which the one-tile forward orders its units slice group by
// slice group: with the latest-tile-first order over all slices, the units in
// flight would each stream another slice's K and V from HBM.
constexpr size_t kSliceMajorKVBytes = size_t(64) << 20;

// Forward kernel choice.  The two-tile kernel (256 query rows per unit, two
// softmax warpgroups) wins once units visit a few key tiles: at d = 64 and 128
// from 1024 rows on (dense) and from a mean of 2048 tokens per sequence
// (packed lists whose sequences do not fit its table, which also hold short
// sequences that fill only tile A); short problems do better with the one-tile
// kernel's 128-row units.  Packed lists that fit the two-tile kernel's
// sequence table (pair_table) take its units on demand, and measured so it
// won from a mean of 200 tokens on (d = 128: 3-16 %, d = 64: 1-12 %), so they
// take it at any length.  rows_*: the dense lengths, or the packed totals over
// the sequence count.
bool use_pair_kernel(bool packed, int d, int64_t rows_q, int64_t rows_kv, bool pair_table = false) {
    if (t_fwd_variant == 1) return false;
    if (t_fwd_variant == 2) return true;
    if (packed && pair_table) return d == 64 || d == 128;
    const int64_t min_rows = packed ? 2048 : 1024;
    return (d == 64 || d == 128) && rows_q >= min_rows && rows_kv >= min_rows;
}

int fail(int status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return status;
}

int ok() {
    t_last_error.clear();
    return SDPA_OK;
}

// ----------------------------------------------------------- per-device state
constexpr int kMaxDevices = 64;
struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    uint32_t *err = nullptr;
    uint32_t *unit_counters = nullptr;  // kUnitCounterSlots
};
std::mutex g_dev_mutex;
DeviceState g_dev[kMaxDevices];

int device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(SDPA_ERR_UNSUPPORTED, "device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(SDPA_ERR_UNSUPPORTED,
                        "device %d has compute capability %d.%d; this library is built for sm_103a",
                        dev, major, minor);
        e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "device attributes: %s", cudaGetErrorString(e));
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_error_word);
        if (e != cudaSuccess)
            return fail(SDPA_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
        s.err = static_cast<uint32_t *>(addr);
        e = cudaGetSymbolAddress(&addr, g_unit_counters);
        if (e != cudaSuccess)
            return fail(SDPA_ERR_CUDA, "cudaGetSymbolAddress(unit counters): %s", cudaGetErrorString(e));
        s.unit_counters = static_cast<uint32_t *>(addr);
        s.ready = true;
    }
    *out = &s;
    return SDPA_OK;
}

// ----------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    return SDPA_OK;
}

// Element kind of a tensor map: 0 bf16, 1 fp16, 2 E4M3 (read as bytes).
static CUtensorMapDataType map_type(int el) {
    return el == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                   : el == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
}
static int elem_bytes(int el) { return el == 2 ? 1 : 2; }

// 3-D map over [dim2][dim1][d] with element stride 1 along d.  The box is
// 128 bytes of a row (64 16-bit or 128 8-bit elements: one swizzle span) x
// box1 x box2, 128-byte swizzle.
int encode_map(CUtensorMap *m, const void *ptr, int el, uint64_t d, uint64_t dim1,
               uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1,
               uint32_t box2) {
    cuuint64_t dims[3] = {d, dim1, dim2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes(el)), box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, map_type(el), 3, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return SDPA_OK;
}

// Dense [rows_per_slice, d] slices stacked `slices` deep; tile = 128 rows of one slice.
int dense_map_el(CUtensorMap *m, const void *ptr, int el, int d, int64_t rows, int64_t slices) {
    if (rows == 0 || slices == 0) {
        memset(m, 0, sizeof(*m));
        return SDPA_OK;
    }
    const uint64_t rb = (uint64_t)d * elem_bytes(el);
    return encode_map(m, ptr, el, d, rows, slices, rb, (uint64_t)rows * rb, 128, 1);
}
int dense_map(CUtensorMap *m, const void *ptr, bool bf16, int d, int64_t rows, int64_t slices) {
    return dense_map_el(m, ptr, bf16 ? 0 : 1, d, rows, slices);
}

// Packed [tokens, h, d]; tile = 128 tokens of one head.  The token extent is
// the packed total, so reads past it are zero-filled.
int packed_map_el(CUtensorMap *m, const void *ptr, int el, int d, int h, int64_t tokens) {
    if (tokens == 0) {
        memset(m, 0, sizeof(*m));
        return SDPA_OK;
    }
    const uint64_t rb = (uint64_t)d * elem_bytes(el);
    return encode_map(m, ptr, el, d, h, tokens, rb, (uint64_t)h * rb, 1, 128);
}
int packed_map(CUtensorMap *m, const void *ptr, bool bf16, int d, int h, int64_t tokens) {
    return packed_map_el(m, ptr, bf16 ? 0 : 1, d, h, tokens);
}

// fp32 dQ accumulator [rows][d] as a 2-D map with 16 x 32 boxes (64-byte rows,
// 64-byte swizzle) for TMA reduce-add.
int acc_map(CUtensorMap *m, float *acc, int d, int64_t rows) {
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 4};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, acc, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled (dQ accumulator) failed (%d)", (int)r);
    return SDPA_OK;
}

// Backward row terms (four fp32 per query row, in the row order of lse) as a
// 3-D map over [dim2][dim1][4]; a box is 128 rows of one slice or head, 16
// bytes each, unswizzled.  Rows past the extent read as zeros.
int rowx_map(CUtensorMap *m, float4 *rowx, uint64_t dim1, uint64_t dim2, uint32_t box1,
             uint32_t box2) {
    cuuint64_t dims[3] = {4, dim1, dim2};
    cuuint64_t strides[2] = {16, (cuuint64_t)dim1 * 16};
    cuuint32_t box[3] = {4, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, rowx, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled (row terms) failed (%d)", (int)r);
    return SDPA_OK;
}

// ----------------------------------------------------------- validation
struct Span {
    const void *p;
    size_t bytes;
    const char *name;
    uintptr_t align = 16;
};

bool overlaps(const Span &a, const Span &b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    auto a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

int check_common(int d, int dtype, float scale) {
    if (dtype != SDPA_BF16 && dtype != SDPA_FP16)
        return fail(SDPA_ERR_UNSUPPORTED, "dtype %d is not SDPA_BF16 or SDPA_FP16", dtype);
    if (d != 64 && d != 128) return fail(SDPA_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(SDPA_ERR_INVALID_ARG, "attn_scale must be finite and > 0 (got %g)", (double)scale);
    return SDPA_OK;
}

int check_causal(int causal) {
    if (causal != 0 && causal != 1) return fail(SDPA_ERR_INVALID_ARG, "causal must be 0 or 1 (got %d)", causal);
    return SDPA_OK;
}

// Mask kind, left window and head grouping of the extended entry points.
int check_mask_heads(int mask, int window_left, int h, int h_kv) {
    if (mask != SDPA_MASK_NONE && mask != SDPA_MASK_CAUSAL && mask != SDPA_MASK_CAUSAL_BOTTOM_RIGHT)
        return fail(SDPA_ERR_INVALID_ARG, "mask must be SDPA_MASK_NONE, SDPA_MASK_CAUSAL or "
                                          "SDPA_MASK_CAUSAL_BOTTOM_RIGHT (got %d)", mask);
    if (window_left < -1) return fail(SDPA_ERR_INVALID_ARG, "window_left must be -1 or >= 0 (got %d)", window_left);
    if (h < 0 || h_kv < 0) return fail(SDPA_ERR_INVALID_ARG, "negative head count (h=%d h_kv=%d)", h, h_kv);
    if (h > 0 && (h_kv == 0 || h % h_kv != 0))
        return fail(SDPA_ERR_INVALID_ARG, "h=%d is not a multiple of h_kv=%d", h, h_kv);
    return SDPA_OK;
}

int check_ptrs(const Span *in, int n_in, const Span *out, int n_out) {
    for (int i = 0; i < n_in + n_out; ++i) {
        const Span &s = i < n_in ? in[i] : out[i - n_in];
        if (s.bytes == 0) continue;
        if (!s.p) return fail(SDPA_ERR_INVALID_ARG, "%s is NULL", s.name);
        if (reinterpret_cast<uintptr_t>(s.p) & (s.align - 1))
            return fail(SDPA_ERR_MISALIGNED, "%s is not %d-byte aligned", s.name, (int)s.align);
    }
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j)
            if (overlaps(out[i], in[j]))
                return fail(SDPA_ERR_INVALID_ARG, "output %s overlaps input %s", out[i].name, in[j].name);
        for (int j = i + 1; j < n_out; ++j)
            if (overlaps(out[i], out[j]))
                return fail(SDPA_ERR_INVALID_ARG, "outputs %s and %s overlap", out[i].name, out[j].name);
    }
    return SDPA_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

// Backward CTA order (bwd.cu): key/value slices per group, and the working
// set (dQ accumulator, Q, dO, K, V) below which one group holds every slice.
constexpr int kBwdSliceGroup = 4;
constexpr size_t kBwdOneGroupBytes = size_t(64) << 20;
// Mean (query head, query tile) pairs per unit up to which the backward takes
// the persistent kernel, whose tiles run a few percent slower than the
// one-CTA-per-unit kernel's but whose units cost less to start and end: in
// measured sweeps it was ahead for dense problems up to a mean of 8 (by 3-13
// %), even at 8.5-16 and behind beyond, and for packed lists up to a mean of
// about 2 (by 35-105 %: short sequences), behind from 4 (by 5-7 %).
constexpr double kPersistMaxMeanTilesDense = 8.0;
constexpr double kPersistMaxMeanTilesPacked = 3.0;
thread_local int t_bwd_used = 0;  // main kernel of this thread's last backward
thread_local int t_bwd_grid_limit = 0;  // most CTAs of the persistent kernel, 0 = one per SM

// Query tiles that see key tile kt of a sequence (the backward's unit length
// per query head, as the main kernels count it).
int64_t unit_query_tiles(int mask, int window, int Lq, int Lkv, int kt) {
    const int delta = mask == SDPA_MASK_CAUSAL_BOTTOM_RIGHT ? Lkv - Lq : 0;
    const int k0 = kt * kTileN;
    const int k_last = std::min(k0 + kTileN, Lkv) - 1;
    const int row_lo = mask != SDPA_MASK_NONE ? std::max(0, k0 - delta) : 0;
    const int row_hi = window >= 0 ? std::min(Lq, k_last - delta + window + 1) : Lq;
    if (row_hi <= row_lo) return 0;
    return (row_hi + kTileM - 1) / kTileM - row_lo / kTileM;
}

// Main-kernel form of a backward call (sets p.persist, p.grid, p.unit_ctr).
// units: length of the unit list (an upper bound for packed inputs);
// short_units: the units are short enough for the persistent kernel;
// fits: the persistent kernel can take this problem.
void choose_bwd_kernel(BwdParams &p, const DeviceState &dev, int64_t units, bool short_units, bool fits) {
    const bool persist = fits && units > 0 && (t_bwd_variant == 2 || (t_bwd_variant == 0 && short_units));
    p.persist = persist ? 1 : 0;
    if (persist) {
        const int ctas = t_bwd_grid_limit > 0 ? std::min(t_bwd_grid_limit, dev.sm_count) : dev.sm_count;
        p.grid = (int)std::min<int64_t>(units, ctas);
        p.unit_ctr = dev.unit_counters + (g_unit_counter_next.fetch_add(1) % kUnitCounterSlots);
    } else {
        p.grid = (int)units;
        p.unit_ctr = nullptr;
    }
    t_bwd_used = persist ? 2 : 1;
}

// Dense two-tile lists of equal units (no mask, no window) whose count leaves
// a partial last wave on the grid: those last units are cut into two 128-row
// units each (their count is added to FwdParams::n_units) when their halves
// fill at most one wave, so the launch ends about half a unit earlier.  Under a causal mask or a window
// the list runs heaviest first and its last units are already short.
int pair_tail_split(int units, int grid, int mask, int window) {
    if (mask != SDPA_MASK_NONE || window >= 0 || units <= grid) return 0;
    const int rest = units % grid;
    return (rest > 0 && 2 * rest <= grid) ? rest : 0;
}

int launch_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return ok();
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return fail(SDPA_ERR_UNSUPPORTED, "%s: no sm_103a kernel image for this device (%s)", what,
                    cudaGetErrorString(e));
    return fail(SDPA_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
}

// Runs a forward on the chosen kernel: launch(true) starts the two-tile kernel,
// launch(false) the one-tile kernel, each with its own unit count and grid.
// A two-tile build refused for its register split (fwd_pair_refused_regs) is
// replaced by the one-tile kernel under the automatic choice; an explicit
// two-tile request reports the mismatch instead.
template <class Launch>
int run_forward(bool pair, Launch &&launch, const char *what) {
    if (!pair) return launch_status(launch(false), what);
    const cudaError_t e = launch(true);
    const int refused = fwd_pair_refused_regs();
    if (e == cudaErrorInvalidConfiguration && refused != 0) {
        if (t_fwd_variant == 0) return launch_status(launch(false), what);
        return fail(SDPA_ERR_UNSUPPORTED,
                    "%s: the two-tile forward kernel was built with %d registers per thread, but "
                    "its register split hands out exactly %d, so it is not launched",
                    what, refused, fwd_pair_split_regs());
    }
    return launch_status(e, what);
}

}  // namespace

// Lets other translation units of the library set the message that
// sdpa_last_error() returns on this thread.
int report_error(int status, const char *message) { return fail(status, "%s", message); }

}  // namespace sdpa

using namespace sdpa;

extern "C" {

const char *sdpa_last_error(void) { return t_last_error.c_str(); }

const char *sdpa_version(void) { return "sdpa_gb300 0.24 sm_103a"; }

int sdpa_set_forward_variant(int variant) {
    if (variant < 0 || variant > 2)
        return fail(SDPA_ERR_INVALID_ARG, "forward variant %d (0 auto, 1 one-tile, 2 two-tile)", variant);
    t_fwd_variant = variant;
    return ok();
}

int sdpa_set_backward_variant(int variant) {
    if (variant < 0 || variant > 2)
        return fail(SDPA_ERR_INVALID_ARG, "backward variant %d (0 auto, 1 one CTA per key tile, 2 persistent)",
                    variant);
    t_bwd_variant = variant;
    return ok();
}

int sdpa_last_backward_variant(void) { return t_bwd_used; }

int sdpa_set_backward_grid_limit(int max_ctas) {
    if (max_ctas < 0) return fail(SDPA_ERR_INVALID_ARG, "backward grid limit %d (0 = one CTA per SM)", max_ctas);
    t_bwd_grid_limit = max_ctas;
    return ok();
}

void sdpa_set_kernel_timer(void *start_event, void *stop_event) {
    t_timer.start = static_cast<cudaEvent_t>(start_event);
    t_timer.stop = static_cast<cudaEvent_t>(stop_event);
    if (!t_timer.start || !t_timer.stop) t_timer = KernelTimer{};
}

int sdpa_check_device_error(sdpa_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    uint32_t word = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
    if (word == 0) return ok();
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    static const char *names[] = {"?", "fwd", "bwd_preprocess", "bwd_main", "bwd_dq_convert", "bwd_dq",
                                  "selftest"};
    const uint32_t tag = word >> 16;
    return fail(SDPA_ERR_TIMEOUT, "kernel %s gave up on a bounded wait (site %u)",
                tag < 7 ? names[tag] : "?", word & 0xffffu);
}

int sdpa_selftest_wait_timeout(int limit_us, sdpa_stream_t stream) {
    if (limit_us < 1 || limit_us > 2000000)
        return fail(SDPA_ERR_INVALID_ARG, "limit_us must be in [1, 2000000] (got %d)", limit_us);
    DeviceState *dev = nullptr;
    int st = device_state(&dev);
    if (st) return st;
    return launch_status(launch_wait_selftest(dev->err, (uint64_t)limit_us * 1000ull,
                                              static_cast<cudaStream_t>(stream)),
                         "sdpa_selftest_wait_timeout");
}

int sdpa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int b, int h,
                int h_kv, int s_q, int s_kv, int d, float attn_scale, int mask, int window_left,
                int dtype, sdpa_stream_t stream) {
    int st = check_common(d, dtype, attn_scale);
    if (st) return st;
    if ((st = check_mask_heads(mask, window_left, h, h_kv))) return st;
    if (b < 0 || s_q < 0 || s_kv < 0)
        return fail(SDPA_ERR_INVALID_ARG, "negative size (b=%d s_q=%d s_kv=%d)", b, s_q, s_kv);
    const int64_t bh = (int64_t)b * h, bh_kv = (int64_t)b * h_kv;
    if (bh == 0 || s_q == 0) return ok();
    // left windows take the two-tile kernel at d = 128 only (its walking instantiations)
    const bool pair = use_pair_kernel(false, d, s_q, s_kv) && (window_left < 0 || d == 128);
    const int64_t q_tiles = (s_q + kTileM - 1) / kTileM;  // 128-row units: the most units
    if (bh > INT32_MAX || q_tiles * bh > INT32_MAX)
        return fail(SDPA_ERR_INVALID_ARG, "problem too large for one launch");
    const size_t qbytes = (size_t)bh * s_q * d * 2, kvbytes = (size_t)bh_kv * s_kv * d * 2;
    const Span in[3] = {{q, qbytes, "q"}, {k, kvbytes, "k"}, {v, kvbytes, "v"}};
    const Span out[2] = {{o, qbytes, "o"}, {lse, lse ? (size_t)bh * s_q * 4 : 0, "lse"}};
    if ((st = check_ptrs(in, 3, out, 2))) return st;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev))) return st;
    if ((st = get_encoder())) return st;
    const bool bf16 = dtype == SDPA_BF16;
    CUtensorMap tq, tk, tv;
    if ((st = dense_map(&tq, q, bf16, d, s_q, bh))) return st;
    if ((st = dense_map(&tk, k, bf16, d, s_kv, bh_kv))) return st;
    if ((st = dense_map(&tv, v, bf16, d, s_kv, bh_kv))) return st;
    FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.err = dev->err;
    p.bh = (int)bh;
    p.h = h;
    p.h_kv = h_kv;
    p.group = h / h_kv;
    p.s_q = s_q;
    p.s_kv = s_kv;
    const bool slice_major = 2 * kvbytes > kSliceMajorKVBytes;
    p.mask = mask;
    p.window = window_left;
    p.scale_log2 = attn_scale * kLog2e;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    auto launch = [&](bool two) {
        const int rows = two ? fwd_pair_rows() : kTileM;
        p.q_tiles = (s_q + rows - 1) / rows;
        const int units = (int)(p.q_tiles * bh);
        const int grid = std::min(units, dev->sm_count);
        p.n_units = units + (two ? pair_tail_split(units, grid, mask, window_left) : 0);
        return two ? launch_fwd_pair(tq, tk, tv, p, d, bf16, false, grid, cs, t_timer)
                   : launch_fwd(tq, tk, tv, p, d, bf16, false, grid, slice_major, cs, t_timer);
    };
    return run_forward(pair, launch, "sdpa_fwd");
}

int sdpa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int b, int h,
             int s_q, int s_kv, int d, float attn_scale, int causal, int dtype,
             sdpa_stream_t stream) {
    int st = check_causal(causal);
    if (st) return st;
    return sdpa_fwd_ex(q, k, v, o, lse, b, h, h, s_q, s_kv, d, attn_scale,
                       causal ? SDPA_MASK_CAUSAL : SDPA_MASK_NONE, -1, dtype, stream);
}

static int check_varlen_sizes(const int32_t *cu_q, const int32_t *cu_kv, int num_seqs, int total_q,
                              int total_kv, int max_q, int max_kv, int h) {
    if (num_seqs < 0 || total_q < 0 || total_kv < 0 || max_q < 0 || max_kv < 0 || h < 0)
        return fail(SDPA_ERR_INVALID_ARG, "negative size in varlen arguments");
    if (cu_kv && !cu_q)
        return fail(SDPA_ERR_INVALID_ARG, "cu_seqlens_kv given without cu_seqlens_q");
    if (num_seqs > 0 && (!cu_q || !cu_kv))
        return fail(SDPA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_kv are required");
    if (max_q > total_q || max_kv > total_kv)
        return fail(SDPA_ERR_INVALID_ARG, "max_seqlen exceeds the packed total");
    if (total_q > 0 && max_q == 0)
        return fail(SDPA_ERR_INVALID_ARG, "max_seqlen_q is 0 but total_q is %d", total_q);
    if (total_kv > 0 && max_kv == 0)
        return fail(SDPA_ERR_INVALID_ARG, "max_seqlen_kv is 0 but total_kv is %d", total_kv);
    if (num_seqs == 0 && (total_q > 0 || total_kv > 0))
        return fail(SDPA_ERR_INVALID_ARG, "tokens given but num_seqs is 0");
    return SDPA_OK;
}

int sdpa_varlen_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                       const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv, int num_seqs,
                       int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv, int h,
                       int h_kv, int d, float attn_scale, int mask, int window_left, int dtype,
                       sdpa_stream_t stream) {
    int st = check_common(d, dtype, attn_scale);
    if (st) return st;
    if ((st = check_mask_heads(mask, window_left, h, h_kv))) return st;
    if ((st = check_varlen_sizes(cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                                 max_seqlen_q, max_seqlen_kv, h)))
        return st;
    if (h == 0 || total_q == 0 || num_seqs == 0) return ok();
    const bool pair = use_pair_kernel(true, d, (int64_t)total_q / num_seqs, (int64_t)total_kv / num_seqs,
                                      window_left < 0 && num_seqs + 1 <= fwd_pair_table_cap(d, false)) &&
                      (window_left < 0 || d == 128);
    const int64_t q_tiles = (max_seqlen_q + kTileM - 1) / kTileM;  // 128-row units: the most
    const int64_t slices = (int64_t)num_seqs * h;
    if (slices > INT32_MAX || q_tiles * slices > INT32_MAX)
        return fail(SDPA_ERR_INVALID_ARG, "problem too large for one launch");
    const size_t qbytes = (size_t)total_q * h * d * 2, kvbytes = (size_t)total_kv * h_kv * d * 2;
    const Span in[5] = {{q, qbytes, "q"}, {k, kvbytes, "k"}, {v, kvbytes, "v"},
                        {cu_seqlens_q, (size_t)(num_seqs + 1) * 4, "cu_seqlens_q", 4},
                        {cu_seqlens_kv, (size_t)(num_seqs + 1) * 4, "cu_seqlens_kv", 4}};
    const Span out[2] = {{o, qbytes, "o"}, {lse, lse ? (size_t)total_q * h * 4 : 0, "lse"}};
    if ((st = check_ptrs(in, 5, out, 2))) return st;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev))) return st;
    if ((st = get_encoder())) return st;
    const bool bf16 = dtype == SDPA_BF16;
    CUtensorMap tq, tk, tv;
    if ((st = packed_map(&tq, q, bf16, d, h, total_q))) return st;
    if ((st = packed_map(&tk, k, bf16, d, h_kv, total_kv))) return st;
    if ((st = packed_map(&tv, v, bf16, d, h_kv, total_kv))) return st;
    FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.cu_q = cu_seqlens_q;
    p.cu_kv = cu_seqlens_kv;
    p.err = dev->err;
    p.bh = (int)slices;
    p.h = h;
    p.h_kv = h_kv;
    p.group = h / h_kv;
    p.num_seqs = num_seqs;
    const bool slice_major = 2 * kvbytes > kSliceMajorKVBytes;
    p.mask = mask;
    p.window = window_left;
    p.scale_log2 = attn_scale * kLog2e;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    auto launch = [&](bool two) {
        const int rows = two ? fwd_pair_rows() : kTileM;
        p.q_tiles = (max_seqlen_q + rows - 1) / rows;
        p.n_units = (int)(p.q_tiles * slices);
        const int grid = std::min(p.n_units, dev->sm_count);
        return two ? launch_fwd_pair(tq, tk, tv, p, d, bf16, true, grid, cs, t_timer)
                   : launch_fwd(tq, tk, tv, p, d, bf16, true, grid, slice_major, cs, t_timer);
    };
    return run_forward(pair, launch, "sdpa_varlen_fwd");
}

int sdpa_varlen_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv, int num_seqs,
                    int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv, int h, int d,
                    float attn_scale, int causal, int dtype, sdpa_stream_t stream) {
    int st = check_causal(causal);
    if (st) return st;
    return sdpa_varlen_fwd_ex(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q,
                              total_kv, max_seqlen_q, max_seqlen_kv, h, h, d, attn_scale,
                              causal ? SDPA_MASK_CAUSAL : SDPA_MASK_NONE, -1, dtype, stream);
}

// Checks of the FP8 forward's extra arguments.
static int check_fp8(int d, int out_dtype, float scale, const float *dq, const float *dk,
                     const float *dv, const float *so) {
    if (d != 128) return fail(SDPA_ERR_UNSUPPORTED, "the FP8 forward takes d = 128 (got d=%d)", d);
    if (out_dtype != SDPA_BF16 && out_dtype != SDPA_FP16 && out_dtype != SDPA_FP8_E4M3)
        return fail(SDPA_ERR_UNSUPPORTED, "out_dtype %d is not SDPA_BF16, SDPA_FP16 or SDPA_FP8_E4M3",
                    out_dtype);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(SDPA_ERR_INVALID_ARG, "attn_scale must be finite and > 0 (got %g)", (double)scale);
    if (!dq || !dk || !dv) return fail(SDPA_ERR_INVALID_ARG, "descale_q, descale_k and descale_v are required");
    if (out_dtype == SDPA_FP8_E4M3 && !so)
        return fail(SDPA_ERR_INVALID_ARG, "scale_o is required for an SDPA_FP8_E4M3 output");
    return SDPA_OK;
}

int sdpa_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                 const float *descale_q, const float *descale_k, const float *descale_v,
                 const float *scale_o, float *amax_o, int b, int h, int h_kv, int s_q, int s_kv,
                 int d, float attn_scale, int mask, int window_left, int out_dtype,
                 sdpa_stream_t stream) {
    int st = check_fp8(d, out_dtype, attn_scale, descale_q, descale_k, descale_v, scale_o);
    if (st) return st;
    if ((st = check_mask_heads(mask, window_left, h, h_kv))) return st;
    if (b < 0 || s_q < 0 || s_kv < 0)
        return fail(SDPA_ERR_INVALID_ARG, "negative size (b=%d s_q=%d s_kv=%d)", b, s_q, s_kv);
    const int64_t bh = (int64_t)b * h, bh_kv = (int64_t)b * h_kv;
    if (bh == 0 || s_q == 0) return ok();
    // FP8 with a left window runs the one-tile kernel
    const bool pair = window_left < 0 && use_pair_kernel(false, d, s_q, s_kv);
    const int64_t q_tiles = (s_q + kTileM - 1) / kTileM;  // 128-row units: the most units
    if (bh > INT32_MAX || q_tiles * bh > INT32_MAX)
        return fail(SDPA_ERR_INVALID_ARG, "problem too large for one launch");
    const size_t ob = out_dtype == SDPA_FP8_E4M3 ? 1 : 2;
    const size_t qbytes = (size_t)bh * s_q * d, kvbytes = (size_t)bh_kv * s_kv * d;
    const Span in[7] = {{q, qbytes, "q"}, {k, kvbytes, "k"}, {v, kvbytes, "v"},
                        {descale_q, 4, "descale_q", 4}, {descale_k, 4, "descale_k", 4},
                        {descale_v, 4, "descale_v", 4}, {scale_o, scale_o ? 4u : 0u, "scale_o", 4}};
    const Span out[3] = {{o, qbytes * ob, "o"}, {lse, lse ? (size_t)bh * s_q * 4 : 0, "lse"},
                         {amax_o, amax_o ? 4u : 0u, "amax_o", 4}};
    if ((st = check_ptrs(in, 7, out, 3))) return st;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev))) return st;
    if ((st = get_encoder())) return st;
    CUtensorMap tq, tk, tv;
    if ((st = dense_map_el(&tq, q, 2, d, s_q, bh))) return st;
    if ((st = dense_map_el(&tk, k, 2, d, s_kv, bh_kv))) return st;
    if ((st = dense_map_el(&tv, v, 2, d, s_kv, bh_kv))) return st;
    FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.err = dev->err;
    p.bh = (int)bh;
    p.h = h;
    p.h_kv = h_kv;
    p.group = h / h_kv;
    p.s_q = s_q;
    p.s_kv = s_kv;
    const bool slice_major = 2 * kvbytes > kSliceMajorKVBytes;
    p.mask = mask;
    p.window = window_left;
    p.scale_log2 = attn_scale * kLog2e;
    p.descale_q = descale_q;
    p.descale_k = descale_k;
    p.descale_v = descale_v;
    p.scale_o = scale_o;
    p.amax_o = amax_o;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (amax_o && cudaMemsetAsync(amax_o, 0, 4, cs) != cudaSuccess)
        return fail(SDPA_ERR_CUDA, "clearing amax_o failed");
    auto launch = [&](bool two) {
        const int rows = two ? fwd_pair_rows() : kTileM;
        p.q_tiles = (s_q + rows - 1) / rows;
        const int units = (int)(p.q_tiles * bh);
        const int grid = std::min(units, dev->sm_count);
        p.n_units = units + (two ? pair_tail_split(units, grid, mask, window_left) : 0);
        return two ? launch_fwd_pair_fp8(tq, tk, tv, p, out_dtype, false, grid, cs, t_timer)
                   : launch_fwd_fp8(tq, tk, tv, p, out_dtype, false, grid, slice_major, cs, t_timer);
    };
    return run_forward(pair, launch, "sdpa_fwd_fp8");
}

int sdpa_varlen_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                        const float *descale_q, const float *descale_k, const float *descale_v,
                        const float *scale_o, float *amax_o, const int32_t *cu_seqlens_q,
                        const int32_t *cu_seqlens_kv, int num_seqs, int total_q, int total_kv,
                        int max_seqlen_q, int max_seqlen_kv, int h, int h_kv, int d,
                        float attn_scale, int mask, int window_left, int out_dtype,
                        sdpa_stream_t stream) {
    int st = check_fp8(d, out_dtype, attn_scale, descale_q, descale_k, descale_v, scale_o);
    if (st) return st;
    if ((st = check_mask_heads(mask, window_left, h, h_kv))) return st;
    if ((st = check_varlen_sizes(cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                                 max_seqlen_q, max_seqlen_kv, h)))
        return st;
    if (h == 0 || total_q == 0 || num_seqs == 0) return ok();
    const bool pair = window_left < 0 &&
                      use_pair_kernel(true, d, (int64_t)total_q / num_seqs, (int64_t)total_kv / num_seqs,
                                      num_seqs + 1 <= fwd_pair_table_cap(d, true));
    const int64_t q_tiles = (max_seqlen_q + kTileM - 1) / kTileM;  // 128-row units: the most
    const int64_t slices = (int64_t)num_seqs * h;
    if (slices > INT32_MAX || q_tiles * slices > INT32_MAX)
        return fail(SDPA_ERR_INVALID_ARG, "problem too large for one launch");
    const size_t ob = out_dtype == SDPA_FP8_E4M3 ? 1 : 2;
    const size_t qbytes = (size_t)total_q * h * d, kvbytes = (size_t)total_kv * h_kv * d;
    const Span in[9] = {{q, qbytes, "q"}, {k, kvbytes, "k"}, {v, kvbytes, "v"},
                        {cu_seqlens_q, (size_t)(num_seqs + 1) * 4, "cu_seqlens_q", 4},
                        {cu_seqlens_kv, (size_t)(num_seqs + 1) * 4, "cu_seqlens_kv", 4},
                        {descale_q, 4, "descale_q", 4}, {descale_k, 4, "descale_k", 4},
                        {descale_v, 4, "descale_v", 4}, {scale_o, scale_o ? 4u : 0u, "scale_o", 4}};
    const Span out[3] = {{o, qbytes * ob, "o"}, {lse, lse ? (size_t)total_q * h * 4 : 0, "lse"},
                         {amax_o, amax_o ? 4u : 0u, "amax_o", 4}};
    if ((st = check_ptrs(in, 9, out, 3))) return st;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev))) return st;
    if ((st = get_encoder())) return st;
    CUtensorMap tq, tk, tv;
    if ((st = packed_map_el(&tq, q, 2, d, h, total_q))) return st;
    if ((st = packed_map_el(&tk, k, 2, d, h_kv, total_kv))) return st;
    if ((st = packed_map_el(&tv, v, 2, d, h_kv, total_kv))) return st;
    FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.cu_q = cu_seqlens_q;
    p.cu_kv = cu_seqlens_kv;
    p.err = dev->err;
    p.bh = (int)slices;
    p.h = h;
    p.h_kv = h_kv;
    p.group = h / h_kv;
    p.num_seqs = num_seqs;
    const bool slice_major = 2 * kvbytes > kSliceMajorKVBytes;
    p.mask = mask;
    p.window = window_left;
    p.scale_log2 = attn_scale * kLog2e;
    p.descale_q = descale_q;
    p.descale_k = descale_k;
    p.descale_v = descale_v;
    p.scale_o = scale_o;
    p.amax_o = amax_o;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (amax_o && cudaMemsetAsync(amax_o, 0, 4, cs) != cudaSuccess)
        return fail(SDPA_ERR_CUDA, "clearing amax_o failed");
    auto launch = [&](bool two) {
        const int rows = two ? fwd_pair_rows() : kTileM;
        p.q_tiles = (max_seqlen_q + rows - 1) / rows;
        p.n_units = (int)(p.q_tiles * slices);
        const int grid = std::min(p.n_units, dev->sm_count);
        return two ? launch_fwd_pair_fp8(tq, tk, tv, p, out_dtype, true, grid, cs, t_timer)
                   : launch_fwd_fp8(tq, tk, tv, p, out_dtype, true, grid, slice_major, cs, t_timer);
    };
    return run_forward(pair, launch, "sdpa_varlen_fwd_fp8");
}

static size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t sdpa_bwd_workspace_size(int b, int h, int s_q, int d) {
    if (b < 0 || h < 0 || s_q < 0 || (d != 64 && d != 128)) return (size_t)-1;
    const size_t rows = (size_t)b * h * s_q;
    if (rows == 0) return 0;
    const size_t acc = rows * d * 4, rowx = rows * 16;
    return ((acc + 255) & ~(size_t)255) + ((rowx + 255) & ~(size_t)255);
}

size_t sdpa_varlen_bwd_workspace_size(int total_q, int h, int d) {
    if (total_q < 0 || h < 0 || (d != 64 && d != 128)) return (size_t)-1;
    const size_t rows = (size_t)total_q * h;
    if (rows == 0) return 0;
    const size_t acc = rows * d * 4, rowx = rows * 16;
    return ((acc + 255) & ~(size_t)255) + ((rowx + 255) & ~(size_t)255);
}

// Deterministic mode keeps only the row terms (dQ is written directly).
static size_t ex_workspace(size_t rows, int d, int deterministic) {
    if (rows == 0) return 0;
    const size_t rowx = round256(rows * 16);
    return deterministic ? rowx : round256(rows * d * 4) + rowx;
}

size_t sdpa_bwd_ex_workspace_size(int b, int h, int s_q, int d, int deterministic) {
    if (deterministic != 0 && deterministic != 1) return (size_t)-1;
    if (b < 0 || h < 0 || s_q < 0 || (d != 64 && d != 128)) return (size_t)-1;
    return ex_workspace((size_t)b * h * s_q, d, deterministic);
}

size_t sdpa_varlen_bwd_ex_workspace_size(int total_q, int h, int d, int deterministic) {
    if (deterministic != 0 && deterministic != 1) return (size_t)-1;
    if (total_q < 0 || h < 0 || (d != 64 && d != 128)) return (size_t)-1;
    return ex_workspace((size_t)total_q * h, d, deterministic);
}

int sdpa_bwd_ex(const void *q, const void *k, const void *v, const void *o, const void *dout,
                const float *lse, void *dq, void *dk, void *dv, int b, int h, int h_kv, int s_q,
                int s_kv, int d, float attn_scale, int mask, int window_left, int deterministic,
                int dtype, void *workspace, size_t workspace_bytes, sdpa_stream_t stream) {
    int st = check_common(d, dtype, attn_scale);
    if (st) return st;
    if ((st = check_mask_heads(mask, window_left, h, h_kv))) return st;
    if (deterministic != 0 && deterministic != 1)
        return fail(SDPA_ERR_INVALID_ARG, "deterministic must be 0 or 1 (got %d)", deterministic);
    if (b < 0 || s_q < 0 || s_kv < 0)
        return fail(SDPA_ERR_INVALID_ARG, "negative size (b=%d s_q=%d s_kv=%d)", b, s_q, s_kv);
    const int64_t bh = (int64_t)b * h, bh_kv = (int64_t)b * h_kv;
    if (bh == 0) return ok();
    const int64_t kv_tiles = (s_kv + kTileN - 1) / kTileN;
    if (bh > INT32_MAX || kv_tiles * bh_kv > INT32_MAX || (int64_t)s_q * bh > INT32_MAX)
        return fail(SDPA_ERR_INVALID_ARG, "problem too large for one launch");
    const size_t qbytes = (size_t)bh * s_q * d * 2, kvbytes = (size_t)bh_kv * s_kv * d * 2;
    const size_t need = sdpa_bwd_ex_workspace_size(b, h, s_q, d, deterministic);
    const Span in[6] = {{q, qbytes, "q"}, {k, kvbytes, "k"}, {v, kvbytes, "v"}, {o, qbytes, "o"},
                        {dout, qbytes, "dout"}, {lse, (size_t)bh * s_q * 4, "lse"}};
    const Span out[4] = {{dq, qbytes, "dq"}, {dk, kvbytes, "dk"}, {dv, kvbytes, "dv"},
                         {workspace, need, "workspace"}};
    if ((st = check_ptrs(in, 6, out, 4))) return st;
    if (need > 0 && workspace_bytes < need)
        return fail(SDPA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev))) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (s_q == 0) {
        // no query: the key/value gradients are zero
        if (kvbytes) {
            cudaError_t e = cudaMemsetAsync(dk, 0, kvbytes, cs);
            if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kvbytes, cs);
            if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
        }
        return ok();
    }
    if ((st = get_encoder())) return st;
    const bool bf16 = dtype == SDPA_BF16;
    CUtensorMap tq, tk, tv, tdo;
    if ((st = dense_map(&tq, q, bf16, d, s_q, bh))) return st;
    if ((st = dense_map(&tk, k, bf16, d, s_kv, bh_kv))) return st;
    if ((st = dense_map(&tv, v, bf16, d, s_kv, bh_kv))) return st;
    if ((st = dense_map(&tdo, dout, bf16, d, s_q, bh))) return st;
    BwdParams p{};
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    CUtensorMap tdq, trx;
    if (deterministic) {
        p.dq_acc = nullptr;
        p.rowx = static_cast<float4 *>(workspace);
        memset(&tdq, 0, sizeof(tdq));  // unused: the main kernel adds no dQ
    } else {
        p.dq_acc = static_cast<float *>(workspace);
        p.rowx = reinterpret_cast<float4 *>(static_cast<char *>(workspace) +
                                            round256((size_t)bh * s_q * d * 4));
        if ((st = acc_map(&tdq, p.dq_acc, d, bh * s_q))) return st;
    }
    if ((st = rowx_map(&trx, p.rowx, s_q, bh, 128, 1))) return st;
    p.deterministic = deterministic;
    p.q_tiles = (s_q + kTileM - 1) / kTileM;
    p.err = dev->err;
    p.bh = (int)bh;
    p.h = h;
    p.h_kv = h_kv;
    p.group = h / h_kv;
    p.kv_slices = (int)bh_kv;
    p.s_q = s_q;
    p.s_kv = s_kv;
    p.kv_tiles = (int)kv_tiles;
    p.total_q = (int)(bh * s_q);
    p.mask = mask;
    p.window = window_left;
    p.scale = attn_scale;
    p.scale_log2 = attn_scale * kLog2e;
    // CTA order of the main kernel: groups of four key/value slices keep the
    // resident CTAs' dQ accumulator, Q and dO in L2; a problem whose whole
    // working set fits in half of L2 runs as one group (heaviest units first).
    const size_t working = (size_t)bh * s_q * d * 4 + 2 * qbytes + 2 * kvbytes;
    p.slice_group = working <= kBwdOneGroupBytes ? (int)bh_kv : kBwdSliceGroup;
    p.seq_table = 0;
    int64_t tiles = 0;
    for (int kt = 0; kt < kv_tiles; ++kt) tiles += unit_query_tiles(mask, window_left, s_q, s_kv, kt);
    const double mean_tiles = kv_tiles > 0 ? (double)tiles * p.group / kv_tiles : 0.0;
    choose_bwd_kernel(p, *dev, kv_tiles * bh_kv, mean_tiles <= kPersistMaxMeanTilesDense, true);
    return launch_status(launch_bwd(tq, tk, tv, tdo, tdq, trx, p, d, bf16, false, cs, t_timer), "sdpa_bwd");
}

int sdpa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
             const float *lse, void *dq, void *dk, void *dv, int b, int h, int s_q, int s_kv,
             int d, float attn_scale, int causal, int dtype, void *workspace,
             size_t workspace_bytes, sdpa_stream_t stream) {
    int st = check_causal(causal);
    if (st) return st;
    return sdpa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, b, h, h, s_q, s_kv, d, attn_scale,
                       causal ? SDPA_MASK_CAUSAL : SDPA_MASK_NONE, -1, 0, dtype, workspace,
                       workspace_bytes, stream);
}

int sdpa_varlen_bwd_ex(const void *q, const void *k, const void *v, const void *o,
                       const void *dout, const float *lse, void *dq, void *dk, void *dv,
                       const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv, int num_seqs,
                       int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv, int h,
                       int h_kv, int d, float attn_scale, int mask, int window_left,
                       int deterministic, int dtype, void *workspace, size_t workspace_bytes,
                       sdpa_stream_t stream) {
    int st = check_common(d, dtype, attn_scale);
    if (st) return st;
    if ((st = check_mask_heads(mask, window_left, h, h_kv))) return st;
    if (deterministic != 0 && deterministic != 1)
        return fail(SDPA_ERR_INVALID_ARG, "deterministic must be 0 or 1 (got %d)", deterministic);
    if ((st = check_varlen_sizes(cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                                 max_seqlen_q, max_seqlen_kv, h)))
        return st;
    if (h == 0 || num_seqs == 0 || (total_q == 0 && total_kv == 0)) return ok();
    const int64_t kv_tiles = (max_seqlen_kv + kTileN - 1) / kTileN;
    const int64_t slices = (int64_t)num_seqs * h, kv_slices = (int64_t)num_seqs * h_kv;
    if (slices > INT32_MAX || kv_tiles * kv_slices > INT32_MAX || (int64_t)total_q * h > INT32_MAX)
        return fail(SDPA_ERR_INVALID_ARG, "problem too large for one launch");
    const size_t qbytes = (size_t)total_q * h * d * 2, kvbytes = (size_t)total_kv * h_kv * d * 2;
    const size_t need = sdpa_varlen_bwd_ex_workspace_size(total_q, h, d, deterministic);
    const Span in[8] = {{q, qbytes, "q"}, {k, kvbytes, "k"}, {v, kvbytes, "v"}, {o, qbytes, "o"},
                        {dout, qbytes, "dout"}, {lse, (size_t)total_q * h * 4, "lse"},
                        {cu_seqlens_q, (size_t)(num_seqs + 1) * 4, "cu_seqlens_q", 4},
                        {cu_seqlens_kv, (size_t)(num_seqs + 1) * 4, "cu_seqlens_kv", 4}};
    const Span out[4] = {{dq, qbytes, "dq"}, {dk, kvbytes, "dk"}, {dv, kvbytes, "dv"},
                         {workspace, need, "workspace"}};
    if ((st = check_ptrs(in, 8, out, 4))) return st;
    if (need > 0 && workspace_bytes < need)
        return fail(SDPA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev))) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (total_q == 0) {
        cudaError_t e = cudaMemsetAsync(dk, 0, kvbytes, cs);
        if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kvbytes, cs);
        if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
        return ok();
    }
    if ((st = get_encoder())) return st;
    const bool bf16 = dtype == SDPA_BF16;
    CUtensorMap tq, tk, tv, tdo;
    if ((st = packed_map(&tq, q, bf16, d, h, total_q))) return st;
    if ((st = packed_map(&tk, k, bf16, d, h_kv, total_kv))) return st;
    if ((st = packed_map(&tv, v, bf16, d, h_kv, total_kv))) return st;
    if ((st = packed_map(&tdo, dout, bf16, d, h, total_q))) return st;
    BwdParams p{};
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    CUtensorMap tdq, trx;
    if (deterministic) {
        p.dq_acc = nullptr;
        p.rowx = static_cast<float4 *>(workspace);
        memset(&tdq, 0, sizeof(tdq));  // unused: the main kernel adds no dQ
    } else {
        p.dq_acc = static_cast<float *>(workspace);
        p.rowx = reinterpret_cast<float4 *>(static_cast<char *>(workspace) +
                                            round256((size_t)total_q * h * d * 4));
        if ((st = acc_map(&tdq, p.dq_acc, d, (int64_t)total_q * h))) return st;
    }
    if ((st = rowx_map(&trx, p.rowx, h, total_q, 1, 128))) return st;
    p.deterministic = deterministic;
    p.q_tiles = (max_seqlen_q + kTileM - 1) / kTileM;
    p.cu_q = cu_seqlens_q;
    p.cu_kv = cu_seqlens_kv;
    p.err = dev->err;
    p.bh = (int)slices;
    p.h = h;
    p.h_kv = h_kv;
    p.group = h / h_kv;
    p.kv_slices = (int)kv_slices;
    p.num_seqs = num_seqs;
    p.kv_tiles = (int)kv_tiles;
    p.total_q = total_q;
    p.mask = mask;
    p.window = window_left;
    p.scale = attn_scale;
    p.scale_log2 = attn_scale * kLog2e;
    // CTA grid of the main kernel: the sequences' own key tiles from a per-CTA
    // sequence table (sum over n of ceil(Lkv_n / 128) <= total_kv / 128 +
    // num_seqs, and <= num_seqs times the longest), or the envelope of the
    // longest sequence for lists too long to tabulate.
    p.slice_group = kBwdSliceGroup;
    p.seq_table = num_seqs <= kBwdSeqTableMax ? 1 : 0;
    const int64_t tiles = p.seq_table ? std::min<int64_t>((int64_t)num_seqs * kv_tiles,
                                                          total_kv / kTileN + num_seqs)
                                      : (int64_t)num_seqs * kv_tiles;
    // The persistent kernel (lists of up to kPersistSeqMax sequences) for
    // short sequences.  The lengths stay on the device, so the mean unit
    // length is estimated from the mean sequence length: a sequence of L
    // keys has ceil(L / 128) key tiles, about L / 128 + 1/2, and under a
    // causal mask its key tiles see (tiles + 1) / 2 query tiles on average;
    // a window bounds that by its own width.
    const double seq_tiles = (double)total_kv / num_seqs / kTileN + 0.5;
    double mean_tiles = mask != SDPA_MASK_NONE ? (seq_tiles + 1.0) / 2.0 : seq_tiles;
    if (window_left >= 0) mean_tiles = std::min(mean_tiles, (double)window_left / kTileM + 2.0);
    mean_tiles *= p.group;
    choose_bwd_kernel(p, *dev, tiles * h_kv, mean_tiles <= kPersistMaxMeanTilesPacked,
                      num_seqs <= kPersistSeqMax);
    return launch_status(launch_bwd(tq, tk, tv, tdo, tdq, trx, p, d, bf16, true, cs, t_timer), "sdpa_varlen_bwd");
}

int sdpa_varlen_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                    const float *lse, void *dq, void *dk, void *dv, const int32_t *cu_seqlens_q,
                    const int32_t *cu_seqlens_kv, int num_seqs, int total_q, int total_kv,
                    int max_seqlen_q, int max_seqlen_kv, int h, int d, float attn_scale,
                    int causal, int dtype, void *workspace, size_t workspace_bytes,
                    sdpa_stream_t stream) {
    int st = check_causal(causal);
    if (st) return st;
    return sdpa_varlen_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv,
                              num_seqs, total_q, total_kv, max_seqlen_q, max_seqlen_kv, h, h, d,
                              attn_scale, causal ? SDPA_MASK_CAUSAL : SDPA_MASK_NONE, -1, 0,
                              dtype, workspace, workspace_bytes, stream);
}

}  // extern "C"
