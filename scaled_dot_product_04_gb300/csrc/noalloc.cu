// Allocation-free variant of the dense backward.
//
// sdpa_bwd needs a workspace (the fp32 dQ accumulator and the per-row D
// terms) that the caller allocates.  Some callers cannot allocate device
// memory at all: code running as a plug-in or callback inside another
// runtime that owns every device allocation and hands out no workspace,
// or a latency-critical loop where a cudaMalloc (which may synchronise the
// whole device) is not allowed.  sdpa_bwd_noalloc serves them from a
// fixed scratch array that lives in this library's device image instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads
// the library holds it (kNoAllocScratchBytes) until the process exits.
// Host code cannot use the symbol's name as a device address: the device
// address is fetched once per device with cudaGetSymbolAddress, with that
// device current, and passed to the kernels.  The address belongs to the
// device's context: a cudaDeviceReset destroys that context, and the kept
// address would then name memory of a context that no longer exists, so a
// process that resets a device must not call this entry point on it again.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sdpa.h"

namespace {

// 32 MiB: enough for b*h*s_q up to 63,550 rows at d = 128 (123,361 at d = 64).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

}  // namespace

namespace sdpa {
int report_error(int status, const char *message);  // sets sdpa_last_error()
}

extern "C" int sdpa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                int b, int h, int s_q, int s_kv, int d, float attn_scale,
                                int causal, int dtype, sdpa_stream_t stream) {
    char msg[512];
    const size_t need = sdpa_bwd_workspace_size(b, h, s_q, d);
    if (need == (size_t)-1)  // invalid sizes: let sdpa_bwd report them
        return sdpa_bwd(q, k, v, o, dout, lse, dq, dk, dv, b, h, s_q, s_kv, d, attn_scale,
                        causal, dtype, nullptr, 0, stream);
    if (need > kNoAllocScratchBytes) {
        snprintf(msg, sizeof(msg),
                 "sdpa_bwd_noalloc: this problem needs %zu bytes of scratch but the built-in "
                 "array holds %zu (b*h*s_q*d*4 for the dQ accumulator plus b*h*s_q*16 for the "
                 "row terms, each rounded up to 256 bytes, must fit); use sdpa_bwd with a "
                 "workspace",
                 need, kNoAllocScratchBytes);
        return sdpa::report_error(SDPA_ERR_WORKSPACE, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "sdpa_bwd_noalloc: cudaGetDevice failed (%s)",
                 cudaGetErrorString(e));
        return sdpa::report_error(SDPA_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg),
                 "sdpa_bwd_noalloc: device index %d is outside the %d devices this library "
                 "keeps a scratch address for", dev, kMaxDevices);
        return sdpa::report_error(SDPA_ERR_UNSUPPORTED, msg);
    }
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_scratch_ptr[dev]) {
            // First call on this device, with the device current.
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || ptr == nullptr) {
                snprintf(msg, sizeof(msg),
                         "sdpa_bwd_noalloc: cudaGetSymbolAddress of the scratch array failed (%s)",
                         cudaGetErrorString(e));
                return sdpa::report_error(SDPA_ERR_CUDA, msg);
            }
            g_scratch_ptr[dev] = ptr;
        }
        scratch = g_scratch_ptr[dev];
    }
    // The backward's preprocess kernel zeroes the dQ accumulator and rewrites
    // the D terms on every call, so what an earlier call left in the array
    // does not matter.
    return sdpa_bwd(q, k, v, o, dout, lse, dq, dk, dv, b, h, s_q, s_kv, d, attn_scale, causal,
                    dtype, scratch, kNoAllocScratchBytes, stream);
}
