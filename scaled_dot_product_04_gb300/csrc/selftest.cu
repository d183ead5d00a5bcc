// Failure-detection self-test of the bounded waits.
//
// Every wait of the kernels is an mbarrier poll bounded in time; on expiry the
// waiting thread records (kernel tag << 16 | wait site) in the library's error
// word and raises the CTA's abort flag, and sdpa_check_device_error turns the
// word into SDPA_ERR_TIMEOUT.  This kernel runs that same code on a barrier
// phase that nothing completes, with a short limit, so a test can watch a wait
// expire and the status come back without faulting or hanging the GPU.
#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {
namespace {

__global__ void __launch_bounds__(32, 1) wait_selftest_kernel(uint32_t *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ uint32_t abort_flag;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);  // one arrival would complete phase 0; none comes
        abort_flag = 0u;
        fence_mbar_init();
    }
    __syncwarp();
    WaitCtx w{&abort_flag, err, kTagSelftest, limit_ns};
    const bool ok = mbar_wait(bar, 0, w, 1);
    // The wait gave up, so the abort flag is up and the error word holds the
    // first failure; a second wait returns at once through the abort flag.
    if (!ok && threadIdx.x == 0) mbar_wait(bar, 0, w, 2);
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t *err, uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace sdpa
