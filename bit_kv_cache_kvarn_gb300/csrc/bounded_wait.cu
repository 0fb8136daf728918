// Self-check of the library's bounded device waits: one wait that is made to run out on purpose.
//
// Every device-side wait in libkvarn (TMA data arriving, tensor-core work completing) polls an
// mbarrier with a time limit; when the limit passes, the waiting thread sets a device error word
// and the kernel ends normally, so the CUDA context stays usable and the host learns of the
// failure through kvarn_device_error.  This kernel exercises that path without any fault: thread 0
// arms an mbarrier for 16 bytes of transfer that no copy will ever deliver (nothing is issued), so
// the phase never completes and the wait gives up after the requested limit.  No memory outside
// the block's own shared memory is touched besides the error word.
#include "kvarn_common.cuh"
#include "kvarn_internal.h"

namespace kvarn {

// Set by the self-check kernel when its wait gives up (always, unless the word was already set).
__device__ unsigned int g_selftest_error = 0;

namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        // one arrival (the barrier's whole count) with 16 bytes of pending transfer: the phase
        // stays open because no bulk copy is ever issued against it
        mbar_expect_tx(&bar, 16);
        mbar_wait_for(&bar, 0, &g_selftest_error, limit_ns);
    }
}

}  // namespace

cudaError_t launch_bounded_wait_check(uint32_t limit_us, cudaStream_t stream) {
    bounded_wait_kernel<<<1, 32, 0, stream>>>((uint64_t)limit_us * 1000ull);
    return cudaGetLastError();
}

cudaError_t read_and_clear_selftest_error(unsigned int* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_selftest_error, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace kvarn
