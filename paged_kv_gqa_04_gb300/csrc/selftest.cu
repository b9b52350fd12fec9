// selftest.cu -- self-test of the bounded waits that every kernel of the
// library uses, run as a call of its own (no data, no copies, no tensor
// memory).
//
// One CTA of two warps and two mbarriers on which nothing ever arrives.
// Warp 0 waits with mbar_wait_bounded (limit limit_ns) and must give up: it
// sets PKV_FLAG_WAIT_TIMEOUT and the CTA's abort flag. Warp 1 waits with
// mbar_wait_or_abort and a limit 100 times longer, so it must stop because
// of the abort flag, soon after warp 0. Each warp's waiting time goes to
// elapsed_ns[warp]. Both waits end by construction (the global timer
// bounds them), so the call cannot hang the GPU.
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

__global__ void __launch_bounds__(64, 1) selftest_wait_kernel(uint64_t limit_ns, int32_t* err, uint64_t* elapsed_ns) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int* ab = &abort_flag;
    const uint64_t t0 = global_ns();
    if (warp == 0) {
        const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars[0]), 0, limit_ns));
        if (!got && lane == 0) {
            *ab = 1;
            flag_error(err, PKV_FLAG_WAIT_TIMEOUT);
        }
    } else {
        (void)__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&bars[1]), 0, ab, 100 * limit_ns));
    }
    if (lane == 0) elapsed_ns[warp] = global_ns() - t0;
    __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t limit_ns, int32_t* err, uint64_t* elapsed_ns, cudaStream_t s) {
    selftest_wait_kernel<<<1, 64, 0, s>>>(limit_ns, err, elapsed_ns);
    return cudaGetLastError();
}

}  // namespace pkv
