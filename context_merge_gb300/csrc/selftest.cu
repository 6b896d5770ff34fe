// Self-test of the failure path of the bounded device waits.
//
// Every kernel of the library that waits on an mbarrier does so for a bounded
// number of cycles; when a wait gives up it records (code, site, block) in
// the context's device status word and returns instead of hanging.  This
// entry point makes exactly that happen on purpose, safely: one warp waits
// for a phase of an mbarrier that nothing ever arrives on, with a short
// cycle limit, and returns.  No trap, fault or endless loop is involved, and
// the context stays usable afterwards.
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"
#include "tc_common.cuh"

namespace {

using namespace cpdr::tc;

constexpr int kSelftestSite = 99;

__global__ void wait_timeout_kernel(int32_t *status, long long limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    // phase 0 never completes: poll with the suspending wait until the limit
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(&bar, 0, 100000u)) return;   // cannot happen
        if (clock64() - t0 > limit) {
            if (atomicCAS(status, 0, 1) == 0) {
                status[1] = kSelftestSite;
                status[2] = (int32_t)blockIdx.x;
            }
            return;
        }
    }
}

}  // namespace

extern "C" cpdr_status cpdr_selftest_wait_timeout(const cpdr_ctx *c, long long max_cycles, void *stream) {
    if (!c) return cpdr::fail_with(CPDR_ERR_INVALID, "null context");
    if (!c->has_device) return cpdr::fail_with(CPDR_ERR_INVALID, "context was created with CPDR_FLAG_HOST_ONLY");
    if (max_cycles <= 0 || max_cycles > 4000000000LL)
        return cpdr::fail_with(CPDR_ERR_INVALID, "max_cycles must be in (0, 4e9]");
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(c->dev.status, max_cycles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cpdr::fail_with(CPDR_ERR_CUDA, std::string("cpdr_selftest_wait_timeout: ") +
                                                                  cudaGetErrorString(e));
    return CPDR_OK;
}
