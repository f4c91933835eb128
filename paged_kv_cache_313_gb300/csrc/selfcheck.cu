// selfcheck.cu — a check of the bounded mbarrier wait that every kernel of the
// library relies on to terminate.
//
// One warp initialises an mbarrier expecting one arrival and, unless asked to
// arrive first, waits on it with a caller-given poll limit while nothing ever
// arrives: the wait must give up, report false and count an error, and the
// kernel must return normally (the context stays usable).  With the arrival
// the same wait must succeed.  Nothing here faults, traps or spins without a
// bound.
#include "pa_internal.cuh"
#include "sm100_ptx.cuh"

namespace pa {
namespace {

__global__ void bounded_wait_check_kernel(uint32_t polls, int arrive, int32_t* result, int32_t* error_count) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    __syncthreads();
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar, 0, polls)) != 0;
    if (threadIdx.x == 0) {
        result[0] = ok ? 1 : 0;
        if (!ok) count_error(error_count);
    }
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_check_bounded_wait(int polls, int arrive, int32_t* result, int32_t* error_count, void* stream) {
    if (polls < 1 || polls > (1 << 16) || !result) return PA_ERR_INVALID_ARG;
    int rc = check_device(nullptr);
    if (rc != PA_OK) return rc;
    bounded_wait_check_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint32_t)polls, arrive ? 1 : 0,
                                                                              result, error_count);
    return check_launch();
}
