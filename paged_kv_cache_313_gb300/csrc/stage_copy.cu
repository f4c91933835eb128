// stage_copy.cu — moving a serving step's packed inputs in and outputs out.
//
// A decode step carries about a megabyte of per-step inputs (queries, the new
// tokens' K/V, block tables, lengths) and half as much output.  On GB300 the
// Grace CPU and the GPU share a coherent link, and page-locked host memory is
// mapped into the device's address space, so a kernel can read or write it
// directly.  For transfers this small a copy kernel finishes sooner than the
// copy engine (whose start-up latency dominates), and it is captured into the
// same CUDA graph as the step's kernels, so a served step is one graph launch.
#include "pa_internal.cuh"

namespace pa {
namespace {

// Each thread moves four 16-byte vectors per round, loads first, so that four
// reads per thread are in flight across the link at once.
__global__ void stage_copy_kernel(int4* __restrict__ dst, const int4* __restrict__ src, size_t n16) {
    pdl_trigger();
    pdl_wait();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        int4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = src[i + k * stride];
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[i + k * stride] = v[k];
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

// Device-accessible memory: device, managed, or page-locked host memory.
bool device_accessible(const void* ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the error so that a later call does not report it
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
           (a.type == cudaMemoryTypeHost && a.devicePointer == ptr);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_stage_copy(void* dst, const void* src, size_t bytes, void* stream) {
    if (bytes == 0) return PA_OK;
    if (!dst || !src) return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) || (reinterpret_cast<uintptr_t>(src) & 15u) || (bytes & 15u))
        return PA_ERR_INVALID_ARG;
    int num_sms = 0;
    int rc = check_device(&num_sms);
    if (rc != PA_OK) return rc;
    if (!device_accessible(dst) || !device_accessible(src)) return PA_ERR_INVALID_ARG;
    const size_t n16 = bytes / 16;
    const size_t want = (n16 + 255) / 256;
    const int grid = (int)(want < (size_t)num_sms * 4 ? want : (size_t)num_sms * 4);
    return launch_kernel(stage_copy_kernel, dim3(grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
                         static_cast<int4*>(dst), static_cast<const int4*>(src), n16);
}
