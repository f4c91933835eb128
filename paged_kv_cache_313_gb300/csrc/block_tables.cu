// block_tables.cu — kernel-side block tables for a block manager whose
// blocks are larger than the kernels' ("PagedAttention学习笔记", 代码实现部分 ›
// 块表与槽位映射, 混合块: map_to_kernel_blocks splits one manager block into
// several kernel blocks).
//
// A manager block of ratio * B tokens occupies the same memory as `ratio`
// consecutive kernel blocks of B tokens (the pool [P][ratio*B][Hkv][D] is the
// pool [P*ratio][B][Hkv][D]), so manager block m is kernel blocks m*ratio ..
// m*ratio + ratio - 1 and every slot is unchanged.  One thread per kernel
// table entry.
#include "pa_internal.cuh"

namespace pa {
namespace {

__global__ void map_to_kernel_blocks_kernel(const int32_t* __restrict__ mgr, int num_seqs, int mgr_width,
                                            int ratio, int32_t* __restrict__ kernel_tables, int kernel_width) {
    pdl_trigger();
    pdl_wait();
    const long long total = (long long)num_seqs * kernel_width;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long s = i / kernel_width;
        const int j = (int)(i - s * kernel_width);
        const int m = j / ratio;
        int32_t entry = -1;
        if (m < mgr_width) {
            const int32_t mb = mgr[s * mgr_width + m];
            if (mb >= 0) entry = mb * ratio + (j - m * ratio);
        }
        kernel_tables[i] = entry;
    }
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_map_to_kernel_blocks(const int32_t* mgr_tables, int num_seqs, int mgr_width, int ratio,
                                       int32_t* kernel_tables, int kernel_width, void* stream) {
    if (num_seqs < 0 || mgr_width < 0 || kernel_width < 0 || ratio < 1) return PA_ERR_INVALID_ARG;
    if ((long long)mgr_width * ratio > (1LL << 30)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || kernel_width == 0) return PA_OK;
    if (!kernel_tables || (mgr_width > 0 && !mgr_tables)) return PA_ERR_INVALID_ARG;
    int num_sms = 0;
    int rc = check_device(&num_sms);
    if (rc != PA_OK) return rc;
    const long long total = (long long)num_seqs * kernel_width;
    const long long want = (total + 255) / 256;
    const int grid = (int)(want < 4LL * num_sms ? want : 4LL * num_sms);
    return launch_kernel(map_to_kernel_blocks_kernel, dim3(grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
                         mgr_tables, num_seqs, mgr_width, ratio, kernel_tables, kernel_width);
}
