// decode_noalloc.cu — pa_decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run decode: a
// host runtime with a fixed memory budget that forbids allocation after
// start-up, a plugin inside another framework's allocator, or code that runs
// where allocation would synchronise the device.  For them this entry point
// takes its split-KV scratch (partials and work-queue counters) from a fixed
// array in device global memory that belongs to the library itself.
//
// The array is file-scope and of fixed size (kNoAllocScratchBytes); every GPU
// that loads the library holds it until the process exits.  In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up once per device with cudaGetSymbolAddress, with that device current, on
// the first call made on that device, and cached.
#include <mutex>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB per device
constexpr int kMaxDevicesNoAlloc = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevicesNoAlloc] = {};

// Device address of g_decode_scratch on the current device (set up once per device).
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevicesNoAlloc) return PA_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess) return set_cuda_error(e);
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_decode_noalloc(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads,
                                 int head_dim, int dtype, const void* k_cache, const void* v_cache, int num_blocks,
                                 int block_size, const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int max_context_len, float scale,
                                 int32_t* error_count, void* stream) {
    if (num_seqs < 0 || num_blocks < 0 || max_blocks_per_seq < 0 || max_context_len < 0) return PA_ERR_INVALID_ARG;
    int rc = decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size);  // the shapes pa_decode takes
    if (rc != PA_OK) return rc;
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !context_lens || (max_blocks_per_seq > 0 && !block_tables))
        return PA_ERR_INVALID_ARG;
    int num_sms = 0;
    rc = check_device(&num_sms);
    if (rc != PA_OK) return rc;
    DecodePlan plan =
        plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, num_sms, kNoAllocScratchBytes);
    DecodeWorkspace lay = decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_splits);
    if (lay.total > kNoAllocScratchBytes) return PA_ERR_WORKSPACE;  // beyond the built-in 16 MiB
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != PA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(scratch);
    // The array keeps the previous call's contents: the work-queue counters must start at zero.
    cudaError_t e = cudaMemsetAsync(ws + lay.work, 0, 2 * sizeof(int), st);
    if (e != cudaSuccess) return set_cuda_error(e);
    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.error_count = error_count;
    p.work = reinterpret_cast<int*>(ws + lay.work);
    p.ws_ml = reinterpret_cast<float2*>(ws + lay.ml);
    p.ws_o = reinterpret_cast<float*>(ws + lay.o);
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.group = num_q_heads / num_kv_heads;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_context_len = max_context_len;
    p.partition = plan.partition;
    p.small_partition = plan.small_partition;
    p.small_from = plan.small_from;
    p.max_splits = plan.max_splits;
    p.scale_log2 = scale * 1.4426950408889634f;
    return run_decode(p, dtype, num_sms, st);
}
