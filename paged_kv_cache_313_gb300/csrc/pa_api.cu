// pa_api.cu — the C ABI of libpa.so: argument checks, device checks and
// dispatch to the kernels.  Every entry point validates on the host and
// launches nothing when a check fails.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <set>
#include <utility>

#include "pa_internal.cuh"

namespace pa {

static thread_local int g_last_cuda_error = 0;

int set_cuda_error(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return PA_ERR_CUDA;
}

int check_launch() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PA_OK : set_cuda_error(e);
}

namespace {
constexpr int kMaxDevices = 64;
struct DeviceInfo {
    int checked = 0;  // 0 unknown, 1 ok, -1 not sm_103
    int num_sms = 0;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_device_mutex;
}  // namespace

int check_device(int* num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_device_mutex);
    DeviceInfo& info = g_devices[dev];
    if (info.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return set_cuda_error(e);
        info.checked = (major == 10 && minor == 3) ? 1 : -1;
        info.num_sms = sms;
    }
    if (num_sms) *num_sms = info.num_sms;
    return info.checked == 1 ? PA_OK : PA_ERR_UNSUPPORTED_DEVICE;
}

int ensure_dynamic_smem(const void* kernel, size_t bytes) {
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e);
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kernel, dev})) return PA_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return set_cuda_error(e);
    done.insert({kernel, dev});
    return PA_OK;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

DecodeWorkspace decode_workspace_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_splits) {
    DecodeWorkspace w;
    size_t units = (size_t)num_seqs * num_kv_heads;
    size_t group = (size_t)(num_q_heads / num_kv_heads);
    w.work = 0;
    w.ml = 256;
    w.o = align_up(w.ml + units * max_splits * group * sizeof(float2), 256);
    w.total = align_up(w.o + units * max_splits * group * head_dim * sizeof(float), 256);
    return w;
}

// Items per SM below which decode partitions shrink from 512 to 256 and 128
// tokens (build-time knob; 0, the measured best, keeps 512 whenever the grid
// covers two waves: shorter items spend more of their time in the epilogue).
// Decode partition (tokens per work item) before any shrinking or growing: bf16 pools, and e4m3 pools (whose
// items carry two kv heads).  768 for bf16 measured against 512, 1024 (the e4m3 best) and 1280.
#ifndef PA_DECODE_PARTITION
#define PA_DECODE_PARTITION 768
#endif
#ifndef PA_DECODE_PARTITION_FP8
#define PA_DECODE_PARTITION_FP8 1024
#endif
#ifndef PA_DECODE_ITEMS_PER_SM
#define PA_DECODE_ITEMS_PER_SM 0
#endif
// Percentage of a batch's sequences, the last ones, cut into quarter-length partitions (0: none).  The
// tensor-core decode kernel hands out its items sequence by sequence, so these come last: when the queue runs
// dry each CTA holds a short item, and the CTAs finish closer together.
#ifndef PA_DECODE_SMALL_TAIL_PCT
#define PA_DECODE_SMALL_TAIL_PCT 20
#endif
// The most quarter-length items (counted at the longest context) per SM: bf16 pools, e4m3 pools.
#ifndef PA_DECODE_SMALL_TAIL_ITEMS
#define PA_DECODE_SMALL_TAIL_ITEMS 8
#endif
#ifndef PA_DECODE_SMALL_TAIL_ITEMS_FP8
#define PA_DECODE_SMALL_TAIL_ITEMS_FP8 12
#endif

DecodePlan plan_decode(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_context_len,
                       int num_sms, size_t workspace_cap, int reserved, bool fp8) {
    // Work items are (sequence, partition, kv head).  PA_DECODE_PARTITION-token
    // partitions (1024: measured against 512 and 2048, it halves the partials
    // a long context leaves to merge and is neutral elsewhere) keep each item's
    // stream of K/V long; shrink them while the batch would
    // give fewer than PA_DECODE_ITEMS_PER_SM items per SM (if set) and while
    // the grid would not cover two waves of the GPU; grow them so
    // that no (sequence, head) has more than 128 partials to merge and the
    // split-KV scratch fits `workspace_cap`.  The estimate uses the maximum
    // context for every sequence: the lengths themselves live on the device.
    auto items = [&](int part) {
        long long splits = ((long long)max_context_len + part - 1) / part;
        return (long long)num_seqs * num_kv_heads * (splits < 1 ? 1 : splits);
    };
    // (halving keeps a multiple of 64)
    auto half_of = [](int part) { return std::max(64, (part >> 1) & ~63); };
    int partition = fp8 ? PA_DECODE_PARTITION_FP8 : PA_DECODE_PARTITION;
    while (partition > 128 && items(partition) < (long long)PA_DECODE_ITEMS_PER_SM * num_sms) partition = half_of(partition);
    while (partition > 64 && items(partition) < 2LL * num_sms) partition = half_of(partition);
    auto splits_of = [&](int part) {
        int sp = (int)(((long long)max_context_len + part - 1) / part);
        return sp < 1 ? 1 : sp;
    };
    // the last sequences (PA_DECODE_SMALL_TAIL_PCT % of them, rounded up) use quarter-length partitions, as
    // long as their items, counted at the longest context, stay within four per resident CTA on bf16 pools
    // (six on e4m3 pools, whose longer items leave a coarser tail): a few long contexts cut small would add
    // more per-item work than the shorter tail saves
    auto small_of = [](int part) { return std::max(64, (part / 4) & ~63); };
    const long long small_items_per_seq = (long long)splits_of(small_of(partition)) * num_kv_heads;
    const long long small_cap = (fp8 ? PA_DECODE_SMALL_TAIL_ITEMS_FP8 : PA_DECODE_SMALL_TAIL_ITEMS) * (long long)num_sms;
    long long small_count = ((long long)num_seqs * PA_DECODE_SMALL_TAIL_PCT + 99) / 100;
    if (small_count * small_items_per_seq > small_cap) small_count = small_cap / small_items_per_seq;
    auto slots_of = [&](int part) {  // partial slots per (sequence, kv head)
        return reserved + (small_count > 0 ? splits_of(small_of(part)) : splits_of(part));
    };
    while (slots_of(partition) > 128 && partition < (1 << 29)) partition <<= 1;
    while (slots_of(partition) > 1 + reserved && partition < (1 << 29) &&
           decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, slots_of(partition)).total >
               workspace_cap)
        partition <<= 1;
    return DecodePlan{partition, slots_of(partition), small_count > 0 ? small_of(partition) : partition,
                      num_seqs - (int)small_count};
}

int run_decode(const DecodeParams& p, int dtype, int num_sms, cudaStream_t stream) {
    if (decode_tc_supported(p, dtype)) {
        const int rc = launch_decode_tc(p, num_sms, stream);
        return rc != PA_OK ? rc : launch_decode_merge(p, dtype, num_sms, stream);
    }
    // the CUDA-core kernel launches one CTA per (sequence, kv head, partition): uniform partitions (its
    // workspace, sized for the shorter ones, has room to spare)
    DecodeParams q = p;
    q.small_from = 1 << 30;
    const int rc = launch_decode_fma(q, dtype, stream);
    return rc != PA_OK ? rc : launch_decode_merge(q, dtype, num_sms, stream);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return 100; }

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3";
        default: return "unknown status";
    }
}

int pa_last_cuda_error(void) { return g_last_cuda_error; }

int pa_slot_mapping(const int32_t* block_tables, int num_seqs, int max_blocks_per_seq, const int32_t* seq_idx,
                    const int32_t* pos, int num_tokens, int block_size, int num_blocks, int64_t* slot_mapping,
                    int32_t* error_count, void* stream) {
    if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq < 0 || block_size < 1 || num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!seq_idx || !pos || !slot_mapping || (num_seqs > 0 && max_blocks_per_seq > 0 && !block_tables))
        return PA_ERR_INVALID_ARG;
    int rc = check_device(nullptr);
    if (rc != PA_OK) return rc;
    return launch_slot_mapping(block_tables, num_seqs, max_blocks_per_seq, seq_idx, pos, num_tokens, block_size,
                               num_blocks, slot_mapping, error_count, static_cast<cudaStream_t>(stream));
}

int pa_write_kv(const void* k_new, const void* v_new, int num_tokens, int num_kv_heads, int head_dim, int dtype,
                void* k_cache, void* v_cache, int num_blocks, int block_size, const int64_t* slot_mapping,
                int32_t* error_count, void* stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || num_blocks < 0 || block_size < 1)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    long long row_bytes = (long long)num_kv_heads * head_dim * elem_size(dtype);
    if (row_bytes % 16 != 0 || row_bytes > (1 << 20)) return PA_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_UNSUPPORTED;
    int rc = check_device(nullptr);
    if (rc != PA_OK) return rc;
    return launch_write_kv(k_new, v_new, num_tokens, (int)row_bytes, k_cache, v_cache,
                           (long long)num_blocks * block_size, slot_mapping, error_count,
                           static_cast<cudaStream_t>(stream));
}

int pa_write_kv_paged(const void* k_new, const void* v_new, int num_tokens, int num_kv_heads, int head_dim,
                      int dtype, void* k_cache, void* v_cache, int num_blocks, int block_size,
                      const int32_t* block_tables, int num_seqs, int max_blocks_per_seq, const int32_t* seq_idx,
                      const int32_t* pos, int64_t* slot_mapping, int32_t* error_count, void* stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || num_blocks < 0 || block_size < 1 || num_seqs < 0 ||
        max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !seq_idx || !pos ||
        (num_seqs > 0 && max_blocks_per_seq > 0 && !block_tables))
        return PA_ERR_INVALID_ARG;
    long long row_bytes = (long long)num_kv_heads * head_dim * elem_size(dtype);
    if (row_bytes % 16 != 0 || row_bytes > (1 << 20)) return PA_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_UNSUPPORTED;
    int rc = check_device(nullptr);
    if (rc != PA_OK) return rc;
    return launch_write_kv_paged(k_new, v_new, num_tokens, (int)row_bytes, k_cache, v_cache, block_tables, num_seqs,
                                 max_blocks_per_seq, seq_idx, pos, block_size, num_blocks, slot_mapping, error_count,
                                 static_cast<cudaStream_t>(stream));
}

int pa_write_kv_paged_fp8(const void* k_new, const void* v_new, int num_tokens, int num_kv_heads, int head_dim,
                          void* k_cache, void* v_cache, int num_blocks, int block_size, const int32_t* block_tables,
                          int num_seqs, int max_blocks_per_seq, const int32_t* seq_idx, const int32_t* pos,
                          int64_t* slot_mapping, float k_scale, float v_scale, int32_t* error_count, void* stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || num_blocks < 0 || block_size < 1 || num_seqs < 0 ||
        max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !seq_idx || !pos ||
        (num_seqs > 0 && max_blocks_per_seq > 0 && !block_tables))
        return PA_ERR_INVALID_ARG;
    const long long row = (long long)num_kv_heads * head_dim;  // elements; fp8 row bytes = row
    if (row % 16 != 0 || row > (1 << 20)) return PA_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_UNSUPPORTED;
    int rc = check_device(nullptr);
    if (rc != PA_OK) return rc;
    const float k_inv = 1.0f / k_scale, v_inv = 1.0f / v_scale;
    return launch_write_kv_paged_fp8(k_new, v_new, num_tokens, (int)row, k_cache, v_cache, block_tables, num_seqs,
                                     max_blocks_per_seq, seq_idx, pos, block_size, num_blocks, slot_mapping, k_inv,
                                     v_inv, error_count, static_cast<cudaStream_t>(stream));
}

int pa_copy_blocks(void* k_cache, void* v_cache, int num_blocks, int block_size, int num_kv_heads, int head_dim,
                   int dtype, const int32_t* src_blocks, const int32_t* dst_blocks, const int32_t* num_valid,
                   int num_copies, int32_t* error_count, void* stream) {
    if (num_copies < 0 || num_blocks < 0 || block_size < 1 || num_kv_heads < 1 || head_dim < 1)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_copies == 0) return PA_OK;
    if (!k_cache || !v_cache || !src_blocks || !dst_blocks || !num_valid) return PA_ERR_INVALID_ARG;
    long long row_bytes = (long long)num_kv_heads * head_dim * elem_size(dtype);
    if (row_bytes % 16 != 0 || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_UNSUPPORTED;
    int rc = check_device(nullptr);
    if (rc != PA_OK) return rc;
    return launch_copy_blocks(k_cache, v_cache, num_blocks, block_size, (int)row_bytes, src_blocks, dst_blocks,
                              num_valid, num_copies, error_count, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace pa {
int decode_shape_ok(int num_q_heads, int num_kv_heads, int head_dim, int block_size) {
    if (num_kv_heads < 1 || num_q_heads < num_kv_heads || num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (block_size < 1 || block_size > 1024) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}
}  // namespace pa

extern "C" {

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int max_context_len) {
    if (num_seqs < 0 || max_context_len < 0 || decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size))
        return 0;
    int num_sms = 0;
    if (check_device(&num_sms) != PA_OK) return 0;
    // enough for bf16 and for e4m3 pools, whose plans differ
    size_t total = 0;
    for (bool fp8 : {false, true}) {
        DecodePlan plan =
            plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, num_sms, SIZE_MAX, 0, fp8);
        total = std::max(total, decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_splits).total);
    }
    return total;
}

int pa_decode_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                   int max_context_len, int* partition, int* max_splits) {
    if (num_seqs < 0 || max_context_len < 0) return PA_ERR_INVALID_ARG;
    int rc = decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size);
    if (rc != PA_OK) return rc;
    int num_sms = 0;
    if ((rc = check_device(&num_sms)) != PA_OK) return rc;
    DecodePlan plan = plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, num_sms, SIZE_MAX);
    if (partition) *partition = plan.partition;
    if (max_splits) *max_splits = plan.max_splits;
    return PA_OK;
}

// Checks and parameters shared by pa_decode and pa_decode_write; *p is ready
// for run_decode when PA_OK is returned.
static int prepare_decode(DecodeParams* p, int* num_sms, void* out, const void* q, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int dtype, const void* k_cache, const void* v_cache,
                          int num_blocks, int block_size, const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int max_context_len, float scale, void* workspace,
                          size_t workspace_bytes, int32_t* error_count, bool fp8 = false) {
    if (num_seqs < 0 || num_blocks < 0 || max_blocks_per_seq < 0 || max_context_len < 0) return PA_ERR_INVALID_ARG;
    int rc = decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size);
    if (rc != PA_OK) return rc;
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_cache || !v_cache || !context_lens || (max_blocks_per_seq > 0 && !block_tables))
        return PA_ERR_INVALID_ARG;
    if ((rc = check_device(num_sms)) != PA_OK) return rc;
    DecodePlan plan =
        plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, *num_sms, SIZE_MAX, 0, fp8);
    DecodeWorkspace lay = decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_splits);
    if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PA_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    p->out = out;
    p->q = q;
    p->k_cache = k_cache;
    p->v_cache = v_cache;
    p->block_tables = block_tables;
    p->context_lens = context_lens;
    p->error_count = error_count;
    p->work = reinterpret_cast<int*>(ws + lay.work);
    p->ws_ml = reinterpret_cast<float2*>(ws + lay.ml);
    p->ws_o = reinterpret_cast<float*>(ws + lay.o);
    p->num_seqs = num_seqs;
    p->num_q_heads = num_q_heads;
    p->num_kv_heads = num_kv_heads;
    p->head_dim = head_dim;
    p->group = num_q_heads / num_kv_heads;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->max_blocks_per_seq = max_blocks_per_seq;
    p->max_context_len = max_context_len;
    p->partition = plan.partition;
    p->small_partition = plan.small_partition;
    p->small_from = plan.small_from;
    p->max_splits = plan.max_splits;
    p->scale_log2 = scale * 1.4426950408889634f;
    return PA_OK;
}

int pa_decode(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int dtype,
              const void* k_cache, const void* v_cache, int num_blocks, int block_size,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              int max_context_len, float scale, void* workspace, size_t workspace_bytes, int32_t* error_count,
              void* stream) {
    if (num_seqs == 0 && num_blocks >= 0 && max_blocks_per_seq >= 0 && max_context_len >= 0 &&
        decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size) == PA_OK &&
        (dtype == PA_F32 || dtype == PA_BF16))
        return PA_OK;
    DecodeParams p;
    int num_sms = 0;
    int rc = prepare_decode(&p, &num_sms, out, q, num_seqs, num_q_heads, num_kv_heads, head_dim, dtype, k_cache,
                            v_cache, num_blocks, block_size, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, scale, workspace, workspace_bytes, error_count);
    if (rc != PA_OK) return rc;
    return run_decode(p, dtype, num_sms, static_cast<cudaStream_t>(stream));
}

int pa_decode_fp8(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                  const void* k_cache, const void* v_cache, int num_blocks, int block_size,
                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                  int max_context_len, float scale, float k_scale, float v_scale, void* workspace,
                  size_t workspace_bytes, int32_t* error_count, void* stream) {
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 && num_blocks >= 0 && max_blocks_per_seq >= 0 && max_context_len >= 0 &&
        decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size) == PA_OK)
        return PA_OK;
    DecodeParams p;
    int num_sms = 0;
    int rc = prepare_decode(&p, &num_sms, out, q, num_seqs, num_q_heads, num_kv_heads, head_dim, PA_BF16, k_cache,
                            v_cache, num_blocks, block_size, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, scale, workspace, workspace_bytes, error_count, true);
    if (rc != PA_OK) return rc;
    p.kv_fp8 = 1;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    if (!decode_tc_supported(p, PA_BF16)) return PA_ERR_UNSUPPORTED;
    return run_decode(p, PA_BF16, num_sms, static_cast<cudaStream_t>(stream));
}

int pa_decode_write(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                    int dtype, void* k_cache, void* v_cache, int num_blocks, int block_size,
                    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                    int max_context_len, float scale, const void* k_new, const void* v_new, int64_t* new_slots,
                    void* workspace, size_t workspace_bytes, int32_t* error_count, void* stream) {
    if (num_seqs == 0 && num_blocks >= 0 && max_blocks_per_seq >= 0 && max_context_len >= 0 &&
        decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size) == PA_OK && dtype == PA_BF16)
        return PA_OK;
    if (dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (!k_new || !v_new) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return PA_ERR_UNSUPPORTED;
    DecodeParams p;
    int num_sms = 0;
    int rc = prepare_decode(&p, &num_sms, out, q, num_seqs, num_q_heads, num_kv_heads, head_dim, dtype, k_cache,
                            v_cache, num_blocks, block_size, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, scale, workspace, workspace_bytes, error_count);
    if (rc != PA_OK) return rc;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_write = k_cache;
    p.v_write = v_cache;
    p.new_slots = new_slots;
    if (!decode_tc_supported(p, dtype)) return PA_ERR_UNSUPPORTED;  // the fused write lives in the tensor-core kernel
    return run_decode(p, dtype, num_sms, static_cast<cudaStream_t>(stream));
}

int pa_decode_write_fp8(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        void* k_cache, void* v_cache, int num_blocks, int block_size, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, float scale,
                        float k_scale, float v_scale, const void* k_new, const void* v_new, int64_t* new_slots,
                        void* workspace, size_t workspace_bytes, int32_t* error_count, void* stream) {
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 && num_blocks >= 0 && max_blocks_per_seq >= 0 && max_context_len >= 0 &&
        decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size) == PA_OK)
        return PA_OK;
    if (!k_new || !v_new) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return PA_ERR_UNSUPPORTED;
    DecodeParams p;
    int num_sms = 0;
    int rc = prepare_decode(&p, &num_sms, out, q, num_seqs, num_q_heads, num_kv_heads, head_dim, PA_BF16, k_cache,
                            v_cache, num_blocks, block_size, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, scale, workspace, workspace_bytes, error_count, true);
    if (rc != PA_OK) return rc;
    p.kv_fp8 = 1;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.k_inv = 1.0f / k_scale;  // in float, as the separate quantising write computes it
    p.v_inv = 1.0f / v_scale;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_write = k_cache;
    p.v_write = v_cache;
    p.new_slots = new_slots;
    if (!decode_tc_supported(p, PA_BF16)) return PA_ERR_UNSUPPORTED;
    return run_decode(p, PA_BF16, num_sms, static_cast<cudaStream_t>(stream));
}

size_t pa_prefill_workspace_size(int num_chunks, int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size) {
    (void)num_chunks; (void)max_q_len; (void)num_q_heads; (void)num_kv_heads; (void)head_dim; (void)block_size;
    return 0;
}

int pa_prefill_chunk(void* out, const void* q, const int32_t* cu_q_lens, const int32_t* q_start_pos,
                     const int32_t* seq_of_chunk, int num_chunks, int total_q, int max_q_len, int num_seqs,
                     int num_q_heads, int num_kv_heads, int head_dim, int dtype, const void* k_cache,
                     const void* v_cache, int num_blocks, int block_size, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* context_lens, float scale, void* workspace,
                     size_t workspace_bytes, int32_t* error_count, void* stream) {
    (void)workspace; (void)workspace_bytes;
    if (num_chunks < 0 || total_q < 0 || max_q_len < 0 || num_seqs < 0 || num_blocks < 0 || max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    int rc = decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size);
    if (rc != PA_OK) return rc;
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_chunks == 0 || total_q == 0 || max_q_len == 0) return PA_OK;
    if (!out || !q || !cu_q_lens || !q_start_pos || !seq_of_chunk || !k_cache || !v_cache || !context_lens ||
        !block_tables || num_seqs == 0)
        return PA_ERR_INVALID_ARG;
    if ((rc = check_device(nullptr)) != PA_OK) return rc;
    PrefillParams p;
    p.out = out;
    p.q = q;
    p.cu_q_lens = cu_q_lens;
    p.q_start_pos = q_start_pos;
    p.seq_of_chunk = seq_of_chunk;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.error_count = error_count;
    p.num_chunks = num_chunks;
    p.total_q = total_q;
    p.max_q_len = max_q_len;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.group = num_q_heads / num_kv_heads;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.scale_log2 = scale * 1.4426950408889634f;
    if (prefill_tc_supported(p, dtype)) return launch_prefill_tc(p, static_cast<cudaStream_t>(stream));
    return launch_prefill_fma(p, dtype, static_cast<cudaStream_t>(stream));
}

// ---- cascade decode: shared prefixes read once per group

// 1: the decode kernel reads each group's prefix as one item of its queue
// (groups of at most 32 query rows); 0: the tensor-core prefill kernel's
// prefix mode reads them in a separate launch.
#ifndef PA_CASCADE_PREFIX_IN_DECODE
#define PA_CASCADE_PREFIX_IN_DECODE 1
#endif

// Plan of the cascade: the tail pass uses pa_decode's partitions, and slot 0 of
// every (sequence, kv head) holds the prefix partial, so max_splits grows by one.
static DecodePlan plan_cascade(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_context_len,
                               int num_sms) {
    return plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, num_sms, SIZE_MAX, 1);
}

size_t pa_decode_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                        int block_size, int max_context_len) {
    if (num_seqs < 0 || max_context_len < 0 || decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size))
        return 0;
    int num_sms = 0;
    if (check_device(&num_sms) != PA_OK) return 0;
    DecodePlan plan = plan_cascade(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, num_sms);
    return decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_splits).total;
}

int pa_decode_cascade(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                      int dtype, const void* k_cache, const void* v_cache, int num_blocks, int block_size,
                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                      int max_context_len, const int32_t* group_offsets, int num_groups, int max_group_size,
                      const int32_t* prefix_lens, float scale, void* workspace, size_t workspace_bytes,
                      int32_t* error_count, void* stream) {
    if (num_seqs < 0 || num_blocks < 0 || max_blocks_per_seq < 0 || max_context_len < 0 || num_groups < 0 ||
        max_group_size < 0)
        return PA_ERR_INVALID_ARG;
    int rc = decode_shape_ok(num_q_heads, num_kv_heads, head_dim, block_size);
    if (rc != PA_OK) return rc;
    if (dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !context_lens || !prefix_lens || !block_tables ||
        (num_groups > 0 && !group_offsets))
        return PA_ERR_INVALID_ARG;
    int num_sms = 0;
    if ((rc = check_device(&num_sms)) != PA_OK) return rc;
    DecodePlan plan = plan_cascade(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, num_sms);
    DecodeWorkspace lay = decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_splits);
    if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PA_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

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
    p.max_splits = plan.max_splits;
    p.small_partition = plan.small_partition;
    p.small_from = plan.small_from;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.prefix_lens = prefix_lens;
    p.split_base = 1;
    p.check_groups = num_groups > 0 ? group_offsets : nullptr;
    p.check_num_groups = num_groups;

    PrefillParams pp;
    pp.out = nullptr;
    pp.q = q;
    pp.cu_q_lens = group_offsets;
    pp.q_start_pos = nullptr;
    pp.seq_of_chunk = nullptr;
    pp.k_cache = k_cache;
    pp.v_cache = v_cache;
    pp.block_tables = block_tables;
    pp.context_lens = context_lens;
    pp.error_count = error_count;
    pp.num_chunks = num_groups;
    pp.total_q = num_seqs;
    pp.max_q_len = max_group_size;
    pp.num_seqs = num_seqs;
    pp.num_q_heads = num_q_heads;
    pp.num_kv_heads = num_kv_heads;
    pp.head_dim = head_dim;
    pp.group = p.group;
    pp.num_blocks = num_blocks;
    pp.block_size = block_size;
    pp.max_blocks_per_seq = max_blocks_per_seq;
    pp.scale_log2 = p.scale_log2;
    pp.prefix_lens = prefix_lens;
    pp.part_o = p.ws_o;
    pp.part_ml = p.ws_ml;
    pp.part_splits = plan.max_splits;
    if (!decode_tc_supported(p, dtype) || !prefill_tc_supported(pp, dtype)) return PA_ERR_UNSUPPORTED;

    // prefix pass (each group's shared prefix once, on the tensor cores), tail pass, merge
    if (PA_CASCADE_PREFIX_IN_DECODE && max_group_size * p.group <= 32) {
        // the shared prefixes are items of the decode kernel's own queue (one per group and kv head)
        p.group_offsets = group_offsets;
        p.num_groups = num_groups;
        return run_decode(p, dtype, num_sms, st);
    }
    if (num_groups > 0 && max_group_size > 0 && (rc = launch_prefill_tc(pp, st)) != PA_OK) return rc;
    return run_decode(p, dtype, num_sms, st);
}

}  // extern "C"
