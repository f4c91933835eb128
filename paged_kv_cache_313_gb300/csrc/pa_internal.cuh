// pa_internal.cuh — shared declarations of the libpa.so translation units:
// status plumbing, device properties, launch parameter structs and small
// device helpers.  Not part of the public ABI (that is include/pa.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------- host side
int set_cuda_error(cudaError_t e);  // records e for pa_last_cuda_error(), returns PA_ERR_CUDA
int check_launch();                 // PA_OK or PA_ERR_CUDA after a kernel launch
int check_device(int* num_sms);     // PA_OK on an sm_103 device (cached per device)
// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device (once per kernel and device).
int ensure_dynamic_smem(const void* kernel, size_t bytes);

// Programmatic dependent launch.  The hot-path kernels are launched with
// programmatic stream serialisation, so a kernel's launch and CTA start-up
// overlap the tail of the kernel before it on the stream.  Every such kernel
// executes pdl_wait() before its first global-memory access (the wait returns
// once the preceding grid has completed and its writes are visible, and at
// once when there is no programmatic predecessor) and pdl_trigger() at its
// start, which lets the next kernel begin launching.  Build with
// -DPA_USE_PDL=0 for plain launches.
#ifndef PA_USE_PDL
#define PA_USE_PDL 1
#endif

template <typename... KArgs, typename... Args>
int launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                  Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PA_USE_PDL ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    return e == cudaSuccess ? PA_OK : set_cuda_error(e);
}

inline int elem_size(int dtype) { return dtype == PA_F32 ? 4 : 2; }

// Shapes pa_decode takes: PA_OK, PA_ERR_INVALID_ARG (head counts that do not
// group) or PA_ERR_UNSUPPORTED (head_dim, block_size or group out of range).
int decode_shape_ok(int num_q_heads, int num_kv_heads, int head_dim, int block_size);

// Split-KV partition policy shared by pa_decode and pa_decode_workspace_size.
struct DecodePlan {
    int partition;        // tokens per split (multiple of 64)
    int max_splits;       // partial slots per (sequence, kv head): the most partitions any sequence can have
    int small_partition;  // the shorter partitions of the batch's last sequences (multiple of 64)
    int small_from;       // first sequence cut into small_partition-token partitions (num_seqs: none)
};
// `workspace_cap`: largest split-KV scratch the caller can offer (SIZE_MAX: any); `reserved`: partial slots
// per (sequence, kv head) used before the partitions' (the cascade's prefix slot); `fp8`: the plan of e4m3
// pools (pa_decode_fp8, pa_decode_write_fp8).
DecodePlan plan_decode(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_context_len,
                       int num_sms, size_t workspace_cap, int reserved = 0, bool fp8 = false);

// Workspace layout of pa_decode (byte offsets from the 256-aligned base).
struct DecodeWorkspace {
    size_t work;      // int32 [2]: the persistent decode kernel's work-queue counters
    size_t ml;        // float2 [num_seqs][num_kv_heads][max_splits][G]  (running max in log2 units, sum)
    size_t o;         // float  [num_seqs][num_kv_heads][max_splits][G][head_dim]
    size_t total;
};
DecodeWorkspace decode_workspace_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_splits);

struct DecodeParams {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* error_count;
    int* work;          // work[0]: next item, work[1]: finished CTAs (persistent kernel)
    float2* ws_ml;
    float* ws_o;
    // Cascade tail pass: sequence s attends only tokens [prefix_lens[s], L); the
    // shared prefix's partial sits in workspace slot 0 and the partitions'
    // partials from slot split_base = 1 on.  nullptr / 0 for plain decode.
    const int32_t* prefix_lens = nullptr;
    int split_base = 0;
    // Cascade prefix items: group g = sequences [group_offsets[g], group_offsets[g+1]) shares
    // prefix_lens[group_offsets[g]] leading tokens; the decode kernel reads them once per group.
    const int32_t* group_offsets = nullptr;
    int num_groups = 0;
    // Cascade (either prefix path): the groups again, for the merge kernel's check that every member maps the
    // first member's physical blocks over its shared prefix (a member that does not is counted in error_count).
    const int32_t* check_groups = nullptr;
    int check_num_groups = 0;
    // pa_decode_write: the newest token of each sequence (position L - 1) has its K and V rows in
    // k_new / v_new [num_seqs][num_kv_heads][head_dim]; the decode kernel writes them into the pools
    // (k_write / v_write = k_cache / v_cache) and attends with them; new_slots[s] gets the slot.
    const void* k_new = nullptr;
    const void* v_new = nullptr;
    void* k_write = nullptr;
    void* v_write = nullptr;
    int64_t* new_slots = nullptr;
    // fp8 pools: k_cache / v_cache hold e4m3 codes read back as code * k_scale / code * v_scale
    int kv_fp8 = 0;
    float k_scale = 1.f, v_scale = 1.f;
    // fp8 pools with a fused write (k_new set): the new rows are stored as e4m3(x * k_inv) / e4m3(x * v_inv),
    // the reciprocals computed in float on the host as the separate quantising write computes them
    float k_inv = 1.f, v_inv = 1.f;
    int num_seqs, num_q_heads, num_kv_heads, head_dim, group;
    int num_blocks, block_size, max_blocks_per_seq, max_context_len;
    int partition, max_splits;
    // Sequences s >= small_from are cut into small_partition-token partitions instead (the tensor-core
    // kernel's queue ends with them, so the last items handed out are short); 1 << 30: none.
    int small_partition = 0, small_from = 1 << 30;
    float scale_log2;  // scale * log2(e): scores are kept in base-2 units
};

struct PrefillParams {
    void* out;
    const void* q;
    const int32_t* cu_q_lens;
    const int32_t* q_start_pos;
    const int32_t* seq_of_chunk;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* error_count;
    int num_chunks, total_q, max_q_len, num_seqs;
    int num_q_heads, num_kv_heads, head_dim, group;
    int num_blocks, block_size, max_blocks_per_seq;
    float scale_log2;
    // Cascade prefix pass (pa_decode_cascade) when prefix_lens is set: chunk c
    // is the group of decode sequences [cu_q_lens[c], cu_q_lens[c+1]), whose
    // queries are those rows of q; every member attends keys [0, P) with
    // P = prefix_lens[first member], read through the first member's table,
    // and its partial (o, m, l) goes to slot 0 of part_o / part_ml (laid out
    // like the decode workspace, part_splits slots per (sequence, kv head))
    // instead of out.
    const int32_t* prefix_lens = nullptr;
    float* part_o = nullptr;
    float2* part_ml = nullptr;
    int part_splits = 0;
};

// Kernel launchers (defined in the .cu files).
int launch_prefill_fma(const PrefillParams& p, int dtype, cudaStream_t stream);
int launch_slot_mapping(const int32_t* block_tables, int num_seqs, int max_blocks_per_seq, const int32_t* seq_idx,
                        const int32_t* pos, int num_tokens, int block_size, int num_blocks, int64_t* slot_mapping,
                        int32_t* error_count, cudaStream_t stream);
int launch_write_kv(const void* k_new, const void* v_new, int num_tokens, int row_bytes, void* k_cache,
                    void* v_cache, long long num_slots, const int64_t* slot_mapping, int32_t* error_count,
                    cudaStream_t stream);
int launch_write_kv_paged(const void* k_new, const void* v_new, int num_tokens, int row_bytes, void* k_cache,
                          void* v_cache, const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                          const int32_t* seq_idx, const int32_t* pos, int block_size, int num_blocks,
                          int64_t* slot_mapping, int32_t* error_count, cudaStream_t stream);
int launch_write_kv_paged_fp8(const void* k_new, const void* v_new, int num_tokens, int row_elems, void* k_cache,
                              void* v_cache, const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                              const int32_t* seq_idx, const int32_t* pos, int block_size, int num_blocks,
                              int64_t* slot_mapping, float k_inv, float v_inv, int32_t* error_count,
                              cudaStream_t stream);
int launch_copy_blocks(void* k_cache, void* v_cache, int num_blocks, int block_size, int row_bytes,
                       const int32_t* src, const int32_t* dst, const int32_t* num_valid, int num_copies,
                       int32_t* error_count, cudaStream_t stream);
int launch_decode_fma(const DecodeParams& p, int dtype, cudaStream_t stream);
bool decode_tc_supported(const DecodeParams& p, int dtype);
int launch_decode_tc(const DecodeParams& p, int num_sms, cudaStream_t stream);
int launch_decode_merge(const DecodeParams& p, int dtype, int num_sms, cudaStream_t stream);
// The decode kernel for these parameters (tensor-core or FMA), then the
// split-KV merge when there is more than one partition.
int run_decode(const DecodeParams& p, int dtype, int num_sms, cudaStream_t stream);
bool prefill_tc_supported(const PrefillParams& p, int dtype);
int launch_prefill_tc(const PrefillParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- device side
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ float from_float<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);  // round to nearest even
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Two floats to their nearest e4m3 codes (ties to even, magnitudes beyond 448 held at 448), lo in the low byte.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Four bf16 values (two 32-bit words, element 0 in the low half of x.x) to four e4m3 codes of x * inv, the
// product rounded to float: the fp8 pools' stored form, code = e4m3(x * (1/scale)).
__device__ __forceinline__ uint32_t e4m3x4_of_bf16x4(uint2 x, float inv) {
    const uint16_t a = pack_e4m3x2(__fmul_rn(__uint_as_float(x.x << 16), inv),
                                   __fmul_rn(__uint_as_float(x.x & 0xFFFF0000u), inv));
    const uint16_t b = pack_e4m3x2(__fmul_rn(__uint_as_float(x.y << 16), inv),
                                   __fmul_rn(__uint_as_float(x.y & 0xFFFF0000u), inv));
    return (uint32_t)a | ((uint32_t)b << 16);
}

__device__ __forceinline__ void count_error(int32_t* error_count, int n = 1) {
    if (error_count != nullptr && n != 0) atomicAdd(error_count, n);
}

// Number of token partitions of a context of length L (>= 1 so that an empty
// context still has one owner that writes its zero output).
__device__ __forceinline__ int num_partitions(int L, int partition) {
    return L <= 0 ? 1 : (L + partition - 1) / partition;
}

}  // namespace pa
