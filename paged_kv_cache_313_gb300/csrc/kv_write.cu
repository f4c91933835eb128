// kv_write.cu — the write side of the paged cache: slot mapping, the slot-
// mapped K/V scatter and the copy-on-write block copy.
//
// Slot mapping follows "PagedAttention学习笔记", 代码实现部分 › BlockTable
// (compute_slot_mapping): slot = block_table[seq][pos / B] * B + pos % B, -1 for
// tokens that are not written.  The scatter follows "KV cache 显存管理：为什么
// PagedAttention 是 vLLM 的核心", 对 ModelRunner 的影响 (the slot says where the
// current token's K/V goes).  The block copy follows "什么是 PagedAttention？",
// 共享但不污染状态 (copy the valid entries of a shared partial block).
//
// All three are pure data movement: HBM-bound, 16-byte vector accesses, no
// shared-memory staging needed since every byte is touched exactly once.
#include "pa_internal.cuh"

namespace pa {
namespace {

// Slot of new token t, -1 when it is not written (pos < 0) or when its
// sequence, logical block or table entry is out of range (counted).
__device__ __forceinline__ long long slot_of(const int32_t* __restrict__ block_tables, int num_seqs,
                                             int max_blocks_per_seq, const int32_t* __restrict__ seq_idx,
                                             const int32_t* __restrict__ pos, int t, int block_size, int num_blocks,
                                             int32_t* error_count) {
    const int p = pos[t];
    if (p < 0) return -1;
    const int s = seq_idx[t];
    const int logical_block = p / block_size;
    const int offset = p - logical_block * block_size;
    if (s >= 0 && s < num_seqs && logical_block < max_blocks_per_seq) {
        const int physical = block_tables[(long long)s * max_blocks_per_seq + logical_block];
        if (physical >= 0 && physical < num_blocks) return (long long)physical * block_size + offset;
    }
    count_error(error_count);
    return -1;
}

__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables, int num_seqs, int max_blocks_per_seq,
                                    const int32_t* __restrict__ seq_idx, const int32_t* __restrict__ pos,
                                    int num_tokens, int block_size, int num_blocks, int64_t* __restrict__ slots,
                                    int32_t* error_count) {
    pdl_trigger();
    pdl_wait();
    int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= num_tokens) return;
    slots[t] = slot_of(block_tables, num_seqs, max_blocks_per_seq, seq_idx, pos, t, block_size, num_blocks,
                       error_count);
}

// Slot mapping and K/V scatter in one launch: one CTA per token; thread 0
// resolves the slot (and records it when `slots` is given), then the CTA
// copies the token's K and V rows with 16-byte accesses.
__global__ void write_kv_paged_kernel(const int4* __restrict__ k_new, const int4* __restrict__ v_new, int row_vecs,
                                      int4* __restrict__ k_cache, int4* __restrict__ v_cache,
                                      const int32_t* __restrict__ block_tables, int num_seqs,
                                      int max_blocks_per_seq, const int32_t* __restrict__ seq_idx,
                                      const int32_t* __restrict__ pos, int block_size, int num_blocks,
                                      int64_t* __restrict__ slots, int32_t* error_count) {
    pdl_trigger();
    pdl_wait();
    __shared__ long long s_slot;
    const int t = blockIdx.x;
    if (threadIdx.x == 0) {
        s_slot = slot_of(block_tables, num_seqs, max_blocks_per_seq, seq_idx, pos, t, block_size, num_blocks,
                         error_count);
        if (slots) slots[t] = s_slot;
    }
    __syncthreads();
    const long long slot = s_slot;
    if (slot < 0) return;
    const int4* ks = k_new + (long long)t * row_vecs;
    const int4* vs = v_new + (long long)t * row_vecs;
    int4* kd = k_cache + slot * row_vecs;
    int4* vd = v_cache + slot * row_vecs;
    for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) {
        int4 k = __ldg(ks + i);
        int4 v = __ldg(vs + i);
        kd[i] = k;
        vd[i] = v;
    }
}

// One CTA per token: its K row and V row (row_bytes each, a multiple of 16)
// are copied with 16-byte loads and stores.
__global__ void write_kv_kernel(const int4* __restrict__ k_new, const int4* __restrict__ v_new, int row_vecs,
                                int4* __restrict__ k_cache, int4* __restrict__ v_cache, long long num_slots,
                                const int64_t* __restrict__ slots, int32_t* error_count) {
    pdl_trigger();
    pdl_wait();
    int t = blockIdx.x;
    long long slot = slots[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0) count_error(error_count);
        return;
    }
    const int4* ks = k_new + (long long)t * row_vecs;
    const int4* vs = v_new + (long long)t * row_vecs;
    int4* kd = k_cache + slot * row_vecs;
    int4* vd = v_cache + slot * row_vecs;
    for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) {
        int4 k = __ldg(ks + i);
        int4 v = __ldg(vs + i);
        kd[i] = k;
        vd[i] = v;
    }
}

// pa_write_kv_paged_fp8: slot mapping, then each bf16 element x of the token's
// K and V rows stored as e4m3(x * inv_scale) into uint8 pools.  One CTA per
// token; a thread converts eight elements (16 bytes in, 8 bytes out).
__global__ void write_kv_paged_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                          int row_vec8, uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                                          const int32_t* __restrict__ block_tables, int num_seqs,
                                          int max_blocks_per_seq, const int32_t* __restrict__ seq_idx,
                                          const int32_t* __restrict__ pos, int block_size, int num_blocks,
                                          int64_t* __restrict__ slots, float k_inv, float v_inv,
                                          int32_t* error_count) {
    pdl_trigger();
    pdl_wait();
    __shared__ long long s_slot;
    const int t = blockIdx.x;
    if (threadIdx.x == 0) {
        s_slot = slot_of(block_tables, num_seqs, max_blocks_per_seq, seq_idx, pos, t, block_size, num_blocks,
                         error_count);
        if (slots) slots[t] = s_slot;
    }
    __syncthreads();
    const long long slot = s_slot;
    if (slot < 0) return;
    for (int i = threadIdx.x; i < 2 * row_vec8; i += blockDim.x) {
        const bool isv = i >= row_vec8;
        const int j = isv ? i - row_vec8 : i;
        const uint4 x = isv ? __ldg(v_new + (long long)t * row_vec8 + j) : __ldg(k_new + (long long)t * row_vec8 + j);
        const float inv = isv ? v_inv : k_inv;
        const uint2 out = make_uint2(e4m3x4_of_bf16x4(make_uint2(x.x, x.y), inv),
                                     e4m3x4_of_bf16x4(make_uint2(x.z, x.w), inv));
        (isv ? v_cache : k_cache)[slot * row_vec8 + j] = out;
    }
}

// One CTA per copy: num_valid token rows of the source block, both pools.
__global__ void copy_blocks_kernel(int4* __restrict__ k_cache, int4* __restrict__ v_cache, int num_blocks,
                                   int block_size, int row_vecs, const int32_t* __restrict__ src,
                                   const int32_t* __restrict__ dst, const int32_t* __restrict__ num_valid,
                                   int32_t* error_count) {
    int c = blockIdx.x;
    int s = src[c], d = dst[c], n = num_valid[c];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks || n < 0 || n > block_size) {
        if (threadIdx.x == 0) count_error(error_count);
        return;
    }
    long long block_vecs = (long long)block_size * row_vecs;
    long long count = (long long)n * row_vecs;
    const int4* ks = k_cache + s * block_vecs;
    const int4* vs = v_cache + s * block_vecs;
    int4* kd = k_cache + d * block_vecs;
    int4* vd = v_cache + d * block_vecs;
    for (long long i = threadIdx.x; i < count; i += blockDim.x) {
        kd[i] = ks[i];
        vd[i] = vs[i];
    }
}

}  // namespace

int launch_slot_mapping(const int32_t* block_tables, int num_seqs, int max_blocks_per_seq, const int32_t* seq_idx,
                        const int32_t* pos, int num_tokens, int block_size, int num_blocks, int64_t* slot_mapping,
                        int32_t* error_count, cudaStream_t stream) {
    const int threads = 256;
    return launch_kernel(slot_mapping_kernel, dim3((num_tokens + threads - 1) / threads), dim3(threads), 0, stream,
                         block_tables, num_seqs, max_blocks_per_seq, seq_idx, pos, num_tokens, block_size,
                         num_blocks, slot_mapping, error_count);
}

int launch_write_kv(const void* k_new, const void* v_new, int num_tokens, int row_bytes, void* k_cache,
                    void* v_cache, long long num_slots, const int64_t* slot_mapping, int32_t* error_count,
                    cudaStream_t stream) {
    int row_vecs = row_bytes / 16;
    int threads = row_vecs >= 256 ? 256 : ((row_vecs + 31) / 32) * 32;
    return launch_kernel(write_kv_kernel, dim3(num_tokens), dim3(threads), 0, stream,
                         static_cast<const int4*>(k_new), static_cast<const int4*>(v_new), row_vecs,
                         static_cast<int4*>(k_cache), static_cast<int4*>(v_cache), num_slots, slot_mapping,
                         error_count);
}

int launch_write_kv_paged(const void* k_new, const void* v_new, int num_tokens, int row_bytes, void* k_cache,
                          void* v_cache, const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                          const int32_t* seq_idx, const int32_t* pos, int block_size, int num_blocks,
                          int64_t* slot_mapping, int32_t* error_count, cudaStream_t stream) {
    int row_vecs = row_bytes / 16;
    int threads = row_vecs >= 256 ? 256 : ((row_vecs + 31) / 32) * 32;
    return launch_kernel(write_kv_paged_kernel, dim3(num_tokens), dim3(threads), 0, stream,
                         static_cast<const int4*>(k_new), static_cast<const int4*>(v_new), row_vecs,
                         static_cast<int4*>(k_cache), static_cast<int4*>(v_cache), block_tables, num_seqs,
                         max_blocks_per_seq, seq_idx, pos, block_size, num_blocks, slot_mapping, error_count);
}

int launch_write_kv_paged_fp8(const void* k_new, const void* v_new, int num_tokens, int row_elems, void* k_cache,
                              void* v_cache, const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                              const int32_t* seq_idx, const int32_t* pos, int block_size, int num_blocks,
                              int64_t* slot_mapping, float k_inv, float v_inv, int32_t* error_count,
                              cudaStream_t stream) {
    const int row_vec8 = row_elems / 8;
    const int threads = 2 * row_vec8 >= 256 ? 256 : ((2 * row_vec8 + 31) / 32) * 32;
    return launch_kernel(write_kv_paged_fp8_kernel, dim3(num_tokens), dim3(threads), 0, stream,
                         static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), row_vec8,
                         static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), block_tables, num_seqs,
                         max_blocks_per_seq, seq_idx, pos, block_size, num_blocks, slot_mapping, k_inv, v_inv,
                         error_count);
}

int launch_copy_blocks(void* k_cache, void* v_cache, int num_blocks, int block_size, int row_bytes,
                       const int32_t* src, const int32_t* dst, const int32_t* num_valid, int num_copies,
                       int32_t* error_count, cudaStream_t stream) {
    copy_blocks_kernel<<<num_copies, 256, 0, stream>>>(static_cast<int4*>(k_cache), static_cast<int4*>(v_cache),
                                                       num_blocks, block_size, row_bytes / 16, src, dst, num_valid,
                                                       error_count);
    return check_launch();
}

}  // namespace pa
