// decode_common.cuh — pieces shared by the decode kernels.
//
// A decode work item is one (sequence, kv head, partition of the context).
// It produces, for each of the G query heads of that kv head, the partial
// softmax state of its tokens: the running max m (base-2 units), the sum
// l = sum_j 2^(x_j - m) and the normalised partial output o = sum_j
// 2^(x_j - m) v_j / l.  With one partition the item writes the output
// directly; otherwise it stores its partial in the workspace and
// decode_merge.cu combines the partials of each (sequence, query head) after
// the decode kernel (online softmax: "PagedAttention学习笔记", 与
// FlashAttention 的关系 names tiling and online softmax as the compatible
// kernel technique).
#pragma once

#include "pa_internal.cuh"

namespace pa {

// Effective context length of sequence s: clamped to what the grid and the
// block table can cover; clamping counts one error when `report` is set.
__device__ __forceinline__ int decode_context(const DecodeParams& p, int s, bool report) {
    int L = p.context_lens[s];
    int cap = min(p.max_context_len, p.max_blocks_per_seq * p.block_size);
    if (L < 0 || L > cap) {
        if (report) count_error(p.error_count);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// Decode range of sequence s (context L): tokens [*prefix, L) where *prefix is
// the cascade prefix length (0 without one), clamped to [0, L).  Returns the
// first token of partition 0, *prefix rounded down to a multiple of 64 so that
// partitions stay block aligned; tokens below *prefix are masked.
__device__ __forceinline__ int decode_start(const DecodeParams& p, int s, int L, int* prefix) {
    int pre = p.prefix_lens ? p.prefix_lens[s] : 0;
    pre = pre < 0 ? 0 : (pre > L ? L : pre);
    *prefix = pre;
    return pre & ~63;
}

// Tokens per partition of sequence s: the batch's last sequences (from small_from on) use shorter ones.
__device__ __forceinline__ int partition_of(const DecodeParams& p, int s) {
    return s >= p.small_from ? p.small_partition : p.partition;
}

__device__ __forceinline__ size_t decode_unit(const DecodeParams& p, int s, int kvh) {
    return (size_t)s * p.num_kv_heads + kvh;
}

}  // namespace pa
