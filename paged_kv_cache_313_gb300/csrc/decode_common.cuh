// decode_common.cuh — pieces shared by the decode kernels: context clamping
// and the cross-partition log-sum-exp merge.
//
// A decode work item is one (sequence, kv head, partition of the context).
// It produces, for each of the G query heads of that kv head, the partial
// softmax state of its tokens: the running max m (base-2 units), the sum
// l = sum_j 2^(x_j - m) and the normalised partial output o = sum_j
// 2^(x_j - m) v_j / l.  With one partition the item writes the output
// directly.  Otherwise every item stores its partial in the workspace and
// takes a ticket; the item that takes the last ticket merges all partials of
// its (sequence, kv head) in partition order:
//     m* = max_i m_i,  w_i = l_i 2^(m_i - m*),  out = sum_i w_i o_i / sum_i w_i
// (online softmax: "PagedAttention学习笔记", 与 FlashAttention 的关系 names
// tiling and online softmax as the compatible kernel technique).  No thread
// ever waits for another CTA, so nothing can spin; the merging item resets
// the ticket counter so the workspace is ready for the next call.
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

__device__ __forceinline__ size_t decode_unit(const DecodeParams& p, int s, int kvh) {
    return (size_t)s * p.num_kv_heads + kvh;
}

// Ticket + merge, executed by `nthreads` threads (thread index `tid`, warps
// `tid/32`) that synchronise with `bar()`.  Each participating thread must
// have finished storing this item's partial (ws_o, ws_ml) before the call.
// `w_smem` holds group * max_splits floats; `flag_smem` one int.
template <typename T, typename Barrier>
__device__ void decode_ticket_merge(const DecodeParams& p, int s, int kvh, int nsplit, float* w_smem,
                                    int* flag_smem, int tid, int nthreads, Barrier bar) {
    const size_t unit = decode_unit(p, s, kvh);
    __threadfence();  // make this item's partial visible device-wide before the ticket
    bar();
    if (tid == 0) {
        int ticket = atomicAdd(&p.counters[unit], 1);
        *flag_smem = (ticket == nsplit - 1);
    }
    bar();
    const bool last = *flag_smem != 0;
    if (last) {
        __threadfence();
        const int G = p.group, D = p.head_dim;
        const int warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;
        const float2* ml = p.ws_ml + unit * p.max_splits * G;
        for (int g = warp; g < G; g += nwarps) {
            float m = -INFINITY;
            for (int i = lane; i < nsplit; i += 32) {
                float2 v = __ldcg(ml + (size_t)i * G + g);
                if (v.y > 0.f) m = fmaxf(m, v.x);
            }
            m = warp_max(m);
            float wsum = 0.f;
            for (int i = lane; i < nsplit; i += 32) {
                float2 v = __ldcg(ml + (size_t)i * G + g);
                float w = (v.y > 0.f) ? v.y * exp2f(v.x - m) : 0.f;
                w_smem[g * p.max_splits + i] = w;
                wsum += w;
            }
            wsum = warp_sum(wsum);
            float inv = wsum > 0.f ? 1.f / wsum : 0.f;
            for (int i = lane; i < nsplit; i += 32) w_smem[g * p.max_splits + i] *= inv;
        }
        bar();
        const float* o = p.ws_o + unit * p.max_splits * G * D;
        T* out = static_cast<T*>(p.out) + ((size_t)s * p.num_q_heads + (size_t)kvh * G) * D;
        for (int idx = tid; idx < G * D; idx += nthreads) {
            int g = idx / D;
            float acc = 0.f;
            for (int i = 0; i < nsplit; ++i) acc += w_smem[g * p.max_splits + i] * __ldcg(o + ((size_t)i * G) * D + idx);
            out[idx] = from_float<T>(acc);
        }
        if (tid == 0) p.counters[unit] = 0;
    }
    bar();  // w_smem / flag_smem free for the next item
}

struct CtaBarrier {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Whole-CTA form used by the one-item-per-CTA kernels.
template <typename T>
__device__ void decode_merge_if_last(const DecodeParams& p, int s, int kvh, int nsplit, float* w_smem) {
    __shared__ int s_is_last;
    decode_ticket_merge<T>(p, s, kvh, nsplit, w_smem, &s_is_last, threadIdx.x, blockDim.x, CtaBarrier{});
}

}  // namespace pa
