// decode_common.cuh — pieces shared by the decode kernels: context clamping
// and the cross-partition log-sum-exp merge.
//
// Each CTA of a decode kernel owns one (sequence, kv head, partition) and
// produces, for each of the G query heads of that kv head, the partial
// softmax state of its tokens: the running max m (base-2 units), the sum
// l = sum_j 2^(x_j - m) and the normalised partial output o = sum_j
// 2^(x_j - m) v_j / l.  With one partition the CTA writes the output directly.
// Otherwise every CTA stores its partial in the workspace and takes a ticket;
// the CTA that takes the last ticket merges all partials of its (sequence,
// kv head) in partition order:
//     m* = max_i m_i,  w_i = l_i 2^(m_i - m*),  out = sum_i w_i o_i / sum_i w_i
// (online softmax: "PagedAttention学习笔记", 与 FlashAttention 的关系 names
// tiling and online softmax as the compatible kernel technique).  No CTA ever
// waits for another, so nothing can spin; the last CTA resets the ticket
// counter so the workspace is ready for the next call.
#pragma once

#include "pa_internal.cuh"

namespace pa {

// Effective context length of sequence s: clamped to what the grid and the
// block table can cover; clamping counts one error (reported by partition 0).
__device__ __forceinline__ int decode_context(const DecodeParams& p, int s, int split) {
    int L = p.context_lens[s];
    int cap = min(p.max_context_len, p.max_blocks_per_seq * p.block_size);
    if (L < 0 || L > cap) {
        if (split == 0 && threadIdx.x == 0) count_error(p.error_count);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

__device__ __forceinline__ size_t decode_unit(const DecodeParams& p, int s, int kvh) {
    return (size_t)s * p.num_kv_heads + kvh;
}

// Called by every thread of a CTA after it stored its partial (ws_o, ws_ml)
// for partition `split`.  If this CTA holds the last ticket it merges all
// `nsplit` partials into out.  `w_smem` must hold group * max_splits floats.
template <typename T>
__device__ void decode_merge_if_last(const DecodeParams& p, int s, int kvh, int nsplit, float* w_smem) {
    __shared__ int s_is_last;
    const size_t unit = decode_unit(p, s, kvh);
    __threadfence();  // make this CTA's partial visible device-wide before the ticket
    __syncthreads();
    if (threadIdx.x == 0) {
        int ticket = atomicAdd(&p.counters[unit], 1);
        s_is_last = (ticket == nsplit - 1);
    }
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();

    const int G = p.group, D = p.head_dim;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
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
    __syncthreads();
    const float* o = p.ws_o + unit * p.max_splits * G * D;
    T* out = static_cast<T*>(p.out) + ((size_t)s * p.num_q_heads + (size_t)kvh * G) * D;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        int g = idx / D;
        float acc = 0.f;
        for (int i = 0; i < nsplit; ++i) acc += w_smem[g * p.max_splits + i] * __ldcg(o + ((size_t)i * G) * D + idx);
        out[idx] = from_float<T>(acc);
    }
    if (threadIdx.x == 0) p.counters[unit] = 0;
}

}  // namespace pa
