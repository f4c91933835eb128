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
constexpr int kMergeUnroll = 4;

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
            // nsplit <= 128 (both decode kernels refuse more): four (m, l) pairs per lane, loaded at once
            float2 v[4];
            float m = -INFINITY;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = lane + 32 * k;
                v[k] = i < nsplit ? __ldcg(ml + (size_t)i * G + g) : make_float2(-INFINITY, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (v[k].y > 0.f) m = fmaxf(m, v[k].x);
            m = warp_max(m);
            float w[4], wsum = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                w[k] = (v[k].y > 0.f) ? v[k].y * exp2f(v[k].x - m) : 0.f;
                wsum += w[k];
            }
            wsum = warp_sum(wsum);
            const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (lane + 32 * k < nsplit) w_smem[g * p.max_splits + lane + 32 * k] = w[k] * inv;
        }
        bar();
        // out = sum_i w_i o_i over the partials in partition order: four
        // columns per float4, two float4 columns per thread and kMergeUnroll
        // splits per round, all of whose loads are in flight together (a
        // dependent load per split would make the merge of a long context the
        // launch's critical path)
        const float4* o = reinterpret_cast<const float4*>(p.ws_o + unit * p.max_splits * G * D);
        const int cols4 = G * D / 4;  // float4 columns of one partial
        T* out = static_cast<T*>(p.out) + ((size_t)s * p.num_q_heads + (size_t)kvh * G) * D;
        for (int c0 = tid; c0 < cols4; c0 += 2 * nthreads) {
            const int c1 = c0 + nthreads < cols4 ? c0 + nthreads : c0;  // a duplicate column is never stored
            const float* w0 = w_smem + (c0 * 4 / D) * p.max_splits;
            const float* w1 = w_smem + (c1 * 4 / D) * p.max_splits;
            float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
            for (int i = 0; i < nsplit; i += kMergeUnroll) {
                const int n = nsplit - i < kMergeUnroll ? nsplit - i : kMergeUnroll;
                float4 v0[kMergeUnroll], v1[kMergeUnroll];
#pragma unroll
                for (int u = 0; u < kMergeUnroll; ++u) {
                    if (u < n) {
                        v0[u] = __ldcg(o + (size_t)(i + u) * cols4 + c0);
                        v1[u] = __ldcg(o + (size_t)(i + u) * cols4 + c1);
                    }
                }
#pragma unroll
                for (int u = 0; u < kMergeUnroll; ++u) {
                    if (u < n) {
                        const float a = w0[i + u], b = w1[i + u];
                        acc0.x = fmaf(a, v0[u].x, acc0.x);
                        acc0.y = fmaf(a, v0[u].y, acc0.y);
                        acc0.z = fmaf(a, v0[u].z, acc0.z);
                        acc0.w = fmaf(a, v0[u].w, acc0.w);
                        acc1.x = fmaf(b, v1[u].x, acc1.x);
                        acc1.y = fmaf(b, v1[u].y, acc1.y);
                        acc1.z = fmaf(b, v1[u].z, acc1.z);
                        acc1.w = fmaf(b, v1[u].w, acc1.w);
                    }
                }
            }
            out[c0 * 4 + 0] = from_float<T>(acc0.x);
            out[c0 * 4 + 1] = from_float<T>(acc0.y);
            out[c0 * 4 + 2] = from_float<T>(acc0.z);
            out[c0 * 4 + 3] = from_float<T>(acc0.w);
            if (c1 != c0) {
                out[c1 * 4 + 0] = from_float<T>(acc1.x);
                out[c1 * 4 + 1] = from_float<T>(acc1.y);
                out[c1 * 4 + 2] = from_float<T>(acc1.z);
                out[c1 * 4 + 3] = from_float<T>(acc1.w);
            }
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
