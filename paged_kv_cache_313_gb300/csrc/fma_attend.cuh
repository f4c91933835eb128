// fma_attend.cuh — the CUDA-core attention loop shared by the fp32 decode
// kernel and the CUDA-core prefill kernel.
//
// A CTA of kFmaThreads threads attends the G query heads of one kv head over
// the tokens [j0, j1) of one sequence.  Tokens are walked in sub-chunks of
// kFmaSub: the sub-chunk's block-table entries are resolved once ("KV cache
// 显存管理…", PagedAttention 改变了什么: token -> logical block -> physical block
// -> offset -> address), scores are computed one warp per token (lanes across
// head_dim), and an online-softmax state is carried across sub-chunks:
//     m' = max(m, max_j x_j),  l' = l 2^(m-m') + sum_j 2^(x_j-m'),
//     acc' = acc 2^(m-m') + sum_j 2^(x_j-m') v_j
// with x_j = scale*log2(e) * q.k_j (base-2 units).
#pragma once

#include "pa_internal.cuh"

namespace pa {

constexpr int kFmaThreads = 128;
constexpr int kFmaSub = 256;     // tokens per sub-chunk
constexpr int kFmaMaxGroup = 16; // query heads per kv head

template <int D>
struct FmaShape {
    static constexpr int kItems = kFmaMaxGroup * D / kFmaThreads;  // (g, d) outputs per thread (upper bound)
    static constexpr int kPerLane = D / 32;
    // dynamic shared memory: q [16][D], p [16][kSub], blocks [kSub+1]
    static constexpr size_t kSmemBytes =
        sizeof(float) * (kFmaMaxGroup * D + kFmaMaxGroup * kFmaSub) + sizeof(int) * (kFmaSub + 1);
    __device__ static float* q_s(float* smem) { return smem; }
    __device__ static float* p_s(float* smem) { return smem + kFmaMaxGroup * D; }
    __device__ static int* blk_s(float* smem) {
        return reinterpret_cast<int*>(smem + kFmaMaxGroup * D + kFmaMaxGroup * kFmaSub);
    }
};

// Attend q (G rows of D, storage type T) to tokens [j0, j1).  On return (after
// a __syncthreads) m_s[g], l_s[g] hold the softmax state and acc[it] the
// unnormalised output of item threadIdx.x + it*kFmaThreads = g*D + d.
template <typename T, int D>
__device__ void fma_attend(const T* __restrict__ q, int G, const T* __restrict__ kc, const T* __restrict__ vc,
                           const int32_t* __restrict__ table, int block_size, int num_kv_heads, int kvh,
                           int num_blocks, int j0, int j1, float scale_log2, int32_t* error_count, float* smem,
                           float (&acc)[FmaShape<D>::kItems], float* m_s, float* l_s, float* alpha_s) {
    using S = FmaShape<D>;
    constexpr int kPerLane = S::kPerLane;
    float* q_s = S::q_s(smem);
    float* p_s = S::p_s(smem);
    int* blk_s = S::blk_s(smem);
    const int B = block_size, Hkv = num_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < G * D; i += kFmaThreads) q_s[i] = to_float(q[i]);
    if (threadIdx.x < kFmaMaxGroup) { m_s[threadIdx.x] = -INFINITY; l_s[threadIdx.x] = 0.f; }
#pragma unroll
    for (int i = 0; i < S::kItems; ++i) acc[i] = 0.f;

    for (int c0 = j0; c0 < j1; c0 += kFmaSub) {
        const int n = min(kFmaSub, j1 - c0);
        const int lb0 = c0 / B, lb1 = (c0 + n - 1) / B;
        __syncthreads();  // q staged / previous sub-chunk fully consumed
        for (int i = threadIdx.x; i <= lb1 - lb0; i += kFmaThreads) {
            int pb = table[lb0 + i];
            if (pb < 0 || pb >= num_blocks) { count_error(error_count); pb = -1; }
            blk_s[i] = pb;
        }
        __syncthreads();
        // two tokens per warp and round (t and t + 4), both K rows loaded before either is used
        constexpr int kWarps = kFmaThreads / 32;
        for (int t0 = warp; t0 < n; t0 += 2 * kWarps) {
            float kr[2][kPerLane];
            int pbs[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = t0 + u * kWarps, j = c0 + t;
                pbs[u] = t < n ? blk_s[j / B - lb0] : -1;
#pragma unroll
                for (int e = 0; e < kPerLane; ++e) kr[u][e] = 0.f;
                if (pbs[u] >= 0) {
                    const T* krow = kc + (((size_t)pbs[u] * B + (j % B)) * Hkv + kvh) * D + lane * kPerLane;
#pragma unroll
                    for (int e = 0; e < kPerLane; ++e) kr[u][e] = to_float(krow[e]);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = t0 + u * kWarps;
                if (t >= n) break;
                for (int g = 0; g < G; ++g) {
                    float part = 0.f;
#pragma unroll
                    for (int e = 0; e < kPerLane; ++e) part = fmaf(q_s[g * D + lane * kPerLane + e], kr[u][e], part);
                    part = warp_sum(part);
                    if (lane == 0) p_s[g * kFmaSub + t] = pbs[u] >= 0 ? part * scale_log2 : -INFINITY;
                }
            }
        }
        __syncthreads();
        for (int g = warp; g < G; g += kFmaThreads / 32) {
            float mx = -INFINITY;
            for (int t = lane; t < n; t += 32) mx = fmaxf(mx, p_s[g * kFmaSub + t]);
            mx = warp_max(mx);
            const float m_old = m_s[g];
            const float m_new = fmaxf(m_old, mx);
            float sum = 0.f;
            for (int t = lane; t < n; t += 32) {
                float e = m_new == -INFINITY ? 0.f : exp2f(p_s[g * kFmaSub + t] - m_new);
                p_s[g * kFmaSub + t] = e;
                sum += e;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                float a = m_old == -INFINITY ? 0.f : exp2f(m_old - m_new);
                alpha_s[g] = a;
                l_s[g] = l_s[g] * a + sum;
                m_s[g] = m_new;
            }
        }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < S::kItems; ++it) {
            const int idx = threadIdx.x + it * kFmaThreads;
            if (idx < G * D) {
                const int g = idx / D, d = idx % D;
                float a = acc[it] * alpha_s[g];
                // eight tokens' V loads go out together, then their products are added in token order (the
                // sum is the same as one token at a time; only the loads no longer wait on each other)
                auto v_of = [&](int t) {
                    const int j = c0 + t;
                    const int pb = blk_s[j / B - lb0];
                    return pb >= 0 ? to_float(vc[(((size_t)pb * B + (j % B)) * Hkv + kvh) * D + d]) : 0.f;
                };
                int t = 0;
                for (; t + 8 <= n; t += 8) {
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) v[u] = v_of(t + u);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (blk_s[(c0 + t + u) / B - lb0] >= 0) a = fmaf(p_s[g * kFmaSub + t + u], v[u], a);
                }
                for (; t < n; ++t)
                    if (blk_s[(c0 + t) / B - lb0] >= 0) a = fmaf(p_s[g * kFmaSub + t], v_of(t), a);
                acc[it] = a;
            }
        }
    }
    __syncthreads();
}

}  // namespace pa
