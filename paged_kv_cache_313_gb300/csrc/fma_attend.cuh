// fma_attend.cuh — the CUDA-core attention loop shared by the fp32 decode
// kernel and the CUDA-core prefill kernel.
//
// A CTA of kFmaThreads threads attends the G query heads of one kv head over
// the tokens [j0, j1) of one sequence.  Tokens are walked in sub-chunks of
// kFmaSub: the sub-chunk's block-table entries are resolved once ("KV cache
// 显存管理…", PagedAttention 改变了什么: token -> logical block -> physical block
// -> offset -> address), K and then V rows are staged into shared memory
// kFmaPiece tokens at a time by all threads together (one round trip to memory
// per piece instead of one per token), scores are computed one warp per token
// (lanes across head_dim), and an online-softmax state is carried across
// sub-chunks:
//     m' = max(m, max_j x_j),  l' = l 2^(m-m') + sum_j 2^(x_j-m'),
//     acc' = acc 2^(m-m') + sum_j 2^(x_j-m') v_j
// with x_j = scale*log2(e) * q.k_j (base-2 units).
#pragma once

#include "pa_internal.cuh"

namespace pa {

constexpr int kFmaThreads = 128;
constexpr int kFmaSub = 256;     // tokens per sub-chunk
constexpr int kFmaPiece = 64;    // tokens of K (or V) rows staged in shared memory at a time
constexpr int kFmaMaxGroup = 16; // query heads per kv head

template <int D>
struct FmaShape {
    static constexpr int kItems = kFmaMaxGroup * D / kFmaThreads;  // (g, d) outputs per thread (upper bound)
    static constexpr int kPerLane = D / 32;
    // dynamic shared memory: q [16][D], p [16][kSub], rows [kPiece][D] (room for fp32), blocks [kSub+1]
    static constexpr size_t kSmemBytes =
        sizeof(float) * (kFmaMaxGroup * D + kFmaMaxGroup * kFmaSub + kFmaPiece * D) + sizeof(int) * (kFmaSub + 1);
    __device__ static float* q_s(float* smem) { return smem; }
    __device__ static float* p_s(float* smem) { return smem + kFmaMaxGroup * D; }
    __device__ static float* row_s(float* smem) { return smem + kFmaMaxGroup * D + kFmaMaxGroup * kFmaSub; }
    __device__ static int* blk_s(float* smem) {
        return reinterpret_cast<int*>(smem + kFmaMaxGroup * D + kFmaMaxGroup * kFmaSub + kFmaPiece * D);
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
    T* rows = reinterpret_cast<T*>(S::row_s(smem));  // [kFmaPiece][D], rows of the piece's tokens
    const bool vec16 = ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & 15u) == 0;
    // rows of tokens [c0 + p0, c0 + p0 + np) of `pool` (this kv head) into `rows`, zeros for a token without a
    // valid block; every thread's loads go out together.  Bracketed by barriers: the previous piece's readers
    // are done before, and the rows are visible to every warp after.
    auto stage_rows = [&](const T* __restrict__ pool, int c0, int p0, int np, int lb0) {
        __syncthreads();
        if (vec16) {
            constexpr int kChunks = D * (int)sizeof(T) / 16;  // 16-byte pieces of a row
            for (int i = threadIdx.x; i < np * kChunks; i += kFmaThreads) {
                const int t = i / kChunks, c = i - t * kChunks, j = c0 + p0 + t;
                const int pb = blk_s[j / B - lb0];
                int4 v = make_int4(0, 0, 0, 0);
                if (pb >= 0)
                    v = reinterpret_cast<const int4*>(pool + (((size_t)pb * B + (j % B)) * Hkv + kvh) * D)[c];
                reinterpret_cast<int4*>(rows + t * D)[c] = v;
            }
        } else {
            for (int i = threadIdx.x; i < np * D; i += kFmaThreads) {
                const int t = i / D, d = i - t * D, j = c0 + p0 + t;
                const int pb = blk_s[j / B - lb0];
                rows[t * D + d] = pb >= 0 ? pool[(((size_t)pb * B + (j % B)) * Hkv + kvh) * D + d] : T{};
            }
        }
        __syncthreads();
    };

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
        // scores, kFmaPiece tokens at a time: the piece's K rows staged, then one warp per token
        for (int p0 = 0; p0 < n; p0 += kFmaPiece) {
            const int np = min(kFmaPiece, n - p0);
            stage_rows(kc, c0, p0, np, lb0);
            for (int t = warp; t < np; t += kFmaThreads / 32) {
                const int j = c0 + p0 + t;
                const int pb = blk_s[j / B - lb0];
                float kr[kPerLane];
#pragma unroll
                for (int e = 0; e < kPerLane; ++e) kr[e] = to_float(rows[t * D + lane * kPerLane + e]);
                for (int g = 0; g < G; ++g) {
                    float part = 0.f;
#pragma unroll
                    for (int e = 0; e < kPerLane; ++e) part = fmaf(q_s[g * D + lane * kPerLane + e], kr[e], part);
                    part = warp_sum(part);
                    if (lane == 0) p_s[g * kFmaSub + p0 + t] = pb >= 0 ? part * scale_log2 : -INFINITY;
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
        // P V, kFmaPiece tokens at a time: the piece's V rows staged, then each thread adds its (head, column)
        // item over the piece's tokens in token order (tokens without a valid block are skipped)
        for (int p0 = 0; p0 < n; p0 += kFmaPiece) {
            const int np = min(kFmaPiece, n - p0);
            stage_rows(vc, c0, p0, np, lb0);
#pragma unroll
            for (int it = 0; it < S::kItems; ++it) {
                const int idx = threadIdx.x + it * kFmaThreads;
                if (idx < G * D) {
                    const int g = idx / D, d = idx % D;
                    float a = p0 == 0 ? acc[it] * alpha_s[g] : acc[it];
                    for (int t = 0; t < np; ++t)
                        if (blk_s[(c0 + p0 + t) / B - lb0] >= 0)
                            a = fmaf(p_s[g * kFmaSub + p0 + t], to_float(rows[t * D + d]), a);
                    acc[it] = a;
                }
            }
        }
    }
    __syncthreads();
}

}  // namespace pa
