// decode_merge.cu — the split-KV combine of paged decode.
//
// A sequence whose context spans nsplit > 1 partitions leaves, per query head
// g and partition i, a partial state (m_i, l_i, o_i) in the workspace
// (decode_common.cuh).  The exact attention output is their log-sum-exp
// combine ("PagedAttention学习笔记", 与 FlashAttention 的关系: the formula is
// unchanged, only tiled with an online softmax):
//     m* = max_i m_i,   w_i = l_i 2^(m_i - m*),   out = sum_i w_i o_i / sum_i w_i
// (partitions with l_i = 0 hold no valid token and get w_i = 0).  In a
// cascade (pa_decode_cascade) slot 0 holds the shared prefix's partial and the
// tail's partitions follow it.
//
// The prefix is read through the group's first member's block table, so in
// a cascade every member must map the same physical blocks over its prefix
// ("什么是 PagedAttention？", 共享但不污染状态: branches share the prefix's
// blocks; a block copied on write is private and belongs to the tail).  The
// warp of each grouped sequence's head 0 checks that against the tables and
// counts a member that breaks it in error_count (its output then used the
// first member's K/V for the prefix).
//
// One warp per (sequence, query head) at a time, grid-stride over all of
// them (a grid of at most a few CTAs per SM, so sequences with a single
// partition cost one length check, not a CTA).  Each lane holds the weights
// of partitions lane, lane+32, ...; for head_dim 128 each lane sums one
// float4 column over the partitions, eight partitions' loads in flight at a
// time, in partition order (deterministic).
#include "decode_common.cuh"

namespace pa {
namespace {

constexpr int kMergeThreads = 128;
constexpr int kMergeUnroll = 8;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(DecodeParams p) {
    constexpr int kCols = D / 4;   // float4 columns of a head's row: 32 (D = 128) or 16 (D = 64)
    constexpr int kLanes = kCols;  // lanes that hold a column; the others idle in the sum
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (kMergeThreads / 32);
    const int G = p.group, Hq = p.num_q_heads;
    const long long units = (long long)p.num_seqs * Hq;
    for (long long u = blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5); u < units; u += warps) {
        const int s = (int)(u / Hq), h = (int)(u - (long long)s * Hq);
        const int L = decode_context(p, s, false);
        int pre;
        const int nsplit = num_partitions(L - decode_start(p, s, L, &pre), partition_of(p, s));
        if (nsplit <= 1 && pre == 0) continue;  // the decode kernel wrote this output directly
        // partial slots [0, split_base) hold the cascade prefix (valid when pre > 0), then the partitions
        const int first = pre > 0 ? 0 : p.split_base, ntot = p.split_base + nsplit;
        const int kvh = h / G, g = h - kvh * G;
        const size_t base = decode_unit(p, s, kvh) * p.max_splits * G + g;  // (slot 0, head g)
        // the first kMergeUnroll partials' loads go out together with the (m, l) loads
        const float4* o = reinterpret_cast<const float4*>(p.ws_o + base * D) + (lane < kLanes ? lane : 0);
        const size_t stride4 = (size_t)G * D / 4;
        float4 x[kMergeUnroll];
#pragma unroll
        for (int k = 0; k < kMergeUnroll; ++k)
            if (first + k < ntot) x[k] = __ldcg(o + (size_t)(first + k) * stride4);
        // weights w_i = l_i 2^(m_i - m*) / sum: at most 128 slots, four per lane
        float2 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = lane + 32 * k;
            v[k] = i >= first && i < ntot ? __ldcg(p.ws_ml + base + (size_t)i * G) : make_float2(-INFINITY, 0.f);
        }
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (v[k].y > 0.f) m = fmaxf(m, v[k].x);
        m = warp_max(m);
        float w[4], wsum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w[k] = v[k].y > 0.f ? v[k].y * exp2f(v[k].x - m) : 0.f;
            wsum += w[k];
        }
        wsum = warp_sum(wsum);
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] *= inv;
        // out = sum_i w_i o_i, in slot order
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i0 = first; i0 < ntot; i0 += kMergeUnroll) {
            if (i0 != first) {
#pragma unroll
                for (int k = 0; k < kMergeUnroll; ++k)
                    if (i0 + k < ntot) x[k] = __ldcg(o + (size_t)(i0 + k) * stride4);
            }
#pragma unroll
            for (int k = 0; k < kMergeUnroll; ++k) {
                const int i = i0 + k;
                // weight of slot i lives in lane i % 32, register i / 32
                const int slot = i >> 5;
                const float wsrc = slot == 0 ? w[0] : slot == 1 ? w[1] : slot == 2 ? w[2] : w[3];
                const float wi = __shfl_sync(0xffffffffu, wsrc, i & 31);
                if (i < ntot) {
                    acc.x = fmaf(wi, x[k].x, acc.x);
                    acc.y = fmaf(wi, x[k].y, acc.y);
                    acc.z = fmaf(wi, x[k].z, acc.z);
                    acc.w = fmaf(wi, x[k].w, acc.w);
                }
            }
        }
        if (lane < kLanes) {
            T* out = static_cast<T*>(p.out) + ((size_t)s * Hq + h) * D + lane * 4;
            out[0] = from_float<T>(acc.x);
            out[1] = from_float<T>(acc.y);
            out[2] = from_float<T>(acc.z);
            out[3] = from_float<T>(acc.w);
        }
        if (h == 0 && pre > 0 && p.check_groups != nullptr) {
            // the first member of s's group (groups are ranges [check_groups[g], check_groups[g + 1]))
            int first = -1;
            for (int g0 = 0; g0 < p.check_num_groups && first < 0; g0 += 32) {
                const int gi = g0 + lane;
                const int lo = gi < p.check_num_groups ? p.check_groups[gi] : 0;
                const int hi = gi < p.check_num_groups ? p.check_groups[gi + 1] : 0;
                const unsigned hit = __ballot_sync(0xffffffffu, lo <= s && s < hi);
                if (hit) first = __shfl_sync(0xffffffffu, lo, __ffs(hit) - 1);
            }
            if (first >= 0 && first != s) {
                const int nb = (pre + p.block_size - 1) / p.block_size;  // blocks holding prefix tokens
                const int32_t* mine = p.block_tables + (size_t)s * p.max_blocks_per_seq;
                const int32_t* ref = p.block_tables + (size_t)first * p.max_blocks_per_seq;
                bool differ = false;
#pragma unroll 4
                for (int b = lane; b < nb; b += 32) differ |= __ldg(mine + b) != __ldg(ref + b);
                if (__any_sync(0xffffffffu, differ) && lane == 0) count_error(p.error_count);
            }
        }
    }
}

template <typename T>
int launch_merge(const DecodeParams& p, int grid, cudaStream_t stream) {
    const dim3 g(grid), b(kMergeThreads);
    if (p.head_dim == 64) return launch_kernel(decode_merge_kernel<T, 64>, g, b, 0, stream, p);
    return launch_kernel(decode_merge_kernel<T, 128>, g, b, 0, stream, p);
}

}  // namespace

int launch_decode_merge(const DecodeParams& p, int dtype, int num_sms, cudaStream_t stream) {
    if (p.max_splits <= 1 && p.prefix_lens == nullptr) return PA_OK;
    if (p.max_splits > 128) return PA_ERR_UNSUPPORTED;
    const long long units = (long long)p.num_seqs * p.num_q_heads;
    const long long want = (units + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
    const int grid = (int)(want < 8LL * num_sms ? want : 8LL * num_sms);
    return dtype == PA_F32 ? launch_merge<float>(p, grid, stream) : launch_merge<__nv_bfloat16>(p, grid, stream);
}

}  // namespace pa
