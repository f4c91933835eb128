// prefill_fma.cu — causal chunked prefill on the CUDA cores (fp32 FMA): the
// path for fp32 pools and for shapes the tensor-core prefill kernel does not
// take.
//
// One CTA per (query of a chunk, kv head).  Query i of chunk c sits at
// absolute position p = q_start_pos[c] + i of sequence seq_of_chunk[c] and
// attends keys 0..p through the block table (fma_attend.cuh); the chunk's own
// keys were scattered into the pool by the write step.
#include "fma_attend.cuh"

namespace pa {
namespace {

// Checks one chunk's descriptors; returns the number of keys its last query
// may read (its own context, clamped to what the table covers), -1 if the
// chunk is unusable.
__device__ __forceinline__ int chunk_limit(const PrefillParams& p, int c, int& s, int& start, int& n) {
    const int r0 = p.cu_q_lens[c];
    n = p.cu_q_lens[c + 1] - r0;
    s = p.seq_of_chunk[c];
    start = p.q_start_pos[c];
    if (n < 0 || r0 < 0 || r0 + n > p.total_q || n > p.max_q_len || s < 0 || s >= p.num_seqs || start < 0)
        return -1;
    return min(p.context_lens[s], p.max_blocks_per_seq * p.block_size);
}

template <typename T, int D>
__global__ void __launch_bounds__(kFmaThreads) prefill_fma_kernel(PrefillParams p) {
    using S = FmaShape<D>;
    pdl_trigger();
    pdl_wait();
    const int i = blockIdx.x, c = blockIdx.y, kvh = blockIdx.z;
    int s, start, n;
    const int cap = chunk_limit(p, c, s, start, n);
    if (cap < 0) {
        if (i == 0 && kvh == 0 && threadIdx.x == 0) count_error(p.error_count);
        return;
    }
    if (i >= n) return;
    const int G = p.group;
    int L = start + i + 1;  // causal: keys 0..start+i
    if (L > cap) {
        if (threadIdx.x == 0 && kvh == 0) count_error(p.error_count);
        L = cap;
    }
    const int row = p.cu_q_lens[c] + i;

    extern __shared__ float smem[];
    __shared__ float m_s[kFmaMaxGroup], l_s[kFmaMaxGroup], alpha_s[kFmaMaxGroup];
    float acc[S::kItems];
    const size_t off = ((size_t)row * p.num_q_heads + (size_t)kvh * G) * D;
    fma_attend<T, D>(static_cast<const T*>(p.q) + off, G, static_cast<const T*>(p.k_cache),
                     static_cast<const T*>(p.v_cache), p.block_tables + (size_t)s * p.max_blocks_per_seq,
                     p.block_size, p.num_kv_heads, kvh, p.num_blocks, 0, L, p.scale_log2, p.error_count, smem, acc,
                     m_s, l_s, alpha_s);
    T* out = static_cast<T*>(p.out) + off;
#pragma unroll
    for (int it = 0; it < S::kItems; ++it) {
        const int idx = threadIdx.x + it * kFmaThreads;
        if (idx < G * D) {
            const float l = l_s[idx / D];
            out[idx] = from_float<T>(l > 0.f ? acc[it] / l : 0.f);
        }
    }
}

template <typename T, int D>
int launch(const PrefillParams& p, cudaStream_t stream) {
    const size_t smem = FmaShape<D>::kSmemBytes;
    int rc = ensure_dynamic_smem(reinterpret_cast<const void*>(prefill_fma_kernel<T, D>), smem);
    if (rc != PA_OK) return rc;
    dim3 grid(p.max_q_len, p.num_chunks, p.num_kv_heads);
    return launch_kernel(prefill_fma_kernel<T, D>, grid, dim3(kFmaThreads), smem, stream, p);
}

}  // namespace

int launch_prefill_fma(const PrefillParams& p, int dtype, cudaStream_t stream) {
    if (p.group > kFmaMaxGroup || p.num_chunks > 65535 || p.num_kv_heads > 65535 || p.prefix_lens != nullptr)
        return PA_ERR_UNSUPPORTED;
    if (dtype == PA_F32) return p.head_dim == 64 ? launch<float, 64>(p, stream) : launch<float, 128>(p, stream);
    return p.head_dim == 64 ? launch<__nv_bfloat16, 64>(p, stream) : launch<__nv_bfloat16, 128>(p, stream);
}

}  // namespace pa
