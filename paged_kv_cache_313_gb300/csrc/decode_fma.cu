// decode_fma.cu — paged decode on the CUDA cores (fp32 FMA), any block size,
// fp32 or bf16 storage.  This is the path for fp32 pools and for block sizes
// the tensor-core decode kernel does not take.
//
// One CTA per (sequence, kv head, partition): it attends the G query heads of
// its kv head over its partition's tokens (fma_attend.cuh), then either
// writes the output (single partition) or stores its partial softmax state
// for the split-KV merge (decode_merge.cu).
#include "decode_common.cuh"
#include "fma_attend.cuh"

namespace pa {
namespace {

template <typename T, int D>
__global__ void __launch_bounds__(kFmaThreads) decode_fma_kernel(DecodeParams p) {
    using S = FmaShape<D>;
    pdl_trigger();
    pdl_wait();
    const int s = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
    const int G = p.group;
    const int L = decode_context(p, s, split == 0 && threadIdx.x == 0);
    const int nsplit = num_partitions(L, p.partition);
    if (split >= nsplit) return;
    const int j0 = split * p.partition;
    const int j1 = min(L, j0 + p.partition);

    extern __shared__ float smem[];
    __shared__ float m_s[kFmaMaxGroup], l_s[kFmaMaxGroup], alpha_s[kFmaMaxGroup];
    float acc[S::kItems];
    const T* q = static_cast<const T*>(p.q) + ((size_t)s * p.num_q_heads + (size_t)kvh * G) * D;
    fma_attend<T, D>(q, G, static_cast<const T*>(p.k_cache), static_cast<const T*>(p.v_cache),
                     p.block_tables + (size_t)s * p.max_blocks_per_seq, p.block_size, p.num_kv_heads, kvh,
                     p.num_blocks, j0, j1, p.scale_log2, p.error_count, smem, acc, m_s, l_s, alpha_s);

    if (nsplit == 1) {
        T* out = static_cast<T*>(p.out) + ((size_t)s * p.num_q_heads + (size_t)kvh * G) * D;
#pragma unroll
        for (int it = 0; it < S::kItems; ++it) {
            const int idx = threadIdx.x + it * kFmaThreads;
            if (idx < G * D) {
                const float l = l_s[idx / D];
                out[idx] = from_float<T>(l > 0.f ? acc[it] / l : 0.f);
            }
        }
        return;
    }
    const size_t unit = decode_unit(p, s, kvh);
    float* wo = p.ws_o + (unit * p.max_splits + split) * G * D;
#pragma unroll
    for (int it = 0; it < S::kItems; ++it) {
        const int idx = threadIdx.x + it * kFmaThreads;
        if (idx < G * D) {
            const float l = l_s[idx / D];
            wo[idx] = l > 0.f ? acc[it] / l : 0.f;
        }
    }
    if (threadIdx.x < G)
        p.ws_ml[(unit * p.max_splits + split) * G + threadIdx.x] = make_float2(m_s[threadIdx.x], l_s[threadIdx.x]);
}

template <typename T, int D>
int launch_fma(const DecodeParams& p, cudaStream_t stream) {
    const size_t smem = FmaShape<D>::kSmemBytes;
    int rc = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_fma_kernel<T, D>), smem);
    if (rc != PA_OK) return rc;
    dim3 grid(p.num_seqs, p.num_kv_heads, p.max_splits);
    return launch_kernel(decode_fma_kernel<T, D>, grid, dim3(kFmaThreads), smem, stream, p);
}

}  // namespace

int launch_decode_fma(const DecodeParams& p, int dtype, cudaStream_t stream) {
    if (p.group > kFmaMaxGroup || p.max_splits > 128 || p.prefix_lens != nullptr) return PA_ERR_UNSUPPORTED;
    if (p.num_kv_heads > 65535 || p.max_splits > 65535) return PA_ERR_UNSUPPORTED;
    if (dtype == PA_F32) return p.head_dim == 64 ? launch_fma<float, 64>(p, stream) : launch_fma<float, 128>(p, stream);
    return p.head_dim == 64 ? launch_fma<__nv_bfloat16, 64>(p, stream) : launch_fma<__nv_bfloat16, 128>(p, stream);
}

}  // namespace pa
