// decode_tc.cu — paged decode for bf16 pools on GB300: TMA-staged K/V blocks
// and warp-level bf16 tensor-core MMAs for the per-block contractions.
//
// What it computes ("PagedAttention学习笔记", 三、算法流程与数据结构: the kernel
// reads Q and the block table, gathers K/V block by block, then softmax(QK^T)V;
// "KV cache 显存管理…", PagedAttention 改变了什么: token -> logical block ->
// physical block -> offset):  for sequence s, query head h and its kv head
// h/G, out = softmax_j(scale q.k_j) v_j over the sequence's context.
//
// Design (one CTA per (sequence, kv head, partition of the context)):
//  * Warp 4 is the producer.  For each 64-token stage it resolves the stage's
//    block-table entries (staged once in shared memory) and issues one 2-D TMA
//    copy per (block, 64-column half) of K and of V: a physical block of one
//    kv head is B rows of head_dim contiguous bf16 at a row stride of
//    Hkv*head_dim, i.e. a box of the pool viewed as a [P*B, Hkv*D] matrix.
//    Boxes land 128-byte-swizzled, so ldmatrix reads are bank-conflict free.
//    A 3-deep ring of stages (mbarrier full/empty pairs) keeps ~96 KB per CTA
//    in flight; two CTAs fit on an SM.
//  * Warps 0-3 are consumers, 16 tokens of each stage apiece.  The G <= 8
//    query heads of the kv head form the N=8 side of m16n8k16 MMAs:
//        S^T[16 tok x 8 heads] = K[16 tok x D] . Q^T        (D/16 MMAs)
//        O^T[D x 8 heads]     += V^T[D x 16 tok] . P^T       (D/16 MMAs)
//    P^T goes from the S^T accumulator layout to the B-operand layout with one
//    movmatrix transpose per 8x8 half.  Softmax is online, in base-2 units,
//    with the running max per head shared by the 8 lanes that hold it.
//  * Tokens past the context or in blocks with an invalid table entry get
//    score -inf and their V rows are zeroed before the PV MMA, so stale or
//    non-finite pool contents never reach the output.
//  * The four consumer warps' states are merged in shared memory; the CTA
//    then writes the output (single partition) or its partial state for the
//    ticketed cross-partition merge in decode_common.cuh.
#include <cudaTypedefs.h>

#include "decode_common.cuh"
#include "sm100_ptx.cuh"

namespace pa {
namespace {

template <int D>
struct TcCfg {
    static constexpr int kHalves = D / 64;              // 64-column (128-byte) halves of a row
    static constexpr int kStageTok = 64;
    static constexpr int kStages = 3;
    static constexpr int kConsumerWarps = 4;
    static constexpr int kThreads = (kConsumerWarps + 1) * 32;
    static constexpr int kHalfBytes = kStageTok * 128;    // one half of a stage's K (or V) tile
    static constexpr int kTileBytes = kHalves * kHalfBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;    // K + V
    static constexpr int kMaxTable = 512;                 // block ids per partition
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kRingBytes + kMaxTable * 4 + 2 * kStages * 8;
    // after the loop the ring is reused: per-warp O^T [warp][head][D] floats, then merge weights
    static constexpr int kReduceBytes = kConsumerWarps * 8 * D * 4;
    static_assert(kReduceBytes + 8 * 128 * 4 <= kRingBytes, "reduction scratch must fit in the ring");
};

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
    // 128-byte swizzle: 16-byte chunk c of 128-byte row r sits at chunk c ^ (r & 7)
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(TcCfg<D>::kThreads, 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const DecodeParams p) {
    using C = TcCfg<D>;
    constexpr int KT = D / 16;  // 16-wide k steps (QK^T) and m tiles (PV)
    const int s = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
    const int G = p.group;
    const int L = decode_context(p, s, split);
    const int nsplit = num_partitions(L, p.partition);
    if (split >= nsplit) return;
    const int j0 = split * p.partition;
    const int ntok = max(0, min(L, j0 + p.partition) - j0);
    const int nstage = (ntok + C::kStageTok - 1) / C::kStageTok;
    const int B = p.block_size;
    const int nblk = (ntok + B - 1) / B;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* tbl = reinterpret_cast<int*>(smem + C::kRingBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(tbl + C::kMaxTable);
    uint64_t* empty = full + C::kStages;
    __shared__ float red_m[C::kConsumerWarps][8], red_l[C::kConsumerWarps][8];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq + j0 / B;
    for (int i = threadIdx.x; i < nblk; i += C::kThreads) {
        int pb = table[i];
        if (pb < 0 || pb >= p.num_blocks) {
            count_error(p.error_count);
            pb = -1;
        }
        tbl[i] = pb;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], C::kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == C::kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && nstage > 0) {
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            for (int st = 0; st < nstage; ++st) {
                const int slot = st % C::kStages;
                if (st >= C::kStages && !mbar_wait(&empty[slot], ((st / C::kStages) - 1) & 1)) {
                    count_error(p.error_count);
                    break;  // consumers time out on their side and finish
                }
                const int t0 = st * C::kStageTok;
                const int b0 = t0 / B;
                const int nb = (min(C::kStageTok, ntok - t0) + B - 1) / B;
                uint32_t bytes = 0;
                for (int b = 0; b < nb; ++b)
                    if (tbl[b0 + b] >= 0) bytes += 2u * C::kHalves * B * 128u;
                mbar_arrive_expect_tx(&full[slot], bytes);
                uint8_t* kdst = smem + slot * C::kStageBytes;
                uint8_t* vdst = kdst + C::kTileBytes;
                for (int b = 0; b < nb; ++b) {
                    const int pb = tbl[b0 + b];
                    if (pb < 0) continue;
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h) {
                        const int x = kvh * D + h * 64;
                        tma_load_2d(kdst + h * C::kHalfBytes + b * B * 128, &tmk, x, pb * B, &full[slot]);
                        tma_load_2d(vdst + h * C::kHalfBytes + b * B * 128, &tmv, x, pb * B, &full[slot]);
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int g4 = lane >> 2, c4 = lane & 3;
        const int row0 = warp * 16;  // this warp's 16 token rows in every stage
        uint32_t qb[KT][2];
        {
            const __nv_bfloat16* q =
                static_cast<const __nv_bfloat16*>(p.q) + ((size_t)s * p.num_q_heads + (size_t)kvh * G) * D;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                if (g4 < G) {
                    qb[kk][0] = *reinterpret_cast<const uint32_t*>(q + g4 * D + kk * 16 + 2 * c4);
                    qb[kk][1] = *reinterpret_cast<const uint32_t*>(q + g4 * D + kk * 16 + 2 * c4 + 8);
                } else {
                    qb[kk][0] = qb[kk][1] = 0u;
                }
            }
        }
        float o[KT][4];
#pragma unroll
        for (int i = 0; i < KT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2*c4 and 2*c4+1
        const float sl2 = p.scale_log2;

        for (int st = 0; st < nstage; ++st) {
            const int slot = st % C::kStages;
            if (!mbar_wait(&full[slot], (st / C::kStages) & 1) && lane == 0) count_error(p.error_count);
            const int base = st * C::kStageTok + row0;  // partition-relative token of row 0
            if (base < ntok) {
                const uint8_t* kt = smem + slot * C::kStageBytes;
                uint8_t* vt = const_cast<uint8_t*>(kt) + C::kTileBytes;
                auto row_valid = [&](int r) { return base + r < ntok && tbl[(base + r) / B] >= 0; };
                // zero V rows that carry no valid token (past the context or in an unloaded block)
                {
                    const int r = lane >> 1;
                    if (!row_valid(r)) {
                        int4 z = make_int4(0, 0, 0, 0);
#pragma unroll
                        for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                *reinterpret_cast<int4*>(vt + h * C::kHalfBytes + (row0 + r) * 128 +
                                                         ((lane & 1) * 4 + c) * 16) = z;
                    }
                    __syncwarp();
                }
                // S^T = K Q^T
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const uint32_t r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t kbase = smem_u32(kt);
#pragma unroll
                    for (int kk = 0; kk < KT; ++kk) {
                        const uint32_t half = kk >> 2, ch = (kk & 3) * 2 + (lane >> 4);
                        uint32_t a[4];
                        ldmatrix_x4(a, kbase + half * C::kHalfBytes + swz(r, ch));
                        mma_bf16_16816(sc, a, qb[kk][0], qb[kk][1]);
                    }
                }
                const bool vlo = row_valid(g4), vhi = row_valid(g4 + 8);
                const float x0 = vlo ? sc[0] * sl2 : -INFINITY, x1 = vlo ? sc[1] * sl2 : -INFINITY;
                const float x2 = vhi ? sc[2] * sl2 : -INFINITY, x3 = vhi ? sc[3] * sl2 : -INFINITY;
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float a0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
                const float a1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
                const float p0 = mn0 == -INFINITY ? 0.f : exp2f(x0 - mn0);
                const float p2 = mn0 == -INFINITY ? 0.f : exp2f(x2 - mn0);
                const float p1 = mn1 == -INFINITY ? 0.f : exp2f(x1 - mn1);
                const float p3 = mn1 == -INFINITY ? 0.f : exp2f(x3 - mn1);
                l0 = l0 * a0 + p0 + p2;
                l1 = l1 * a1 + p1 + p3;
                m0 = mn0;
                m1 = mn1;
#pragma unroll
                for (int mt = 0; mt < KT; ++mt) {
                    o[mt][0] *= a0;
                    o[mt][1] *= a1;
                    o[mt][2] *= a0;
                    o[mt][3] *= a1;
                }
                const uint32_t b0 = movmatrix_trans(pack_bf16x2(p0, p1));
                const uint32_t b1 = movmatrix_trans(pack_bf16x2(p2, p3));
                // O^T += V^T P^T
                {
                    const uint32_t r = row0 + (lane & 7) + (lane >> 4) * 8;
                    const uint32_t vbase = smem_u32(vt);
#pragma unroll
                    for (int mt = 0; mt < KT; ++mt) {
                        const uint32_t half = mt >> 2, ch = (mt & 3) * 2 + ((lane >> 3) & 1);
                        uint32_t a[4];
                        ldmatrix_x4_trans(a, vbase + half * C::kHalfBytes + swz(r, ch));
                        mma_bf16_16816(o[mt], a, b0, b1);
                    }
                }
                fence_proxy_async_smem();  // generic-proxy zeroing before the next TMA write of this slot
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // ---- merge the four warps' states
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if (g4 == 0) {
            red_m[warp][2 * c4] = m0;
            red_m[warp][2 * c4 + 1] = m1;
            red_l[warp][2 * c4] = l0;
            red_l[warp][2 * c4 + 1] = l1;
        }
        consumer_bar();  // also: every consumer is done reading the ring
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kConsumerWarps; ++w) {
            M0 = fmaxf(M0, red_m[w][2 * c4]);
            M1 = fmaxf(M1, red_m[w][2 * c4 + 1]);
        }
        const float f0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M0);
        const float f1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M1);
        float* ored = reinterpret_cast<float*>(smem);  // [warp][head 0..7][D]
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
            const int d = mt * 16 + g4;
            ored[(warp * 8 + 2 * c4) * D + d] = o[mt][0] * f0;
            ored[(warp * 8 + 2 * c4 + 1) * D + d] = o[mt][1] * f1;
            ored[(warp * 8 + 2 * c4) * D + d + 8] = o[mt][2] * f0;
            ored[(warp * 8 + 2 * c4 + 1) * D + d + 8] = o[mt][3] * f1;
        }
        consumer_bar();
        const size_t unit = decode_unit(p, s, kvh);
        __nv_bfloat16* out =
            static_cast<__nv_bfloat16*>(p.out) + ((size_t)s * p.num_q_heads + (size_t)kvh * G) * D;
        float* wo = p.ws_o + (unit * p.max_splits + split) * G * D;
        for (int idx = threadIdx.x; idx < G * D; idx += 32 * C::kConsumerWarps) {
            const int h = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::kConsumerWarps; ++w) M = fmaxf(M, red_m[w][h]);
            float Ls = 0.f, acc = 0.f;
#pragma unroll
            for (int w = 0; w < C::kConsumerWarps; ++w) {
                const float mw = red_m[w][h];
                if (mw != -INFINITY) Ls += red_l[w][h] * exp2f(mw - M);
                acc += ored[(w * 8 + h) * D + d];
            }
            const float val = Ls > 0.f ? acc / Ls : 0.f;
            if (nsplit == 1) {
                out[idx] = __float2bfloat16_rn(val);
            } else {
                wo[idx] = val;
                if (d == 0) p.ws_ml[(unit * p.max_splits + split) * G + h] = make_float2(M, Ls);
            }
        }
    }
    if (nsplit > 1) decode_merge_if_last<__nv_bfloat16>(p, s, kvh, nsplit, reinterpret_cast<float*>(smem + C::kReduceBytes));
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// The pool viewed as a [num_blocks*B, Hkv*D] bf16 matrix; a box is one
// block's B rows x 64 columns, 128-byte swizzled in shared memory.
int pool_tensor_map(CUtensorMap* map, const void* pool, int num_blocks, int block_size, int num_kv_heads, int head_dim) {
    auto enc = tensor_map_encoder();
    if (!enc) return PA_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)num_kv_heads * head_dim, (cuuint64_t)num_blocks * block_size};
    cuuint64_t strides[1] = {(cuuint64_t)num_kv_heads * head_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)block_size};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

template <int D>
int launch(const DecodeParams& p, cudaStream_t stream) {
    using C = TcCfg<D>;
    CUtensorMap tmk, tmv;
    int rc = pool_tensor_map(&tmk, p.k_cache, p.num_blocks, p.block_size, p.num_kv_heads, D);
    if (rc != PA_OK) return rc;
    if ((rc = pool_tensor_map(&tmv, p.v_cache, p.num_blocks, p.block_size, p.num_kv_heads, D)) != PA_OK) return rc;
    if ((rc = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_tc_kernel<D>), C::kSmemBytes)) != PA_OK)
        return rc;
    dim3 grid(p.num_seqs, p.num_kv_heads, p.max_splits);
    decode_tc_kernel<D><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tmk, tmv, p);
    return check_launch();
}

}  // namespace

bool decode_tc_supported(const DecodeParams& p, int dtype) {
    const int B = p.block_size;
    if (dtype != PA_BF16 || (p.head_dim != 64 && p.head_dim != 128) || p.group > 8) return false;
    if (B != 8 && B != 16 && B != 32 && B != 64) return false;
    if (p.partition % 64 != 0 || p.partition / B > TcCfg<128>::kMaxTable) return false;
    if (((uintptr_t)p.k_cache & 15) || ((uintptr_t)p.v_cache & 15) || ((uintptr_t)p.q & 3)) return false;
    if ((long long)p.num_blocks * B >= (1LL << 31)) return false;
    return p.num_kv_heads <= 65535 && p.max_splits <= 128;
}

int launch_decode_tc(const DecodeParams& p, cudaStream_t stream) {
    return p.head_dim == 64 ? launch<64>(p, stream) : launch<128>(p, stream);
}

}  // namespace pa
