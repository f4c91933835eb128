/*
 * pa.h — C ABI of libpa.so, the GB300 (sm_103a) paged-attention hot path.
 *
 * Sources (page title, then section):
 *   [P1] "什么是 PagedAttention？"
 *   [P2] "PagedAttention学习笔记"
 *   [P3] "KV cache 显存管理：为什么 PagedAttention 是 vLLM 的核心"
 *
 * The operation: the KV cache lives in fixed-size physical blocks of
 * block_size (B) token slots; each sequence's block table maps its logical
 * block i (tokens iB .. iB+B-1) to a physical block ([P2] §2.1; [P3]
 * "分页思想：逻辑连续，物理不连续").  New tokens are scattered to
 * slot = physical_block * B + pos % B ([P2] 代码实现部分 › BlockTable), and
 * attention gathers K/V through the table: logical_block = pos / B,
 * offset = pos % B, physical = block_table[seq][logical_block] ([P3]
 * "PagedAttention 改变了什么"), computing the unchanged softmax(scale QK^T)V
 * ([P2] "与 FlashAttention 的关系").  The argument list follows the kernel
 * inputs of [P3] "对 ModelRunner 的影响": the new tokens, each sequence's
 * context length and block table, the physical block pool and the write slots.
 *
 * Conventions for every entry point:
 *  - Tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *    row-major.  The library allocates no device memory; scratch comes from
 *    the caller's workspace.  An attention output (`out`) may instead be
 *    page-locked host memory mapped into the device's address space (as
 *    cudaHostAlloc gives on this platform): the kernels then store the
 *    results straight into host memory, visible to the host once the stream
 *    has been synchronised.
 *  - K and V pools are separate arrays laid out [num_blocks][block_size]
 *    [num_kv_heads][head_dim]: element (slot, h, d) is at
 *    (slot*num_kv_heads + h)*head_dim + d.  Query head h reads KV head
 *    h / (num_q_heads / num_kv_heads).
 *  - Block tables are int32 [num_seqs][max_blocks_per_seq]; entries past a
 *    sequence's last block are ignored (conventionally -1).
 *  - context_lens[s] counts every token sequence s attends to, including the
 *    token(s) written in the same step (write first, then attend).
 *  - dtype is PA_F32 or PA_BF16 and applies to q, k/v (new and pooled) and out.
 *  - stream is a cudaStream_t passed as void*; NULL means the legacy default
 *    stream.  All calls are asynchronous on that stream.
 *  - Return value: PA_OK, or an error status; nothing is launched when the
 *    host-side checks fail.  PA_ERR_CUDA carries the CUDA error code in
 *    pa_last_cuda_error() (per calling thread).
 *  - Optional error_count (device int32, may be NULL): kernels add the number
 *    of invalid indices they met (out-of-range sequence, logical block, table
 *    entry or slot).  Invalid entries are skipped, never dereferenced.
 *  - The device must be compute capability 10.3 (GB300); otherwise
 *    PA_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,        /* null pointer, negative size, inconsistent shape */
    PA_ERR_UNSUPPORTED = 2,        /* head_dim / block_size / group size / dtype not built */
    PA_ERR_CUDA = 3,               /* a CUDA runtime call failed, see pa_last_cuda_error() */
    PA_ERR_WORKSPACE = 4,          /* workspace missing or smaller than required */
    PA_ERR_UNSUPPORTED_DEVICE = 5  /* current device is not sm_103 */
};

enum pa_dtype { PA_F32 = 0, PA_BF16 = 1 };

/* Library ABI version (major*100 + minor). */
PA_API int pa_version(void);

/* Static, human-readable name of a status code. */
PA_API const char* pa_status_string(int status);

/* cudaError_t of the last PA_ERR_CUDA returned on this thread (0 if none). */
PA_API int pa_last_cuda_error(void);

/*
 * Slot mapping ([P2] 代码实现部分 › "块表与槽位映射：BlockTable",
 * compute_slot_mapping; [P2] 三、算法流程与数据结构).
 * For each new token t of sequence seq_idx[t] at position pos[t]:
 *     slot_mapping[t] = block_tables[seq_idx[t]][pos[t] / B] * B + pos[t] % B
 * pos[t] < 0 marks padding: slot -1, not an error ([P2] writes -1 for tokens
 * another rank owns).  An out-of-range sequence, a logical block at or beyond
 * max_blocks_per_seq, or a table entry outside [0, num_blocks) gives slot -1
 * and counts one error.
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]   (read)
 *   seq_idx, pos  int32 [num_tokens]                     (read)
 *   slot_mapping  int64 [num_tokens]                     (written)
 * num_tokens == 0 is a no-op.  block_size >= 1.
 */
PA_API int pa_slot_mapping(const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                    const int32_t* seq_idx, const int32_t* pos, int num_tokens, int block_size,
                    int num_blocks, int64_t* slot_mapping, int32_t* error_count, void* stream);

/*
 * Paged KV write ([P3] "对 ModelRunner 的影响": the slot says where the
 * current token's K/V is written).  Bit-exact copy:
 *     k_cache[slot_mapping[t]] = k_new[t],  v_cache[slot_mapping[t]] = v_new[t]
 * for every t with slot_mapping[t] >= 0; a row is num_kv_heads*head_dim
 * elements.  Slots at or beyond num_blocks*block_size count one error and
 * are skipped.  Slots must be distinct (the same slot twice is a race).
 *   k_new, v_new      [num_tokens][num_kv_heads][head_dim]            (read)
 *   k_cache, v_cache  [num_blocks][block_size][num_kv_heads][head_dim] (written at the slots)
 * Needs num_kv_heads*head_dim*sizeof(dtype) to be a multiple of 16 bytes and
 * all four arrays 16-byte aligned, else PA_ERR_UNSUPPORTED.
 */
PA_API int pa_write_kv(const void* k_new, const void* v_new, int num_tokens, int num_kv_heads, int head_dim,
                int dtype, void* k_cache, void* v_cache, int num_blocks, int block_size,
                const int64_t* slot_mapping, int32_t* error_count, void* stream);

/*
 * pa_slot_mapping and pa_write_kv in one launch (the two steps the pages put
 * between the scheduler and the attention kernel, fused): for every new
 * token t the slot is resolved from (block_tables, seq_idx, pos) exactly as
 * pa_slot_mapping does and the token's K and V rows are written there exactly
 * as pa_write_kv does.  slot_mapping (int64 [num_tokens]) receives the slots
 * when non-NULL.  Argument meaning, layouts, ownership and error counting are
 * those of the two calls; the pools must not alias k_new / v_new.
 */
PA_API int pa_write_kv_paged(const void* k_new, const void* v_new, int num_tokens, int num_kv_heads, int head_dim,
                             int dtype, void* k_cache, void* v_cache, int num_blocks, int block_size,
                             const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                             const int32_t* seq_idx, const int32_t* pos, int64_t* slot_mapping,
                             int32_t* error_count, void* stream);

/*
 * fp8 KV pools ("KV cache 显存管理…": the pool's size is layers x tokens x kv
 * heads x head_dim x 2 x dtype_size; an e4m3 pool halves dtype_size).  The
 * pools hold one e4m3 code per element (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, largest finite 448) and read back as
 * code * scale, one scale per pool.  This call is pa_write_kv_paged for such
 * pools: every element x of the bf16 rows k_new / v_new ([num_tokens]
 * [num_kv_heads][head_dim]) is stored as the e4m3 code nearest to
 * x * (1.0f / scale) (float arithmetic; ties to the even code; magnitudes
 * beyond 448 are held at 448), k_cache / v_cache being uint8
 * [num_blocks][block_size][num_kv_heads][head_dim].  Scales must be finite
 * and positive.
 */
PA_API int pa_write_kv_paged_fp8(const void* k_new, const void* v_new, int num_tokens, int num_kv_heads,
                                 int head_dim, void* k_cache, void* v_cache, int num_blocks, int block_size,
                                 const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                                 const int32_t* seq_idx, const int32_t* pos, int64_t* slot_mapping, float k_scale,
                                 float v_scale, int32_t* error_count, void* stream);

/*
 * Bytes of workspace pa_decode needs for these sizes (split-KV partial
 * results plus two work-queue counters).  Deterministic:
 * the same arguments on the same device always give the same size.
 */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_context_len);

/*
 * The split-KV plan pa_decode uses for these sizes: *partition receives the
 * partition length in tokens (a multiple of 64) and *max_splits the number of
 * partitions of a max_context_len context (1: no merge kernel is launched).
 * Returns PA_OK, PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED for sizes pa_decode
 * rejects, or PA_ERR_UNSUPPORTED_DEVICE without a compute capability 10.3
 * device.  Either output pointer may be NULL.
 */
PA_API int pa_decode_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int max_context_len, int* partition, int* max_splits);

/*
 * Paged decode attention, one query token per sequence ([P2] 三、算法流程与
 * 数据结构: the kernel reads Q and the block table, gathers K/V block by
 * block, then softmax(QK^T)V; [P3] "PagedAttention 改变了什么" for the
 * address chain).  For sequence s and query head h, with L = context_lens[s]
 * and kv = h / (num_q_heads/num_kv_heads):
 *     out[s][h] = sum_{j<L} softmax_j(scale * q[s][h] . K[s][j][kv]) V[s][j][kv]
 * where K[s][j] is pool row block_tables[s][j/B]*B + j%B.  L == 0 gives zeros.
 *   out, q        [num_seqs][num_q_heads][head_dim]   (out written, q read)
 *   context_lens  int32 [num_seqs]; every entry must be <= max_context_len
 *                 and <= max_blocks_per_seq*B (larger entries are clamped and
 *                 counted as errors; pass error_count to see them)
 * Long contexts are split into partitions processed in parallel and merged
 * with a log-sum-exp combine in a fixed order (deterministic) by a second
 * kernel on the same stream.  workspace must
 * hold pa_decode_workspace_size(...) bytes, be 256-byte aligned, and be zeroed
 * once before its first use; the library leaves it zeroed-for-reuse after
 * every call.  One workspace must not serve two calls that may overlap on the
 * GPU.  Supported: head_dim 64 or 128, block_size 1..1024,
 * num_q_heads/num_kv_heads in 1..16 (other shapes: PA_ERR_UNSUPPORTED).
 * bf16 pools with block_size 8, 16, 32 or 64 and up to 8 query heads per kv
 * head run on the tensor-core kernel; every other supported shape, and fp32,
 * runs on the CUDA-core kernel.
 */
PA_API int pa_decode(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
              int dtype, const void* k_cache, const void* v_cache, int num_blocks, int block_size,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              int max_context_len, float scale, void* workspace, size_t workspace_bytes,
              int32_t* error_count, void* stream);

/*
 * Cascade decode for sequences that share a prefix (parallel sampling, beam
 * search, a common system prompt): "什么是 PagedAttention？", 共享但不污染状态
 * (several sequences map the same physical blocks).  Computes exactly what
 * pa_decode computes, but each group's shared prefix is read from memory once
 * for all of the group's sequences instead of once per sequence:
 *   - groups: sequences [group_offsets[g], group_offsets[g+1]) form group g
 *     (int32 [num_groups+1], non-decreasing, each group a contiguous range of
 *     sequence indices; sequences outside every group, or in a group of one,
 *     are plain decode);
 *   - prefix_lens: int32 [num_seqs], the number of leading context tokens a
 *     sequence shares with its group (0: none).  All members of a group must
 *     have the same prefix length and map the same physical blocks for those
 *     tokens (a block copied on write is private and belongs to the tail); the
 *     prefix is read through the group's first member's block table.  A member
 *     whose prefix length differs from the first member's, or whose table
 *     differs from the first member's over the prefix's blocks, is counted in
 *     error_count (its output is then not its own prefix's).
 *   - max_group_size >= the largest group.
 * Two kernels run on `stream`: the decode kernel, whose queue holds one item
 * per (group, kv head) for the shared prefix (the group's G x members query
 * rows against the prefix's keys, at most 32 rows) followed by the
 * (sequence, partition, kv head) items of every sequence's own tokens
 * [prefix_len, L), and the log-sum-exp merge of the two.  A group wider than
 * 32 query rows has its prefix read by a third, tensor-core prefill-style
 * kernel first.  workspace: pa_decode_cascade_workspace_size
 * bytes, 256-byte aligned, zeroed once.  Supported: bf16, head_dim 128,
 * num_q_heads/num_kv_heads in {1, 2, 4, 8}, block_size 8..64; otherwise
 * PA_ERR_UNSUPPORTED (use pa_decode).
 */
PA_API size_t pa_decode_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                               int block_size, int max_context_len);
PA_API int pa_decode_cascade(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads,
                             int head_dim, int dtype, const void* k_cache, const void* v_cache, int num_blocks,
                             int block_size, const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, int max_context_len, const int32_t* group_offsets,
                             int num_groups, int max_group_size, const int32_t* prefix_lens, float scale,
                             void* workspace, size_t workspace_bytes, int32_t* error_count, void* stream);

/*
 * pa_decode over fp8 pools (see pa_write_kv_paged_fp8): k_cache / v_cache are
 * uint8 [num_blocks][block_size][num_kv_heads][head_dim] e4m3 codes read back
 * as code * k_scale and code * v_scale; q and out are bf16.  The same
 * attention as pa_decode on the read-back values: the kernel loads half the
 * bytes, converts the codes to f16 in registers and runs the products with
 * f16 tensor-core MMAs (q * scale * log2(e) rounded to f16, so |q * scale|
 * must stay below 4e4).  Workspace: pa_decode_workspace_size(...).  Supported:
 * head_dim 128, num_q_heads/num_kv_heads <= 8, block_size 8, 16, 32 or 64;
 * otherwise PA_ERR_UNSUPPORTED.
 */
PA_API int pa_decode_fp8(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                         const void* k_cache, const void* v_cache, int num_blocks, int block_size,
                         const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                         int max_context_len, float scale, float k_scale, float v_scale, void* workspace,
                         size_t workspace_bytes, int32_t* error_count, void* stream);

/*
 * pa_decode fused with the KV write of the step's decode tokens: sequence s's
 * newest token (position L-1, L = context_lens[s]) has its K and V rows in
 * k_new / v_new ([num_seqs][num_kv_heads][head_dim], read).  The decode
 * kernel writes them into k_cache / v_cache at the slot the block table gives
 * (block_tables[s][(L-1)/B]*B + (L-1)%B, exactly pa_slot_mapping +
 * pa_write_kv for that token) and attends with them, so the step needs no
 * separate write launch for its decode tokens ("KV cache 显存管理…",
 * 对 ModelRunner 的影响: the write slots and the attention inputs arrive
 * together).  new_slots (int64 [num_seqs], may be NULL) receives the slots.
 * Everything else is pa_decode's.  A sequence whose newest token falls in a
 * block with an invalid table entry is counted in error_count and nothing is
 * written for it.  Supported: bf16 and the shapes of the tensor-core decode
 * kernel (head_dim 64 or 128, num_q_heads/num_kv_heads <= 8, block_size 8,
 * 16, 32 or 64); otherwise PA_ERR_UNSUPPORTED (use pa_write_kv + pa_decode).
 */
PA_API int pa_decode_write(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                           int dtype, void* k_cache, void* v_cache, int num_blocks, int block_size,
                           const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                           int max_context_len, float scale, const void* k_new, const void* v_new,
                           int64_t* new_slots, void* workspace, size_t workspace_bytes, int32_t* error_count,
                           void* stream);

/*
 * pa_decode_fp8 fused with the quantising KV write of the step's decode
 * tokens: sequence s's newest token (position L-1) has its bf16 K and V rows in
 * k_new / v_new ([num_seqs][num_kv_heads][head_dim], read).  The decode kernel
 * stores them into the e4m3 pools k_cache / v_cache at the slot the block
 * table gives, as code = e4m3(x * (1/k_scale)) and e4m3(x * (1/v_scale)) with
 * the reciprocal and the product rounded to float (exactly what
 * pa_write_kv_paged_fp8 stores), and attends with those codes, so the step
 * needs no separate write launch for its decode tokens ("KV cache 显存管理…",
 * KV size formula: dtype_size a free factor; 对 ModelRunner 的影响: the write
 * slots and the attention inputs arrive together).  new_slots (int64
 * [num_seqs], may be NULL) receives the slots.  Everything else is
 * pa_decode_fp8's: same shapes, scales, workspace and error behaviour; a
 * sequence whose newest token falls in a block with an invalid table entry is
 * counted in error_count and nothing is written for it.  k_scale and v_scale
 * must be positive and finite (else PA_ERR_INVALID_ARG); k_new and v_new
 * 16-byte aligned (else PA_ERR_UNSUPPORTED).
 */
PA_API int pa_decode_write_fp8(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads,
                               int head_dim, void* k_cache, void* v_cache, int num_blocks, int block_size,
                               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                               int max_context_len, float scale, float k_scale, float v_scale, const void* k_new,
                               const void* v_new, int64_t* new_slots, void* workspace, size_t workspace_bytes,
                               int32_t* error_count, void* stream);

/*
 * pa_decode for callers that cannot allocate device memory.  The pages have
 * no counterpart: this is a deployment aid, not part of the method.
 *
 * Some callers cannot call cudaMalloc where decode runs (a runtime that
 * forbids allocation after start-up, a plugin living inside another
 * framework's memory budget, or a caller that must not trigger the implicit
 * synchronisation an allocation can cause).  This entry point computes the
 * same attention as pa_decode, with the same arguments minus the workspace,
 * within the same tolerances (bitwise equal to pa_decode whenever the split
 * plan is unchanged; where the plan below makes partitions longer, the
 * partials are rounded and merged differently in the last bits).  Its
 * split-KV scratch is a fixed 16 MiB array in device global
 * memory owned by the library, which every GPU that loads the library keeps
 * until the process exits.  It allocates nothing (no cudaMalloc / cudaFree,
 * no allocating library routine).
 *  - The partitions are made longer (fewer partials) where that keeps the
 *    scratch within 16 MiB; sizes whose scratch exceeds 16 MiB even with a
 *    single partition are rejected with PA_ERR_WORKSPACE before anything is
 *    launched.
 *  - The first call on a device looks up the array's device address on that
 *    device (cudaGetSymbolAddress) and caches it for the life of the process;
 *    make that first call before any stream capture on the device.  A device
 *    reset (cudaDeviceReset, or a reset of the primary context) invalidates
 *    the cached address: do not call this entry point on that device after
 *    one.
 *  - The array is shared by every call and keeps the last call's contents;
 *    each call clears its work-queue counters (an asynchronous memset on
 *    `stream`) before launching.  Calls that may overlap on the GPU (other
 *    streams, other host threads) race on the array: serialise them.
 */
PA_API int pa_decode_noalloc(void* out, const void* q, int num_seqs, int num_q_heads, int num_kv_heads,
                             int head_dim, int dtype, const void* k_cache, const void* v_cache, int num_blocks,
                             int block_size, const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, int max_context_len, float scale,
                             int32_t* error_count, void* stream);

/*
 * Causal chunked-prefill attention over the paged pool ([P1] 工作原理:
 * prefill takes blocks for the input length; the chunk's own K/V are written
 * by pa_write_kv first).  Chunk c holds queries cu_q_lens[c] ..
 * cu_q_lens[c+1]-1 of sequence seq_of_chunk[c]; query i of the chunk sits at
 * absolute position p = q_start_pos[c] + i and attends keys 0..p of that
 * sequence through its block table:
 *     out[r][h] = sum_{j<=p} softmax_j(scale * q[r][h] . K[j][kv]) V[j][kv]
 * Needs q_start_pos[c] + n_c <= context_lens[seq_of_chunk[c]] (else the
 * chunk is clamped and counted as an error).
 *   out, q        [total_q][num_q_heads][head_dim]
 *   cu_q_lens     int32 [num_chunks+1], cu_q_lens[0] = 0, nondecreasing,
 *                 cu_q_lens[num_chunks] = total_q; max_q_len bounds n_c
 *   q_start_pos, seq_of_chunk  int32 [num_chunks]
 * workspace: pa_prefill_workspace_size(...) bytes (may be 0, then NULL is fine).
 */
PA_API size_t pa_prefill_workspace_size(int num_chunks, int max_q_len, int num_q_heads, int num_kv_heads,
                                 int head_dim, int block_size);

PA_API int pa_prefill_chunk(void* out, const void* q, const int32_t* cu_q_lens, const int32_t* q_start_pos,
                     const int32_t* seq_of_chunk, int num_chunks, int total_q, int max_q_len,
                     int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int dtype,
                     const void* k_cache, const void* v_cache, int num_blocks, int block_size,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                     float scale, void* workspace, size_t workspace_bytes, int32_t* error_count,
                     void* stream);

/*
 * Kernel-side block tables for a block manager whose blocks hold `ratio`
 * kernel blocks ("PagedAttention学习笔记", 代码实现部分 › 块表与槽位映射, 混合块:
 * map_to_kernel_blocks).  The manager's pool [P][ratio*B][Hkv][D] is the same
 * memory as the kernels' pool [P*ratio][B][Hkv][D], so manager block m maps to
 * kernel blocks m*ratio .. m*ratio+ratio-1 and every slot is unchanged:
 *   kernel_tables[s][j] = mgr_tables[s][j / ratio] * ratio + j % ratio
 * (-1 where the manager entry is -1 or j / ratio >= mgr_width).
 *   mgr_tables     int32 [num_seqs][mgr_width], read
 *   kernel_tables  int32 [num_seqs][kernel_width], written (kernel_width is
 *                  normally mgr_width * ratio)
 * Returns PA_ERR_INVALID_ARG for negative sizes or ratio < 1.
 */
PA_API int pa_map_to_kernel_blocks(const int32_t* mgr_tables, int num_seqs, int mgr_width, int ratio,
                                   int32_t* kernel_tables, int kernel_width, void* stream);

/*
 * Copy `bytes` from src to dst with a kernel on `stream`, where either buffer
 * may be page-locked host memory (which the device addresses directly: on
 * GB300 the CPU and GPU share a coherent link) or device memory.  For the
 * per-step transfers of a serving loop (a packed input buffer in, the outputs
 * out, a megabyte or less) this finishes sooner than the copy engine and can
 * be captured into the same CUDA graph as the step.  Not part of the method:
 * a deployment aid.  Both pointers and bytes must be multiples of 16;
 * pageable (unregistered) host memory is rejected with PA_ERR_INVALID_ARG.
 */
PA_API int pa_stage_copy(void* dst, const void* src, size_t bytes, void* stream);

/*
 * Copy-on-write block copy ([P1] 共享但不污染状态: a write into a shared
 * partial block first copies its valid entries into a private block).  For
 * each i < num_copies, token slots 0..num_valid[i]-1 of physical block
 * src_blocks[i] are copied to dst_blocks[i], in both pools.  Destinations
 * must be distinct and must not be sources.  Out-of-range blocks or
 * num_valid outside [0, block_size] count one error and are skipped.
 *   src_blocks, dst_blocks, num_valid  int32 [num_copies]  (device, read)
 */
PA_API int pa_copy_blocks(void* k_cache, void* v_cache, int num_blocks, int block_size, int num_kv_heads,
                   int head_dim, int dtype, const int32_t* src_blocks, const int32_t* dst_blocks,
                   const int32_t* num_valid, int num_copies, int32_t* error_count, void* stream);

/*
 * Self-check of the bounded wait that lets every kernel of this library
 * terminate (no counterpart on the pages: it checks the library's own error
 * path, without a fault).  Every kernel waits on its mbarriers with a poll
 * limit; a wait that runs out counts an error in error_count and the kernel
 * finishes.  This launches one warp that waits, with `polls` polls (1..65536,
 * each a suspended try-wait of at most about 20 us), on a barrier nothing
 * arrives on (arrive == 0) or that it arrived on first (arrive != 0).
 *   result       device int32 [1]: 1 if the wait saw its phase complete, 0 if
 *                it gave up
 *   error_count  device int32 [1] or NULL: incremented when the wait gave up
 * PA_ERR_INVALID_ARG for polls out of range or a NULL result.
 */
PA_API int pa_check_bounded_wait(int polls, int arrive, int32_t* result, int32_t* error_count, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
