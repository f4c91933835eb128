// prefill_tc.cu — causal chunked prefill over the paged pool on the 5th-gen
// tensor cores (tcgen05, accumulators in TMEM), bf16.
//
// What it computes ("什么是 PagedAttention？", 工作原理: prefill takes blocks for
// the input length; "KV cache 显存管理…", PagedAttention 改变了什么: keys are
// found through the block table): query i of chunk c, at absolute position
// p = q_start_pos[c] + i, attends keys 0..p of its sequence, the chunk's own
// keys included (they were written to the pool first).
//
// A work item is a (128-row query tile, kv head, chunk).  The G query heads
// that share a kv head are packed into the tile's rows: row r is position
// i0 + r/G, head r%G, so every K/V tile is loaded once for all G heads.  The
// kernel is persistent: one CTA per SM walks its share of the items (the
// heaviest tile of every chunk first), its K/V rings, barriers and tensor
// memory carrying on from item to item, so one item's epilogue overlaps the
// next item's loads and a CTA is set up once.
// Key tiles are 128 keys, gathered block by block from the pool by TMA
// (one box per physical block and 64-column half, 128-byte swizzled).
//
// Warp roles (352 threads):
//   warp 0    TMA producer of the Q tile (once) and of K tiles into a 3-deep
//             ring (released after their QK^T MMA); it also publishes each
//             key tile's validity mask to the softmax warps.
//   warp 10   TMA producer of V tiles into a 3-deep ring (released after their
//             PV MMA); separate from warp 0 so K never queues behind V.
//   warp 1    TMEM owner and MMA issuer (one thread):
//               S_j = Q K_j^T      M=128 N=128 K=128   -> TMEM S[j%2]
//               O  += P_j V_j      M=128 N=128 K=128   A = P_j from TMEM
//             S is double-buffered, so QK^T of tile j+1 runs on the tensor
//             cores while the softmax warps work on tile j.  P_j is written
//             over S_j in tensor memory and read from there as the A operand
//             of the PV MMA, so shared memory holds only Q, K and V.
//   warps 2-9 softmax, two threads per query row (TMEM lane = row), one for
//             keys 0-63 and one for keys 64-127 of every tile, each with its
//             own running max and sum and its own O accumulator (O_a, O_b),
//             combined once at the end: read S, mask (causal and context),
//             online softmax in base-2 units with a lazy rescale (a half's O is
//             rescaled only when its max grows by more than 2^8), write P as
//             bf16 into tensor memory, zero V rows past the last valid key,
//             and finally normalise O and store the output rows.
// All waits are bounded (an error is counted and the kernel still finishes);
// TMEM is always freed.  Before the CTA exits, the producers wait (bounded)
// for the last phase they armed on each of their barriers and the MMA warp
// commits once more and waits for that commit, so no bulk copy is landing in
// shared memory and no MMA is writing tensor memory when the CTA frees its
// tensor memory and exits.
#include "pa_internal.cuh"
#include "sm100_ptx.cuh"

namespace pa {
namespace {

constexpr int kTileQ = 128;      // query rows per tile
constexpr int kTileK = 128;      // keys per tile
constexpr int kD = 128;          // head_dim handled by this kernel
constexpr int kHalf = 128 * 128; // bytes of one 64-column half of a 128-row tile
constexpr int kTileBytes = 2 * kHalf;
constexpr int kThreads = 352;  // K producer, MMA issuer, 8 softmax warps, V producer
constexpr int kVWarp = 10;
constexpr uint32_t kTmemCols = 512;        // S0 | S1 | O_a | O_b
constexpr uint32_t kTmemOa = 256;          // keys 0-63 of every tile, softmax state of the row's first half
constexpr uint32_t kTmemOb = 384;          // keys 64-127, the second half's state
constexpr float kRescaleThreshold = 8.0f;  // base-2 units


// shared memory layout (offsets from a 1024-aligned base).  P lives in tensor
// memory (over the S buffer it was computed from), so shared memory holds Q
// and 3-deep K and V rings.
constexpr int kKStages = 3;
constexpr int kVStages = 3;
constexpr int kMaskSlots = 8;  // the producer runs at most 5 key tiles ahead of the softmax's mask reads
constexpr int kQ = 0;
constexpr int kK = kQ + kTileBytes;
constexpr int kV = kK + kKStages * kTileBytes;
constexpr int kBars = kV + kVStages * kTileBytes;
// barriers: q_full, k_full[3], k_empty[3], v_full[3], v_empty[3], s_full[2], p_full[2], o_done[2], m_full[8],
// q_empty, o_free, mma_drain
constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + kMaskSlots + 3;
constexpr int kMask = kBars + kNumBars * 8;  // uint32 [8][4]: key-validity mask of tile j in slot j%8
constexpr int kTmemSlot = kMask + kMaskSlots * 4 * 4;
constexpr size_t kSmemBytes = 1024 + kTmemSlot + 16;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// Dense tiles exponentiate in bf16 pairs (one instruction per two keys; P is
// rounded to bf16 for its MMA either way, the pair form also rounds x - m).
#ifndef PA_PREFILL_EXP2_PAIRS
#define PA_PREFILL_EXP2_PAIRS 1
#endif

// A 32-byte global store (8 words; the address 32-byte aligned): an output row leaves the epilogue in whole
// 32-byte sectors, half the store instructions of 16-byte stores.
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// the eight softmax warps (256 threads) only
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

struct Bars {
    uint64_t* base;
    __device__ uint64_t* q_full() const { return base; }
    __device__ uint64_t* k_full(int i) const { return base + 1 + i; }
    __device__ uint64_t* k_empty(int i) const { return base + 1 + kKStages + i; }
    __device__ uint64_t* v_full(int i) const { return base + 1 + 2 * kKStages + i; }
    __device__ uint64_t* v_empty(int i) const { return base + 1 + 2 * kKStages + kVStages + i; }
    __device__ uint64_t* s_full(int i) const { return base + 1 + 2 * kKStages + 2 * kVStages + i; }
    // P of tile j written into S buffer j%2
    __device__ uint64_t* p_full(int i) const { return base + 3 + 2 * kKStages + 2 * kVStages + i; }
    // the PV that read P buffer i is done
    __device__ uint64_t* o_done(int i) const { return base + 5 + 2 * kKStages + 2 * kVStages + i; }
    // mask slot i published
    __device__ uint64_t* m_full(int i) const { return base + 7 + 2 * kKStages + 2 * kVStages + i; }
    // the Q buffer may be refilled: every QK^T of the item has completed
    __device__ uint64_t* q_empty() const { return base + 7 + 2 * kKStages + 2 * kVStages + kMaskSlots; }
    // the softmax warps have read O (and left the S buffers) in an item's epilogue
    __device__ uint64_t* o_free() const { return base + 8 + 2 * kKStages + 2 * kVStages + kMaskSlots; }
    // every tcgen05.mma the MMA warp issued has completed (its last commit, before tensor memory is freed)
    __device__ uint64_t* mma_drain() const { return base + 9 + 2 * kKStages + 2 * kVStages + kMaskSlots; }
};

__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
    pdl_trigger();
    pdl_wait();
    const int G = p.group, B = p.block_size;
    const int pos_per_tile = kTileQ / G;
    const bool prefix_mode = p.prefix_lens != nullptr;

    // ---- work items: (query tile, kv head, chunk), the heaviest (latest) tile of every chunk first,
    // then the next heaviest, ...; CTA b takes one item of every pass of `grid` items, in serpentine
    // order (b in even passes, grid - 1 - b in odd ones) so that heavy and light items pair up.  Every
    // warp walks the same items, so the roles agree without communicating.  (Claiming items from a
    // work queue instead was measured 10-25% slower.)
    const int tiles_max = (p.max_q_len + pos_per_tile - 1) / pos_per_tile;
    const int per_rank = p.num_chunks * p.num_kv_heads;
    const int num_items = tiles_max * per_rank;
    struct Item {
        int kvh, r0, s, start, i0, nq, last_key, nkeys, nt;
    };
    auto item_of = [&](int c) {  // this CTA's item of pass c
        const int b = blockIdx.x, g = gridDim.x;
        return c * g + ((c & 1) ? g - 1 - b : b);
    };
    // false for an empty item (a tile past its chunk's queries, or an invalid chunk)
    auto describe = [&](int k, Item& d) {
        const int rank = k / per_rank, rem = k - rank * per_rank;
        const int c = rem / p.num_kv_heads;
        d.kvh = rem - c * p.num_kv_heads;
        d.r0 = p.cu_q_lens[c];
        const int n = p.cu_q_lens[c + 1] - d.r0;
        d.s = prefix_mode ? d.r0 : p.seq_of_chunk[c];
        d.start = prefix_mode ? 0 : p.q_start_pos[c];
        bool chunk_ok =
            n >= 0 && d.r0 >= 0 && d.r0 + n <= p.total_q && n <= p.max_q_len && d.s >= 0 && d.s < p.num_seqs;
        if (chunk_ok && prefix_mode && n > 0) d.start = p.prefix_lens[d.s];  // the group's shared prefix length
        chunk_ok = chunk_ok && d.start >= 0;
        if (!chunk_ok) {
            if (rank == 0 && d.kvh == 0 && threadIdx.x == 0) count_error(p.error_count);
            return false;
        }
        const int ntiles_q = (n + pos_per_tile - 1) / pos_per_tile;
        if (rank >= ntiles_q) return false;
        d.i0 = (ntiles_q - 1 - rank) * pos_per_tile;
        d.nq = min(pos_per_tile, n - d.i0);
        const int cap = min(p.context_lens[d.s], p.max_blocks_per_seq * B);
        // the tile's last query position; a cascade prefix pass reads keys [0, start) for every row
        d.last_key = prefix_mode ? d.start - 1 : d.start + d.i0 + d.nq - 1;
        if (d.last_key >= cap) {
            if (threadIdx.x == 0) count_error(p.error_count);
            d.last_key = cap - 1;
        }
        d.nkeys = d.last_key + 1;  // keys 0..last_key are read
        d.nt = d.nkeys > 0 ? (d.nkeys + kTileK - 1) / kTileK : 0;
        return true;
    };

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Bars bars{reinterpret_cast<uint64_t*>(smem + kBars)};
    uint32_t* vmask = reinterpret_cast<uint32_t*>(smem + kMask);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bars.q_full(), 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(bars.k_full(i), 1);
            mbar_init(bars.k_empty(i), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(bars.v_full(i), 1);
            mbar_init(bars.v_empty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars.s_full(i), 1);
            mbar_init(bars.p_full(i), 8);
            mbar_init(bars.o_done(i), 1);
        }
        for (int i = 0; i < kMaskSlots; ++i) mbar_init(bars.m_full(i), 1);
        mbar_init(bars.q_empty(), 1);
        mbar_init(bars.o_free(), 8);
        mbar_init(bars.mma_drain(), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0 || warp == kVWarp) {
        // ============================================================ producers
        // warp 0 loads Q, the K tiles and publishes each tile's key mask; warp kVWarp loads the V
        // tiles.  Each waits only on its own ring, so K streams ahead of V.
        const bool v_side = warp == kVWarp;
        const int bpt = kTileK / B;  // blocks per key tile
        // Per key tile the producer only waits for its ring slot and issues the copies: the block ids of
        // a 32-entry chunk of the table are loaded one per lane when the chunk is reached, and the
        // tiles under that chunk get their key masks and byte counts lane-parallel (lane t for the
        // chunk's tile t).  The rings run on across items.
        const int tpc = 32 / bpt;  // key tiles per 32-entry chunk of the table
        if (lane == 0) {
            if (!v_side) {
                tma_prefetch_desc(&tmq);
                tma_prefetch_desc(&tmk);
            } else {
                tma_prefetch_desc(&tmv);
            }
        }
        int gt = 0, gi = 0;  // key tiles, and items with keys, taken so far
        uint32_t armed = 0, armed_q = 0;  // phases armed on this producer's ring (K or V) and on q_full
        for (int c = 0; c * (int)gridDim.x < num_items && ok; ++c) {
            const int k = item_of(c);
            Item d;
            if (k >= num_items || !describe(k, d)) continue;
            const int kvh = d.kvh, nkeys = d.nkeys, nt = d.nt;
            const int32_t* table = p.block_tables + (size_t)d.s * p.max_blocks_per_seq;
            const int nblk = (nkeys + B - 1) / B;
            if (!v_side && nt > 0) {  // with no keys nothing is loaded (nor left in flight)
                // the Q tile; its buffer is free once the previous item's last QK^T completed
                if (gi > 0 && !mbar_wait_warp(bars.q_empty(), (gi - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bars.q_full(), 2 * kHalf);
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(smem + kQ + h * kHalf, &tmq, h * 64, kvh * G, d.r0 + d.i0, bars.q_full());
                }
                ++armed_q;
            }
            int pb_lane = -1;
            uint32_t lbytes = 0, lvm[4] = {0u, 0u, 0u, 0u};
            for (int j = 0; j < nt; ++j) {
                const int g = gt + j;  // the CTA's key tile number: ring slots and phases
                const int chunk = j / tpc, l = j - chunk * tpc;
                if (l == 0) {
                    const int idx = chunk * 32 + lane;
                    pb_lane = -1;
                    if (idx < nblk) {
                        pb_lane = table[idx];
                        if (pb_lane < 0 || pb_lane >= p.num_blocks) {
                            if (!v_side) count_error(p.error_count);
                            pb_lane = -1;
                        }
                    }
                    const int jt = chunk * tpc + lane;  // this lane's key tile
                    lbytes = 0;
#pragma unroll
                    for (int w = 0; w < 4; ++w) lvm[w] = 0u;
                    for (int b = 0; b < bpt; ++b) {
                        const int pb = __shfl_sync(0xffffffffu, pb_lane, (lane * bpt + b) & 31);
                        if (lane < tpc && jt * bpt + b < nblk && pb >= 0) {
                            lbytes += 2u * B * 128u;
                            const int k0 = b * B, k1 = min((b + 1) * B, nkeys - jt * kTileK);
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                const int lo = max(k0, 32 * w), hi = min(k1, 32 * w + 32);
                                if (lo < hi) lvm[w] |= (hi - lo == 32 ? ~0u : ((1u << (hi - lo)) - 1u)) << (lo - 32 * w);
                            }
                        }
                    }
                }
                const uint32_t bytes = __shfl_sync(0xffffffffu, lbytes, l);
                // lanes [0, 2 bpt) copy the tile's blocks, one (block, 64-column half) box each
                const int blk = lane >> 1, h = lane & 1;
                const int my_pb = __shfl_sync(0xffffffffu, pb_lane, (l * bpt + (lane < 2 * bpt ? blk : 0)) & 31);
                const bool my_load = lane < 2 * bpt && j * bpt + blk < nblk && my_pb >= 0;
                if (!v_side) {
                    // K tile j (its slot is free once S_{j-3} completed; S_{j-3} was issued after PV_{j-5}, so
                    // the softmax warps have finished tile j-5 and read every mask up to j-5: the mask ring
                    // of 8 slots is never overwritten unread)
                    uint32_t vm[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) vm[w] = __shfl_sync(0xffffffffu, lvm[w], l);
                    const int st = g % kKStages;
                    if (g >= kKStages && !mbar_wait_warp(bars.k_empty(st), ((g / kKStages) - 1) & 1)) ok = false;
                    if (!ok) break;
                    if (lane == 0) {
                        for (int w = 0; w < 4; ++w) vmask[(g % kMaskSlots) * 4 + w] = vm[w];
                        mbar_arrive(bars.m_full(g % kMaskSlots));
                        mbar_arrive_expect_tx(bars.k_full(st), bytes);
                    }
                    ++armed;
                    __syncwarp();  // armed before any copy is issued
                    if (my_load)
                        tma_load_2d(smem + kK + st * kTileBytes + h * kHalf + blk * B * 128, &tmk, kvh * kD + h * 64,
                                    my_pb * B, bars.k_full(st));
                } else {
                    // V tile j (its slot is free once PV_{j-kVStages} completed)
                    const int vs = g % kVStages;
                    if (g >= kVStages && !mbar_wait_warp(bars.v_empty(vs), ((g / kVStages) - 1) & 1)) ok = false;
                    if (!ok) break;
                    if (lane == 0) mbar_arrive_expect_tx(bars.v_full(vs), bytes);
                    ++armed;
                    __syncwarp();
                    if (my_load)
                        tma_load_2d(smem + kV + vs * kTileBytes + h * kHalf + blk * B * 128, &tmv, kvh * kD + h * 64,
                                    my_pb * B, bars.v_full(vs));
                }
                __syncwarp();
            }
            gt += nt;
            if (nt > 0) ++gi;
        }
        if (!ok && lane == 0) count_error(p.error_count);
        // drain: every copy this warp issued has landed before the CTA exits (at once on the normal path,
        // where the MMA warp waited for every armed phase; after a timeout, copies still in flight)
        if (lane == 0) {
            const bool drained = v_side ? drain_ring(bars.v_full(0), kVStages, armed)
                                        : drain_ring(bars.k_full(0), kKStages, armed) &&
                                              drain_ring(bars.q_full(), 1, armed_q);
            if (!drained) count_error(p.error_count);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        // The whole warp runs the loop with warp-uniform descriptors; one elected lane issues every
        // MMA and commit.  (Run by lane 0 alone, the same loop spent about 75 cycles per MMA issued.)
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity)) != 0;
        };
        constexpr uint32_t idesc_s = umma_idesc_bf16(128, 128, false, false);
        constexpr uint32_t idesc_o = umma_idesc_bf16(128, 128, false, true);
        const uint32_t q_base = smem_u32(smem + kQ), k_base = smem_u32(smem + kK);
        const uint32_t v_base = smem_u32(smem + kV);
        const uint32_t t_oa = tmem + kTmemOa, t_ob = tmem + kTmemOb;
        // descriptors of k-step 0; a k-step adds its byte offset >> 4 to the start-address field
        const uint64_t dq0 = umma_desc_sw128(q_base, 16, 1024);
        const uint64_t dk0 = umma_desc_sw128(k_base, 16, 1024);
        const uint64_t dv0 = umma_desc_sw128(v_base, kHalf, 1024);
        int gt = 0, gi = 0;  // key tiles, and items with keys, taken so far
        for (int c = 0; c * (int)gridDim.x < num_items && ok; ++c) {
            const int k = item_of(c);
            Item d;
            if (k >= num_items || !describe(k, d) || d.nt == 0) continue;
            const int nt = d.nt;
            if (!wait_all(bars.q_full(), gi & 1)) {
                ok = false;
                break;
            }
            // the previous item's epilogue has read O and left the S buffers
            if (gi > 0 && !wait_all(bars.o_free(), (gi - 1) & 1)) {
                ok = false;
                break;
            }
            for (int j = 0; j <= nt && ok; ++j) {
                if (j < nt) {  // S_j = Q K_j^T into S[g%2]
                    // S[g%2] last held P_{g-2}, read by PV_{g-2}, which was issued before this MMA (the
                    // tensor core runs one thread's MMAs in order)
                    const int g = gt + j, st = g % kKStages, sb = g & 1;
                    if (!wait_all(bars.k_full(st), (g / kKStages) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dk = dk0 + (uint64_t)((st * kTileBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint64_t off = (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
                        umma_bf16_warp(tmem + sb * 128, dq0 + off, dk + off, idesc_s, kk > 0);
                    }
                    umma_commit_warp(bars.s_full(sb));
                    umma_commit_warp(bars.k_empty(st));
                    if (j == nt - 1) umma_commit_warp(bars.q_empty());  // every QK^T of the item is done with Q
                }
                if (j >= 1) {  // O += P_{j-1} V_{j-1}, P from tensor memory
                    const int jj = j - 1, g = gt + jj, vs = g % kVStages, pb = g & 1;
                    // V (usually landed long before) first, so that its poll is not on the path from P
                    if (!wait_all(bars.v_full(vs), (g / kVStages) & 1)) { ok = false; break; }
                    if (!wait_all(bars.p_full(pb), (g >> 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dv = dv0 + (uint64_t)((vs * kTileBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTileK / 16; ++kk) {
                        // keys 16kk..16kk+15: P columns 8kk.. (keys 0-63) or 64 + 8(kk-4).. (keys 64-127);
                        // keys 0-63 into O_a, keys 64-127 into O_b: each half of the row keeps its own max
                        const uint32_t pa = tmem + pb * 128 + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
                        umma_bf16_ta_warp(kk < 4 ? t_oa : t_ob, pa, dv + (uint64_t)((kk * 2048) >> 4), idesc_o,
                                          jj > 0 || (kk & 3) > 0);
                    }
                    umma_commit_warp(bars.o_done(pb));
                    umma_commit_warp(bars.v_empty(vs));
                }
            }
            gt += nt;
            ++gi;
        }
        if (!ok && lane == 0) count_error(p.error_count);
        // drain: one more commit tracks every MMA issued so far; tensor memory is freed (below) only after
        // it arrives, also when the loop above stopped at a timeout with MMAs still running
        umma_commit_warp(bars.mma_drain());
        if (!wait_all(bars.mma_drain(), 0) && lane == 0) count_error(p.error_count);
        __syncwarp();
    } else {
        // ============================================================ softmax / epilogue
        // Eight warps: warps 2-5 take keys 0-63 of every tile (every row), warps 6-9
        // keys 64-127.  Each half of a row runs its own online softmax (own max and
        // sum) and its keys accumulate into their own O (O_a, O_b), so the two
        // threads of a row never wait for each other inside the key loop; their
        // states are combined once, in the epilogue.  Every thread runs every
        // iteration and the named barrier, even after a wait timed out, so the
        // barrier can never be left one-sided.
        const int quarter = warp & 3;       // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;   // which 64 columns of the row
        const int r = quarter * 32 + lane;  // the query row this thread works on
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int col0 = half * 64;
        const uint32_t t_own = tmem + lane_off + (half ? kTmemOb : kTmemOa);  // this half's O, row r
        const float sl2 = p.scale_log2;
        const bool out_al32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
        int gt = 0;  // key tiles taken so far
        for (int c = 0; c * (int)gridDim.x < num_items; ++c) {
            const int k = item_of(c);
            Item d;
            if (k >= num_items || !describe(k, d)) continue;
            const int kvh = d.kvh, r0 = d.r0, start = d.start, i0 = d.i0, nq = d.nq, last_key = d.last_key, nt = d.nt;
            const int pos = i0 + r / G;  // chunk-relative position
            const bool row_ok = pos - i0 < nq;
            const int my_last = prefix_mode ? last_key : min(start + pos, last_key);  // last key this row may see
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nt; ++j) {
                const int g = gt + j, st = g & 1;
                // validity of the tile's 128 keys (inside the context, in a block with a valid table
                // entry), published by the producer
                if (ok && !mbar_wait(bars.m_full(g % kMaskSlots), (g / kMaskSlots) & 1)) ok = false;
                uint32_t vm[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) vm[w] = vmask[(g % kMaskSlots) * 4 + w];
                if (ok && !mbar_wait(bars.s_full(st), (g >> 1) & 1)) ok = false;
                tc_fence_after();
                float sv[64];
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    float t[32];
                    tmem_ld32(tmem + lane_off + st * 128 + col0 + q2 * 32, t);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sv[q2 * 32 + i] = t[i];
                }
                tmem_wait_ld();
                const int kbase = j * kTileK + col0;
                const uint32_t w0 = vm[half * 2], w1 = vm[half * 2 + 1];
                // dense: every key of my 64 is valid and causally visible, and the scale is positive,
                // so the max can be taken on raw scores and the scale folded into one FMA later
                const bool dense = (w0 & w1) == ~0u && kbase + 63 <= my_last && sl2 > 0.f;
                // row max over my 64 keys in eight independent chains (a single chain of 64 dependent
                // maxima was a third of the softmax's time)
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
                if (dense) {
#pragma unroll
                    for (int k = 0; k < 64; k += 2) mx8[(k >> 1) & 7] = fmax3(mx8[(k >> 1) & 7], sv[k], sv[k + 1]);
                } else {
#pragma unroll
                    for (int k = 0; k < 64; ++k) {
                        const bool valid = (((k < 32 ? w0 : w1) >> (k & 31)) & 1u) && kbase + k <= my_last;
                        sv[k] = valid ? sv[k] * sl2 : -INFINITY;
                        mx8[k & 7] = fmaxf(mx8[k & 7], sv[k]);
                    }
                }
                float mpart = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                    fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                if (dense) mpart *= sl2;
                const float mt = mpart;
                if (mt > m_run + kRescaleThreshold) {  // also true for the first finite max
                    if (m_run != -INFINITY) {
                        const float alpha = fast_exp2(m_run - mt);
                        l_run *= alpha;
                        if (j > 0) {
                            // every PV issued so far (the last is PV_{j-1}) must be done before O changes
                            if (ok && !mbar_wait(bars.o_done((g - 1) & 1), ((g - 1) >> 1) & 1)) ok = false;
                            tc_fence_after();
#pragma unroll 1
                            for (int q2 = 0; q2 < 8; ++q2) {  // all 128 columns of this half's O row
                                float t[16];
                                tmem_ld16(t_own + q2 * 16, t);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 16; ++i) t[i] *= alpha;
                                tmem_st16(t_own + q2 * 16, t);
                            }
                            tmem_wait_st();
                        }
                    }
                    m_run = mt;
                }
                // P = 2^(x - m) in bf16, my 64 keys of row r packed in pairs into 32 columns of S buffer j%2
                // (its first 32 columns for keys 0-63, columns 64-95 for keys 64-127: each thread
                // overwrites only S values it has already read)
                float lsum = 0.f;
                const float neg_m = -m_run;
                {
                    uint32_t pk[32];
                    float ls4[4] = {0.f, 0.f, 0.f, 0.f};
                    if (PA_PREFILL_EXP2_PAIRS && dense) {
                        // two keys per instruction throughout: x - m by a paired FMA, rounded to a bf16
                        // pair, 2^x of the pair (which is P itself), and the sum of the same bf16 values
                        // by a paired add
                        const unsigned long long s2 = f32x2_pack(sl2, sl2), m2 = f32x2_pack(neg_m, neg_m);
                        unsigned long long acc2[2] = {f32x2_pack(0.f, 0.f), f32x2_pack(0.f, 0.f)};
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float y0, y1;
                            f32x2_unpack(fma_f32x2(f32x2_pack(sv[2 * i], sv[2 * i + 1]), s2, m2), y0, y1);
                            const uint32_t e = exp2_bf16x2(pack_bf16x2(y0, y1));
                            pk[i] = e;
                            acc2[i & 1] = add_f32x2(
                                acc2[i & 1], f32x2_pack(__uint_as_float(e << 16), __uint_as_float(e & 0xFFFF0000u)));
                        }
                        float a0, a1, b0, b1;
                        f32x2_unpack(acc2[0], a0, a1);
                        f32x2_unpack(acc2[1], b0, b1);
                        ls4[0] = a0;
                        ls4[1] = a1;
                        ls4[2] = b0;
                        ls4[3] = b1;
                    } else {
                        if (dense) {
#pragma unroll
                            for (int k = 0; k < 64; ++k) sv[k] = fast_exp2(fmaf(sv[k], sl2, neg_m));
                        } else {
#pragma unroll
                            for (int k = 0; k < 64; ++k)
                                sv[k] = (sv[k] == -INFINITY || m_run == -INFINITY) ? 0.f : fast_exp2(sv[k] + neg_m);
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            ls4[i & 3] += sv[2 * i] + sv[2 * i + 1];
                            pk[i] = pack_bf16x2(sv[2 * i], sv[2 * i + 1]);
                        }
                    }
                    lsum = (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
                    tmem_st32u(tmem + lane_off + st * 128 + col0, pk);
                    tmem_wait_st();
                }
                l_run += lsum;
                // V rows that carry no valid key for any query row are zeroed (stale or non-finite pool
                // bytes); only then does this tile need its V to have landed here
                const bool need_zero = (vm[0] & vm[1] & vm[2] & vm[3]) != ~0u;
                const int vs = g % kVStages;
                if (need_zero && ok && !mbar_wait(bars.v_full(vs), (g / kVStages) & 1)) ok = false;
                if (need_zero && ok && half == 0 && !((vm[r >> 5] >> (r & 31)) & 1u)) {
                    uint8_t* vrow = smem + kV + vs * kTileBytes;
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) *reinterpret_cast<uint4*>(vrow + h * kHalf + r * 128 + c8 * 16) = z;
                }
                if (need_zero) fence_proxy_async_smem();  // the zeroed rows before the PV MMA reads them
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(bars.p_full(st));
            }
            // ---- epilogue: O / l -> out (each thread stores its 64 columns of the row)
            const int g_last = gt + nt - 1;
            if (ok && nt > 0 && !mbar_wait(bars.o_done(g_last & 1), (g_last >> 1) & 1)) ok = false;
            tc_fence_after();
            // combine the halves: M = max(m_a, m_b), O = (f_a O_a + f_b O_b) / (f_a l_a + f_b l_b),
            // f_x = 2^(m_x - M); the states cross through TMEM columns 0-3 of S0 (free now: the MMA warp
            // starts the next item only after o_free)
            // (an item without keys has no state to combine and must not touch tensor memory, which the MMA
            // warp may already be filling for the next item)
            float m_oth = -INFINITY, l_oth = 0.f;
            if (nt > 0) {
                tmem_st1(tmem + lane_off + half, m_run);
                tmem_st1(tmem + lane_off + 2 + half, l_run);
                tmem_wait_st();
                tc_fence_before();
                softmax_bar();
                tc_fence_after();
                m_oth = tmem_ld1(tmem + lane_off + (half ^ 1));
                l_oth = tmem_ld1(tmem + lane_off + 2 + (half ^ 1));
                tmem_wait_ld();
            }
            const float m_a = half ? m_oth : m_run, m_b = half ? m_run : m_oth;
            const float l_a = half ? l_oth : l_run, l_b = half ? l_run : l_oth;
            const float m_row = fmaxf(m_a, m_b);
            const float f_a = m_a == -INFINITY ? 0.f : fast_exp2(m_a - m_row);
            const float f_b = m_b == -INFINITY ? 0.f : fast_exp2(m_b - m_row);
            const float l_row = f_a * l_a + f_b * l_b;
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
            const float wa = f_a * inv, wb = f_b * inv;  // weights of O_a and O_b in this row's output
            // member sequence r0 + pos, head r % G of a cascade prefix pass: its partial (o, m, l) goes to
            // workspace slot 0; a member whose own prefix length differs from the group's gets an empty one
            const int sm = r0 + pos;
            const bool same = prefix_mode && row_ok && p.prefix_lens[sm] == start;
            if (prefix_mode && row_ok && !same && half == 0 && r % G == 0) count_error(p.error_count);
            const size_t slot = ((size_t)sm * p.num_kv_heads + kvh) * p.part_splits * G + (r % G);
            if (prefix_mode && row_ok && half == 0)
                p.part_ml[slot] = same ? make_float2(m_row, l_row) : make_float2(-INFINITY, 0.f);
            __nv_bfloat16* out = prefix_mode ? nullptr
                                             : static_cast<__nv_bfloat16*>(p.out) +
                                                   ((size_t)(r0 + pos) * p.num_q_heads + (size_t)kvh * G + (r % G)) * kD +
                                                   col0;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {  // my 64 output columns, 16 at a time
                float t[16];
                if (nt > 0) {
                    float u[16];
                    tmem_ld16(tmem + lane_off + kTmemOa + col0 + q4 * 16, t);
                    tmem_ld16(tmem + lane_off + kTmemOb + col0 + q4 * 16, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) t[i] = t[i] * wa + u[i] * wb;
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) t[i] = 0.f;
                }
                if (!row_ok) continue;
                // (the workspace partials are 256-byte aligned; the output takes 32-byte stores when its base
                // allows, 16-byte ones otherwise)
                if (prefix_mode) {
                    float* po = p.part_o + slot * kD + col0 + q4 * 16;
                    const float f = same ? 1.f : 0.f;
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        uint32_t w8[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) w8[i] = __float_as_uint(t[h8 * 8 + i] * f);
                        st_global_v8(po + h8 * 8, w8);
                    }
                } else {
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(t[2 * i], t[2 * i + 1]);
                    if (out_al32) {
                        st_global_v8(out + q4 * 16, pk);
                    } else {
                        uint4* o4 = reinterpret_cast<uint4*>(out + q4 * 16);
                        o4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        o4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            }
            if (nt > 0) {  // O has been read: the MMA warp may start the next item
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(bars.o_free());
            }
            gt += nt;
        }
        if (!ok && lane == 0) count_error(p.error_count);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool prefill_tc_supported(const PrefillParams& p, int dtype) {
    const int G = p.group, B = p.block_size;
    if (dtype != PA_BF16 || p.head_dim != kD) return false;
    if (G != 1 && G != 2 && G != 4 && G != 8) return false;
    if (B != 8 && B != 16 && B != 32 && B != 64 && B != 128) return false;
    if (((uintptr_t)p.q & 15) || ((uintptr_t)p.k_cache & 15) || ((uintptr_t)p.v_cache & 15) ||
        ((uintptr_t)p.out & 15))
        return false;
    if ((long long)p.num_blocks * B >= (1LL << 31)) return false;
    return p.num_chunks <= 65535 && p.num_kv_heads <= 65535;
}

int launch_prefill_tc(const PrefillParams& p, cudaStream_t stream) {
    CUtensorMap tmq, tmk, tmv;
    {
        auto enc = tensor_map_encoder();
        if (!enc) return PA_ERR_CUDA;
        const int G = p.group;
        // q as [total_q][Hq][D]: a box is 128/G positions x the G heads of one kv head x 64 columns
        cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.num_q_heads, (cuuint64_t)p.total_q};
        cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.num_q_heads * kD * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kTileQ / G)};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = enc(&tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.q), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return PA_ERR_UNSUPPORTED;
    }
    int rc = pool_tensor_map(&tmk, p.k_cache, p.num_blocks, p.block_size, p.num_kv_heads, kD);
    if (rc != PA_OK) return rc;
    if ((rc = pool_tensor_map(&tmv, p.v_cache, p.num_blocks, p.block_size, p.num_kv_heads, kD)) != PA_OK) return rc;
    if ((rc = ensure_dynamic_smem(reinterpret_cast<const void*>(prefill_tc_kernel), kSmemBytes)) != PA_OK) return rc;
    // persistent: one CTA per SM (or per work item, if fewer), each walking its share of the items
    const int pos_per_tile = kTileQ / p.group;
    const long long items = (long long)((p.max_q_len + pos_per_tile - 1) / pos_per_tile) * p.num_chunks *
                            p.num_kv_heads;
    if (items == 0) return PA_OK;
    int dev = 0, num_sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return check_launch();
    const int grid = (int)(items < num_sms ? items : num_sms);
    return launch_kernel(prefill_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, tmq, tmk, tmv, p);
}

}  // namespace pa
