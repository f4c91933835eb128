// decode_tc.cu — paged decode for bf16 and e4m3 pools on GB300: a persistent
// kernel with TMA-staged K/V blocks and warp-level tensor-core MMAs.
//
// What it computes ("PagedAttention学习笔记", 三、算法流程与数据结构: the kernel
// reads Q and the block table, gathers K/V block by block, then softmax(QK^T)V;
// "KV cache 显存管理…", PagedAttention 改变了什么: token -> logical block ->
// physical block -> offset):  for sequence s, query head h and its kv head
// h/G, out = softmax_j(scale q.k_j) v_j over the sequence's context.
//
// Work decomposition.  A work item is (sequence, partition of its context,
// kv head) — or, for e4m3 pools with an even number of kv heads, a pair of
// adjacent kv heads, whose rows sit side by side in the pool so that one box
// per block carries both; partitions are `partition` tokens (a multiple of
// 64).  Items are numbered densely: first partition 0 of every (sequence, kv
// head), numbered directly, then the later partitions sequence-major then
// partition then kv head, through a prefix sum of the per-sequence counts
// that every CTA's consumer warps compute once from context_lens while its
// producer starts on its first item.  Persistent CTAs (two per SM; three for
// single-head e4m3 items) start on the item of their own index and take the
// rest from a global counter in the workspace, so long and short sequences
// balance dynamically.  The cascade's queues, which begin with shared-prefix
// items, run on a separate instantiation (kPrefix), so that the prefix items'
// code does not shape the plain decode kernel's.
//
// Inside a CTA:
//  * Warp 4 is the producer.  For each 64-token stage it waits for a free
//    ring slot, publishes the stage's description (sequence, kv head,
//    valid-token mask) and issues one 3-D TMA copy per block of K and of V —
//    a physical block of one kv head is B rows of head_dim contiguous
//    elements at a row stride of Hkv*head_dim, one box {128 bytes, B rows,
//    row bytes/128 segments} of the pool viewed as [128-byte segment][row]
//    [128 bytes] — from separate lanes, so the boxes go out together (with an
//    L2 evict-first policy: each K/V byte is read once per call); on an
//    item's first stage it adds a 1-D bulk copy of the item's G query rows.
//    Everything else is off the per-stage path: the next item is claimed two
//    stages before the current one's last and described (with its first 32
//    block-table entries loaded, one per lane) a stage later, and the
//    valid-token masks of the stages covering a 32-entry chunk of the table
//    are worked out lane-parallel when the chunk is reached.  Claiming late
//    keeps a CTA from holding more than the rest of one item when the queue
//    runs dry.  Boxes land 128-byte swizzled (ldmatrix reads are bank-conflict
//    free) in a ring of kStages stages, completion counted on mbarriers; the
//    producer streams straight across item boundaries.
//  * Warps 0-3 consume 16 tokens of each stage apiece (two-head items: warps
//    0-1 take the first head and 2-3 the second, 32 tokens apiece).  The G <= 8 query
//    heads form the N=8 side of m16n8k16 tensor-core MMAs:
//        S^T[16 tok x 8 heads] = K[16 tok x D] . Q^T        (D/16 MMAs)
//        O^T[D x 8 heads]     += V^T[D x 16 tok] . P^T       (D/16 MMAs)
//    P^T goes from the accumulator layout to the B-operand layout with one
//    movmatrix transpose per 8x8 half.  Softmax is online, in base-2 units;
//    a warp's 16-token chunks of a stage (two for two-head items, four for a
//    shared prefix) share one step of it: one row max and one rescale of O.
//    bf16 pools use bf16 MMAs; e4m3 pools are widened to f16 in registers
//    (two codes per conversion) and use f16 MMAs, with the queries, already
//    scaled, in f16.
//  * Tokens past the context or in blocks with an invalid table entry are
//    masked (score -inf) and their V rows zeroed before the PV MMA, so stale
//    or non-finite pool contents never reach the output.
//  * On an item's last stage the consumers combine their states (per kv head)
//    through slabs in the K tile of the stage just consumed and write the output (one
//    partition) or a partial for the split-KV merge kernel (decode_merge.cu);
//    no fence, ticket or wait on other CTAs.  The producer keeps filling the
//    other stages of the ring meanwhile.
// Every wait is bounded, the consumers' epilogue barrier included (an
// mbarrier, not a named barrier, so a warp that gave up cannot strand the
// others); a timeout counts an error and the kernel still terminates.  Before
// a CTA exits, its producer waits (bounded) for the last phase it armed on
// every ring slot, so no bulk copy it issued is still landing in shared
// memory when the CTA is gone.  The work counter is reset by the last CTA to
// finish.
#include <atomic>
#include <climits>
#include <type_traits>

#include "decode_common.cuh"
#include "sm100_ptx.cuh"

namespace pa {
namespace {

// Ring depth and CTAs per SM (build-time knobs; the defaults are the measured best).
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 3
#endif
// K/V copies tagged evict-first in L2 (they are read once; tables, queries and partials stay).
#ifndef PA_DECODE_KV_EVICT_FIRST
#define PA_DECODE_KV_EVICT_FIRST 1
#endif
// How many stages before an item's last one the producer claims the next item: bf16 pools, e4m3 pools
// (measured against 1, 2 and 3 for each).
#ifndef PA_DECODE_CLAIM_STAGES
#define PA_DECODE_CLAIM_STAGES 3
#endif
#ifndef PA_DECODE_CLAIM_STAGES_FP8
#define PA_DECODE_CLAIM_STAGES_FP8 1
#endif
// e4m3 pools with an even number of kv heads: items of two kv heads.
#ifndef PA_DECODE_FP8_PAIRS
#define PA_DECODE_FP8_PAIRS 1
#endif
#ifndef PA_DECODE_FP8_STAGES
#define PA_DECODE_FP8_STAGES 3
#endif
#ifndef PA_DECODE_FP8_CTAS_PER_SM
#define PA_DECODE_FP8_CTAS_PER_SM 3
#endif
#ifndef PA_DECODE_CTAS_PER_SM
#define PA_DECODE_CTAS_PER_SM 2
#endif
constexpr int kMaxSeqsPersistent = PA_DECODE_CTAS_PER_SM == 1 ? 2048 : 1024;
constexpr int kMaxSeqsPairs = 768;

struct StageInfo {
    int s, kvh, split, nsplit;
    int flags;  // bit 0: first stage of its item, bit 1: last stage, bit 2: the item writes the output
    int ntok;   // tokens of this stage (0..64)
    unsigned long long valid;  // bit r: token row r holds a valid token
    int new_row;         // pa_decode_write: row of the sequence's newest token in this stage, or -1
    long long new_slot;  // and its pool slot
};

// kFp8: the pools hold e4m3 codes (one byte per element) instead of bf16.
// kPair: an item covers two adjacent kv heads, whose rows sit next to each
// other in the pool, so one box per block carries both (e4m3 pools: a 64-token
// stage of two heads is as many bytes as one of a single bf16 head).
template <int D, bool kFp8, bool kPair = false>
struct TcCfg {
    static constexpr int kRowBytes = kFp8 ? D : 2 * D;   // one token row of one kv head
    static constexpr int kHalves = kRowBytes / 128;       // 128-byte segments (swizzle rows) of a token row
    static constexpr int kHeads = kPair ? 2 : 1;          // kv heads per item
    static constexpr int kSegs = kHalves * kHeads;        // segments per token row of a block's box
    static constexpr int kStageTok = 64;
    // bf16 D=128: 32 KiB stages; bf16 D=64 and e4m3 D=128: 16 KiB stages, so more of them fit
    static constexpr int kStages = kSegs == 2 ? PA_DECODE_STAGES : kFp8 ? PA_DECODE_FP8_STAGES : 2 * PA_DECODE_STAGES;
    // e4m3 pools, one head per item: more, smaller CTAs per SM (more producers and consumers for the
    // same bytes)
    static constexpr int kCtasPerSm = kFp8 && !kPair ? PA_DECODE_FP8_CTAS_PER_SM : PA_DECODE_CTAS_PER_SM;
    static constexpr int kConsumerWarps = 4;
    static constexpr int kWarpsPerHead = kConsumerWarps / kHeads;
    static constexpr int kThreads = (kConsumerWarps + 1) * 32;
    static constexpr int kHalfBytes = kStageTok * 128;   // one half of a stage's K (or V) tile
    static constexpr int kTileBytes = kSegs * kHalfBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;   // K + V
    static constexpr int kQBytes = kHeads * 8 * D * 2;   // up to 8 query rows per kv head of the item
    // shared memory layout (offsets from a 1024-aligned base)
    static constexpr int kRing = 0;
    static constexpr int kQ = kRing + kStages * kStageBytes;
    // pa_decode_write: the newest token's K and V rows of the item, staged next to each stage
    static constexpr int kNew = kQ + kStages * kQBytes;
    static constexpr int kNewBytes = kFp8 ? 0 : 2 * D * 2;  // (no fused write into e4m3 pools)
    static constexpr int kCum = kNew + kStages * kNewBytes;  // int [kMaxSeqs + 1]
    // the consumers' cross-warp (m, l) exchange (two buffers of [warp][8] each), per-warp scan totals, item total
    // sequences per launch (the prefix sum lives in shared memory; two-head items keep a shorter one so
    // that their larger query slots fit)
    static constexpr int kMaxSeqs = kPair ? kMaxSeqsPairs : kMaxSeqsPersistent;
    static constexpr int kRed = kCum + ((kMaxSeqs + 1) * 4 + 63) / 64 * 64;
    static constexpr int kRedBytes = 2 * 2 * kConsumerWarps * 8 * 4;
    static constexpr int kScan = kRed + kRedBytes;
    static constexpr int kInfo = kScan + 64;
    static constexpr int kBars = kInfo + kStages * (int)sizeof(StageInfo);
    // full[kStages], empty[kStages], the consumers' epilogue barrier and the prefix sum's completion
    static constexpr int kCtx = kBars + (2 * kStages + 2) * 8;
    // an SM holds 228 KiB of shared memory, 1 KiB of it reserved per resident CTA, and 1 KiB of each CTA's
    // allocation goes to aligning the base; every array lives in the dynamic allocation
    static constexpr int kSmemCap = 228 * 1024 / kCtasPerSm - 2 * 1024;
    // the clamped context length of every sequence, where it fits (else read from global memory)
    static constexpr int kCtxN = kCtx + kMaxSeqs * 4 <= kSmemCap ? kMaxSeqs : 0;
    static constexpr int kEnd = kCtx + kCtxN * 4;
    static constexpr size_t kSmemBytes = 1024 + kEnd;
    static_assert(kEnd <= kSmemCap, "shared memory budget");
};

// Byte offset, within a stage's K (or V) tile, of 128-byte row r of half 0,
// and the distance between the halves of a row.  The 128-byte swizzle of a
// row depends on r & 7 either way: boxes start 1 KiB aligned and B >= 8.
struct TileRows {
    uint32_t half_stride, block_stride;
    int log2b;
    __device__ __forceinline__ uint32_t row(uint32_t r) const {
        return (r >> log2b) * block_stride + (r & ((1u << log2b) - 1u)) * 128u;
    }
    __device__ __forceinline__ uint32_t at(uint32_t r, uint32_t half, uint32_t chunk) const {
        return row(r) + half * half_stride + ((chunk ^ (r & 7u)) << 4);
    }
};

// Item -> (sequence, partition, kv head) through the prefix sum cum[0..N] of
// the per-sequence item counts: the largest s with cum[s] <= item.
__device__ __forceinline__ void decode_item(const int* cum, int N, int Hkv, int item, int& s, int& split, int& kvh) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= item) lo = mid; else hi = mid - 1;
    }
    s = lo;
    int r = item - cum[lo];
    split = r / Hkv;
    kvh = r - split * Hkv;
}

// kPrefix: the cascade's kernel, whose queue begins with shared-prefix items (a separate instantiation, so that
// the prefix items' four-chunk code does not shape the plain decode kernel's)
template <int D, bool kFp8, bool kPair, bool kPrefix>
__global__ void __launch_bounds__(TcCfg<D, kFp8, kPair>::kThreads, TcCfg<D, kFp8, kPair>::kCtasPerSm)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const DecodeParams p, int* work) {
    using C = TcCfg<D, kFp8, kPair>;
    static_assert(!kFp8 || D == 128, "fp8 pools: head_dim 128");
    static_assert(!kPair || kFp8, "kv-head pairs: e4m3 pools");
    constexpr int KT = D / 16;  // 16-wide k steps (QK^T) and m tiles (PV)
    const int N = p.num_seqs, Hkv = p.num_kv_heads, G = p.group, B = p.block_size;
    const int HkvI = Hkv / C::kHeads;  // items per partition

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* cum = reinterpret_cast<int*>(smem + C::kCum);
    int* ctx = reinterpret_cast<int*>(smem + C::kCtx);  // clamped context lengths (when C::kCtxN > 0)
    StageInfo* info = reinterpret_cast<StageInfo*>(smem + C::kInfo);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBars);
    uint64_t* empty = full + C::kStages;
    uint64_t* cons_bar = empty + C::kStages;  // the consumer warps' epilogue barrier (bounded)
    uint64_t* cum_bar = cons_bar + 1;         // the consumers' prefix sum (cum, ctx, s_total) is written
    auto red_m = reinterpret_cast<float(*)[C::kConsumerWarps][8]>(smem + C::kRed);
    auto red_l = reinterpret_cast<float(*)[C::kConsumerWarps][8]>(smem + C::kRed + C::kRedBytes / 2);
    int* warp_tot = reinterpret_cast<int*>(smem + C::kScan);
    int& s_total = warp_tot[C::kThreads / 32];
    static_assert(C::kThreads / 32 + 1 <= 16, "scan totals");
    auto context_of = [&](int s) { return C::kCtxN ? ctx[s] : decode_context(p, s, false); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], C::kConsumerWarps);
        }
        mbar_init(cons_bar, C::kConsumerWarps);
        mbar_init(cum_bar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // ---- Item numbering.  Plain decode: items [0, N*HkvI) are the partition-0 items, (sequence i / HkvI,
    // kv head slot i % HkvI), numbered without any table, so that a CTA's first copies wait only for its own
    // sequence's context length and table entries; then the (sequence, partition >= 1, kv head slot) items
    // through the exclusive prefix sum cum[] of the per-sequence counts of those.  The cascade's kernel
    // numbers every (sequence, partition, kv head) item through cum[], after its groups' prefix items.
    // The consumer warps compute cum[] (and the clamped context lengths) while the producer starts its
    // first item, and signal cum_bar when it is written.  (Queueing every sequence's short last partition
    // after all the whole ones was measured 5-7% slower.)
    constexpr bool kDirect = !kPrefix;
    const int n_first = kDirect ? N * HkvI : 0;  // items numbered directly
    auto counted_items = [&](int L, int s) {
        int pre;
        return (num_partitions(L - decode_start(p, s, L, &pre), partition_of(p, s)) - (kDirect ? 1 : 0)) * HkvI;
    };
    if (warp < C::kConsumerWarps) {
        constexpr int kScanThreads = C::kConsumerWarps * 32;
        auto consumer_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kScanThreads) : "memory"); };
        const int per = (N + kScanThreads - 1) / kScanThreads;
        const int first = threadIdx.x * per;
        int local = 0;
        for (int i = 0; i < per && first + i < N; ++i)
            local += counted_items(decode_context(p, first + i, blockIdx.x == 0), first + i);
        int incl = local;  // inclusive scan over the warp
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) warp_tot[warp] = incl;
        consumer_sync();
        int run = incl - local;
        for (int w = 0; w < warp; ++w) run += warp_tot[w];
        for (int i = 0; i < per && first + i < N; ++i) {
            cum[first + i] = run;
            const int L = decode_context(p, first + i, false);
            if (C::kCtxN) ctx[first + i] = L;
            run += counted_items(L, first + i);
        }
        if (threadIdx.x == kScanThreads - 1) {
            int tot = 0;
            for (int w = 0; w < C::kConsumerWarps; ++w) tot += warp_tot[w];
            s_total = tot;
            cum[N] = tot;
        }
        consumer_sync();
        if (threadIdx.x == 0) mbar_arrive(cum_bar);  // releases every consumer's writes (ordered by the barrier)
    }
    // items: the cascade groups' shared prefixes (one per group and kv head) first, then the
    // (sequence, partition, kv head) items
    const int n_grouped = kPrefix && p.group_offsets ? p.num_groups * Hkv : 0;

    if (warp == C::kConsumerWarps) {
        // ================================================================ producer
        // Per stage the producer only waits for its ring slot, publishes the
        // stage's description and issues the copies: each item's block-table
        // entries are loaded one item ahead, and the valid-token masks of a
        // 32-block chunk of the table are worked out lane-parallel (lane l for
        // the chunk's stage l) when the chunk is reached.
        if (lane == 0) {
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
        }
        struct Item {
            int s, split, kvh, nsplit, pre, j0, ntok, L;
            bool grouped;
        };
        auto describe = [&](int it) {
            Item d;
            d.grouped = it < n_grouped;
            if (d.grouped) {
                // a cascade group's shared prefix for one kv head: tokens [0, P) of its first sequence,
                // the group's G x members query rows at once (members * G <= 32)
                const int g = it / Hkv;
                d.kvh = it - g * Hkv;
                int s0 = p.group_offsets[g];
                int members = p.group_offsets[g + 1] - s0;
                if (s0 < 0 || members < 1 || s0 + members > N || members * G > 32) {
                    if (lane == 0) count_error(p.error_count);
                    s0 = 0;
                    members = 0;
                }
                int pre = 0;
                if (members) decode_start(p, s0, context_of(s0), &pre);
                d.s = s0;
                d.nsplit = members;  // carried to the consumers in StageInfo::nsplit
                d.split = pre;       // and the prefix length in StageInfo::split
                d.pre = pre;
                d.j0 = 0;
                d.ntok = pre;
                d.L = 0;
            } else {
                const int i = it - n_grouped;
                if (i < n_first) {  // a partition-0 item (its context length read from global memory: the
                                    // shared-memory copy may not be written yet)
                    d.s = i / HkvI;
                    d.split = 0;
                    d.kvh = i - d.s * HkvI;
                    d.L = decode_context(p, d.s, false);
                } else {
                    decode_item(cum, N, HkvI, i - n_first, d.s, d.split, d.kvh);
                    d.split += kDirect ? 1 : 0;
                    d.L = context_of(d.s);
                }
                d.kvh *= C::kHeads;  // the item's first kv head
                const int j_first = decode_start(p, d.s, d.L, &d.pre);
                const int part = partition_of(p, d.s);
                d.nsplit = num_partitions(d.L - j_first, part);
                d.j0 = j_first + d.split * part;
                d.ntok = max(0, min(d.L, d.j0 + part) - d.j0);
            }
            return d;
        };
        // raw table entry of block (chunk * 32 + lane) of an item; checked when the chunk is used
        auto load_chunk = [&](const Item& d, int chunk) {
            const int idx = chunk * 32 + lane;
            return idx < (d.ntok + B - 1) / B ? p.block_tables[(size_t)d.s * p.max_blocks_per_seq + d.j0 / B + idx]
                                              : -1;
        };
        const int bps = C::kStageTok / B;   // blocks per stage (B <= 64)
        const int spc = 32 / bps;           // stages per 32-block chunk of the table
        const uint32_t block_bytes = 2u * C::kSegs * B * 128u;  // K and V of one block and the item's kv heads
        const uint64_t kv_policy = l2_policy_evict_first();  // K/V is read once per call

        // the first item is the CTA's own index (no claim on the way to the first copies); later claims take
        // the counter's places after the grid's
        int item = blockIdx.x;
        int nxt = 0;  // the item after this one (lane 0), claimed a few stages before this one's last
        bool ok = true;
        // the item count, known once the consumers' prefix sum is in; items below n_grouped + n_first exist
        // without it
        int total = -1;
        auto is_item = [&](int it) {
            if (it < n_grouped + n_first) return true;
            if (total < 0) {
                total = 0;
                if (mbar_wait_warp(cum_bar, 0)) total = n_grouped + n_first + s_total;
                else ok = false;
            }
            return it < total;
        };
        Item d{};
        int raw = -1;
        if (is_item(item)) {
            d = describe(item);
            raw = load_chunk(d, 0);
        }
        uint32_t stage_no = 0;  // stages issued by this CTA
        while (ok && is_item(item)) {
            const int nst = max(1, (d.ntok + C::kStageTok - 1) / C::kStageTok);
            const int nblk = (d.ntok + B - 1) / B;
            int pb_lane = -1;                 // physical block of this lane's table entry in the current chunk
            unsigned long long lvalid = 0ull; // lane l: valid-token mask of the chunk's stage l
            int lnvb = 0;                     // and how many of its blocks are loaded
            int item2 = INT_MAX, raw2 = -1;
            Item d2{};
            // The next item is claimed when kClaimStages stages of this one are left to issue and
            // described (with its first table chunk loaded) one stage later, so the claim's latency is hidden
            // while a CTA never holds more than the rest of one item when the queue runs dry.
            constexpr int kClaimStages = kFp8 ? PA_DECODE_CLAIM_STAGES_FP8 : PA_DECODE_CLAIM_STAGES;
            const int claim_at = max(0, nst - kClaimStages), describe_at = min(nst - 1, claim_at + 1);
            for (int st = 0; st < nst; ++st) {
                const int slot = stage_no % C::kStages;
                const int chunk = st / spc, l = st - chunk * spc;
                if (l == 0) {
                    if (chunk > 0) raw = load_chunk(d, chunk);
                    pb_lane = -1;
                    if (chunk * 32 + lane < nblk) {
                        pb_lane = raw;
                        if (raw < 0 || raw >= p.num_blocks) {
                            count_error(p.error_count);
                            pb_lane = -1;
                        }
                    }
                    // lane l: stage chunk * spc + l
                    const int t0l = (chunk * spc + lane) * C::kStageTok;
                    const int ntl = max(0, min(C::kStageTok, d.ntok - t0l));
                    lvalid = 0ull;
                    lnvb = 0;
                    for (int b = 0; b < bps; ++b) {
                        const int pb = __shfl_sync(0xffffffffu, pb_lane, (lane * bps + b) & 31);
                        const int cnt = min(B, ntl - b * B);
                        if (pb >= 0 && cnt > 0) {
                            lvalid |= (cnt >= 64 ? ~0ull : ((1ull << cnt) - 1ull)) << (b * B);
                            ++lnvb;
                        }
                    }
                    const int skip = d.grouped ? 0 : d.pre - (d.j0 + t0l);  // a tail's first stage: mask the prefix
                    if (skip > 0) lvalid &= skip >= 64 ? 0ull : ~((1ull << skip) - 1ull);
                }
                if (stage_no >= (uint32_t)C::kStages &&
                    !mbar_wait_warp(&empty[slot], ((stage_no / C::kStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int t0 = st * C::kStageTok;
                const int nt = max(0, min(C::kStageTok, d.ntok - t0));
                const int nbs = (nt + B - 1) / B;  // blocks of this stage
                const int b0 = l * bps;            // its first block within the chunk
                const unsigned long long valid = __shfl_sync(0xffffffffu, lvalid, l);
                uint32_t bytes = (uint32_t)__shfl_sync(0xffffffffu, lnvb, l) * block_bytes;
                if (st == 0 && !d.grouped) bytes += (uint32_t)(C::kHeads * G * D * 2);
                // pa_decode_write(_fp8): the sequence's newest token (position L - 1) falls in this stage.  bf16
                // pools: its K and V rows are staged next to the stage; e4m3 pools: the consumer warp that owns
                // the row loads and quantises them itself (the rows are prefetched into L2 here)
                int new_row = -1;
                long long new_slot = -1;
                if ((C::kNewBytes || kFp8) && p.k_new && !d.grouped) {
                    const int jn = d.L - 1 - (d.j0 + t0);
                    const bool here = d.L > 0 && jn >= 0 && jn < nt;
                    const int pbn = __shfl_sync(0xffffffffu, pb_lane, (b0 + (here ? jn / B : 0)) & 31);
                    if (here && pbn >= 0) {
                        new_row = jn;
                        new_slot = (long long)pbn * B + (d.L - 1) % B;
                        bytes += (uint32_t)C::kNewBytes;
                        if (kFp8 && lane < 4 * C::kHeads) {  // K and V rows of each kv head: 256 bytes, 2 lines each
                            const int hh = lane >> 2, isv = (lane >> 1) & 1, half = lane & 1;
                            const __nv_bfloat16* row = static_cast<const __nv_bfloat16*>(isv ? p.v_new : p.k_new) +
                                                       ((size_t)d.s * Hkv + d.kvh + hh) * D + half * 64;
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
                        }
                    }
                }
                if (lane == 0) {
                    StageInfo& inf = info[slot];
                    inf.s = d.s;
                    inf.kvh = d.kvh;
                    inf.split = d.split;
                    inf.nsplit = d.nsplit;
                    inf.flags = (st == 0 ? 1 : 0) | (st == nst - 1 ? 2 : 0) |
                                (!d.grouped && d.nsplit == 1 && d.pre == 0 ? 4 : 0) | (d.grouped ? 16 : 0);
                    inf.ntok = nt;
                    inf.valid = valid;
                    inf.new_row = new_row;
                    inf.new_slot = new_slot;
                    mbar_arrive_expect_tx(&full[slot], bytes);
                    if (C::kNewBytes && new_row >= 0) {  // bf16 pools: stage the newest token's rows
                        const size_t row = ((size_t)d.s * Hkv + d.kvh) * D;
                        bulk_load(smem + C::kNew + slot * C::kNewBytes,
                                  static_cast<const __nv_bfloat16*>(p.k_new) + row, (uint32_t)(D * 2), &full[slot]);
                        bulk_load(smem + C::kNew + slot * C::kNewBytes + D * 2,
                                  static_cast<const __nv_bfloat16*>(p.v_new) + row, (uint32_t)(D * 2), &full[slot]);
                    }
                    if (st == 0 && !d.grouped)
                        bulk_load(smem + C::kQ + slot * C::kQBytes,
                                  static_cast<const __nv_bfloat16*>(p.q) +
                                      ((size_t)d.s * p.num_q_heads + (size_t)d.kvh * G) * D,
                                  (uint32_t)(C::kHeads * G * D * 2), &full[slot]);
                }
                __syncwarp();  // the transaction count is armed before any copy is issued
                // lanes [0, nbs) copy the stage's K blocks and lanes [nbs, 2 nbs) its V blocks, so the
                // boxes go out together
                uint8_t* kdst = smem + C::kRing + slot * C::kStageBytes;
                const int isv = lane >= nbs;
                const int b = lane - isv * nbs;
                const int my_pb = __shfl_sync(0xffffffffu, pb_lane, (b0 + (lane < 2 * nbs ? b : 0)) & 31);
                if (lane < 2 * nbs && my_pb >= 0)
                    if (PA_DECODE_KV_EVICT_FIRST)
                        tma_load_3d_hint(kdst + isv * C::kTileBytes + b * C::kSegs * B * 128, isv ? &tmv : &tmk, 0,
                                         my_pb * B, d.kvh * C::kHalves, &full[slot], kv_policy);
                    else
                        tma_load_3d(kdst + isv * C::kTileBytes + b * C::kSegs * B * 128, isv ? &tmv : &tmk, 0,
                                    my_pb * B, d.kvh * C::kHalves, &full[slot]);
                __syncwarp();
                ++stage_no;
                if (st == claim_at && lane == 0) nxt = (int)gridDim.x + atomicAdd(&work[0], 1);
                if (st == describe_at) {
                    item2 = __shfl_sync(0xffffffffu, nxt, 0);
                    if (is_item(item2)) {
                        d2 = describe(item2);
                        raw2 = load_chunk(d2, 0);
                    }
                }
            }
            item = item2;
            d = d2;
            raw = raw2;
        }
        // terminator stage: armed only once its slot is free (the consumers released the slot, so the
        // slot's previous phase of `full` has completed and a new arrival starts the next phase)
        uint32_t armed = stage_no;  // phases of `full` armed so far, in ring order
        {
            const int slot = stage_no % C::kStages;
            const bool free_slot =
                stage_no < (uint32_t)C::kStages || mbar_wait_warp(&empty[slot], ((stage_no / C::kStages) - 1) & 1);
            if (lane == 0) {
                if (!ok || !free_slot) count_error(p.error_count);
                if (free_slot) {
                    info[slot].s = -1;
                    info[slot].flags = 0;
                    mbar_arrive_expect_tx(&full[slot], 0);
                }
            }
            if (free_slot) ++armed;
        }
        // drain: every copy this CTA issued has landed before it exits.  On the normal path the consumers
        // have waited for every armed phase already and this returns at once; after a timeout it keeps
        // the CTA (and its shared memory) alive until the copies in flight complete.
        if (lane == 0 && !drain_ring(full, C::kStages, armed)) count_error(p.error_count);
        __syncwarp();
    } else {
        // ================================================================ consumers
        const int g4 = lane >> 2, c4 = lane & 3;
        // this warp's kv head within the item and its token rows in every stage: 16 rows of the one
        // head, or 32 rows of one of the two
        const int hp = C::kHeads == 2 ? warp >> 1 : 0;
        const int row0 = C::kHeads == 2 ? (warp & 1) * 32 : warp * 16;
        const int tid = threadIdx.x;  // 0..127
        uint32_t qb[KT][2];
        float o[KT][4];
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            qb[i][0] = qb[i][1] = 0u;
            o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        }
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2*c4 and 2*c4+1
        // base-2 score scale: fp8 pools fold the softmax scale into the f16 queries and the K scale here
        const float sl2 = kFp8 ? p.k_scale : p.scale_log2;
        int item_parity = 0;
        // the item epilogue's barrier among the four consumer warps: an mbarrier with a bounded wait, so a
        // consumer warp that gave up on a stage can never leave the others blocked in an epilogue
        BoundedWarpBarrier cbar{cons_bar, 0u};
        const TileRows tr{(uint32_t)B * 128u, (uint32_t)(C::kSegs * B * 128), __ffs(B) - 1};
        for (uint32_t stage_no = 0;; ++stage_no) {
            const int slot = stage_no % C::kStages;
            if (!mbar_wait_warp(&full[slot], (stage_no / C::kStages) & 1)) {
                if (lane == 0) count_error(p.error_count);
                break;
            }
            const StageInfo inf = info[slot];
            if (inf.s < 0) break;
            if (kPrefix && (inf.flags & 17) == 17) {  // first stage of a shared-prefix item: this warp's 8 rows from global
                // row 8*warp + g4 is member (row / G), head (row % G) of the group's first sequence inf.s
                const int rr = warp * 8 + g4, mem = rr / G, head = rr - mem * G;
                const bool row_ok = mem < inf.nsplit;
                const uint32_t* qg = reinterpret_cast<const uint32_t*>(
                    static_cast<const __nv_bfloat16*>(p.q) +
                    ((size_t)(inf.s + (row_ok ? mem : 0)) * p.num_q_heads + (size_t)inf.kvh * G + head) * D);
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    qb[kk][0] = row_ok ? __ldg(qg + kk * 8 + c4) : 0u;
                    qb[kk][1] = row_ok ? __ldg(qg + kk * 8 + c4 + 4) : 0u;
                }
            } else if ((inf.flags & 1) && kFp8) {
                // fp8 pools: q * scale * log2(e) as f16, in the k order the e4m3 K fragments arrive in
                // (lane (g4, c4) of the 32-column group kq holds columns 4c4..4c4+3 and 16+4c4..16+4c4+3:
                // fragment 2kq takes the first two of each four, fragment 2kq+1 the last two)
                const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(smem + C::kQ + slot * C::kQBytes);
                const float qsc = p.scale_log2;
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    const int base = (kk >> 1) * 32 + 4 * c4 + (kk & 1) * 2;
                    if (g4 < G) {
                        const __nv_bfloat16* r = qs + (hp * G + g4) * D;
                        qb[kk][0] = pack_f16x2(__bfloat162float(r[base]) * qsc, __bfloat162float(r[base + 1]) * qsc);
                        qb[kk][1] = pack_f16x2(__bfloat162float(r[base + 16]) * qsc,
                                               __bfloat162float(r[base + 17]) * qsc);
                    } else {
                        qb[kk][0] = qb[kk][1] = 0u;
                    }
                }
            } else if (inf.flags & 1) {  // first stage of an item: load its queries
                const uint8_t* qs = smem + C::kQ + slot * C::kQBytes;
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    if (g4 < G) {
                        qb[kk][0] = *reinterpret_cast<const uint32_t*>(qs + (g4 * D + kk * 16 + 2 * c4) * 2);
                        qb[kk][1] = *reinterpret_cast<const uint32_t*>(qs + (g4 * D + kk * 16 + 2 * c4 + 8) * 2);
                    } else {
                        qb[kk][0] = qb[kk][1] = 0u;
                    }
                }
            }
            if (inf.flags & 1) {  // fresh softmax state
#pragma unroll
                for (int i = 0; i < KT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
            }
            uint8_t* kt = smem + C::kRing + slot * C::kStageBytes;
            uint8_t* vt = kt + C::kTileBytes;
            // pa_decode_write_fp8: the newest token's K and V rows of this warp's kv head, when the token is one of
            // rows [rlo, rhi) of the stage, quantised here (code = e4m3(x * (1/scale)), four elements per lane)
            // into the tiles, before any ldmatrix of the row, and into the pools at its slot
            auto patch_new_fp8 = [&](int rlo, int rhi) {
                if (!kFp8 || inf.new_row < rlo || inf.new_row >= rhi) return;
                const int kvh_h = inf.kvh + hp;
                const size_t roff = ((size_t)inf.s * Hkv + kvh_h) * D;
                const uint2 kx = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.k_new) + roff) + lane);
                const uint2 vx = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.v_new) + roff) + lane);
                const uint32_t kc = e4m3x4_of_bf16x4(kx, p.k_inv), vc = e4m3x4_of_bf16x4(vx, p.v_inv);
                const uint32_t off = tr.at(inf.new_row, hp, lane >> 2) + (lane & 3) * 4;
                *reinterpret_cast<uint32_t*>(kt + off) = kc;
                *reinterpret_cast<uint32_t*>(vt + off) = vc;
                const size_t poff = ((size_t)inf.new_slot * Hkv + kvh_h) * D;
                reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.k_write) + poff)[lane] = kc;
                reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.v_write) + poff)[lane] = vc;
                if (p.new_slots && kvh_h == 0 && lane == 0) p.new_slots[inf.s] = inf.new_slot;
                fence_proxy_async_smem();  // these writes precede the slot's next TMA write
                __syncwarp();
            };
            // NC chunks of 16 token rows from row r0 of the stage (validity bits in `valid`) against this warp's 8
            // query rows, in one online-softmax step: the chunks' scores (independent MMA chains), one row max and
            // one rescale of the output for all of them, then each chunk's P V.  A chunk without a valid token is
            // skipped (it would add nothing); in one with some, the V rows of invalid tokens are zeroed first.
            auto chunks = [&](auto nc, const int r0, const unsigned long long valid) {
                constexpr int NC = decltype(nc)::value;
                uint32_t rows[NC];
                bool zeroed = false;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    rows[c] = (uint32_t)(valid >> (r0 + 16 * c)) & 0xFFFFu;  // (r0 + 16 c <= 48)
                    if (rows[c] != 0u && rows[c] != 0xFFFFu) {  // zero V rows without a valid token
                        zeroed = true;
                        const int r = lane >> 1;
                        if (!((rows[c] >> r) & 1u)) {
                            const int4 z = make_int4(0, 0, 0, 0);
#pragma unroll
                            for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    *reinterpret_cast<int4*>(vt + tr.row(r0 + 16 * c + r) +
                                                             (hp * C::kHalves + h) * tr.half_stride +
                                                             ((lane & 1) * 4 + q) * 16) = z;
                        }
                    }
                }
                if (zeroed) __syncwarp();
                float x[NC][4];
                bool all_active = true;  // (four-chunk path) every chunk holds a valid token
                if constexpr (NC >= 4) {
                    // Four chunks (the 64 tokens of a shared prefix's stage; bf16 pools only): S^T = K Q^T per
                    // chunk (two independent accumulation chains each); with all four active the chunks advance
                    // together, k step by k step, so that their MMA chains overlap (cascade decode 116.2 ->
                    // 114.2 us; the same for the two chunks of an e4m3 pair item measured 1.5 us slower), else they
                    // go one at a time.  Each chain gets the same MMAs in the same order either way.
                    static_assert(!kFp8 || NC < 4, "shared-prefix items read bf16 pools");
#pragma unroll
                    for (int c = 0; c < NC; ++c) all_active = all_active && rows[c] != 0u;
                    float sa[NC][4], sb[NC][4];
#pragma unroll
                    for (int c = 0; c < NC; ++c)
#pragma unroll
                        for (int i = 0; i < 4; ++i) sa[c][i] = sb[c][i] = 0.f;
                    const uint32_t kbase = smem_u32(kt);
                    const uint32_t krow = (lane & 7) + ((lane >> 3) & 1) * 8;
                    auto qk_step = [&](int c, int kk) {  // 16 columns of chunk c: even steps into sa, odd ones into sb
                        const uint32_t half = kk >> 2, ch = (kk & 3) * 2 + (lane >> 4);
                        uint32_t a[4];
                        ldmatrix_x4(a, kbase + tr.at(r0 + 16 * c + krow, half, ch));
                        if (kk & 1) mma_bf16_16816(sb[c], a, qb[kk][0], qb[kk][1]);
                        else mma_bf16_16816(sa[c], a, qb[kk][0], qb[kk][1]);
                    };
                    if (all_active) {
#pragma unroll
                        for (int kk = 0; kk < KT; ++kk)
#pragma unroll
                            for (int c = 0; c < NC; ++c) qk_step(c, kk);
                    } else {
#pragma unroll
                        for (int c = 0; c < NC; ++c) {
                            if (rows[c] == 0u) continue;
#pragma unroll
                            for (int kk = 0; kk < KT; ++kk) qk_step(c, kk);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const bool vlo = rows[c] != 0u && ((rows[c] >> g4) & 1u);
                        const bool vhi = rows[c] != 0u && ((rows[c] >> (g4 + 8)) & 1u);
                        x[c][0] = vlo ? (sa[c][0] + sb[c][0]) * sl2 : -INFINITY;
                        x[c][1] = vlo ? (sa[c][1] + sb[c][1]) * sl2 : -INFINITY;
                        x[c][2] = vhi ? (sa[c][2] + sb[c][2]) * sl2 : -INFINITY;
                        x[c][3] = vhi ? (sa[c][3] + sb[c][3]) * sl2 : -INFINITY;
                    }
                } else {
                    // S^T = K Q^T per chunk (two independent accumulation chains each)
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        if (rows[c] == 0u) {
                            x[c][0] = x[c][1] = x[c][2] = x[c][3] = -INFINITY;
                            continue;
                        }
                        const int r0c = r0 + 16 * c;
                        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                        if constexpr (kFp8) {
                            // one ldmatrix.x4 per 32 e4m3 columns: each register holds four consecutive codes of a row,
                            // the low two feeding fragment 2kq and the high two fragment 2kq+1 (f16 after conversion)
                            const uint32_t r = r0c + (lane & 7) + ((lane >> 3) & 1) * 8;
                            const uint32_t kbase = smem_u32(kt);
#pragma unroll
                            for (int kq = 0; kq < D / 32; ++kq) {
                                uint32_t raw[4], a[4];
                                ldmatrix_x4(raw, kbase + tr.at(r, hp, 2 * kq + (lane >> 4)));
#pragma unroll
                                for (int i = 0; i < 4; ++i) a[i] = e4m3x2_to_f16x2(raw[i] & 0xFFFFu);
                                mma_f16_16816(sa, a, qb[2 * kq][0], qb[2 * kq][1]);
#pragma unroll
                                for (int i = 0; i < 4; ++i) a[i] = e4m3x2_to_f16x2(raw[i] >> 16);
                                mma_f16_16816(sb, a, qb[2 * kq + 1][0], qb[2 * kq + 1][1]);
                            }
                        } else {
                            const uint32_t r = r0c + (lane & 7) + ((lane >> 3) & 1) * 8;
                            const uint32_t kbase = smem_u32(kt);
#pragma unroll
                            for (int kk = 0; kk < KT; ++kk) {
                                const uint32_t half = kk >> 2, ch = (kk & 3) * 2 + (lane >> 4);
                                uint32_t a[4];
                                ldmatrix_x4(a, kbase + tr.at(r, half, ch));
                                if (kk & 1) mma_bf16_16816(sb, a, qb[kk][0], qb[kk][1]);
                                else mma_bf16_16816(sa, a, qb[kk][0], qb[kk][1]);
                            }
                        }
                        const bool vlo = (rows[c] >> g4) & 1u, vhi = (rows[c] >> (g4 + 8)) & 1u;
                        x[c][0] = vlo ? (sa[0] + sb[0]) * sl2 : -INFINITY;
                        x[c][1] = vlo ? (sa[1] + sb[1]) * sl2 : -INFINITY;
                        x[c][2] = vhi ? (sa[2] + sb[2]) * sl2 : -INFINITY;
                        x[c][3] = vhi ? (sa[3] + sb[3]) * sl2 : -INFINITY;
                    }
                }
                float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
                for (int c = 1; c < NC; ++c) {
                    mx0 = fmaxf(mx0, fmaxf(x[c][0], x[c][2]));
                    mx1 = fmaxf(mx1, fmaxf(x[c][1], x[c][3]));
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float a0 = mn0 == -INFINITY ? 1.f : fast_exp2(m0 - mn0);
                const float a1 = mn1 == -INFINITY ? 1.f : fast_exp2(m1 - mn1);
                float s0 = 0.f, s1 = 0.f;  // (x becomes p = 2^(x - m))
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    x[c][0] = mn0 == -INFINITY ? 0.f : fast_exp2(x[c][0] - mn0);
                    x[c][2] = mn0 == -INFINITY ? 0.f : fast_exp2(x[c][2] - mn0);
                    x[c][1] = mn1 == -INFINITY ? 0.f : fast_exp2(x[c][1] - mn1);
                    x[c][3] = mn1 == -INFINITY ? 0.f : fast_exp2(x[c][3] - mn1);
                    s0 += x[c][0] + x[c][2];
                    s1 += x[c][1] + x[c][3];
                }
                l0 = l0 * a0 + s0;
                l1 = l1 * a1 + s1;
                m0 = mn0;
                m1 = mn1;
#pragma unroll
                for (int mt = 0; mt < KT; ++mt) {
                    o[mt][0] *= a0;
                    o[mt][1] *= a1;
                    o[mt][2] *= a0;
                    o[mt][3] *= a1;
                }
                if constexpr (NC >= 4) {
                    // O^T += V^T P^T for four chunks, advancing together when all are active (as the scores above)
                    uint32_t pb0[NC], pb1[NC];  // P^T of each chunk in the B-operand layout
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        pb0[c] = movmatrix_trans(pack_bf16x2(x[c][0], x[c][1]));
                        pb1[c] = movmatrix_trans(pack_bf16x2(x[c][2], x[c][3]));
                    }
                    const uint32_t vbase = smem_u32(vt);
                    const uint32_t vrow = (lane & 7) + (lane >> 4) * 8;
                    auto pv_step = [&](int c, int mt) {  // 16 output columns from chunk c
                        const uint32_t half = mt >> 2, ch = (mt & 3) * 2 + ((lane >> 3) & 1);
                        uint32_t a[4];
                        ldmatrix_x4_trans(a, vbase + tr.at(r0 + 16 * c + vrow, half, ch));
                        mma_bf16_16816(o[mt], a, pb0[c], pb1[c]);
                    };
                    if (all_active) {
#pragma unroll
                        for (int mt = 0; mt < KT; ++mt)
#pragma unroll
                            for (int c = 0; c < NC; ++c) pv_step(c, mt);
                    } else {
#pragma unroll
                        for (int c = 0; c < NC; ++c) {
                            if (rows[c] == 0u) continue;
#pragma unroll
                            for (int mt = 0; mt < KT; ++mt) pv_step(c, mt);
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        if (rows[c] == 0u) continue;
                        const int r0c = r0 + 16 * c;
                        const uint32_t b0 =
                            movmatrix_trans(kFp8 ? pack_f16x2(x[c][0], x[c][1]) : pack_bf16x2(x[c][0], x[c][1]));
                        const uint32_t b1 =
                            movmatrix_trans(kFp8 ? pack_f16x2(x[c][2], x[c][3]) : pack_bf16x2(x[c][2], x[c][3]));
                        if constexpr (kFp8) {
                            // O^T += V^T P^T: ldmatrix.trans of 16-bit pairs gives a lane the codes of tokens 2c4 and
                            // 2c4+1 at columns 2g4 and 2g4+1; a byte permutation regroups them per column, so
                            // fragment 2kv holds the even columns of the 32-column group kv and 2kv+1 the odd ones
                            const uint32_t r = r0c + (lane & 7) + (lane >> 4) * 8;
                            const uint32_t vbase = smem_u32(vt);
#pragma unroll
                            for (int kv = 0; kv < D / 32; ++kv) {
                                uint32_t raw[4], ev[4], od[4];
                                ldmatrix_x4_trans(raw, vbase + tr.at(r, hp, 2 * kv + ((lane >> 3) & 1)));
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const uint32_t t = __byte_perm(raw[i], 0u, 0x3120);
                                    ev[i] = e4m3x2_to_f16x2(t & 0xFFFFu);
                                    od[i] = e4m3x2_to_f16x2(t >> 16);
                                }
                                mma_f16_16816(o[2 * kv], ev, b0, b1);
                                mma_f16_16816(o[2 * kv + 1], od, b0, b1);
                            }
                        } else {  // O^T += V^T P^T
                            const uint32_t r = r0c + (lane & 7) + (lane >> 4) * 8;
                            const uint32_t vbase = smem_u32(vt);
#pragma unroll
                            for (int mt = 0; mt < KT; ++mt) {
                                const uint32_t half = mt >> 2, ch = (mt & 3) * 2 + ((lane >> 3) & 1);
                                uint32_t a[4];
                                ldmatrix_x4_trans(a, vbase + tr.at(r, half, ch));
                                mma_bf16_16816(o[mt], a, b0, b1);
                            }
                        }
                    }
                }
                if (zeroed) fence_proxy_async_smem();  // zeroing before the slot's next TMA write
            };
            if (kPrefix && (inf.flags & 16)) {
                // a shared-prefix item: this warp's 8 query rows against all 64 tokens of the stage (every warp
                // zeroes the invalid V rows of a chunk before it reads them; the writes are identical).  (e4m3
                // pools have no prefix items.)
                if constexpr (kPrefix) chunks(std::integral_constant<int, 4>{}, 0, inf.valid);
            } else if constexpr (C::kHeads == 2) {
                // two chunks of 16 rows of this warp's head
                if (p.k_new) patch_new_fp8(row0, row0 + 32);
                chunks(std::integral_constant<int, 2>{}, row0, inf.valid);
            } else if (row0 < inf.ntok) {
                if (kFp8) {
                    if (p.k_new) patch_new_fp8(row0, row0 + 16);
                } else if (inf.new_row >= row0 && inf.new_row < row0 + 16) {
                    // pa_decode_write: the newest token's staged K and V rows go into this stage's tiles
                    // (128-byte swizzled, before any ldmatrix of the row) and into the pool at its slot
                    const uint8_t* stg = smem + C::kNew + slot * C::kNewBytes;
                    constexpr int kChunks = D / 8;  // 16-byte chunks of a row
                    for (int c = lane; c < 2 * kChunks; c += 32) {
                        const int isv = c >= kChunks, cc = isv ? c - kChunks : c;
                        const int4 v = *reinterpret_cast<const int4*>(stg + isv * D * 2 + cc * 16);
                        *reinterpret_cast<int4*>((isv ? vt : kt) + tr.at(inf.new_row, cc / 8, cc % 8)) = v;
                        __nv_bfloat16* pool = static_cast<__nv_bfloat16*>(isv ? p.v_write : p.k_write);
                        reinterpret_cast<int4*>(pool + ((size_t)inf.new_slot * Hkv + inf.kvh) * D)[cc] = v;
                    }
                    if (p.new_slots && inf.kvh == 0 && lane == 0) p.new_slots[inf.s] = inf.new_slot;
                    fence_proxy_async_smem();  // these writes precede the slot's next TMA write
                    __syncwarp();
                }
                chunks(std::integral_constant<int, 1>{}, row0, inf.valid);
            }
            __syncwarp();
            if (!(inf.flags & 2)) {
                if (lane == 0) mbar_arrive(&empty[slot]);
                continue;
            }
            if (kPrefix && (inf.flags & 16)) {
                // ---------------------------------------- shared-prefix item epilogue
                // This warp's 8 rows are its own: normalise them and store every member's prefix
                // partial (o, m, l) in workspace slot 0.  A member whose own prefix length differs
                // from the group's gets an empty partial and an error count.
                float L0 = l0, L1 = l1;
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    L0 += __shfl_xor_sync(0xffffffffu, L0, off);
                    L1 += __shfl_xor_sync(0xffffffffu, L1, off);
                }
#pragma unroll
                for (int hsel = 0; hsel < 2; ++hsel) {
                    const int rr = warp * 8 + 2 * c4 + hsel, mem = rr / G, head = rr - mem * G;
                    if (mem >= inf.nsplit) continue;
                    const int sm = inf.s + mem;
                    int pre_m;
                    decode_start(p, sm, context_of(sm), &pre_m);
                    const bool same = pre_m == inf.split;  // inf.split carries the group's prefix length
                    const size_t slot0 = decode_unit(p, sm, inf.kvh) * p.max_splits * G + head;
                    const float Ls = hsel ? L1 : L0;
                    const float inv = (same && Ls > 0.f) ? 1.f / Ls : 0.f;
                    float* wo = p.ws_o + slot0 * D;
#pragma unroll
                    for (int mt = 0; mt < KT; ++mt) {
                        wo[mt * 16 + g4] = o[mt][hsel] * inv;
                        wo[mt * 16 + g4 + 8] = o[mt][2 + hsel] * inv;
                    }
                    if (g4 == 0) {
                        p.ws_ml[slot0] = same ? make_float2(hsel ? m1 : m0, Ls) : make_float2(-INFINITY, 0.f);
                        if (!same) count_error(p.error_count);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
                continue;
            }

            // ---------------------------------------------------- item epilogue
            // The four warps' states are combined through four [head][D] fp32
            // slabs in the K tile of the stage just consumed; the stage goes
            // back to the producer only after that.  The (m, l) exchange
            // arrays alternate between items so that a warp running ahead
            // into the next epilogue never overwrites values still being read.
            const int par = item_parity;
            item_parity ^= 1;
            float L0 = l0, L1 = l1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                L0 += __shfl_xor_sync(0xffffffffu, L0, off);
                L1 += __shfl_xor_sync(0xffffffffu, L1, off);
            }
            if (g4 == 0) {
                red_m[par][warp][2 * c4] = m0;
                red_m[par][warp][2 * c4 + 1] = m1;
                red_l[par][warp][2 * c4] = L0;
                red_l[par][warp][2 * c4 + 1] = L1;
            }
            if (!cbar.sync()) {  // every warp is done with this stage's K/V, and the states are visible
                if (lane == 0) count_error(p.error_count);
                break;
            }
            float M0 = -INFINITY, M1 = -INFINITY;  // over the warps that share this warp's kv head
#pragma unroll
            for (int w = hp * C::kWarpsPerHead; w < (hp + 1) * C::kWarpsPerHead; ++w) {
                M0 = fmaxf(M0, red_m[par][w][2 * c4]);
                M1 = fmaxf(M1, red_m[par][w][2 * c4 + 1]);
            }
            const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M0);
            const float f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M1);
            float* slabs = reinterpret_cast<float*>(smem + C::kRing + slot * C::kStageBytes);  // [warp][head][D]
            {
                float* my = slabs + warp * 8 * D;
#pragma unroll
                for (int mt = 0; mt < KT; ++mt) {
                    // the output columns of fragment mt (fp8: even / odd columns of a 32-column group)
                    const int d0 = kFp8 ? (mt >> 1) * 32 + 2 * g4 + (mt & 1) : mt * 16 + g4;
                    const int d1 = kFp8 ? d0 + 16 : d0 + 8;
                    my[(2 * c4) * D + d0] = o[mt][0] * f0;
                    my[(2 * c4 + 1) * D + d0] = o[mt][1] * f1;
                    my[(2 * c4) * D + d1] = o[mt][2] * f0;
                    my[(2 * c4 + 1) * D + d1] = o[mt][3] * f1;
                }
            }
            fence_proxy_async_smem();  // these writes precede the slot's next TMA write
            if (!cbar.sync()) {
                if (lane == 0) count_error(p.error_count);
                break;
            }
            // the item's query rows (G per kv head, the heads' rows adjacent in q and out)
            __nv_bfloat16* out =
                static_cast<__nv_bfloat16*>(p.out) + ((size_t)inf.s * p.num_q_heads + (size_t)inf.kvh * G) * D;
            // four consecutive columns per thread: one pass for G <= 4 (one head), two for G = 8
            for (int idx = 4 * tid; idx < C::kHeads * G * D; idx += 4 * 32 * C::kConsumerWarps) {
                const int hr = idx / D, dc = idx - hr * D;
                const int hh = C::kHeads == 2 ? hr / G : 0, h = hr - hh * G;  // kv head of the item, query row
                const int w0 = hh * C::kWarpsPerHead;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < C::kWarpsPerHead; ++w) M = fmaxf(M, red_m[par][w0 + w][h]);
                float Ls = 0.f;
#pragma unroll
                for (int w = 0; w < C::kWarpsPerHead; ++w) {
                    const float mw = red_m[par][w0 + w][h];
                    if (mw != -INFINITY) Ls += red_l[par][w0 + w][h] * fast_exp2(mw - M);
                }
                float4 acc = *reinterpret_cast<const float4*>(slabs + (w0 * 8 + h) * D + dc);
#pragma unroll
                for (int w = 1; w < C::kWarpsPerHead; ++w) {
                    const float4 v = *reinterpret_cast<const float4*>(slabs + ((w0 + w) * 8 + h) * D + dc);
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                const size_t slot_ws = decode_unit(p, inf.s, inf.kvh + hh) * p.max_splits + inf.split + p.split_base;
                float* wo = p.ws_o + (slot_ws * G + h) * D + dc;
                const float sc = Ls > 0.f ? (kFp8 ? p.v_scale : 1.f) / Ls : 0.f;
                acc.x *= sc;
                acc.y *= sc;
                acc.z *= sc;
                acc.w *= sc;
                if (inf.flags & 4) {
                    *reinterpret_cast<uint2*>(out + idx) =
                        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
                } else {
                    *reinterpret_cast<float4*>(wo) = acc;
                    if (dc == 0) p.ws_ml[slot_ws * G + h] = make_float2(M, Ls);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);  // this warp has read the slabs
        }
    }

    // ---- the last CTA to finish resets the work counter for the next call
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&work[1], 1) == (int)gridDim.x - 1) {
            atomicExch(&work[0], 0);
            atomicExch(&work[1], 0);
        }
    }
}

template <int D, bool kFp8, bool kPair, bool kPrefix = false>
int launch(const DecodeParams& p, int num_sms, cudaStream_t stream) {
    using C = TcCfg<D, kFp8, kPair>;
    CUtensorMap tmk, tmv;
    int rc = pool_tensor_map_rows(&tmk, p.k_cache, p.num_blocks, p.block_size, p.num_kv_heads, D, kFp8, C::kHeads);
    if (rc != PA_OK) return rc;
    if ((rc = pool_tensor_map_rows(&tmv, p.v_cache, p.num_blocks, p.block_size, p.num_kv_heads, D, kFp8,
                                   C::kHeads)) != PA_OK)
        return rc;
    if ((rc = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_tc_kernel<D, kFp8, kPair, kPrefix>), C::kSmemBytes)) !=
        PA_OK)
        return rc;
    // C::kCtasPerSm CTAs per SM (or as many as are resident at once, should fewer fit), never more
    // CTAs than the largest possible item count: a persistent CTA that is not resident from the start finds
    // the queue empty when it runs
    // (occupancy depends only on the kernel and its launch shape, the same on every GB300; the cached value is
    // atomic so that concurrent first calls from several host threads are safe)
    static std::atomic<int> resident_cache{0};
    int resident = resident_cache.load(std::memory_order_relaxed);
    if (resident == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_tc_kernel<D, kFp8, kPair, kPrefix>, C::kThreads,
                                                          C::kSmemBytes) != cudaSuccess)
            return check_launch();
        if (n < 1) return PA_ERR_UNSUPPORTED;
        resident = n < C::kCtasPerSm ? n : C::kCtasPerSm;
        resident_cache.store(resident, std::memory_order_relaxed);
    }
    long long max_items = (long long)p.num_seqs * p.num_kv_heads * p.max_splits;
    const long long slots = (long long)num_sms * resident;
    int grid = (int)(max_items < slots ? max_items : slots);
    return launch_kernel(decode_tc_kernel<D, kFp8, kPair, kPrefix>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream,
                         tmk, tmv, p, p.work);
}

}  // namespace

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

int pool_tensor_map(CUtensorMap* map, const void* pool, int num_blocks, int block_size, int num_kv_heads,
                    int head_dim) {
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

// The pool as a 3-D map for one-box-per-block loads: x = column within a
// 128-byte segment (64), y = pool row (P*B, stride Hkv*D*2 bytes), z = 128-byte
// segment of the row (Hkv*D/64, stride 128 bytes).  A box {64, B, D/64} at
// (0, pb*B, kvh*D/64) is block pb's B rows of kv head kvh, stored
// [segment][row][64] and 128-byte swizzled.
int pool_tensor_map_rows(CUtensorMap* map, const void* pool, int num_blocks, int block_size, int num_kv_heads,
                         int head_dim, bool fp8, int heads_per_box) {
    auto enc = tensor_map_encoder();
    if (!enc) return PA_ERR_CUDA;
    // x: elements of one 128-byte segment; the segments of a row are 128 bytes apart
    const int esz = fp8 ? 1 : 2, seg = 128 / esz, row_bytes = num_kv_heads * head_dim * esz;
    cuuint64_t dims[3] = {(cuuint64_t)seg, (cuuint64_t)num_blocks * block_size, (cuuint64_t)row_bytes / 128};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, 128};
    cuuint32_t box[3] = {(cuuint32_t)seg, (cuuint32_t)block_size, (cuuint32_t)(heads_per_box * head_dim * esz / 128)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void*>(pool), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

bool decode_tc_supported(const DecodeParams& p, int dtype) {
    const int B = p.block_size;
    if (dtype != PA_BF16 || (p.head_dim != 64 && p.head_dim != 128) || p.group > 8) return false;
    // fp8 pools: head_dim 128, plain decode or the fused write (no cascade items)
    if (p.kv_fp8 && (p.head_dim != 128 || p.group_offsets)) return false;
    if (B != 8 && B != 16 && B != 32 && B != 64) return false;
    if (p.partition % 64 != 0 || p.num_seqs > kMaxSeqsPersistent) return false;
    if (p.small_from < p.num_seqs && (p.small_partition % 64 != 0 || p.small_partition < 64)) return false;
    if (((uintptr_t)p.k_cache & 15) || ((uintptr_t)p.v_cache & 15) || ((uintptr_t)p.q & 15) || ((uintptr_t)p.out & 15))
        return false;
    if ((long long)p.num_blocks * B >= (1LL << 31)) return false;
    return p.max_splits <= 128 && p.work != nullptr;
}

int launch_decode_tc(const DecodeParams& p, int num_sms, cudaStream_t stream) {
    if (p.kv_fp8)
        return PA_DECODE_FP8_PAIRS && p.num_kv_heads % 2 == 0 && p.num_seqs <= kMaxSeqsPairs
                   ? launch<128, true, true>(p, num_sms, stream)
                                                             : launch<128, true, false>(p, num_sms, stream);
    if (p.group_offsets)  // cascade prefix items (pa_decode_cascade takes head_dim 128 only)
        return p.head_dim == 128 ? launch<128, false, false, true>(p, num_sms, stream) : PA_ERR_UNSUPPORTED;
    return p.head_dim == 64 ? launch<64, false, false>(p, num_sms, stream)
                            : launch<128, false, false>(p, num_sms, stream);
}

}  // namespace pa
