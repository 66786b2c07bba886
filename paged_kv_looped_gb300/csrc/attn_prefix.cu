// Shared-prefix ("cascade") paged decode attention for sm_103a.
//
// "Faster fuzzy minds" ("When scheduler does the work"): a radix tree lets a
// request that shares a prompt prefix inherit the computed KV, so several page
// tables point at the same physical pages.  Plain paged decode then reads each
// shared page once per request.  Here a host planner finds, from the page
// tables, the 128-token tiles that several requests map to the same pages, as
// runs ("segments") with one member set; the kernel below reads each such tile
// once per kv head and applies it to the queries of every member at once:
//     S = Q K^T   (M = 128 query rows: members x GQA heads, N = 128 tokens, K = D)
//     O = P V     (M = 128 query rows, N = D, K = 128 tokens)
// on the 5th-generation tensor cores (tcgen05.mma, fp32 accumulators in TMEM),
// with K and V tiles brought in by TMA tensor copies in 128-byte-swizzled
// shared memory.  Each run of work (below) writes one (o, log2-sum-exp)
// partial per query row; with private tails every request's own tokens are
// segments too, otherwise the split-K kernel covers them; the combine kernel
// merges everything.
#include <math_constants.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <type_traits>
#include <vector>

#include "rlt.h"
#include "rlt_device.cuh"
#include "rlt_internal.h"
#include "rlt_tc.cuh"

namespace rlt {
namespace {

// Persistent CTAs, one per SM.  The work is a list of items (kv head, segment,
// member block, chunk of chunk_tiles 128-token tiles), kv-head-major; CTA c
// takes the contiguous c-th share of it.  Consecutive items of one (kv head,
// segment, member block) form a "run": one accumulation over their tokens and
// one partial, so a CTA pays its start-up once and its pipeline never drains
// between items.
//
// On this part a kind::f16 tcgen05.mma with M = 128 occupies the tensor pipe
// about equally long for N = 64, 128 or 256, so every MMA here has N = 128:
// S = Q K^T over a 128-token sub-tile (A = Q from TMEM), O += P V with N = D
// (A = P from TMEM, written over the S it came from).  Shared memory holds
// only the K and V rings.  Roles (8 warps):
//   warps 0-7  softmax: warp w owns query rows 32(w%4)..+31 (the TMEM lanes it may
//              touch) and the columns half w/4 of each sub-tile; the two warps of a
//              row quarter swap row maxima and sums through shared memory.  They
//              also write the next run's Q rows into TMEM.
//   warp 8/9   TMA copies of V / K sub-tiles (128 tokens) into 3-slot rings
//   warp 10    MMA issue: S into 2 TMEM S/P buffers, O += P V into the O buffer
//   warp 11    scheduler: decodes the runs into a 4-deep ring of descriptors in
//              shared memory, with the members' request ids
constexpr int kSoftWarps = 8;
constexpr int kLoadVWarp = 8, kLoadKWarp = 9, kMmaWarp = 10, kSchedWarp = 11;
constexpr int kPThreads = 12 * 32;
constexpr int kSub = 128;                   // tokens per sub-tile (= one planner tile)
constexpr int kStagesK = 3, kStagesV = 3;   // ring depths (sub-tiles), measured against 2/4, 2/3, 2/2
constexpr int kPrefetch = 3;                 // sub-tiles fetched into L2 ahead of the ring
constexpr int kHalfKV = kSub * 128;         // one 64-dim column block of a sub-tile (128 rows x 128 B)
constexpr int kKVBytes = 2 * kHalfKV;       // K (or V) of one sub-tile
constexpr int kSBufs = 2;                   // S/P buffers in TMEM
constexpr int kQBufs = 2;
constexpr int kDescs = 4;                   // run descriptors published ahead
constexpr int kDescConsumers = 4 + kSoftWarps;   // K and V producers, the MMA's two cursors, softmax warps
constexpr int kMaxChunkTiles = 32;
constexpr int kKOff = 0;
constexpr int kVOff = kKOff + kStagesK * kKVBytes;
constexpr int kBarOff = kVOff + kStagesV * kKVBytes;
enum PrefixBar {
    kBarFullK = 0,                          // K slot landed (TMA transaction count)
    kBarFreeK = kBarFullK + kStagesK,       // K slot read by its S MMA
    kBarFullV = kBarFreeK + kStagesK,
    kBarFreeV = kBarFullV + kStagesV,       // V slot read by its P.V MMA
    kBarSFull = kBarFreeV + kStagesV,       // S of the sub-tile in buffer i written
    kBarPFull = kBarSFull + kSBufs,         // its P written over it by all 4 softmax warps
    kBarPvDone = kBarPFull + kSBufs,        // its P.V complete
    kBarQFull = kBarPvDone + kSBufs,        // Q buffer i written by all 4 softmax warps
    kBarOFree = kBarQFull + kQBufs,         // O read out by all 4 softmax warps
    kBarDescFull = kBarOFree + 1,           // descriptor i published
    kBarDescFree = kBarDescFull + kDescs,   // descriptor i copied by every consumer
    kBarMemFull = kBarDescFree + kDescs,    // descriptor i's member rows and limits written
    kBarPair = kBarMemFull + kDescs,        // the two softmax warps of row quarter i meet
    kNumBars = kBarPair + 4
};
constexpr int kFlagOff = kBarOff + kNumBars * 8;   // TMEM base address, abort flag
constexpr int kDescOff = (kFlagOff + 16 + 63) / 64 * 64;
constexpr int kMemOff = kDescOff + kDescs * 64;    // q rows of each descriptor's members
constexpr int kLimOff = kMemOff + kDescs * 128 * 4;  // their key counts (causal limits)
constexpr int kXMaxOff = kLimOff + kDescs * 128 * 4;   // row maxima [sub-tile parity][column half][row]
constexpr int kXSumOff = kXMaxOff + 2 * 2 * 128 * 4;   // row sums [column half][row]
constexpr int kSmemP = kXSumOff + 2 * 128 * 4 + 1024;
// TMEM columns: Q[2] (128 rows x 128 bf16, two per column), S/P[2], O
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = kColQ + kQBufs * 64, kColO = kColS + kSBufs * kSub;
static_assert(kColO + 128 == kTmemCols, "TMEM plan");
// O accumulates in TMEM against a per-row reference max that moves only when
// the row's running max exceeds it by more than this (log2 units): p <= 2^8.
constexpr float kRescaleThreshold = 8.f;

static_assert(kSmemP <= 227 * 1024, "shared memory of one CTA");
static_assert(kVOff % 1024 == 0, "swizzled operands");

// One run: tokens [tok_begin, tok_end) of a segment for kv head g and n_mem of
// its members, their query rows held F times (prefix_replication); copy k of a
// row writes its partial to slot `slot + k` of the member's (b, h), and marks
// the slots of the nchunks - 1 following chunks (F each) empty.
struct RunDesc {
    int64_t tok_begin, tok_end;
    int32_t g, nsub, page_row, n_mem, slot, nchunks, F;
    int32_t tail;                            // a one-member segment: a request's private tail
    int32_t once;                            // one member block covers the segment: its tiles are read once
};
static_assert(sizeof(RunDesc) <= 64, "descriptor slot");

struct Run {
    RunDesc d;
    int32_t member_begin;
    int next_item;
};

// The run that starts at work item `item` of a CTA whose items end at item_end; called by
// all 32 lanes of a warp (every lane gets the same run).  Its segment is the last one whose
// first work unit is <= the item's (work units ascend with the segment index): the lanes read
// the rows of 32 segments at once and a ballot picks it, so the plan costs one round trip per
// 32 segments searched instead of one per halving step.
__device__ __forceinline__ Run decode_run(const PrefixParams &pp, int G, int item, int item_end, int lane)
{
    Run r;
    r.d.g = item / pp.work_units;
    const int unit = item - r.d.g * pp.work_units;
    int32_t sd[kSegFields];
#pragma unroll
    for (int f = 0; f < kSegFields; ++f)
        sd[f] = 0;
    for (int base = 0; base < pp.num_segments; base += 32) {
        const int s = base + lane;
        int32_t row[kSegFields];
#pragma unroll
        for (int f = 0; f < kSegFields; ++f)
            row[f] = s < pp.num_segments ? pp.segments[s * kSegFields + f] : 0;
        const unsigned le = __ballot_sync(kFullMask, s < pp.num_segments && row[kSegWorkBegin] <= unit);
        if (le != 0u) {
            const int src = 31 - __clz(le);
#pragma unroll
            for (int f = 0; f < kSegFields; ++f)
                sd[f] = __shfl_sync(kFullMask, row[f], src);
        }
        if (le != kFullMask)
            break;                               // a later segment starts past this unit
    }
    if (pp.num_segments > 0 && __shfl_sync(kFullMask, pp.segments[kSegWorkBegin], 0) > unit) {
#pragma unroll
        for (int f = 0; f < kSegFields; ++f)     // (a malformed plan: segment 0, as a search would)
            sd[f] = pp.segments[f];
    }
    const int num_tiles = sd[kSegNumTiles];
    const int nchunks_seg = max(1, (num_tiles + pp.chunk_tiles - 1) / pp.chunk_tiles);
    const int local = max(0, unit - sd[kSegWorkBegin]);
    const int mb = local / nchunks_seg;
    const int chunk0 = local - mb * nchunks_seg;
    r.d.nchunks = min(nchunks_seg - chunk0, item_end - item);   // items of one member block
    const int per_block = 128 / G;
    const int m0 = mb * per_block;
    r.d.n_mem = min(per_block, sd[kSegMemberCount] - m0);
    r.d.F = prefix_replication(min(per_block, sd[kSegMemberCount]) * G);
    r.member_begin = sd[kSegMemberBegin] + m0;
    r.d.page_row = sd[kSegPageRow];
    r.d.tail = sd[kSegMemberCount] == 1;
    r.d.once = sd[kSegMemberCount] <= per_block;
    r.d.slot = sd[kSegSlotBase] + chunk0 * r.d.F;
    const int t_first = sd[kSegFirstTile] + chunk0 * pp.chunk_tiles;
    const int t_last = sd[kSegFirstTile] + min(num_tiles, (chunk0 + r.d.nchunks) * pp.chunk_tiles);
    r.d.tok_begin = (int64_t)t_first * kPrefixTile;
    r.d.tok_end = min((int64_t)t_last * kPrefixTile, (int64_t)sd[kSegEndToken]);
    if (pp.member_limit != nullptr && r.d.n_mem > 0)   // no key past the block's largest limit
        r.d.tok_end = min(r.d.tok_end, (int64_t)pp.member_limit[r.member_begin + r.d.n_mem - 1]);
    r.d.nsub = (r.d.n_mem > 0 && r.d.tok_end > r.d.tok_begin)
                   ? (int)((r.d.tok_end - r.d.tok_begin + kSub - 1) / kSub) : 0;
    r.next_item = item + max(1, r.d.nchunks);
    return r;
}

// The next run with work at or after *item; false when the CTA's items are done.
__device__ __forceinline__ bool next_run(const PrefixParams &pp, int G, int &item, int item_end, Run &r, int lane)
{
    while (item < item_end) {
        r = decode_run(pp, G, item, item_end, lane);
        item = r.next_item;
        if (r.d.nsub > 0)
            return true;
    }
    return false;
}

// Warp-uniform bounded wait (every lane gets the same answer).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const volatile int *abort)
{
    return __all_sync(kFullMask, mbar_wait_or_abort(bar, parity, abort));
}

// Copy run descriptor r (and, for row >= 0, the member and key count behind query row
// `row` of the run: its copy row % (128 / F), member of that / G) and release its slot.
// Warp-collective; false if the wait gave up.
__device__ __forceinline__ bool take_desc(uint64_t *bars, const unsigned char *base, int r, RunDesc &out,
                                          int row, int G, int &member, int &limit, const volatile int *abort,
                                          int lane)
{
    if (!warp_wait(&bars[kBarDescFull + r % kDescs], (r / kDescs) & 1u, abort))
        return false;
    // the softmax warps also need the member rows, published after the descriptor
    if (row >= 0 && !warp_wait(&bars[kBarMemFull + r % kDescs], (r / kDescs) & 1u, abort))
        return false;
    out = reinterpret_cast<const RunDesc *>(base + kDescOff)[r % kDescs];
    const int mrow = row < 0 ? -1 : (row % (128 / max(out.F, 1))) / G;
    if (mrow >= 0 && mrow < out.n_mem) {
        member = reinterpret_cast<const int32_t *>(base + kMemOff)[(r % kDescs) * 128 + mrow];
        limit = reinterpret_cast<const int32_t *>(base + kLimOff)[(r % kDescs) * 128 + mrow];
    }
    __syncwarp();
    if (lane == 0)
        mbar_arrive(&bars[kBarDescFree + r % kDescs]);
    return true;
}

// Dims 64*half..64*half+63 of this thread's query row (copy row lr = row % (128 / F):
// member lr / G, head lr % G of run d) as 32 words of packed bf16 pairs; zero for rows
// past the run's members.
__device__ __forceinline__ void load_q(const DecodeParams &p, const RunDesc &d, int G, int row, int member,
                                       int half, uint32_t (&w)[32])
{
    const int lr = row % (128 / max(d.F, 1));
    const bool live = d.nsub > 0 && lr < d.n_mem * G;
    const uint4 *src = reinterpret_cast<const uint4 *>(
        p.q + ((int64_t)member * p.num_q_heads + d.g * G + lr % G) * 128 + half * 64);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = live ? src[i] : make_uint4(0u, 0u, 0u, 0u);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
}

// Bring the 128 bytes load_q will read into L2 ahead of time (no registers held).
__device__ __forceinline__ void prefetch_q(const DecodeParams &p, const RunDesc &d, int G, int row, int member,
                                           int half)
{
    const int lr = row % (128 / max(d.F, 1));
    if (d.nsub > 0 && lr < d.n_mem * G) {
        const uint16_t *src = p.q + ((int64_t)member * p.num_q_heads + d.g * G + lr % G) * 128 + half * 64;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
    }
}

// Those words into columns 32*half.. of the TMEM Q buffer at t_q (the A operand
// layout of S = Q K^T: a row's dims in order, two per column, the lower in the low
// half), then the warp's arrive on the buffer's barrier.
__device__ __forceinline__ void store_q(const uint32_t (&w)[32], int half, uint32_t t_q, uint64_t *bar,
                                        int lane)
{
    tc::tmem_st32u(t_q + half * 32, w);
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0)
        mbar_arrive(bar);
}

// The two softmax warps of a row quarter meet (their k-th meeting; k counts from 0 in
// both): shared-memory writes before it are visible to the other warp after it.
// Bounded, like every wait here; false if it gave up.
__device__ __forceinline__ bool pair_sync(uint64_t *bar, int &k, const volatile int *abort, int lane)
{
    __syncwarp();
    if (lane == 0)
        mbar_arrive(bar);
    return warp_wait(bar, (uint32_t)(k++) & 1u, abort);
}

// kAppend: the call fuses the append and runs every request's private tail here (no
// split-K rest), so the producers store each tail's new rows before copying them.
// kL2Ahead: the copy warps prefetch sub-tiles into L2 ahead of their rings (a separate
// instance, so that the others carry none of its code: with it compiled in but switched off
// the long-context call measured 1.5-3 us slower).
template <bool kAppend, bool kL2Ahead>
__global__ void __launch_bounds__(kPThreads, 1)
    decode_prefix_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const DecodeParams p,
                         const PrefixParams pp)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kBarOff);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + kFlagOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kFlagOff + 4);

    // The kernel behind this one (the combine) may be scheduled now.  Until pdl_wait a thread
    // reads only what no kernel still running may write: the plan, lengths, page table and
    // cached K/V rows.  q and k_new / v_new are read, and partials and pool rows written, only
    // by threads that have passed it.
    pdl_launch_dependents();
    const int G = p.num_q_heads / p.num_kv_heads;
    const int64_t n_items = (int64_t)p.num_kv_heads * pp.work_units;
    const int item_begin = (int)((int64_t)blockIdx.x * n_items / gridDim.x);
    const int item_end = (int)((int64_t)(blockIdx.x + 1) * n_items / gridDim.x);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < kBarSFull; ++i)
            mbar_init(&bars[i], 1);
        for (int i = 0; i < kSBufs; ++i) {
            mbar_init(&bars[kBarSFull + i], 1);
            mbar_init(&bars[kBarPFull + i], kSoftWarps);
            mbar_init(&bars[kBarPvDone + i], 1);
        }
        for (int i = 0; i < kQBufs; ++i)
            mbar_init(&bars[kBarQFull + i], kSoftWarps);
        mbar_init(&bars[kBarOFree], kSoftWarps);
        for (int i = 0; i < kDescs; ++i) {
            mbar_init(&bars[kBarDescFull + i], 1);
            mbar_init(&bars[kBarDescFree + i], kDescConsumers);
            mbar_init(&bars[kBarMemFull + i], 1);
        }
        for (int i = 0; i < 4; ++i)
            mbar_init(&bars[kBarPair + i], 2);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 0)
        tc::tmem_alloc(tslot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    bool ok = true;
    int unused = 0;

    if (warp == kSchedWarp) {
        // ---------------------------------------------------------- scheduler
        // Publishes descriptor d once every consumer has copied descriptor d - kDescs.
        RunDesc *descs = reinterpret_cast<RunDesc *>(base + kDescOff);
        int32_t *dmem = reinterpret_cast<int32_t *>(base + kMemOff);
        int32_t *dlim = reinterpret_cast<int32_t *>(base + kLimOff);
        int item = item_begin;
        for (int d = 0;; ++d) {
            if (d >= kDescs &&
                !(ok = warp_wait(&bars[kBarDescFree + d % kDescs], ((d - kDescs) / kDescs) & 1u, abort_flag)))
                break;
            Run r;
            const bool has = next_run(pp, G, item, item_end, r, lane);
            if (!has)
                r.d.nsub = 0;                    // the terminal descriptor
            if (lane == 0) {
                descs[d % kDescs] = r.d;
                // the copies and MMAs need only the descriptor: publish it before the members
                mbar_arrive(&bars[kBarDescFull + d % kDescs]);
            }
            for (int i = lane; has && i < r.d.n_mem; i += 32) {
                int b = pp.members[r.member_begin + i];
                if (b < 0 || b >= pp.num_rows) {
                    record_error(p.err, RLT_DEVERR_BAD_SLOT);
                    b = 0;
                }
                dmem[(d % kDescs) * 128 + i] = b;
                dlim[(d % kDescs) * 128 + i] =
                    pp.member_limit != nullptr ? pp.member_limit[r.member_begin + i] : INT32_MAX;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars[kBarMemFull + d % kDescs]);
            // Fused append, checked once the descriptor is out: a member whose newest token
            // lies in tiles it shares would need a slot of a shared (read-only) page; flagged,
            // not written.  (The slot stays readable until every consumer has released it.)
            for (int i = lane; kAppend && has && !r.d.tail && i < r.d.n_mem; i += 32) {
                const int b = dmem[(d % kDescs) * 128 + i];
                const int len = p.seq_lens[b];
                if (len > 0 && dlim[(d % kDescs) * 128 + i] >= len)
                    record_error(p.err, RLT_DEVERR_BAD_SLOT);
            }
            if (!has)
                break;
        }
        if (!ok)
            *abort_flag = 1;
    } else if (warp == kLoadKWarp || warp == kLoadVWarp) {
        // ------------------------------------------------- TMA producers (K, V)
        // Lane j copies box j/2, column block j&1 of each sub-tile of this warp's tensor.
        // The page-table read for the next sub-tile (of this run or the next) is
        // issued before the wait for the current sub-tile's slot.
        const bool is_v = warp == kLoadVWarp;
        const int stages = is_v ? kStagesV : kStagesK;
        const CUtensorMap *map = is_v ? &vmap : &kmap;
        uint64_t *fullx = bars + (is_v ? kBarFullV : kBarFullK);
        uint64_t *freex = bars + (is_v ? kBarFreeV : kBarFreeK);
        unsigned char *ring = base + (is_v ? kVOff : kKOff);
        if (lane == 0)
            tc::prefetch_tmap(map);
        const int BR = p.page_size < kSub ? p.page_size : kSub;   // rows per TMA box
        const int boxes = kSub / BR;
        // pool row of this lane's box in sub-tile j of run d (-1: no box)
        auto lane_row = [&](const RunDesc &d, int j) -> int {
            if (lane >= 2 * boxes)
                return -1;
            const int64_t tok = d.tok_begin + (int64_t)j * kSub + (lane >> 1) * BR;
            if (tok >= d.tok_end)
                return -1;
            const int64_t idx = tok / p.page_size;
            int64_t page = -1;
            if (d.page_row >= 0 && d.page_row < p.batch && idx < p.max_pages)
                page = p.page_table[(int64_t)d.page_row * p.max_pages + idx];
            if (page < 0 || page >= p.num_pages) {
                record_error(p.err, RLT_DEVERR_BAD_PAGE);
                page = 0;                        // stay in bounds; the result is flagged
            }
            return (int)((page * p.num_kv_heads + d.g) * p.page_size + tok % p.page_size);
        };
        // Fused append (private tails): position of the run's request's new token when the
        // run ends at that request's length, else -1.
        auto new_token = [&](const RunDesc &d) -> int64_t {
            if (!kAppend || !d.tail || d.nsub <= 0 || d.page_row < 0 || d.page_row >= p.batch)
                return -1;
            return p.seq_lens[d.page_row] == d.tok_end ? d.tok_end - 1 : -1;
        };
        int n = 0, r = 0, j = 0;                 // sub-tiles issued; current run and sub-tile
        RunDesc cur;
        ok = take_desc(bars, base, r, cur, -1, G, unused, unused, abort_flag, lane);
        int row_next = ok && cur.nsub > 0 ? lane_row(cur, 0) : -1;
        int64_t nt_next = ok ? new_token(cur) : -1;
        while (ok && cur.nsub > 0) {
            const int row = row_next;
            const int64_t nt = nt_next;
            const int nt_b = cur.page_row, nt_g = cur.g;
            const int64_t sub_begin = cur.tok_begin + (int64_t)j * kSub, tok_end = cur.tok_end;
            // With l2_ahead, sub-tiles past the ring are fetched into L2 ahead of their copies:
            // at a run's start the kPrefetch after the ring's first fill, then one per sub-tile,
            // kPrefetch ahead of the ring, so that each copy into a freed slot reads L2 and a
            // CTA's few sub-tiles are all requested at once, before the kernel ahead finishes.
            int pf_row[kPrefetch];
#pragma unroll
            for (int k = 0; k < kPrefetch; ++k) {
                const int t = j == 0 ? stages + k : (k == kPrefetch - 1 ? j + stages + k : -1);
                pf_row[k] = kL2Ahead && t >= 0 && t < cur.nsub ? lane_row(cur, t) : -1;
            }
            const bool once = cur.once != 0;
            if (j + 1 < cur.nsub) {
                row_next = lane_row(cur, ++j);
            } else {
                j = 0;
                if (!(ok = take_desc(bars, base, ++r, cur, -1, G, unused, unused, abort_flag, lane)))
                    break;
                if (cur.nsub > 0)
                    row_next = lane_row(cur, 0);
                nt_next = new_token(cur);
            }
            const int st = n % stages;
            if (n >= stages && !(ok = warp_wait(&freex[st], ((n / stages) - 1) & 1u, abort_flag)))
                break;
            const int nbox = (int)min((int64_t)boxes, (tok_end - sub_begin + BR - 1) / BR);
            if (lane == 0)
                mbar_arrive_expect_tx(&fullx[st], (uint32_t)(nbox * BR * 128 * 2));
            __syncwarp();
            if (kAppend && nt >= sub_begin && nt < sub_begin + kSub && lane < 2 * nbox &&
                (lane >> 1) == (nt - sub_begin) / BR) {
                // this lane's box holds the new token: its 64 dims go to the pool slot first,
                // then the copy (same thread, ordered by the proxy fence) reads them back
                const int64_t dr = (nt - sub_begin) % BR;
                const int64_t pidx = nt / p.page_size;
                const int64_t pg = pidx < p.max_pages ? p.page_table[(int64_t)nt_b * p.max_pages + pidx] : -1;
                const bool page_valid = pg >= 0 && pg < p.num_pages;   // a bad page is flagged, not written
                pdl_wait();
                const uint4 *src = reinterpret_cast<const uint4 *>((is_v ? p.v_new : p.k_new) +
                                                                   ((int64_t)nt_b * p.num_kv_heads + nt_g) * 128 +
                                                                   (lane & 1) * 64);
                uint4 *dst = reinterpret_cast<uint4 *>(const_cast<uint16_t *>(is_v ? p.v_bank : p.k_bank) +
                                                       ((int64_t)row + dr) * 128 + (lane & 1) * 64);
                if (page_valid) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = src[k];
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            if (lane < 2 * nbox) {
                void *dst = ring + st * kKVBytes + (lane & 1) * kHalfKV + (lane >> 1) * BR * 128;
                if (once)
                    tc::tma_load_2d_once(dst, map, (lane & 1) * 64, row, &fullx[st]);
                else
                    tc::tma_load_2d(dst, map, (lane & 1) * 64, row, &fullx[st]);
            }
            if constexpr (kL2Ahead) {
#pragma unroll
                for (int k = 0; k < kPrefetch; ++k)
                    if (pf_row[k] >= 0)
                        tc::tma_prefetch_l2_2d(map, (lane & 1) * 64, pf_row[k]);
            }
            ++n;
        }
        if (!ok) {
            *abort_flag = 1;
            // copies of the last sub-tiles may still be landing: wait for them (bounded)
            if (lane == 0)
                for (int k = max(0, n - stages); k < n; ++k)
                    mbar_wait(&fullx[k % stages], (k / stages) & 1u);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issuer
        // Event loop over two cursors on the run sequence: S of sub-tile n as soon as
        // K_n has landed, S/P buffer n%2 is free (P.V of n-2 issued; tcgen05 MMAs run
        // in issue order, so S cannot overwrite P before that P.V has read it) and, at
        // a run's start, its Q is written; P.V of sub-tile n as soon as every softmax
        // warp wrote P_n and V_n has landed (and, at a run's start, O was read out).
        // Probes do not block, so neither cursor waits on the other.
        const uint32_t id = tc::instr_desc_bf16(128, 128, false);      // S: B = K, K-major
        const uint32_t id_o = tc::instr_desc_bf16(128, 128, true);     // O: B = V, MN-major
        const uint32_t ka = smem_u32(base + kKOff), va = smem_u32(base + kVOff);
        const RunDesc *descs = reinterpret_cast<const RunDesc *>(base + kDescOff);
        RunDesc sd{}, pd{};
        bool s_have = false, p_have = false, s_done = false, p_done = false;
        int s_r = 0, p_r = 0, s_j = 0, p_j = 0, s_n = 0, p_n = 0;
        uint64_t t_idle = 0;
        // take the next descriptor for a cursor if it is published (non-blocking)
        auto try_take = [&](int r, RunDesc &out, bool &have, bool &done) -> bool {
            if (!__all_sync(kFullMask, mbar_test_wait(&bars[kBarDescFull + r % kDescs], (r / kDescs) & 1u)))
                return false;
            out = descs[r % kDescs];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars[kBarDescFree + r % kDescs]);
            if (out.nsub > 0)
                have = true;
            else
                done = true;
            return true;
        };
        while (!p_done) {
            bool progress = false;
            if (!s_done && !s_have)
                progress |= try_take(s_r, sd, s_have, s_done);
            if (s_have && s_n < p_n + kSBufs) {
                bool ready = mbar_test_wait(&bars[kBarFullK + s_n % kStagesK], (s_n / kStagesK) & 1u);
                if (s_j == 0)
                    ready = ready && mbar_test_wait(&bars[kBarQFull + s_r % kQBufs], (s_r / kQBufs) & 1u);
                if (__all_sync(kFullMask, ready)) {
                    tc::fence_after_sync();
                    if (lane == 0) {
                        const uint32_t qt = tmem + kColQ + (s_r % kQBufs) * 64;
                        const uint32_t kb = ka + (s_n % kStagesK) * kKVBytes;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_bf16_ta(tmem + kColS + (s_n % kSBufs) * kSub, qt + kk * 8,
                                            tc::smem_desc(kb + (kk >> 2) * kHalfKV + (kk & 3) * 32, 16, 1024), id,
                                            kk > 0);
                        tc::mma_commit(&bars[kBarSFull + s_n % kSBufs]);
                        tc::mma_commit(&bars[kBarFreeK + s_n % kStagesK]);
                    }
                    __syncwarp();
                    ++s_n;
                    if (++s_j == sd.nsub) {
                        s_j = 0;
                        s_have = false;
                        ++s_r;
                    }
                    progress = true;
                }
            }
            if (!p_done && !p_have)
                progress |= try_take(p_r, pd, p_have, p_done);
            if (p_have && p_n < s_n) {
                bool ready = mbar_test_wait(&bars[kBarPFull + p_n % kSBufs], (p_n / kSBufs) & 1u) &&
                             mbar_test_wait(&bars[kBarFullV + p_n % kStagesV], (p_n / kStagesV) & 1u);
                if (p_j == 0 && p_r >= 1)
                    ready = ready && mbar_test_wait(&bars[kBarOFree], (p_r - 1) & 1u);
                if (__all_sync(kFullMask, ready)) {
                    tc::fence_after_sync();
                    if (lane == 0) {
                        const uint32_t pt = tmem + kColS + (p_n % kSBufs) * kSub;
                        const uint32_t vb = va + (p_n % kStagesV) * kKVBytes;
#pragma unroll
                        for (int kk = 0; kk < kSub / 16; ++kk)
                            tc::mma_bf16_ta(tmem + kColO, pt + kk * 8, tc::smem_desc(vb + kk * 2048, kHalfKV, 1024),
                                            id_o, (p_j > 0) || (kk > 0));
                        tc::mma_commit(&bars[kBarPvDone + p_n % kSBufs]);
                        tc::mma_commit(&bars[kBarFreeV + p_n % kStagesV]);
                    }
                    __syncwarp();
                    ++p_n;
                    if (++p_j == pd.nsub) {
                        p_j = 0;
                        p_have = false;
                        ++p_r;
                    }
                    progress = true;
                }
            }
            if (progress) {
                t_idle = 0;
            } else {
                __nanosleep(32);
                const uint64_t now = global_ns();
                if (t_idle == 0)
                    t_idle = now;
                else if (__any_sync(kFullMask, now - t_idle > kWaitLimitNs || *abort_flag != 0)) {
                    ok = false;
                    break;
                }
            }
        }
        // every issued MMA must be complete before the CTA gives up its memory: the last
        // P.V commit covers all earlier MMAs (bounded wait; on the normal path it has arrived)
        if (lane == 0 && p_n > 0)
            mbar_wait(&bars[kBarPvDone + (p_n - 1) % kSBufs], ((p_n - 1) / kSBufs) & 1u);
        if (lane == 0 && s_n > p_n)
            mbar_wait(&bars[kBarSFull + (s_n - 1) % kSBufs], ((s_n - 1) / kSBufs) & 1u);
        __syncwarp();
        if (!ok)
            *abort_flag = 1;
    } else {
        // ------------------------------------------------------------- softmax
        // Run r: its first sub-tile's S is waited for with the next run's Q rows already
        // loaded, so that Q goes into TMEM at once (the previous run's S MMAs are then
        // complete); the epilogue of run r-1 is deferred until after run r's first P,
        // so the tensor pipe computes that P.V while O is read out.
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        float *xmax = reinterpret_cast<float *>(base + kXMaxOff);
        float *xsum = reinterpret_cast<float *>(base + kXSumOff);
        uint64_t *pair = &bars[kBarPair + quarter];
        int n = 0, meets = 0;
        RunDesc rd, rn;
        int b_row = 0, b_next = 0, lim_row = INT32_MAX, lim_next = INT32_MAX;
        // the run whose epilogue is pending
        RunDesc ed{};
        int e_b = 0, e_last = -1;
        float e_m = 0.f, e_l = 0.f;
        auto epilogue = [&]() -> bool {
            if (!warp_wait(&bars[kBarPvDone + e_last % kSBufs], (e_last / kSBufs) & 1u, abort_flag))
                return false;
            tc::fence_after_sync();
            const int R = ed.n_mem * G;
            const int RB = 128 / ed.F;
            const int lr = row % RB;              // the row this copy holds
            const bool live = quarter * 32 % RB < R;
            const int64_t slot = ((int64_t)e_b * p.num_q_heads + ed.g * G + lr % G) * p.part_stride + ed.slot +
                                 quarter * 32 / RB;
            float l_tot = e_l;
            if (live) {
                xsum[half * 128 + row] = e_l;
                if (!pair_sync(pair, meets, abort_flag, lane))
                    return false;
                l_tot = e_l + xsum[(half ^ 1) * 128 + row];
                const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;   // a row with no key: o = 0
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float o[16];
                    tc::tmem_ld<16>(t_lane + kColO + half * 64 + c * 16, o);
                    if (c == 3) {
                        // O has left TMEM: the next run's first P.V may overwrite it now
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(&bars[kBarOFree]);
                    }
                    if (lr < R) {
                        float4 *dst = reinterpret_cast<float4 *>(p.o_part + slot * 128 + half * 64 + c * 16);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                                 o[4 * i + 3] * inv);
                    }
                }
            } else {
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars[kBarOFree]);
            }
            if (live && half == 0 && lr < R) {
                p.lse_part[slot] = l_tot > 0.f ? e_m + log2f(l_tot) : -CUDART_INF_F;
                for (int k = 1; k < ed.nchunks; ++k)   // chunks merged into this run's partial
                    p.lse_part[slot + k * ed.F] = -CUDART_INF_F;
            }
            // both warps have read xsum before a later epilogue writes it
            return !live || pair_sync(pair, meets, abort_flag, lane);
        };

        uint32_t qw[32];
        ok = take_desc(bars, base, 0, rd, row, G, b_row, lim_row, abort_flag, lane);
        pdl_wait();                              // q, and the partials this warp writes
        if (ok && rd.nsub > 0) {
            load_q(p, rd, G, row, b_row, half, qw);
            store_q(qw, half, t_lane + kColQ, &bars[kBarQFull], lane);
        }
        for (int r = 0; ok && rd.nsub > 0; ++r) {
            // the next run's Q rows, loaded while this run's first S is computed
            if (!(ok = take_desc(bars, base, r + 1, rn, row, G, b_next, lim_next, abort_flag, lane)))
                break;
            prefetch_q(p, rn, G, row, b_next, half);
            const int R = rd.n_mem * G;
            const int RB = 128 / rd.F;           // rows per copy of the run's query rows
            const int part = quarter * 32 / RB;  // the copy this quarter holds
            const bool live = quarter * 32 % RB < R;   // uniform over the quarter's two warps
            float m_ref = -CUDART_INF_F, l_run = 0.f;   // l_run: this warp's columns only
            if (!(ok = warp_wait(&bars[kBarSFull + n % kSBufs], (n / kSBufs) & 1u, abort_flag)))
                break;
            for (int j = 0; j < rd.nsub; ++j, ++n) {
                if (j > 0 && !(ok = warp_wait(&bars[kBarSFull + n % kSBufs], (n / kSBufs) & 1u, abort_flag)))
                    break;
                const uint32_t t_s = t_lane + kColS + (n % kSBufs) * kSub;
                if (live) {
                    tc::fence_after_sync();
                    const int64_t sub_begin = rd.tok_begin + (int64_t)j * kSub;
                    const int valid = (int)min((int64_t)kSub, rd.tok_end - sub_begin);   // tokens of the sub-tile
                    // this row's own end (its key limit: shared prefix length, or causal limit)
                    const int row_end = (int)max(min((int64_t)valid, (int64_t)lim_row - sub_begin), (int64_t)0);
                    if (valid < kSub && warp == 0) {
                        // ragged end of a private tail: zero the V rows past it, whose memory may
                        // hold anything (0 * NaN would poison O), once this V copy has landed
                        if (!(ok = warp_wait(&bars[kBarFullV + n % kStagesV], (n / kStagesV) & 1u, abort_flag)))
                            break;
                        unsigned char *vst = base + kVOff + (n % kStagesV) * kKVBytes;
                        for (int c = lane; c < (kSub - valid) * 16; c += 32) {
                            const int rr = valid + c / 16, c16 = c % 16;
                            *reinterpret_cast<uint4 *>(vst + (c16 >> 3) * kHalfKV + rr * 128 + (c16 & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async();     // zeroed rows (generic) -> P.V MMA (async proxy)
                    }
                    // The copy `part` of a row owns tokens [part * 128/F, +128/F) of the sub-tile;
                    // the quarter's two warps take one half of them each (WC columns), and each
                    // warp writes P for its columns and zeros over its share of the other copies'.
                    auto subtile = [&](auto fc) -> bool {
                        constexpr int F = decltype(fc)::value;
                        constexpr int WC = 64 / F;                 // this warp's columns
                        // all of them stay in registers from the max to the exp pass: once the
                        // pair has met, the other warp's P stores may overwrite these S columns
                        constexpr int CW = WC;
                        constexpr int NCH = 1;
                        const int c0 = part * (128 / F) + half * WC;
                        float v[CW];
                        float mx = -CUDART_INF_F;
#pragma unroll
                        for (int ch = 0; ch < NCH; ++ch) {
                            const int rv = min(max(row_end - c0 - ch * CW, 0), CW);
                            tc::tmem_ld<CW>(t_s + c0 + ch * CW, v);
#pragma unroll
                            for (int i = 0; i < CW; ++i)
                                if (i < rv)
                                    mx = fmaxf(mx, v[i]);
                        }
                        // the row max over both warps' columns
                        xmax[((n & 1) * 2 + half) * 128 + row] = mx;
                        if (!pair_sync(pair, meets, abort_flag, lane))
                            return false;
                        mx = fmaxf(mx, xmax[((n & 1) * 2 + (half ^ 1)) * 128 + row]) * p.qscale;
                        const bool up = mx > m_ref + kRescaleThreshold;
                        const float m_next = up ? mx : m_ref;   // rows past the members hold garbage, never stored
                        // 1 if the reference stays, 0 at first; 1 while a row has seen no key at all
                        const float scale_o = m_next == -CUDART_INF_F ? 1.f : exp2f(m_ref - m_next);
                        if (__any_sync(kFullMask, up) && j > 0) {
                            // rescale this warp's half of the row's O (P.V of the previous sub-tile landed)
                            if (!warp_wait(&bars[kBarPvDone + (n - 1) % kSBufs], ((n - 1) / kSBufs) & 1u, abort_flag))
                                return false;
                            tc::fence_after_sync();
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                float o[16];
                                uint32_t ow[16];
                                tc::tmem_ld<16>(t_lane + kColO + half * 64 + c * 16, o);
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    ow[i] = __float_as_uint(o[i] * scale_o);
                                tc::tmem_st_nowait<16>(t_lane + kColO + half * 64 + c * 16, ow);
                            }
                            tc::tmem_wait_st();
                        }
                        l_run *= scale_o;
                        m_ref = m_next;
                        // P = 2^(s - m) as bf16 pairs, stored in pieces of at most 16 words
                        float lsum = 0.f;
#pragma unroll
                        for (int ch = 0; ch < NCH; ++ch) {
                            const int rv = min(max(row_end - c0 - ch * CW, 0), CW);
                            uint32_t w[CW / 2];
#pragma unroll
                            for (int i = 0; i < CW / 2; ++i) {
                                const float p0 = 2 * i < rv ? fast_exp2(fmaf(v[2 * i], p.qscale, -m_ref)) : 0.f;
                                const float p1 = 2 * i + 1 < rv ? fast_exp2(fmaf(v[2 * i + 1], p.qscale, -m_ref)) : 0.f;
                                lsum += p0 + p1;
                                w[i] = cvt_bf16x2(p0, p1);
                            }
                            tc::tmem_st_nowait<CW / 2>(t_s + (c0 + ch * CW) / 2, w);
                        }
                        // zeros over this warp's share of the other copies' columns
                        if constexpr (F > 1) {
#pragma unroll
                            for (int k = 0; k < F; ++k)
                                if (k != part)
                                    tc::tmem_zero_nowait<WC / 2>(t_s + k * (64 / F) + half * (WC / 2));
                        }
                        tc::tmem_wait_st();
                        l_run += lsum;
                        tc::fence_before_sync();
                        return true;
                    };
                    const bool good = rd.F == 4   ? subtile(std::integral_constant<int, 4>{})
                                      : rd.F == 2 ? subtile(std::integral_constant<int, 2>{})
                                                  : subtile(std::integral_constant<int, 1>{});
                    if (!(ok = good))
                        break;
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars[kBarPFull + n % kSBufs]);
                // the next run's Q rows (brought into L2 at this run's start) into the Q buffer of
                // the run before this one, whose S MMAs completed before this run's first S
                if (j == 0 && rn.nsub > 0) {
                    load_q(p, rn, G, row, b_next, half, qw);
                    store_q(qw, half, t_lane + kColQ + ((r + 1) % kQBufs) * 64, &bars[kBarQFull + (r + 1) % kQBufs],
                            lane);
                }
                if (j == 0 && e_last >= 0) {
                    // run r-1's epilogue: its last P.V ran while this P was being made
                    if (!(ok = epilogue()))
                        break;
                    e_last = -1;
                }
            }
            if (!ok)
                break;
            ed = rd;
            e_b = b_row;
            e_m = m_ref;
            e_l = l_run;
            e_last = n - 1;
            rd = rn;
            b_row = b_next;
            lim_row = lim_next;
        }
        if (ok && e_last >= 0)
            ok = epilogue();
        if (!ok)
            *abort_flag = 1;
    }

    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 && *abort_flag != 0)
        record_error(p.err, RLT_DEVERR_TIMEOUT);
    if (warp == 0)
        tc::tmem_dealloc(tmem, kTmemCols);
    if (tid == 0)
        pdl_wait();                              // no CTA ends before the grids it depends on
}

// ---------------------------------------------------------- tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D view of one bank: rows of head_dim = 128 bf16, boxes of 64 x box_rows, 128B swizzle.
bool make_map(CUtensorMap *map, const void *bank, int64_t rows, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128 * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(bank), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefix_supported(int head_dim, int group, int page_size)
{
    return head_dim == 128 && (group == 1 || group == 2 || group == 4 || group == 8) &&
           page_size % 16 == 0 && (kPrefixTile % page_size == 0 || page_size % kPrefixTile == 0);
}

size_t prefix_smem_bytes(int, int) { return kSmemP; }

cudaError_t launch_prefix(const DecodeParams &p, const PrefixParams &pp, const void *k_bank,
                          const void *v_bank, int64_t bank_rows, cudaStream_t stream, bool early)
{
    if (pp.num_segments == 0 || pp.work_units == 0)
        return cudaSuccess;
    if (pp.chunk_tiles < 1 || pp.chunk_tiles > kMaxChunkTiles || bank_rows >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    const int box_rows = p.page_size < kSub ? p.page_size : kSub;
    CUtensorMap kmap, vmap;
    if (!make_map(&kmap, k_bank, bank_rows, box_rows) || !make_map(&vmap, v_bank, bank_rows, box_rows))
        return cudaErrorInvalidValue;
    static std::atomic<uint64_t> configured[3]{{0}, {0}, {0}};
    const bool append = p.k_new != nullptr;
    const int which = append ? 0 : pp.l2_ahead != 0 ? 2 : 1;   // (the fused append runs no split-K rest)
    auto kernel = which == 0   ? decode_prefix_kernel<true, false>
                  : which == 1 ? decode_prefix_kernel<false, false>
                               : decode_prefix_kernel<false, true>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || (configured[which].load() & bit) == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemP);
        if (e != cudaSuccess)
            return e;
        configured[which].fetch_or(bit);
    }
    if (pp.ctas < 1)
        return cudaErrorInvalidValue;
    return launch_kernel(kernel, dim3(pp.ctas), dim3(kPThreads), kSmemP, stream, early, kmap, vmap, p, pp);
}

}  // namespace rlt

// ------------------------------------------------------------- host planner

extern "C" RLT_API rlt_status rlt_plan_prefix(const int32_t *page_table, int32_t max_pages,
                                              const int32_t *seq_lens, int32_t batch,
                                              int32_t page_size, int32_t chunk_tiles,
                                              int32_t query_group, int32_t private_tails,
                                              int32_t *segments,
                                              int32_t max_segments, int32_t *members,
                                              int32_t *member_limit, int32_t max_member_entries,
                                              int32_t *request_prefix,
                                              int32_t *sizes)
{
    using rlt::kPrefixTile;
    if (batch < 0 || max_pages < 0 || page_size < 1 || chunk_tiles < 1 ||
        chunk_tiles > rlt::kMaxChunkTiles || query_group < 1 || query_group > 128 ||
        max_segments < 0 || max_member_entries < 0 ||
        sizes == nullptr || (batch > 0 && (page_table == nullptr || seq_lens == nullptr ||
                                           request_prefix == nullptr)))
        return RLT_ERR_INVALID_ARG;
    if (kPrefixTile % page_size != 0 && page_size % kPrefixTile != 0)
        return RLT_ERR_UNSUPPORTED;
    const int per_tile = page_size < kPrefixTile ? kPrefixTile / page_size : 1;

    // requests b and c share tile t when they map it to the same pages (for pages larger
    // than a tile, the same page: the in-page offset is t's in both)
    auto same_tile = [&](int b, int c, int t) {
        const int64_t tok = (int64_t)t * kPrefixTile;
        const int32_t *rb = page_table + (int64_t)b * max_pages, *rc = page_table + (int64_t)c * max_pages;
        for (int j = 0; j < per_tile; ++j) {
            const int64_t idx = (tok + (int64_t)j * page_size) / page_size;
            if (rb[idx] != rc[idx])
                return false;
        }
        return true;
    };
    std::vector<int> full_tiles(batch);
    for (int b = 0; b < batch; ++b) {
        const int64_t L = std::min<int64_t>(std::max(seq_lens[b], 0), (int64_t)max_pages * page_size);
        full_tiles[b] = (int)(L / kPrefixTile);
    }

    // mem: member requests; lim: each member's key count in the segment (its shared tokens)
    struct Seg {
        int first, tiles, parent;
        std::vector<int> mem;
        int64_t end_token;
        std::vector<int64_t> lim;
        int page_row = -1;                     // whose pages the kernel reads (-1: the last member)
    };
    std::vector<Seg> segs;
    std::vector<int> deepest(batch, -1);       // segment holding each request's last shared tile
    struct Group { std::vector<int> mem; int seg; };
    std::vector<Group> level, next;
    {
        Group root{{}, -1};
        for (int b = 0; b < batch; ++b)
            if (full_tiles[b] > 0)
                root.mem.push_back(b);
        if (root.mem.size() >= 2)
            level.push_back(root);
    }
    // walk the trie of tiles from position 0: at tile t each group of requests that agreed
    // on tiles 0..t-1 splits by tile t's pages (a bucket: the requests whose tile t matches
    // the first remaining one's); buckets of >= 2 requests go on
    std::vector<int> rest, bucket, others;
    for (int t = 0; !level.empty(); ++t) {
        next.clear();
        for (const Group &grp : level) {
            rest.clear();
            for (int b : grp.mem)
                if (full_tiles[b] > t)
                    rest.push_back(b);
            while (rest.size() >= 2) {
                const int rep = rest[0];
                bucket.clear();
                others.clear();
                for (int b : rest)
                    (b == rep || same_tile(b, rep, t) ? bucket : others).push_back(b);
                rest.swap(others);
                if (bucket.size() < 2)
                    continue;                      // not shared: that request's prefix ends here
                int s;
                if (grp.seg >= 0 && bucket == segs[grp.seg].mem &&
                    segs[grp.seg].first + segs[grp.seg].tiles == t) {
                    s = grp.seg;                   // same members: the segment grows
                    segs[s].tiles++;
                } else {
                    s = (int)segs.size();
                    segs.push_back({t, 1, grp.seg, bucket, 0, {}});
                }
                for (int b : bucket)
                    deepest[b] = s;
                next.push_back({bucket, s});
            }
        }
        level.swap(next);
    }

    for (Seg &sg : segs) {
        sg.end_token = (int64_t)(sg.first + sg.tiles) * kPrefixTile;
        sg.lim.assign(sg.mem.size(), sg.end_token);
    }

    // A chain of segments that only shrinks (each the only child of the one before:
    // requests leaving a common prefix one after another, as in a radix tree over one
    // prompt) becomes ONE segment whose members carry their own key limits: the tiles
    // are still read once, and the kernel runs one long accumulation instead of one
    // short run per link.  Merged only where all members fit one member block of the
    // kernel (128 / query_group), so that no tile is read more often than before.
    const int per_block = 128 / query_group;
    {
        std::vector<std::vector<int>> kids(segs.size());
        for (size_t s = 0; s < segs.size(); ++s)
            if (segs[s].parent >= 0)
                kids[segs[s].parent].push_back((int)s);
        std::vector<int> into(segs.size(), -1);
        std::vector<Seg> out;
        for (size_t s = 0; s < segs.size(); ++s) {    // parents precede children
            if (into[s] >= 0)
                continue;
            const int idx = (int)out.size();
            Seg m = segs[s];
            m.parent = m.parent < 0 ? -1 : into[m.parent];
            into[s] = idx;
            std::map<int, size_t> pos;
            for (size_t i = 0; i < m.mem.size(); ++i)
                pos[m.mem[i]] = i;
            int cur = (int)s;
            if ((int)m.mem.size() <= per_block) {
                while (kids[cur].size() == 1) {
                    const int c = kids[cur][0];
                    m.tiles += segs[c].tiles;
                    m.end_token = segs[c].end_token;
                    for (int b : segs[c].mem)
                        m.lim[pos[b]] = segs[c].end_token;
                    into[c] = idx;
                    cur = c;
                }
            }
            // members by ascending limit: a member block then ends at its last member's
            // limit, and the page row (the longest member) holds every tile's pages
            std::vector<size_t> order(m.mem.size());
            for (size_t i = 0; i < order.size(); ++i)
                order[i] = i;
            std::stable_sort(order.begin(), order.end(),
                             [&](size_t a, size_t b) { return m.lim[a] < m.lim[b]; });
            Seg sorted = m;
            for (size_t i = 0; i < order.size(); ++i) {
                sorted.mem[i] = m.mem[order[i]];
                sorted.lim[i] = m.lim[order[i]];
            }
            out.push_back(sorted);
        }
        segs.swap(out);
        for (int b = 0; b < batch; ++b)
            deepest[b] = -1;
        for (size_t s = 0; s < segs.size(); ++s)
            for (int b : segs[s].mem)
                deepest[b] = (int)s;
    }
    // Without private tails the split-K kernel takes each request's rest in 16-token tiles,
    // so a member's shared prefix need not end on a 128-token tile: at the segment where its
    // sharing ends, its key limit goes on page by page while its page is the page row's (the
    // tensor-core kernel reads the segment's tiles from the page row's pages) and another
    // member of the segment maps that page too (a member that goes on to a deeper segment
    // reads that part of the tile there as well).  The pages a request shares with others past its last
    // whole shared tile are then read once per kv head here instead of once per request by
    // the split-K kernel; the segment's last tile may end mid-tile (end token), the kernel
    // masks each member's keys past its limit.  (With private tails every token past the
    // shared tiles belongs to a tail segment that starts on a tile; a segment of several
    // member blocks keeps its limits on its tiles.)
    if (!private_tails && page_size < kPrefixTile) {
        std::vector<int64_t> L(batch);
        for (int b = 0; b < batch; ++b)
            L[b] = std::min<int64_t>(std::max(seq_lens[b], 0), (int64_t)max_pages * page_size);
        auto page_of = [&](int b, int64_t tok) { return page_table[(int64_t)b * max_pages + tok / page_size]; };
        for (size_t s = 0; s < segs.size(); ++s) {
            Seg &sg = segs[s];
            if ((int)sg.mem.size() > per_block)
                continue;                          // several member blocks: limits stay on tiles
            const int pr = sg.mem.back();
            for (;;) {
                bool grew = false;
                for (size_t i = 0; i < sg.mem.size(); ++i) {
                    const int b = sg.mem[i];
                    const int64_t tok = sg.lim[i];
                    if (deepest[b] != (int)s || tok % page_size != 0 || tok + page_size > std::min(L[b], L[pr]) ||
                        page_of(b, tok) != page_of(pr, tok))
                        continue;
                    bool other = false;            // a second member maps this page here
                    for (size_t k = 0; k < sg.mem.size() && !other; ++k) {
                        const int c = sg.mem[k];
                        other = c != b && tok + page_size <= L[c] && page_of(c, tok) == page_of(b, tok);
                    }
                    if (!other)
                        continue;
                    sg.lim[i] = tok + page_size;
                    grew = true;
                }
                if (!grew)
                    break;
            }
            int64_t end = sg.end_token;
            for (int64_t x : sg.lim)
                end = std::max(end, x);
            sg.end_token = end;
            sg.tiles = (int)((end + kPrefixTile - 1) / kPrefixTile) - sg.first;
            // members stay in ascending limit order (a member block ends at its last member's
            // limit); the page row keeps its role even if another member's limit now exceeds
            // its own (that member's extension follows the page row's pages)
            sg.page_row = pr;
            std::vector<size_t> order(sg.mem.size());
            for (size_t i = 0; i < order.size(); ++i)
                order[i] = i;
            std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) { return sg.lim[a] < sg.lim[b]; });
            Seg sorted = sg;
            for (size_t i = 0; i < order.size(); ++i) {
                sorted.mem[i] = sg.mem[order[i]];
                sorted.lim[i] = sg.lim[order[i]];
            }
            sg = sorted;
        }
    }
    std::vector<int64_t> covered(batch, 0);
    for (int b = 0; b < batch; ++b) {
        if (deepest[b] < 0)
            continue;
        const Seg &sg = segs[deepest[b]];
        for (size_t i = 0; i < sg.mem.size(); ++i)
            if (sg.mem[i] == b)
                covered[b] = sg.lim[i];
    }
    if (private_tails) {
        // every request's own remaining tokens become a one-member segment
        for (int b = 0; b < batch; ++b) {
            const int64_t L = std::min<int64_t>(std::max(seq_lens[b], 0), (int64_t)max_pages * page_size);
            if (L <= covered[b])
                continue;
            const int first = (int)(covered[b] / kPrefixTile);
            const int tiles = (int)((L + kPrefixTile - 1) / kPrefixTile) - first;
            segs.push_back({first, tiles, deepest[b], {b}, L, {L}});
            deepest[b] = (int)segs.size() - 1;
            covered[b] = L;
        }
    }
    const int nseg = (int)segs.size();
    // per member, a segment has `chunks` partial slots per copy of its query rows
    std::vector<int> chunks(nseg), slot_base(nseg), slots(nseg);
    int64_t member_entries = 0;
    int max_chunks = 0, max_members = 0;
    for (int s = 0; s < nseg; ++s) {               // parents precede children
        chunks[s] = (segs[s].tiles + chunk_tiles - 1) / chunk_tiles;
        slots[s] = chunks[s] *
                   rlt::prefix_replication(std::min<int>((int)segs[s].mem.size(), per_block) * query_group);
        slot_base[s] = segs[s].parent < 0 ? 0 : slot_base[segs[s].parent] + slots[segs[s].parent];
        member_entries += (int64_t)segs[s].mem.size();
        max_chunks = std::max(max_chunks, chunks[s]);
        max_members = std::max(max_members, (int)segs[s].mem.size());
    }
    // work units: (segment, chunk, member block); a member block holds 128 / query_group members
    std::vector<int64_t> work_begin(nseg + 1, 0);
    for (int s = 0; s < nseg; ++s)
        work_begin[s + 1] = work_begin[s] + (int64_t)chunks[s] *
                                                ((segs[s].mem.size() + per_block - 1) / per_block);
    sizes[0] = nseg;
    sizes[1] = (int32_t)member_entries;
    sizes[2] = max_chunks;
    sizes[3] = 0;
    sizes[4] = max_members;
    sizes[6] = (int32_t)work_begin[nseg];
    int max_slots = 0;
    int64_t max_rest = 0;
    for (int b = 0; b < batch; ++b) {
        const int s = deepest[b];
        request_prefix[2 * b] = (int32_t)covered[b];
        request_prefix[2 * b + 1] = s < 0 ? 0 : slot_base[s] + slots[s];
        max_slots = std::max(max_slots, request_prefix[2 * b + 1]);
        const int64_t L = std::min<int64_t>(std::max(seq_lens[b], 0), (int64_t)max_pages * page_size);
        max_rest = std::max(max_rest, L - covered[b]);
    }
    sizes[3] = max_slots;
    sizes[5] = (int32_t)max_rest;
    if (nseg > max_segments || member_entries > max_member_entries)
        return RLT_ERR_OUT_OF_RANGE;               // sizes[] tells the caller what is needed
    if (nseg > 0 && (segments == nullptr || members == nullptr || member_limit == nullptr))
        return RLT_ERR_INVALID_ARG;
    int64_t m = 0;
    for (int s = 0; s < nseg; ++s) {
        int32_t *row = segments + (int64_t)s * rlt::kSegFields;
        row[rlt::kSegFirstTile] = segs[s].first;
        row[rlt::kSegNumTiles] = segs[s].tiles;
        row[rlt::kSegSlotBase] = slot_base[s];
        row[rlt::kSegMemberBegin] = (int32_t)m;
        row[rlt::kSegMemberCount] = (int32_t)segs[s].mem.size();
        row[rlt::kSegPageRow] = segs[s].page_row >= 0 ? segs[s].page_row : segs[s].mem.back();
        row[rlt::kSegEndToken] = (int32_t)segs[s].end_token;
        row[rlt::kSegWorkBegin] = (int32_t)work_begin[s];
        for (size_t i = 0; i < segs[s].mem.size(); ++i, ++m) {
            members[m] = segs[s].mem[i];
            member_limit[m] = (int32_t)segs[s].lim[i];
        }
    }
    return RLT_OK;
}

// ------------------------------------------------------ extend planner

// Work of a causal extend (span) attention for the tensor-core kernel: one
// segment per request with new tokens, covering its whole key range, whose
// "members" are its new tokens (rows of the packed q, request by request) with
// their causal key counts.  Each member block (128 / query_group new tokens)
// needs keys only up to its last token's limit; its rows' partial slots are
// the chunks up to there (row_prefix[row] = {limit, slots}, row_len[row] =
// limit), so the combine merges exactly what the kernel wrote.
extern "C" RLT_API rlt_status rlt_plan_extend(const int32_t *seq_lens, const int32_t *new_lens,
                                              int32_t batch, int32_t page_size, int32_t chunk_tiles,
                                              int32_t query_group, int32_t *segments, int32_t max_segments,
                                              int32_t *members, int32_t *member_limit,
                                              int32_t max_member_entries, int32_t *row_prefix,
                                              int32_t *row_len, int32_t *sizes)
{
    using rlt::kPrefixTile;
    if (batch < 0 || page_size < 1 || chunk_tiles < 1 || chunk_tiles > rlt::kMaxChunkTiles ||
        query_group < 1 || query_group > 128 || 128 % query_group != 0 || max_segments < 0 ||
        max_member_entries < 0 || sizes == nullptr ||
        (batch > 0 && (seq_lens == nullptr || new_lens == nullptr)))
        return RLT_ERR_INVALID_ARG;
    if (kPrefixTile % page_size != 0 && page_size % kPrefixTile != 0)
        return RLT_ERR_UNSUPPORTED;
    const int per_block = 128 / query_group;
    const int64_t chunk_tokens = (int64_t)chunk_tiles * kPrefixTile;
    int64_t nseg = 0, rows = 0, units = 0;
    int max_chunks = 0, max_members = 0, max_slots = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t L = seq_lens[b], n = new_lens[b];
        if (n < 0 || L < n || L > INT32_MAX)
            return RLT_ERR_INVALID_ARG;
        if (n == 0)
            continue;
        const int tiles = (int)((L + kPrefixTile - 1) / kPrefixTile);
        const int chunks = (tiles + chunk_tiles - 1) / chunk_tiles;
        ++nseg;
        rows += n;
        units += (int64_t)chunks * ((n + per_block - 1) / per_block);
        max_chunks = std::max(max_chunks, chunks);
        max_members = std::max(max_members, (int)n);
        max_slots = std::max(max_slots, chunks * rlt::prefix_replication(
                                                     (int)std::min<int64_t>(n, per_block) * query_group));
    }
    if (rows > INT32_MAX || units > INT32_MAX)
        return RLT_ERR_OUT_OF_RANGE;
    sizes[0] = (int32_t)nseg;
    sizes[1] = (int32_t)rows;
    sizes[2] = max_chunks;
    sizes[3] = max_slots;             // partial slots per row: every chunk of the longest key range, per copy
    sizes[4] = max_members;
    sizes[5] = 0;                     // no split-K rest
    sizes[6] = (int32_t)units;
    if (nseg > max_segments || rows > max_member_entries)
        return RLT_ERR_OUT_OF_RANGE;  // sizes[] tells the caller what is needed
    if (nseg > 0 && (segments == nullptr || members == nullptr || member_limit == nullptr ||
                     row_prefix == nullptr || row_len == nullptr))
        return RLT_ERR_INVALID_ARG;
    int64_t s = 0, m = 0, work = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t L = seq_lens[b], n = new_lens[b];
        if (n == 0)
            continue;
        const int tiles = (int)((L + kPrefixTile - 1) / kPrefixTile);
        const int chunks = (tiles + chunk_tiles - 1) / chunk_tiles;
        const int F = rlt::prefix_replication((int)std::min<int64_t>(n, per_block) * query_group);
        int32_t *row = segments + s * rlt::kSegFields;
        row[rlt::kSegFirstTile] = 0;
        row[rlt::kSegNumTiles] = tiles;
        row[rlt::kSegSlotBase] = 0;
        row[rlt::kSegMemberBegin] = (int32_t)m;
        row[rlt::kSegMemberCount] = (int32_t)n;
        row[rlt::kSegPageRow] = b;
        row[rlt::kSegEndToken] = (int32_t)L;
        row[rlt::kSegWorkBegin] = (int32_t)work;
        for (int64_t i = 0; i < n; ++i) {
            const int64_t limit = L - n + i + 1;
            const int64_t last = std::min(n, (i / per_block + 1) * per_block) - 1;   // block's last token
            const int64_t block_end = L - n + last + 1;
            members[m + i] = (int32_t)(m + i);                 // packed q row of this new token
            member_limit[m + i] = (int32_t)limit;
            row_prefix[2 * (m + i)] = (int32_t)limit;
            row_prefix[2 * (m + i) + 1] = (int32_t)((block_end + chunk_tokens - 1) / chunk_tokens) * F;
            row_len[m + i] = (int32_t)limit;
        }
        work += (int64_t)chunks * ((n + per_block - 1) / per_block);
        m += n;
        ++s;
    }
    return RLT_OK;
}
