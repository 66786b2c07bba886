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
// shared memory.  Each CTA writes one (o, log2-sum-exp) partial per query row;
// the split-K kernel covers each request's remaining tokens and the combine
// kernel merges everything.
#include <math_constants.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <vector>

#include "rlt.h"
#include "rlt_device.cuh"
#include "rlt_internal.h"
#include "rlt_tc.cuh"

namespace rlt {
namespace {

constexpr int kPThreads = 128;              // 4 warps, one TMEM lane quadrant each
constexpr int kPStages = 2;                 // K/V tile ring depth
constexpr int kHalf = 128 * 128;            // one 64-element column block of a 128-row tile
constexpr int kTileBytesP = 2 * kHalf;      // K (or V) tile: 128 tokens x 128 dims, bf16
constexpr int kStageBytesP = 2 * kTileBytesP;
constexpr int kMaxChunkTiles = 32;
constexpr int kMaxBoxes = 8;                // 128-token tile = up to 8 page boxes (page_size 16)
constexpr int kQOff = 0, kPOff = kTileBytesP, kStageOff = 2 * kTileBytesP;
constexpr int kRowsOff = kStageOff + kPStages * kStageBytesP;
constexpr int kMemOff = kRowsOff + kMaxChunkTiles * kMaxBoxes * 4;
constexpr int kBarOff = kMemOff + kPThreads * 4;
constexpr int kSmemP = kBarOff + 64 + 1024;  // + alignment slack for the 1024-byte base
constexpr uint32_t kTmemCols = 256;          // S in columns [0,128), O in [128,256)

__global__ void __launch_bounds__(kPThreads, 1)
    decode_prefix_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const DecodeParams p,
                         const PrefixParams pp)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *qs = base + kQOff;
    unsigned char *ps = base + kPOff;
    unsigned char *stages = base + kStageOff;
    int32_t *box_rows = reinterpret_cast<int32_t *>(base + kRowsOff);
    int32_t *mem = reinterpret_cast<int32_t *>(base + kMemOff);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kBarOff);   // full[2], s_done, o_done
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 4);

    const int G = p.num_q_heads / p.num_kv_heads;
    const int chunk = blockIdx.x, g = blockIdx.y;
    const int seg = blockIdx.z / pp.member_blocks, mb = blockIdx.z % pp.member_blocks;
    if (seg >= pp.num_segments)
        return;
    const int32_t *sd = pp.segments + seg * kSegFields;
    const int num_tiles = sd[kSegNumTiles];
    const int t0 = chunk * pp.chunk_tiles;
    if (t0 >= num_tiles)
        return;
    const int nt = min(pp.chunk_tiles, num_tiles - t0);
    const int per_block = kPThreads / G;
    const int m0 = mb * per_block;
    const int n_mem = min(per_block, sd[kSegMemberCount] - m0);
    if (n_mem <= 0)
        return;
    const int R = n_mem * G;                    // live query rows of this CTA
    const int page_row = sd[kSegPageRow];
    const int first_tile = sd[kSegFirstTile] + t0;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int BR = p.page_size < kPrefixTile ? p.page_size : kPrefixTile;   // rows per TMA box
    const int boxes = kPrefixTile / BR;

    for (int i = tid; i < n_mem; i += kPThreads)
        mem[i] = pp.members[sd[kSegMemberBegin] + m0 + i];
    for (int i = tid; i < nt * boxes; i += kPThreads) {
        const int64_t tok = (int64_t)(first_tile + i / boxes) * kPrefixTile + (i % boxes) * BR;
        const int64_t idx = tok / p.page_size;
        int64_t page = idx < p.max_pages ? p.page_table[(int64_t)page_row * p.max_pages + idx] : -1;
        if (page < 0 || page >= p.num_pages) {
            record_error(p.err, RLT_DEVERR_BAD_PAGE);
            page = 0;                            // stay in bounds; the result is flagged
        }
        box_rows[i] = (int32_t)((page * p.num_kv_heads + g) * p.page_size + tok % p.page_size);
    }
    if (tid == 0) {
        for (int i = 0; i < 4; ++i)
            mbar_init(&bars[i], 1);
        mbar_init_fence();
    }
    if (warp == 0)
        tc::tmem_alloc(tslot, kTmemCols);
    __syncthreads();

    // Query rows r = member * G + head, K-major, 128-byte swizzled (rows >= R unused).
    for (int i = tid; i < R * 16; i += kPThreads) {
        const int r = i >> 4, c16 = i & 15;
        const int b = mem[r / G], h = r % G;
        const uint4 v = *reinterpret_cast<const uint4 *>(
            p.q + ((int64_t)b * p.num_q_heads + g * G + h) * 128 + c16 * 8);
        *reinterpret_cast<uint4 *>(qs + (c16 >> 3) * kHalf + tc::sw128_offset(r, (c16 & 7) * 8)) = v;
    }
    fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    // Warp 0 loads tile i into stage i % 2: lane j copies box j/4, column block (j/2)&1,
    // of K (j even) or V (j odd); lane 0 arms the barrier first.
    auto load_tile = [&](int i) {
        uint64_t *full = &bars[i % kPStages];
        unsigned char *st = stages + (i % kPStages) * kStageBytesP;
        if (lane == 0)
            mbar_arrive_expect_tx(full, kStageBytesP);
        __syncwarp();
        if (lane < 4 * boxes) {
            const int box = lane >> 2, half = (lane >> 1) & 1, is_v = lane & 1;
            tc::tma_load_2d(st + is_v * kTileBytesP + half * kHalf + box * BR * 128,
                            is_v ? &vmap : &kmap, half * 64, box_rows[i * boxes + box], full);
        }
    };
    int issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            tc::prefetch_tmap(&kmap);
            tc::prefetch_tmap(&vmap);
        }
        for (; issued < kPStages && issued < nt; ++issued)
            load_tile(issued);
    }

    const uint32_t id_s = tc::instr_desc_bf16(128, 128, false);
    const uint32_t id_o = tc::instr_desc_bf16(128, 128, true);
    const uint32_t qa = smem_u32(qs), pa = smem_u32(ps);
    const int row = warp * 32 + lane;
    const bool warp_live = warp * 32 < R;
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);

    float acc[128];
#pragma unroll
    for (int j = 0; j < 128; ++j)
        acc[j] = 0.f;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    uint32_t ph_full = 0, ph_s = 0, ph_o = 0;
    bool ok = true, pending_s = false, pending_o = false;
    int consumed = 0;

    for (int i = 0; i < nt; ++i) {
        const int s = i % kPStages;
        const uint32_t ka = smem_u32(stages + s * kStageBytesP);
        const uint32_t va = ka + kTileBytesP;
        if (tid == 0) {
            ok = mbar_wait(&bars[s], (ph_full >> s) & 1u);
            if (ok) {
                ph_full ^= 1u << s;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16(tmem, tc::smem_desc(qa + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024),
                                 tc::smem_desc(ka + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024), id_s,
                                 kk > 0);
                tc::mma_commit(&bars[2]);
            }
        }
        ok = __syncthreads_and(ok) != 0;
        if (!ok)
            break;
        ++consumed;
        pending_s = true;
        ok = mbar_wait(&bars[2], ph_s);
        if (ok) {
            ph_s ^= 1u;
            pending_s = false;
        }
        if (!__syncthreads_and(ok)) {
            ok = false;
            break;
        }
        tc::fence_after_sync();

        // Softmax of this thread's query row over the tile's 128 tokens (log2 domain).
        float m_new = m_run, alpha = 1.f;
        if (warp_live) {
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[32];
                tc::tmem_ld32(t_row + c * 32, v);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    mx = fmaxf(mx, v[j]);
            }
            m_new = fmaxf(m_run, mx * p.qscale);
            alpha = exp2f(m_run - m_new);
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[32];
                tc::tmem_ld32(t_row + c * 32, v);
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float p0 = exp2f(fmaf(v[2 * j], p.qscale, -m_new));
                    const float p1 = exp2f(fmaf(v[2 * j + 1], p.qscale, -m_new));
                    lsum += p0 + p1;
                    w[j] = pack_bf16x2(p0, p1);
                }
                if (row < R) {
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        *reinterpret_cast<uint4 *>(ps + (c >> 1) * kHalf +
                                                   tc::sw128_offset(row, (c & 1) * 32 + q8 * 8)) =
                            make_uint4(w[4 * q8], w[4 * q8 + 1], w[4 * q8 + 2], w[4 * q8 + 3]);
                }
            }
            l_run = l_run * alpha + lsum;
        }
        fence_proxy_async();                    // P (generic writes) -> MMA (async proxy)
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16(tmem + 128, tc::smem_desc(pa + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024),
                             tc::smem_desc(va + kk * 2048, kHalf, 1024), id_o, kk > 0);
            tc::mma_commit(&bars[3]);
        }
        pending_o = true;
        ok = mbar_wait(&bars[3], ph_o);
        if (ok) {
            ph_o ^= 1u;
            pending_o = false;
        }
        if (!__syncthreads_and(ok)) {
            ok = false;
            break;
        }
        tc::fence_after_sync();
        if (warp_live) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[32];
                tc::tmem_ld32(t_row + 128 + c * 32, v);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    acc[c * 32 + j] = fmaf(acc[c * 32 + j], alpha, v[j]);
            }
        }
        m_run = m_new;
        // both MMAs reading stage s are complete: refill it
        if (warp == 0 && issued < nt) {
            load_tile(issued);
            ++issued;
        }
    }

    if (!ok) {
        // A wait ran out: flag it, let this CTA's copies still in flight land
        // (bounded), and skip the partial.
        if (tid == 0) {
            record_error(p.err, RLT_DEVERR_TIMEOUT);
            for (int k = consumed; k < issued; ++k) {
                const int s = k % kPStages;
                mbar_wait(&bars[s], (ph_full >> s) & 1u);
                ph_full ^= 1u << s;
            }
            if (pending_s)
                mbar_wait(&bars[2], ph_s);      // MMAs still reading shared memory
            if (pending_o)
                mbar_wait(&bars[3], ph_o);
        }
    } else if (warp_live && row < R) {
        const int b = mem[row / G], h = row % G;
        const int64_t slot = ((int64_t)b * p.num_q_heads + g * G + h) * p.part_stride +
                             pp.segments[seg * kSegFields + kSegSlotBase] + chunk;
        const float inv = 1.f / l_run;
        float4 *dst = reinterpret_cast<float4 *>(p.o_part + slot * 128);
#pragma unroll
        for (int j = 0; j < 32; ++j)
            dst[j] = make_float4(acc[4 * j] * inv, acc[4 * j + 1] * inv, acc[4 * j + 2] * inv,
                                 acc[4 * j + 3] * inv);
        p.lse_part[slot] = m_run + log2f(l_run);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0)
        tc::tmem_dealloc(tmem, kTmemCols);
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

cudaError_t launch_prefix(const DecodeParams &p, const PrefixParams &pp, int max_chunks,
                          const void *k_bank, const void *v_bank, int64_t bank_rows,
                          cudaStream_t stream)
{
    if (pp.num_segments == 0 || max_chunks == 0)
        return cudaSuccess;
    if (pp.chunk_tiles < 1 || pp.chunk_tiles > kMaxChunkTiles || bank_rows >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    const int box_rows = p.page_size < kPrefixTile ? p.page_size : kPrefixTile;
    CUtensorMap kmap, vmap;
    if (!make_map(&kmap, k_bank, bank_rows, box_rows) || !make_map(&vmap, v_bank, bank_rows, box_rows))
        return cudaErrorInvalidValue;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || (configured.load() & bit) == 0) {
        e = cudaFuncSetAttribute(decode_prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemP);
        if (e != cudaSuccess)
            return e;
        configured.fetch_or(bit);
    }
    const dim3 grid(max_chunks, p.num_kv_heads, pp.num_segments * pp.member_blocks);
    decode_prefix_kernel<<<grid, kPThreads, kSmemP, stream>>>(kmap, vmap, p, pp);
    return cudaGetLastError();
}

}  // namespace rlt

// ------------------------------------------------------------- host planner

extern "C" RLT_API rlt_status rlt_plan_prefix(const int32_t *page_table, int32_t max_pages,
                                              const int32_t *seq_lens, int32_t batch,
                                              int32_t page_size, int32_t chunk_tiles,
                                              int32_t *segments, int32_t max_segments,
                                              int32_t *members, int32_t max_member_entries,
                                              int32_t *request_prefix, int32_t *sizes)
{
    using rlt::kPrefixTile;
    if (batch < 0 || max_pages < 0 || page_size < 1 || chunk_tiles < 1 ||
        chunk_tiles > rlt::kMaxChunkTiles || max_segments < 0 || max_member_entries < 0 ||
        sizes == nullptr || (batch > 0 && (page_table == nullptr || seq_lens == nullptr ||
                                           request_prefix == nullptr)))
        return RLT_ERR_INVALID_ARG;
    if (kPrefixTile % page_size != 0 && page_size % kPrefixTile != 0)
        return RLT_ERR_UNSUPPORTED;
    const int per_tile = page_size < kPrefixTile ? kPrefixTile / page_size : 1;

    // tile t of request b is keyed by the page ids (and, for big pages, the offset) it covers
    auto key = [&](int b, int t) {
        std::vector<int32_t> k;
        const int64_t tok = (int64_t)t * kPrefixTile;
        for (int j = 0; j < per_tile; ++j)
            k.push_back(page_table[(int64_t)b * max_pages + (tok + (int64_t)j * page_size) / page_size]);
        if (page_size > kPrefixTile)
            k.push_back((int32_t)(tok % page_size));
        return k;
    };
    auto full_tiles = [&](int b) {
        const int64_t L = std::min<int64_t>(std::max(seq_lens[b], 0), (int64_t)max_pages * page_size);
        return (int)(L / kPrefixTile);
    };

    struct Seg { int first, tiles, parent; std::vector<int> mem; };
    std::vector<Seg> segs;
    std::vector<int> deepest(batch, -1);       // segment holding each request's last shared tile
    struct Group { std::vector<int> mem; int seg; };
    std::vector<Group> level;
    {
        Group root{{}, -1};
        for (int b = 0; b < batch; ++b)
            if (full_tiles(b) > 0)
                root.mem.push_back(b);
        if (root.mem.size() >= 2)
            level.push_back(root);
    }
    for (int t = 0; !level.empty(); ++t) {
        std::vector<Group> next;
        for (const Group &grp : level) {
            std::map<std::vector<int32_t>, std::vector<int>> buckets;
            for (int b : grp.mem)
                if (full_tiles(b) > t)
                    buckets[key(b, t)].push_back(b);
            for (auto &kv : buckets) {
                if (kv.second.size() < 2)
                    continue;                      // not shared: that request's prefix ends here
                int s;
                if (grp.seg >= 0 && kv.second == segs[grp.seg].mem &&
                    segs[grp.seg].first + segs[grp.seg].tiles == t) {
                    s = grp.seg;                   // same members: the segment grows
                    segs[s].tiles++;
                } else {
                    s = (int)segs.size();
                    segs.push_back({t, 1, grp.seg, kv.second});
                }
                for (int b : kv.second)
                    deepest[b] = s;
                next.push_back({kv.second, s});
            }
        }
        level.swap(next);
    }

    const int nseg = (int)segs.size();
    std::vector<int> chunks(nseg), slot_base(nseg);
    int64_t member_entries = 0;
    int max_chunks = 0, max_members = 0;
    for (int s = 0; s < nseg; ++s) {               // parents precede children
        chunks[s] = (segs[s].tiles + chunk_tiles - 1) / chunk_tiles;
        slot_base[s] = segs[s].parent < 0 ? 0 : slot_base[segs[s].parent] + chunks[segs[s].parent];
        member_entries += (int64_t)segs[s].mem.size();
        max_chunks = std::max(max_chunks, chunks[s]);
        max_members = std::max(max_members, (int)segs[s].mem.size());
    }
    sizes[0] = nseg;
    sizes[1] = (int32_t)member_entries;
    sizes[2] = max_chunks;
    sizes[3] = 0;
    sizes[4] = max_members;
    int max_slots = 0;
    for (int b = 0; b < batch; ++b) {
        const int s = deepest[b];
        request_prefix[2 * b] = s < 0 ? 0 : (segs[s].first + segs[s].tiles) * kPrefixTile;
        request_prefix[2 * b + 1] = s < 0 ? 0 : slot_base[s] + chunks[s];
        max_slots = std::max(max_slots, request_prefix[2 * b + 1]);
    }
    sizes[3] = max_slots;
    if (nseg > max_segments || member_entries > max_member_entries)
        return RLT_ERR_OUT_OF_RANGE;               // sizes[] tells the caller what is needed
    int64_t m = 0;
    for (int s = 0; s < nseg; ++s) {
        int32_t *row = segments + (int64_t)s * rlt::kSegFields;
        row[rlt::kSegFirstTile] = segs[s].first;
        row[rlt::kSegNumTiles] = segs[s].tiles;
        row[rlt::kSegSlotBase] = slot_base[s];
        row[rlt::kSegMemberBegin] = (int32_t)m;
        row[rlt::kSegMemberCount] = (int32_t)segs[s].mem.size();
        row[rlt::kSegPageRow] = segs[s].mem[0];
        for (int b : segs[s].mem)
            members[m++] = b;
    }
    return RLT_OK;
}
