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

// Roles: warps 0-3 own query rows 0..127 (softmax, rescale, output; warp w may
// only touch TMEM lanes 32w..32w+31), warp 4 issues the MMAs, warp 5 issues the
// TMA copies.  Work goes in 64-token sub-tiles (half a planner tile).
constexpr int kSoftWarps = 4;
constexpr int kPThreads = (kSoftWarps + 3) * 32;
// The MMA warp spins on its barriers: it shares a scheduler (warp id mod 4) with softmax warp 2,
// which has live rows only for more than 64 query rows.
constexpr int kLoadVWarp = kSoftWarps, kLoadKWarp = kSoftWarps + 1, kMmaWarp = kSoftWarps + 2;
constexpr int kSub = 64;                    // tokens per sub-tile
constexpr int kStagesP = 4;                 // K/V sub-tile ring depth
constexpr int kHalfQ = 128 * 128;           // one 64-element column block of the 128 Q rows
constexpr int kHalfKV = kSub * 128;         // one 64-dim column block of a sub-tile (64 rows x 128 B)
constexpr int kKVBytes = 2 * kHalfKV;       // K (or V) of one sub-tile
constexpr int kStageBytesP = 2 * kKVBytes;  // one K slot + one V slot
constexpr int kPBytes = 128 * kSub * 2;     // P of one sub-tile: 128 rows x 64 tokens, bf16
constexpr int kMaxChunkTiles = 32;
constexpr int kMaxBoxes = 2 * kMaxChunkTiles * 4;   // sub-tiles x boxes (page_size 16: 4 per sub-tile)
constexpr int kQOff = 0;
constexpr int kSBufs = 4;                   // S buffers in TMEM: S runs up to 4 sub-tiles ahead
constexpr int kPBufs = 3;                   // P buffers in shared memory
constexpr int kPOff = kQOff + 2 * kHalfQ;
constexpr int kStageOff = kPOff + kPBufs * kPBytes;
constexpr int kRowsOff = kStageOff + kStagesP * kStageBytesP;
constexpr int kMemOff = kRowsOff + kMaxBoxes * 4;
constexpr int kBarOff = kMemOff + 128 * 4;
// K and V have rings of their own: a K slot is free once S has read it, a V slot once P.V has
constexpr int kNumBars = 4 * kStagesP + 2 * kSBufs + kPBufs;   // K/V rings, s_full, p_full, o_full
constexpr int kSmemP = kBarOff + kNumBars * 8 + 16 + 1024;
constexpr uint32_t kTmemCols = 512;         // S[4] x 64 cols, O x 128 cols
constexpr uint32_t kColS = 0, kColO = kSBufs * kSub;
// O accumulates in TMEM against a per-row reference max that moves only when
// the row's running max exceeds it by more than this (log2 units): p <= 2^8.
constexpr float kRescaleThreshold = 8.f;

constexpr int kQBarrier = 1;                // named barrier: Q staged (softmax warps + MMA warp)

__device__ __forceinline__ void named_barrier_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__global__ void __launch_bounds__(kPThreads, 1)
    decode_prefix_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const DecodeParams p,
                         const PrefixParams pp)
{
    // the split-K kernel that follows may start on SMs this grid leaves idle
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *qs = base + kQOff;
    unsigned char *pbuf = base + kPOff;
    unsigned char *stages = base + kStageOff;
    int32_t *box_rows = reinterpret_cast<int32_t *>(base + kRowsOff);
    int32_t *mem = reinterpret_cast<int32_t *>(base + kMemOff);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kBarOff);
    uint64_t *full_k = bars, *free_k = bars + kStagesP, *full_v = bars + 2 * kStagesP,
             *free_v = bars + 3 * kStagesP;
    uint64_t *s_full = bars + 4 * kStagesP, *p_full = s_full + kSBufs, *o_full = p_full + kSBufs;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

    // work unit -> (segment, chunk, member block) through the segments' work offsets
    const int G = p.num_q_heads / p.num_kv_heads;
    const int g = blockIdx.y;
    const int unit = blockIdx.x;
    int lo = 0, hi = pp.num_segments - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pp.segments[mid * kSegFields + kSegWorkBegin] <= unit)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int32_t *sd = pp.segments + lo * kSegFields;
    const int per_block = 128 / G;
    const int mblocks = (sd[kSegMemberCount] + per_block - 1) / per_block;
    const int local = unit - sd[kSegWorkBegin];
    const int chunk = local / mblocks, mb = local % mblocks;
    const int num_tiles = sd[kSegNumTiles];
    const int t0 = chunk * pp.chunk_tiles;
    if (t0 >= num_tiles || local < 0)
        return;
    const int nt = min(pp.chunk_tiles, num_tiles - t0);
    const int m0 = mb * per_block;
    const int n_mem = min(per_block, sd[kSegMemberCount] - m0);
    if (n_mem <= 0)
        return;
    const int R = n_mem * G;                    // live query rows of this CTA
    const int page_row = sd[kSegPageRow];
    const int first_tile = sd[kSegFirstTile] + t0;
    // tokens [tok_begin, tok_end) of this CTA; a private tail segment ends mid-tile
    const int64_t tok_begin = (int64_t)first_tile * kPrefixTile;
    const int64_t tok_end = min((int64_t)(first_tile + nt) * kPrefixTile, (int64_t)sd[kSegEndToken]);
    if (tok_end <= tok_begin)
        return;
    const int nsub = (int)((tok_end - tok_begin + kSub - 1) / kSub);   // 64-token sub-tiles

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int BR = p.page_size < kSub ? p.page_size : kSub;    // rows per TMA box
    const int boxes = kSub / BR;                                // boxes per sub-tile

    for (int i = tid; i < n_mem; i += kPThreads)
        mem[i] = pp.members[sd[kSegMemberBegin] + m0 + i];
    for (int i = tid; i < nsub * boxes; i += kPThreads) {
        const int64_t tok = tok_begin + (int64_t)(i / boxes) * kSub + (i % boxes) * BR;
        if (tok >= tok_end) {
            box_rows[i] = -1;                    // past the request's last token: not loaded
            continue;
        }
        const int64_t idx = tok / p.page_size;
        int64_t page = idx < p.max_pages ? p.page_table[(int64_t)page_row * p.max_pages + idx] : -1;
        if (page < 0 || page >= p.num_pages) {
            record_error(p.err, RLT_DEVERR_BAD_PAGE);
            page = 0;                            // stay in bounds; the result is flagged
        }
        box_rows[i] = (int32_t)((page * p.num_kv_heads + g) * p.page_size + tok % p.page_size);
    }
    if (tid == 0) {
        for (int i = 0; i < 4 * kStagesP; ++i)
            mbar_init(&bars[i], 1);
        for (int i = 0; i < kSBufs; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], (R + 31) / 32);   // one arrive per softmax warp with live rows
        }
        for (int i = 0; i < kPBufs; ++i)
            mbar_init(&o_full[i], 1);
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

    if (warp < kSoftWarps) {
        // Query rows r = member * G + head, K-major, 128-byte swizzled (rows >= R unused),
        // staged while the producers already stream K and V.
        for (int i = tid; i < R * 16; i += kSoftWarps * 32) {
            const int r = i >> 4, c16 = i & 15;
            const int b = mem[r / G], h = r % G;
            const uint4 v = *reinterpret_cast<const uint4 *>(
                p.q + ((int64_t)b * p.num_q_heads + g * G + h) * 128 + c16 * 8);
            *reinterpret_cast<uint4 *>(qs + (c16 >> 3) * kHalfQ + tc::sw128_offset(r, (c16 & 7) * 8)) = v;
        }
        fence_proxy_async();
        named_barrier_sync(kQBarrier, (kSoftWarps + 1) * 32);
    }

    if (warp == kLoadKWarp || warp == kLoadVWarp) {
        // ------------------------------------------------- TMA producers (K, V)
        // Lane j copies box j/2, column block j&1 of this warp's tensor.
        const bool is_v = warp == kLoadVWarp;
        const CUtensorMap *map = is_v ? &vmap : &kmap;
        uint64_t *fullx = is_v ? full_v : full_k, *freex = is_v ? free_v : free_k;
        unsigned char *ring = stages + (is_v ? kStagesP * kKVBytes : 0);
        if (lane == 0)
            tc::prefetch_tmap(map);
        int j = 0;
        for (; j < nsub && ok; ++j) {
            const int st = j % kStagesP;
            if (j >= kStagesP)
                ok = mbar_wait_or_abort(&freex[st], ((j / kStagesP) - 1) & 1u, abort_flag);
            if (!ok)
                break;
            const int64_t sub_begin = tok_begin + (int64_t)j * kSub;
            const int nbox = (int)min((int64_t)boxes, (tok_end - sub_begin + BR - 1) / BR);
            if (lane == 0)
                mbar_arrive_expect_tx(&fullx[st], (uint32_t)(nbox * BR * 128 * 2));
            __syncwarp();
            if (lane < 2 * nbox) {
                const int box = lane >> 1, half = lane & 1;
                tc::tma_load_2d(ring + st * kKVBytes + half * kHalfKV + box * BR * 128, map, half * 64,
                                box_rows[j * boxes + box], &fullx[st]);
            }
        }
        if (!ok) {
            *abort_flag = 1;
            // copies of the last (up to 4) sub-tiles may still be landing: wait for them (bounded)
            if (lane == 0)
                for (int k = max(0, j - kStagesP); k < j; ++k)
                    mbar_wait(&fullx[k % kStagesP], (k / kStagesP) & 1u);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issuer
        const uint32_t id_s = tc::instr_desc_bf16(128, kSub, false);
        const uint32_t id_o = tc::instr_desc_bf16(128, 128, true);
        const uint32_t qa = smem_u32(qs), pa = smem_u32(pbuf), sa = smem_u32(stages);
        named_barrier_sync(kQBarrier, (kSoftWarps + 1) * 32);   // Q staged
        // Event loop: issue S_k as soon as K_k has landed and S buffer k%4 is free
        // (P.V of k-4 issued), and P.V_j as soon as every softmax warp wrote P_j
        // and V_j has landed.  Probes do not block, so neither waits on the other.
        int s_next = 0, pv_next = 0;
        uint64_t t_idle = 0;
        while (pv_next < nsub) {
            bool progress = false;
            if (s_next < nsub && s_next < pv_next + kSBufs &&
                __all_sync(kFullMask, mbar_test_wait(&full_k[s_next % kStagesP], (s_next / kStagesP) & 1u))) {
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t ka = sa + (s_next % kStagesP) * kKVBytes;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_bf16(tmem + kColS + (s_next % kSBufs) * kSub,
                                     tc::smem_desc(qa + (kk >> 2) * kHalfQ + (kk & 3) * 32, 16, 1024),
                                     tc::smem_desc(ka + (kk >> 2) * kHalfKV + (kk & 3) * 32, 16, 1024), id_s,
                                     kk > 0);
                    tc::mma_commit(&s_full[s_next % kSBufs]);
                    tc::mma_commit(&free_k[s_next % kStagesP]);
                }
                __syncwarp();
                ++s_next;
                progress = true;
            }
            const int j = pv_next;
            if (j < s_next &&
                __all_sync(kFullMask, mbar_test_wait(&p_full[j % kSBufs], (j / kSBufs) & 1u) &&
                                          mbar_test_wait(&full_v[j % kStagesP], (j / kStagesP) & 1u))) {
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t va = sa + (kStagesP + j % kStagesP) * kKVBytes;
                    const uint32_t pj = pa + (j % kPBufs) * kPBytes;
#pragma unroll
                    for (int kk = 0; kk < kSub / 16; ++kk)
                        tc::mma_bf16(tmem + kColO, tc::smem_desc(pj + kk * 32, 16, 1024),
                                     tc::smem_desc(va + kk * 2048, kHalfKV, 1024), id_o, (j > 0) || (kk > 0));
                    tc::mma_commit(&o_full[j % kPBufs]);
                    tc::mma_commit(&free_v[j % kStagesP]);
                }
                __syncwarp();
                ++pv_next;
                progress = true;
            }
            if (progress) {
                t_idle = 0;
            } else {
                __nanosleep(32);
                const uint64_t now = global_ns();
                if (t_idle == 0)
                    t_idle = now;
                else if (now - t_idle > kWaitLimitNs || *abort_flag != 0) {
                    ok = false;
                    break;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            // let issued MMAs finish before the CTA gives up its shared memory (bounded)
            if (lane == 0 && pv_next > 0)
                mbar_wait(&o_full[(pv_next - 1) % kPBufs], ((pv_next - 1) / kPBufs) & 1u);
        }
    } else if (warp * 32 < R) {
        // ------------------------------------------- softmax warps with live rows
        const int row = warp * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        float m_ref = -CUDART_INF_F, l_run = 0.f;

        for (int j = 0; j < nsub && ok; ++j) {
            ok = mbar_wait_or_abort(&s_full[j % kSBufs], (j / kSBufs) & 1u, abort_flag);
            if (!ok)
                break;
            tc::fence_after_sync();
            float v[64];
            tc::tmem_ld64(t_lane + kColS + (j % kSBufs) * kSub, v);
            const int valid = (int)min((int64_t)kSub, tok_end - (tok_begin + (int64_t)j * kSub));
            if (valid < kSub) {
                // ragged end of a private tail: mask the missing tokens, and zero their V
                // rows, whose memory may hold anything (0 * NaN would poison O)
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    v[i] = i < valid ? v[i] : -CUDART_INF_F;
                if (warp == 0) {
                    // after this sub-tile's V copy has landed (it may write garbage rows too)
                    ok = __all_sync(kFullMask, mbar_wait_or_abort(&full_v[j % kStagesP], (j / kStagesP) & 1u,
                                                                  abort_flag));
                    if (!ok)
                        break;
                    unsigned char *vst = stages + (kStagesP + j % kStagesP) * kKVBytes;
                    for (int c = lane; c < (kSub - valid) * 16; c += 32) {
                        const int r = valid + c / 16, c16 = c % 16;
                        *reinterpret_cast<uint4 *>(vst + (c16 >> 3) * kHalfKV + r * 128 + (c16 & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int i = 0; i < 64; ++i)
                mx = fmaxf(mx, v[i]);
            mx *= p.qscale;
            const bool up = mx > m_ref + kRescaleThreshold;
            const float m_next = up ? mx : m_ref;   // rows >= R hold garbage and are never stored
            const float scale_o = exp2f(m_ref - m_next);   // 1 if the reference stays, 0 at first
            if (__any_sync(kFullMask, up) && j > 0) {
                // rescale this row's O (PV of sub-tile j-1 must have landed)
                ok = mbar_wait_or_abort(&o_full[(j - 1) % kPBufs], ((j - 1) / kPBufs) & 1u, abort_flag);
                if (!__all_sync(kFullMask, ok)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float o[32];
                    tc::tmem_ld32(t_lane + kColO + c * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] *= scale_o;
                    tc::tmem_st32(t_lane + kColO + c * 32, o);
                }
            }
            l_run *= scale_o;
            m_ref = m_next;
            float lsum = 0.f;
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float p0 = fast_exp2(fmaf(v[2 * i], p.qscale, -m_ref));
                const float p1 = fast_exp2(fmaf(v[2 * i + 1], p.qscale, -m_ref));
                lsum += p0 + p1;
                w[i] = cvt_bf16x2(p0, p1);
            }
            l_run += lsum;
            if (j >= kPBufs) {   // P[j%3] was read by the P.V of sub-tile j-3
                ok = mbar_wait_or_abort(&o_full[j % kPBufs], ((j - kPBufs) / kPBufs) & 1u, abort_flag);
                if (!__all_sync(kFullMask, ok)) {
                    ok = false;
                    break;
                }
            }
            if (row < R) {
                unsigned char *pj = pbuf + (j % kPBufs) * kPBytes;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    *reinterpret_cast<uint4 *>(pj + tc::sw128_offset(row, c8 * 8)) =
                        make_uint4(w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
            }
            fence_proxy_async();                // P (generic writes) -> MMA (async proxy)
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[j % kSBufs]);
        }
        if (ok) {
            ok = mbar_wait_or_abort(&o_full[(nsub - 1) % kPBufs], ((nsub - 1) / kPBufs) & 1u, abort_flag);
            ok = __all_sync(kFullMask, ok);
        }
        if (!ok)
            *abort_flag = 1;
        if (__all_sync(kFullMask, ok && *abort_flag == 0)) {   // warp-uniform: TMEM loads below
            tc::fence_after_sync();
            const int b = row < R ? mem[row / G] : 0, h = row % G;
            const int64_t slot = ((int64_t)b * p.num_q_heads + g * G + h) * p.part_stride +
                                 sd[kSegSlotBase] + chunk;
            const float inv = 1.f / l_run;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tc::tmem_ld32(t_lane + kColO + c * 32, o);
                if (row < R) {
                    float4 *dst = reinterpret_cast<float4 *>(p.o_part + slot * 128 + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                             o[4 * i + 3] * inv);
                }
            }
            if (row < R)
                p.lse_part[slot] = m_ref + log2f(l_run);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 && *abort_flag != 0)
        record_error(p.err, RLT_DEVERR_TIMEOUT);
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

cudaError_t launch_prefix(const DecodeParams &p, const PrefixParams &pp, const void *k_bank,
                          const void *v_bank, int64_t bank_rows, cudaStream_t stream)
{
    if (pp.num_segments == 0 || pp.work_units == 0)
        return cudaSuccess;
    if (pp.chunk_tiles < 1 || pp.chunk_tiles > kMaxChunkTiles || bank_rows >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    const int box_rows = p.page_size < kSub ? p.page_size : kSub;
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
    const dim3 grid(pp.work_units, p.num_kv_heads, 1);
    decode_prefix_kernel<<<grid, kPThreads, kSmemP, stream>>>(kmap, vmap, p, pp);
    return cudaGetLastError();
}

}  // namespace rlt

// ------------------------------------------------------------- host planner

extern "C" RLT_API rlt_status rlt_plan_prefix(const int32_t *page_table, int32_t max_pages,
                                              const int32_t *seq_lens, int32_t batch,
                                              int32_t page_size, int32_t chunk_tiles,
                                              int32_t query_group, int32_t private_tails,
                                              int32_t *segments,
                                              int32_t max_segments, int32_t *members,
                                              int32_t max_member_entries, int32_t *request_prefix,
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

    struct Seg { int first, tiles, parent; std::vector<int> mem; int64_t end_token; };
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
                    segs.push_back({t, 1, grp.seg, kv.second, 0});
                }
                for (int b : kv.second)
                    deepest[b] = s;
                next.push_back({kv.second, s});
            }
        }
        level.swap(next);
    }

    for (Seg &sg : segs)
        sg.end_token = (int64_t)(sg.first + sg.tiles) * kPrefixTile;
    std::vector<int64_t> covered(batch, 0);
    for (int b = 0; b < batch; ++b)
        if (deepest[b] >= 0)
            covered[b] = segs[deepest[b]].end_token;
    if (private_tails) {
        // every request's own remaining tokens become a one-member segment
        for (int b = 0; b < batch; ++b) {
            const int64_t L = std::min<int64_t>(std::max(seq_lens[b], 0), (int64_t)max_pages * page_size);
            if (L <= covered[b])
                continue;
            const int first = (int)(covered[b] / kPrefixTile);
            const int tiles = (int)((L + kPrefixTile - 1) / kPrefixTile) - first;
            segs.push_back({first, tiles, deepest[b], {b}, L});
            deepest[b] = (int)segs.size() - 1;
            covered[b] = L;
        }
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
    // work units: (segment, chunk, member block); a member block holds 128 / query_group members
    const int per_block = 128 / query_group;
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
        request_prefix[2 * b + 1] = s < 0 ? 0 : slot_base[s] + chunks[s];
        max_slots = std::max(max_slots, request_prefix[2 * b + 1]);
        const int64_t L = std::min<int64_t>(std::max(seq_lens[b], 0), (int64_t)max_pages * page_size);
        max_rest = std::max(max_rest, L - covered[b]);
    }
    sizes[3] = max_slots;
    sizes[5] = (int32_t)max_rest;
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
        row[rlt::kSegEndToken] = (int32_t)segs[s].end_token;
        row[rlt::kSegWorkBegin] = (int32_t)work_begin[s];
        for (int b : segs[s].mem)
            members[m++] = b;
    }
    return RLT_OK;
}
