// Merging of (o, log2-sum-exp) partials by the combine kernels.
//
// Attention of one query row over disjoint key sets K_1..K_n, given each set's
// softmax-weighted mean o_i and log2-sum-exp l_i, is
//     o = sum_i 2^(l_i - M) o_i / sum_i 2^(l_i - M),   lse = M + log2 sum_i 2^(l_i - M),
// M = max_i l_i: the identity that makes split-K decode ("Faster fuzzy minds", "When
// scheduler does the work": attention over the pages a request maps) exact up to
// rounding.
#pragma once

#include <math_constants.h>

#include "rlt_device.cuh"
#include "rlt_internal.h"

namespace rlt {

constexpr float kLn2 = 0.6931471805599453f;

// Tokens [tok0, L) of request b that the split-K kernels cover, and n_pre, the
// partials the shared-prefix kernel wrote for it.  seq_lens[b] is clamped to
// the page-table row and the split grid (a clamp is recorded as an error).
struct Span {
    int tok0, L, n_pre;
};

__device__ __forceinline__ Span request_span(const DecodeParams &p, int b, bool report)
{
    int len = p.seq_lens[b];
    bool bad = false;
    const int64_t cap_pages = (int64_t)p.max_pages * p.page_size;
    if (len < 0 || len > cap_pages) {
        len = len < 0 ? 0 : (int)cap_pages;
        bad = true;
    }
    Span sp{0, len, 0};
    if (p.request_prefix != nullptr) {
        sp.tok0 = min(max(p.request_prefix[2 * b], 0), len);
        sp.n_pre = p.request_prefix[2 * b + 1];
    }
    const int64_t cap_grid = (int64_t)p.max_splits * p.tiles_per_split * kTileTokens;
    if (sp.L - sp.tok0 > cap_grid) {
        sp.L = (int)(sp.tok0 + cap_grid);
        bad = true;
    }
    if (bad && report)
        record_error(p.err, RLT_DEVERR_BAD_LEN);
    return sp;
}

// Split-K partials of a request: one per split of its tokens [tok0, L).
__device__ __forceinline__ int split_count(const DecodeParams &p, const Span &sp)
{
    const int n_tiles = (sp.L - sp.tok0 + kTileTokens - 1) / kTileTokens;
    return (n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
}

// The prefix partials of a request, clamped to the slots the workspace holds (a plan
// inconsistent with it is recorded as an error).
__device__ __forceinline__ int prefix_partials(const DecodeParams &p, const Span &sp, bool report)
{
    int n_pre = sp.n_pre;
    if (n_pre < 0 || n_pre > p.prefix_slots) {
        if (report)
            record_error(p.err, RLT_DEVERR_BAD_SLOT);
        n_pre = n_pre < 0 ? 0 : p.prefix_slots;
    }
    return n_pre;
}

// Row bh (request x query head) merged by one warp from its n_pre prefix partials and n
// split-K partials (n_pre + n <= 32): lane s holds slot s's log2-sum-exp.  Up to kLoads
// slots every partial is read together with the log-sum-exps (one dependent round trip);
// past that the live slots' partials are read in slot order, kLoads loads in flight per
// lane.  Writes out[bh] (bf16) and lse_out[bh] (natural log); a row with no slot gets
// out = 0, lse = -inf.
template <int D, int kLoads>
__device__ __forceinline__ void merge_row_warp(const DecodeParams &p, int64_t bh, int n_pre, int n, int lane)
{
    constexpr int DPL = D / 32;
    uint16_t *o = p.out + bh * D + lane * DPL;
    if (n_pre + n == 0) {                        // empty request: out = 0, lse = -inf
        if constexpr (DPL == 4)
            *reinterpret_cast<uint2 *>(o) = make_uint2(0u, 0u);
        else
            *reinterpret_cast<uint32_t *>(o) = 0u;
        if (lane == 0 && p.lse_out != nullptr)
            p.lse_out[bh] = -CUDART_INF_F;
        return;
    }
    const int total = n_pre + n;                 // <= prefix_slots + max_splits <= 32
    const int64_t row = bh * p.part_stride;
    const int my_slot = lane < n_pre ? lane : p.prefix_slots + (lane - n_pre);
    auto slot_part = [&](int s) -> const float * {
        return p.o_part + (row + (s < n_pre ? s : p.prefix_slots + (s - n_pre))) * D + lane * DPL;
    };
    float acc[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        acc[d] = 0.f;
    if (total <= kLoads) {
        // every slot's partial is read together with the log-sum-exps (one round trip); a slot
        // without a partial may hold anything, so it is skipped, never scaled by zero
        float v[kLoads][DPL];
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            if (i < total) {
                if constexpr (DPL == 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4 *>(slot_part(i)));
                    v[i][0] = x.x; v[i][1] = x.y; v[i][2] = x.z; v[i][3] = x.w;
                } else {
                    const float2 x = __ldcg(reinterpret_cast<const float2 *>(slot_part(i)));
                    v[i][0] = x.x; v[i][1] = x.y;
                }
            }
        }
        const float l = lane < total ? __ldcg(p.lse_part + row + my_slot) : -CUDART_INF_F;
        const float M = warp_max_xor(l, 1);
        const float w = l != -CUDART_INF_F ? exp2f(l - M) : 0.f;
        const float ls = warp_sum_xor(w, 1);
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            const float wi = __shfl_sync(kFullMask, w, i);
            if (i < total && wi > 0.f) {
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    acc[d] = fmaf(wi, v[i][d], acc[d]);
            }
        }
        const float inv = ls > 0.f ? 1.f / ls : 0.f;
        if constexpr (DPL == 4) {
            uint2 x;
            x.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            x.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2 *>(o) = x;
        } else {
            *reinterpret_cast<uint32_t *>(o) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        }
        if (lane == 0 && p.lse_out != nullptr)
            p.lse_out[bh] = ls > 0.f ? (M + log2f(ls)) * kLn2 : -CUDART_INF_F;
        return;
    }
    const float l = lane < total ? __ldcg(p.lse_part + row + my_slot) : -CUDART_INF_F;
    const float M = warp_max_xor(l, 1);
    const float w = l != -CUDART_INF_F ? exp2f(l - M) : 0.f;
    const float ls = warp_sum_xor(w, 1);
    unsigned live = __ballot_sync(kFullMask, l != -CUDART_INF_F);
    while (live != 0u) {
        int sl[kLoads];
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            sl[i] = live != 0u ? __ffs(live) - 1 : -1;
            live &= live - 1u;
        }
        float v[kLoads][DPL];
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            const int s = sl[i] >= 0 ? sl[i] : 0;
            const int slot = s < n_pre ? s : p.prefix_slots + (s - n_pre);
            const float *op = p.o_part + (row + slot) * D + lane * DPL;
            if constexpr (DPL == 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (sl[i] >= 0)
                    x = __ldcg(reinterpret_cast<const float4 *>(op));
                v[i][0] = x.x; v[i][1] = x.y; v[i][2] = x.z; v[i][3] = x.w;
            } else {
                float2 x = make_float2(0.f, 0.f);
                if (sl[i] >= 0)
                    x = __ldcg(reinterpret_cast<const float2 *>(op));
                v[i][0] = x.x; v[i][1] = x.y;
            }
        }
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            const float wi = __shfl_sync(kFullMask, w, sl[i] >= 0 ? sl[i] : 0);
            if (sl[i] >= 0) {
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    acc[d] = fmaf(wi, v[i][d], acc[d]);
            }
        }
    }
    const float inv = ls > 0.f ? 1.f / ls : 0.f;
    if constexpr (DPL == 4) {
        uint2 x;
        x.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        x.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(o) = x;
    } else {
        *reinterpret_cast<uint32_t *>(o) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0 && p.lse_out != nullptr)
        p.lse_out[bh] = ls > 0.f ? (M + log2f(ls)) * kLn2 : -CUDART_INF_F;
}

}  // namespace rlt
