// Paged GQA decode attention for sm_103a: split-K partial kernel + LSE combine.
//
// What it computes ("Faster fuzzy minds", "When scheduler does the work" and
// "Recurrent depth"): for every request b and query head h, softmax(q K^T *
// scale) V over the seq_lens[b] cached tokens of b, gathered page by page
// through the page table from one (layer, plane) bank of the pool.
//
// Design (HBM-bound: every K/V byte is read once and used by the G query heads
// of its kv head):
//  * One CTA per (split, kv head, request); a split is a run of 16-token tiles.
//  * Pool layout [page][kv_head][offset][D] makes the 16 rows of a tile one
//    contiguous chunk, so each tile is two `cp.async.bulk` copies (K and V) of
//    16*D*2 bytes straight into shared memory, completing on an mbarrier.
//  * The 4 warps of a CTA take tiles round-robin; each warp runs its own
//    2-stage copy ring and its own online softmax, so no CTA-wide barrier is
//    crossed until the final merge.
//  * Inside a tile a half-warp holds 8 token rows, each lane D/16 dims:
//    16-byte (D=128) shared loads without bank conflicts, scores reduced by a
//    transpose butterfly (8 shuffles for 8 tokens), probabilities broadcast
//    through shared memory for the P.V accumulation.  The dot products and the
//    accumulation run on packed fp32 pairs (f32x2 FMA), half the instructions.
//  * Splits write (o, log2-sum-exp) partials; the combine kernel merges them.
//    Requests with one split write their output directly.
#include <math_constants.h>

#include <atomic>

#include "rlt_device.cuh"
#include "rlt_internal.h"
#include "rlt_merge.cuh"

namespace rlt {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;                   // copy ring depth per warp

template <int D, int G>
struct Cfg {
    static constexpr int kDpl = D / 16;                          // dims per lane
    static constexpr int kTileBytes = kTileTokens * D * 2;       // K (or V) rows of a tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kPipeBytes = kWarps * kStages * kStageBytes;
    static constexpr int kMergeStride = D + 4;                   // floats per (warp, head)
    static constexpr int kMergeBytes = kWarps * G * kMergeStride * 4;
    static constexpr int kRegionBytes = kPipeBytes > kMergeBytes ? kPipeBytes : kMergeBytes;
    static constexpr int kPBytes = kWarps * G * kTileTokens * 4;
    static constexpr int kBarOffset = kRegionBytes + kPBytes;
    static constexpr int kSmemBytes = kBarOffset + kWarps * kStages * 8;
};

template <int DPL>
__device__ __forceinline__ void load_frag(const unsigned char *src, float (&f)[DPL])
{
    if constexpr (DPL == 8) {
        const uint4 w = *reinterpret_cast<const uint4 *>(src);
        f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
        f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
    } else {
        static_assert(DPL == 4, "head_dim 64 or 128");
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    }
}

template <int DPL>
__device__ __forceinline__ void load_frag_global(const uint16_t *src, float (&f)[DPL])
{
    load_frag<DPL>(reinterpret_cast<const unsigned char *>(src), f);
}

// Pairs of fp32 in one 64-bit register: Blackwell's packed f32x2 FMA / MUL do two
// lanes' worth of work per instruction (each half rounded as its own fmaf / fmul).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 f2_unpack(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return make_float2(lo, hi);
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// A tile row's DPL bf16 dims of this lane as DPL/2 fp32 pairs (bf16 -> fp32 is exact).
template <int DPL>
__device__ __forceinline__ void load_frag2(const unsigned char *src, uint64_t (&f)[DPL / 2])
{
    if constexpr (DPL == 8) {
        const uint4 w = *reinterpret_cast<const uint4 *>(src);
        f[0] = f2_pack(bf16_lo(w.x), bf16_hi(w.x));
        f[1] = f2_pack(bf16_lo(w.y), bf16_hi(w.y));
        f[2] = f2_pack(bf16_lo(w.z), bf16_hi(w.z));
        f[3] = f2_pack(bf16_lo(w.w), bf16_hi(w.w));
    } else {
        static_assert(DPL == 4, "head_dim 64 or 128");
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        f[0] = f2_pack(bf16_lo(w.x), bf16_hi(w.x));
        f[1] = f2_pack(bf16_lo(w.y), bf16_hi(w.y));
    }
}

// Merge the partials of one (request, query head): its shared-prefix slots
// [0, n_pre) and split-K slots [prefix_slots, prefix_slots + n); a slot whose
// lse is -inf holds no partial (a tensor-core run marks the chunk slots it merged
// that way).  Four warps per pair.  The slots are taken in windows of
// kCombineWindow: every thread reads its slots' lse values at once, the live ones
// are listed in shared memory, and then only those partials are read, each warp
// with all of its loads in flight; the warps' (sum, vector) fold at the end.
// Partials are read through L2 (they may come from other CTAs of a running grid).
constexpr int kCombineWarps = 4;
constexpr int kCombineThreads = kCombineWarps * 32;
constexpr int kCombineWindow = 1024;
constexpr int kCombinePer = kCombineWindow / kCombineThreads;   // lse values per thread per window

template <int D>
struct MergeSmem {
    float red_m[kCombineWarps], red_l[kCombineWarps];
    alignas(16) float red_o[kCombineWarps][D];
    int live_slot[kCombineWindow];
    float live_w[kCombineWindow];
    int live_off[kCombinePer * kCombineWarps + 1];
};

// Merge row bh (total = n_pre + n >= 1 slots) and write out[bh] and lse_out[bh].  Called by
// all kCombineThreads threads of the CTA; sm may alias other shared memory of the caller.
template <int D>
__device__ void merge_row(const DecodeParams &p, int64_t bh, int n_pre, int n, MergeSmem<D> &sm)
{
    constexpr int DPL = D / 32;
    constexpr int kPer = kCombinePer;
    float *red_m = sm.red_m, *red_l = sm.red_l;
    auto &red_o = sm.red_o;
    int *live_slot = sm.live_slot, *live_off = sm.live_off;
    float *live_w = sm.live_w;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = n_pre + n;
    __syncthreads();                             // the shared buffers of an earlier merge are free
    auto slot_of = [&](int s) -> int64_t {
        return bh * p.part_stride + (s < n_pre ? s : p.prefix_slots + (s - n_pre));
    };

    // the largest lse over all slots (independent loads); the first window's values stay
    // in registers for the live-slot list below
    float l0[kPer];
    float M = -CUDART_INF_F;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int s = i * kCombineThreads + threadIdx.x;
        l0[i] = s < total ? __ldcg(p.lse_part + slot_of(s)) : -CUDART_INF_F;
        M = fmaxf(M, l0[i]);
    }
    for (int s = kCombineWindow + threadIdx.x; s < total; s += kCombineThreads)
        M = fmaxf(M, __ldcg(p.lse_part + slot_of(s)));
    M = warp_max_xor(M, 1);
    if (lane == 0)
        red_m[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w)
        M = fmaxf(M, red_m[w]);

    float acc[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        acc[d] = 0.f;
    float ls = 0.f;
    for (int w0 = 0; M != -CUDART_INF_F && w0 < total; w0 += kCombineWindow) {
        // list this window's live slots in slot order with their weights: a ballot per
        // (value index, warp), one scan of the 32 counts, then each live lane's place
        float l[kPer];
        unsigned bal[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int s = w0 + i * kCombineThreads + threadIdx.x;
            l[i] = w0 == 0 ? l0[i] : s < total ? __ldcg(p.lse_part + slot_of(s)) : -CUDART_INF_F;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            bal[i] = __ballot_sync(kFullMask, l[i] != -CUDART_INF_F);
            if (lane == 0)
                live_off[i * kCombineWarps + warp] = __popc(bal[i]);
        }
        __syncthreads();
        if (warp == 0) {
            static_assert(kPer * kCombineWarps == 32, "one count per lane");
            const int c = live_off[lane];
            int x = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFullMask, x, o);
                if (lane >= o)
                    x += y;
            }
            __syncwarp();
            live_off[lane] = x - c;               // exclusive prefix
            if (lane == 31)
                live_off[32] = x;                 // live slots in the window
        }
        __syncthreads();
        const unsigned below = (1u << lane) - 1u;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (l[i] != -CUDART_INF_F) {
                const int k = live_off[i * kCombineWarps + warp] + __popc(bal[i] & below);
                live_slot[k] = w0 + i * kCombineThreads + threadIdx.x;
                live_w[k] = exp2f(l[i] - M);
            }
        }
        __syncthreads();
        // warps take the live partials in turn, sixteen loads in flight
        const int nl = live_off[32];
        for (int k0 = warp * 16; k0 < nl; k0 += kCombineWarps * 16) {
            float o[16][DPL];
            float wk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k = k0 + i;
                wk[i] = k < nl ? live_w[k] : 0.f;
                const float *op = p.o_part + slot_of(k < nl ? live_slot[k] : 0) * D + lane * DPL;
                if constexpr (DPL == 4) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (k < nl)
                        v = __ldcg(reinterpret_cast<const float4 *>(op));
                    o[i][0] = v.x; o[i][1] = v.y; o[i][2] = v.z; o[i][3] = v.w;
                } else {
                    float2 v = make_float2(0.f, 0.f);
                    if (k < nl)
                        v = __ldcg(reinterpret_cast<const float2 *>(op));
                    o[i][0] = v.x; o[i][1] = v.y;
                }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                ls += wk[i];
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    acc[d] = fmaf(wk[i], o[i][d], acc[d]);
            }
        }
        __syncthreads();                         // the list is rebuilt for the next window
    }
    if (lane == 0)
        red_l[warp] = ls;
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        red_o[warp][lane * DPL + d] = acc[d];
    __syncthreads();
    if (warp != 0)
        return;
    ls = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w)
        ls += red_l[w];
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < kCombineWarps; ++w)
            a += red_o[w][lane * DPL + d];
        acc[d] = a;
    }
    const float inv = ls > 0.f ? 1.f / ls : 0.f;
    uint16_t *o = p.out + bh * D + lane * DPL;
    if constexpr (DPL == 4) {
        uint2 w;
        w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(o) = w;
    } else {
        *reinterpret_cast<uint32_t *>(o) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0 && p.lse_out != nullptr)
        p.lse_out[bh] = ls > 0.f ? (M + log2f(ls)) * kLn2 : -CUDART_INF_F;
}


// acc[h] += p[h][t] * V_t for the 8 rows t of this lane's half of a tile.  In
// the last tile of a request, rows past its end are skipped: that pool memory
// may hold anything, even NaN patterns, and 0 * NaN would poison the sum.
template <int D, int G, bool kMasked>
__device__ __forceinline__ void pv_tile(const unsigned char *vs, const float *pbuf, int half,
                                        int j, int valid, uint64_t (&acc)[G][D / 32])
{
    constexpr int DPL = D / 16;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        if (kMasked && half * 8 + r >= valid)
            continue;
        uint64_t vf[DPL / 2];
        load_frag2<DPL>(vs + ((half * 8 + r) * D + j * DPL) * 2, vf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float pw = pbuf[h * kTileTokens + half * 8 + r];
            const uint64_t pw2 = f2_pack(pw, pw);
#pragma unroll
            for (int d = 0; d < DPL / 2; ++d)
                acc[h][d] = f2_fma(pw2, vf[d], acc[h][d]);
        }
    }
}

template <int D, int G, bool kFault>
__device__ __forceinline__ void decode_partial_body(const DecodeParams &p);

// The split-K kernel.  In shared-prefix mode it covers each request's tokens
// past its shared segments and runs beside the tensor-core kernel, on a second
// stream; the combine waits for both.  kFault: the instance that the timeout
// test's fault switch launches (one copy left unissued, the wait limit from the
// call); every other call runs the instance without either, whose registers
// the switch does not disturb.
template <int D, int G, bool kFault>
__global__ void __launch_bounds__(kThreads) decode_partial_kernel(const DecodeParams p)
{
    decode_partial_body<D, G, kFault>(p);
}

template <int D, int G, bool kFault>
__device__ __forceinline__ void decode_partial_body(const DecodeParams &p)
{
    using C = Cfg<D, G>;
    constexpr int DPL = C::kDpl;
    extern __shared__ __align__(128) unsigned char smem[];

    // The kernel behind this one (the combine, or the next call) may be scheduled now.
    pdl_launch_dependents();
    const int split = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;                // which 8 rows of a tile
    const int j = lane & 15;                   // which D/16 dims

    // In shared-prefix mode the first tok0 tokens were covered by the prefix kernel,
    // which wrote n_pre partials; this kernel covers [tok0, L).
    const Span sp = request_span(p, b, split == 0 && g == 0 && threadIdx.x == 0);
    const int L = sp.L, tok0 = sp.tok0, n_pre = sp.n_pre;
    const int n_tiles = (L - tok0 + kTileTokens - 1) / kTileTokens;
    const int n_splits = (n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    // A fused append needs the new token past the shared prefix: inside it, its slot
    // would be a shared (read-only) page's.  Flagged, not written.
    if (p.k_new != nullptr && L > 0 && L - 1 < tok0 && split == 0 && g == 0 && threadIdx.x == 0)
        record_error(p.err, RLT_DEVERR_BAD_SLOT);

    // Until pdl_wait this CTA reads only what no kernel still running may write: the
    // lengths, page table, prefix plan and cached K/V rows of the bank.  q, k_new and
    // v_new are read, and out, the partials and the pool written, only after it.
    if (n_splits == 0 && n_pre == 0) {          // empty request: out = 0, lse = -inf
        if (split == 0) {
            pdl_wait();
            for (int i = threadIdx.x; i < G * D / 2; i += kThreads) {
                const int h = i / (D / 2), d2 = i % (D / 2);
                reinterpret_cast<uint32_t *>(
                    p.out + ((int64_t)b * p.num_q_heads + g * G + h) * D)[d2] = 0u;
            }
            if (p.lse_out != nullptr && threadIdx.x < G)
                p.lse_out[(int64_t)b * p.num_q_heads + g * G + threadIdx.x] = -CUDART_INF_F;
        }
        return;
    }
    if (split >= n_splits) {
        if (split == 0)
            pdl_wait();                         // every grid waits in at least one CTA
        return;
    }

    const int tile_begin = split * p.tiles_per_split;
    const int tile_end = min(tile_begin + p.tiles_per_split, n_tiles);
    const int my_first = tile_begin + warp;      // tile index counted from tok0
    const int my_count = my_first < tile_end ? (tile_end - my_first + kWarps - 1) / kWarps : 0;

    unsigned char *pipe = smem + warp * kStages * C::kStageBytes;
    float *pbuf = reinterpret_cast<float *>(smem + C::kRegionBytes) + warp * G * kTileTokens;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOffset) + warp * kStages;

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s)
            mbar_init(&bars[s], 1);
        mbar_init_fence();
    }
    __syncwarp();

    // Page and in-page offset of this warp's i-th tile live in lane i.
    int my_page = -1, my_off = 0;
    if (lane < my_count) {
        const int tok = tok0 + (my_first + lane * kWarps) * kTileTokens;
        const int page = p.page_table[(int64_t)b * p.max_pages + tok / p.page_size];
        if (page >= 0 && (int64_t)page < p.num_pages)
            my_page = page;
        else
            record_error(p.err, RLT_DEVERR_BAD_PAGE);
        my_off = tok % p.page_size;
    }

    // Fused append: the new token (position L - 1) falls in tile t_new of [tok0, L); the
    // warp whose i_new-th tile that is loads row r_new of it from k_new / v_new instead of
    // the pool (the tile's other rows come from the pool as usual, in one or two pieces)
    // and, once the tile has landed, stores that row to the pool slot.
    int i_new = -1, r_new = 0;
    if (p.k_new != nullptr && L > tok0 && L == p.seq_lens[b]) {      // not on a clamped length
        const int t_new = (L - 1 - tok0) / kTileTokens;
        if (t_new >= my_first && t_new < tile_end && (t_new - my_first) % kWarps == 0) {
            i_new = (t_new - my_first) / kWarps;
            r_new = (L - 1 - tok0) % kTileTokens;
        }
    }

    auto issue = [&](int i) {
        const int page = __shfl_sync(kFullMask, my_page, i);
        const int off = __shfl_sync(kFullMask, my_off, i);
        if (lane == 0 && page >= 0) {
            uint64_t *bar = &bars[i % kStages];
            unsigned char *dst = pipe + (i % kStages) * C::kStageBytes;
            const int64_t row = ((int64_t)page * p.num_kv_heads + g) * p.page_size + off;
            mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
            if (kFault && i == 0 && warp == 0 && split == 0 && g == 0 && b == 0) {
                // fault injection (timeout test only): this stage's bytes never arrive
            } else if (i != i_new) {
                bulk_load_once(dst, p.k_bank + row * D, C::kTileBytes, bar);
                bulk_load_once(dst + C::kTileBytes, p.v_bank + row * D, C::kTileBytes, bar);
            } else {
                constexpr uint32_t kRow = D * 2;
                const int64_t nrow = ((int64_t)b * p.num_kv_heads + g) * D;
                for (int kv = 0; kv < 2; ++kv) {
                    const uint16_t *bank = kv == 0 ? p.k_bank : p.v_bank;
                    unsigned char *d = dst + kv * C::kTileBytes;
                    if (r_new > 0)
                        bulk_load(d, bank + row * D, r_new * kRow, bar);
                    bulk_load(d + r_new * kRow, (kv == 0 ? p.k_new : p.v_new) + nrow, kRow, bar);
                    if (r_new < kTileTokens - 1)
                        bulk_load(d + (r_new + 1) * kRow, bank + (row + r_new + 1) * D,
                                  (kTileTokens - 1 - r_new) * kRow, bar);
                }
            }
        }
    };

    // The first ring stages go out before the wait for the kernels ahead (their K/V rows
    // are already in the pool); the tile that takes the fused append's new row from
    // k_new / v_new goes out after it.
    const int n_prologue = my_count < kStages ? my_count : kStages;
    const int n_early = (i_new >= 0 && i_new < n_prologue) ? i_new : n_prologue;
    int issued = 0;
    for (; issued < n_early; ++issued)
        issue(issued);
    pdl_wait();
    for (; issued < n_prologue; ++issued)
        issue(issued);

    // Query heads g*G .. g*G+G-1, this lane's dims, pre-scaled into log2 units, as fp32
    // pairs; the accumulators are fp32 pairs too.
    uint64_t q[G][DPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float qf[DPL];
        load_frag_global<DPL>(p.q + ((int64_t)b * p.num_q_heads + g * G + h) * D + j * DPL, qf);
#pragma unroll
        for (int d = 0; d < DPL / 2; ++d)
            q[h][d] = f2_pack(qf[2 * d] * p.qscale, qf[2 * d + 1] * p.qscale);
    }

    float m[G], l[G];
    uint64_t acc2[G][DPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -CUDART_INF_F;
        l[h] = 0.f;
#pragma unroll
        for (int d = 0; d < DPL / 2; ++d)
            acc2[h][d] = f2_pack(0.f, 0.f);
    }

    uint32_t phase = 0;                        // bit s: parity of stage s's next phase
    const uint64_t wait_ns = kFault ? p.wait_limit_ns : kWaitLimitNs;
    int failed_at = -1;

    for (int i = 0; i < my_count; ++i) {
        const int s = i % kStages;
        const int page = __shfl_sync(kFullMask, my_page, i);
        if (page >= 0) {
            const bool arrived = __all_sync(kFullMask, mbar_wait(&bars[s], (phase >> s) & 1u, wait_ns));
            if (!arrived) {
                failed_at = i;
                break;
            }
            phase ^= 1u << s;

            const int valid = min(kTileTokens, L - tok0 - (my_first + i * kWarps) * kTileTokens);
            const unsigned char *ks = pipe + s * C::kStageBytes;
            const unsigned char *vs = ks + C::kTileBytes;
            if (i == i_new) {                   // warp-uniform: the new row to its pool slot
                const int off = __shfl_sync(kFullMask, my_off, i);
                const int vec = lane & 15;
                if (vec < D / 8) {
                    const uint4 v = reinterpret_cast<const uint4 *>((lane < 16 ? ks : vs) + r_new * D * 2)[vec];
                    const int64_t slot_row = ((int64_t)page * p.num_kv_heads + g) * p.page_size + off + r_new;
                    uint16_t *dst = const_cast<uint16_t *>(lane < 16 ? p.k_bank : p.v_bank) + slot_row * D;
                    reinterpret_cast<uint4 *>(dst)[vec] = v;
                }
            }

            // Partial dot products of this lane's dims for its half's 8 rows.
            // At head_dim 128 with one or two query heads per kv head the 8 rows' K fragments are read
            // first, so that their shared-memory loads overlap (measured on the G = 1 ouro
            // workload: 177.9 -> 175.6 us per call); larger groups have the registers busy.
            float sc[G][8];
            constexpr int kAhead = (D == 128 && G <= 2) ? 8 : 1;
            uint64_t k_ahead[kAhead][DPL / 2];
            if constexpr (kAhead == 8) {
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    load_frag2<DPL>(ks + ((half * 8 + r) * D + j * DPL) * 2, k_ahead[r]);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                uint64_t kf[DPL / 2];
                if constexpr (kAhead == 8) {
#pragma unroll
                    for (int d = 0; d < DPL / 2; ++d)
                        kf[d] = k_ahead[r][d];
                } else {
                    load_frag2<DPL>(ks + ((half * 8 + r) * D + j * DPL) * 2, kf);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    uint64_t a = f2_mul(q[h][0], kf[0]);
#pragma unroll
                    for (int d = 1; d < DPL / 2; ++d)
                        a = f2_fma(q[h][d], kf[d], a);
                    const float2 a2 = f2_unpack(a);
                    sc[h][r] = a2.x + a2.y;
                }
            }
            // Transpose butterfly over the 16 lanes of the half: afterwards lane j
            // holds the full score of row j>>1 (lanes j and j^1 agree).
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const bool up = j & 8;
                    const float send = up ? sc[h][k] : sc[h][k + 4];
                    const float keep = up ? sc[h][k + 4] : sc[h][k];
                    sc[h][k] = keep + __shfl_xor_sync(kFullMask, send, 8);
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const bool up = j & 4;
                    const float send = up ? sc[h][k] : sc[h][k + 2];
                    const float keep = up ? sc[h][k + 2] : sc[h][k];
                    sc[h][k] = keep + __shfl_xor_sync(kFullMask, send, 4);
                }
                {
                    const bool up = j & 2;
                    const float send = up ? sc[h][0] : sc[h][1];
                    const float keep = up ? sc[h][1] : sc[h][0];
                    sc[h][0] = keep + __shfl_xor_sync(kFullMask, send, 2);
                }
                sc[h][0] += __shfl_xor_sync(kFullMask, sc[h][0], 1);
            }

            // Online softmax update (log2 domain), one running max per head.
            const int t = half * 8 + (j >> 1);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float s_t = t < valid ? sc[h][0] : -CUDART_INF_F;
                const float m_new = fmaxf(m[h], warp_max_xor(s_t, 2));
                const float alpha = exp2f(m[h] - m_new);
                const float pr = exp2f(s_t - m_new);
                l[h] = l[h] * alpha + ((j & 1) ? 0.f : pr);
                const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll
                for (int d = 0; d < DPL / 2; ++d)
                    acc2[h][d] = f2_mul(acc2[h][d], alpha2);
                m[h] = m_new;
                if ((j & 1) == 0)
                    pbuf[h * kTileTokens + t] = pr;
            }
            __syncwarp();

            // acc += p_t * V_t over this half's rows.
            if (valid == kTileTokens)
                pv_tile<D, G, false>(vs, pbuf, half, j, valid, acc2);
            else
                pv_tile<D, G, true>(vs, pbuf, half, j, valid, acc2);
        }
        __syncwarp();
        fence_proxy_async();                   // our reads of stage s before its next refill
        if (issued < my_count && issued == i + kStages) {
            issue(issued);
            ++issued;
        }
    }

    if (failed_at >= 0) {
        // A copy never arrived: record it, then wait (bounded) for this warp's
        // copies still in flight before the shared memory is given up.
        if (lane == 0)
            record_error(p.err, RLT_DEVERR_TIMEOUT);
        for (int k = failed_at; k < issued; ++k) {
            const int s = k % kStages;
            if (__shfl_sync(kFullMask, my_page, k) >= 0) {
                mbar_wait(&bars[s], (phase >> s) & 1u, wait_ns);
                phase ^= 1u << s;
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -CUDART_INF_F;
            l[h] = 0.f;
        }
    }

    float acc[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int d = 0; d < DPL / 2; ++d) {
            const float2 v = f2_unpack(acc2[h][d]);
            acc[h][2 * d] = v.x;
            acc[h][2 * d + 1] = v.y;
        }
    // Fold the two halves (same dims, different rows) and the per-lane sums.
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int d = 0; d < DPL; ++d)
            acc[h][d] += __shfl_xor_sync(kFullMask, acc[h][d], 16);
        l[h] = warp_sum_xor(l[h], 1);
    }

    // Merge the 4 warps through shared memory (aliases the copy rings).
    __syncthreads();
    float *mg = reinterpret_cast<float *>(smem);
    if (half == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int d = 0; d < DPL; ++d)
                mg[(warp * G + h) * C::kMergeStride + j * DPL + d] = acc[h][d];
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mg[(warp * G + h) * C::kMergeStride + D] = m[h];
            mg[(warp * G + h) * C::kMergeStride + D + 1] = l[h];
        }
    }
    __syncthreads();

    for (int item = threadIdx.x; item < G * D / 4; item += kThreads) {
        const int h = item / (D / 4);
        const int d0 = (item % (D / 4)) * 4;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            M = fmaxf(M, mg[(w * G + h) * C::kMergeStride + D]);
        float ls = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float *row = mg + (w * G + h) * C::kMergeStride;
                const float sc = exp2f(row[D] - M);
                ls = fmaf(row[D + 1], sc, ls);
                o0 = fmaf(row[d0 + 0], sc, o0);
                o1 = fmaf(row[d0 + 1], sc, o1);
                o2 = fmaf(row[d0 + 2], sc, o2);
                o3 = fmaf(row[d0 + 3], sc, o3);
            }
        }
        const float inv = ls > 0.f ? 1.f / ls : 0.f;
        const float lse2 = ls > 0.f ? M + log2f(ls) : -CUDART_INF_F;
        const int64_t bh = (int64_t)b * p.num_q_heads + g * G + h;
        if (n_splits == 1 && n_pre == 0) {
            uint2 w;
            w.x = pack_bf16x2(o0 * inv, o1 * inv);
            w.y = pack_bf16x2(o2 * inv, o3 * inv);
            *reinterpret_cast<uint2 *>(p.out + bh * D + d0) = w;
            if (d0 == 0 && p.lse_out != nullptr)
                p.lse_out[bh] = lse2 * kLn2;
        } else {
            const int64_t slot = bh * p.part_stride + p.prefix_slots + split;
            *reinterpret_cast<float4 *>(p.o_part + slot * D + d0) =
                make_float4(o0 * inv, o1 * inv, o2 * inv, o3 * inv);
            if (d0 == 0)
                p.lse_part[slot] = lse2;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeParams p)
{
    __shared__ MergeSmem<D> sm;
    pdl_launch_dependents();
    const int64_t bh = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = (int)(bh / p.num_q_heads);
    const Span sp = request_span(p, b, false);   // inputs of the call: read before the wait
    const int n_pre = sp.n_pre;
    const int n = split_count(p, sp);
    pdl_wait();                                  // the partial kernels of this call are done
    if (n_pre == 0 && n == 1)
        return;                                  // written by the partial kernel
    if (n_pre + n == 0) {                        // empty request: out = 0, lse = -inf
        if (warp == 0) {
            for (int d = lane; d < D / 2; d += 32)
                reinterpret_cast<uint32_t *>(p.out + bh * D)[d] = 0u;
            if (lane == 0 && p.lse_out != nullptr)
                p.lse_out[bh] = -CUDART_INF_F;
        }
        return;
    }
    merge_row<D>(p, bh, n_pre, n, sm);
}

// The same merge when every row's partial slots fit one warp (prefix slots + splits <= 32):
// a warp per row, four rows per CTA, no shared memory.  Lane s holds slot s's log2-sum-exp;
// the live slots' partials are then read in slot order, kLoads loads in flight per lane.
template <int D, int kLoads>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_warp_kernel(const DecodeParams p)
{
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t bh = (int64_t)blockIdx.x * kCombineWarps + warp;
    const bool live = bh < (int64_t)p.batch * p.num_q_heads;
    // the lengths and the plan are inputs of the call: read before the wait
    int n_pre = 0, n = 0;
    if (live) {
        const Span sp = request_span(p, (int)(bh / p.num_q_heads), false);
        n_pre = prefix_partials(p, sp, lane == 0);
        n = split_count(p, sp);
    }
    pdl_wait();                                  // the partial kernels of this call are done
    if (!live || (n_pre == 0 && n == 1))
        return;                                  // (written by the partial kernel)
    merge_row_warp<D, kLoads>(p, bh, n_pre, n, lane);
}

template <int D>
cudaError_t launch_combine_typed(const DecodeParams &p, cudaStream_t stream)
{
    const int64_t pairs = (int64_t)p.batch * p.num_q_heads;
    const unsigned grid = (unsigned)((pairs + kCombineWarps - 1) / kCombineWarps);
    // A warp per row when the slots fit; with few rows each warp keeps more of its row's
    // partial reads in flight (measured: huginn's 512 rows 33.8 -> 32.3 us per call with 16,
    // ouro's 1024 rows 181.2 -> 180.4; gqa's 8192 rows 514 with 8, 515 with 16).
    // Launched as a programmatic dependent of the call's partial kernels: it is resident
    // while they finish and waits for them in pdl_wait.
    if ((int64_t)p.prefix_slots + p.max_splits <= 32) {
        if (pairs >= 4096)
            return launch_kernel(decode_combine_warp_kernel<D, 8>, dim3(grid), dim3(kCombineThreads), 0, stream,
                                 true, p);
        return launch_kernel(decode_combine_warp_kernel<D, 16>, dim3(grid), dim3(kCombineThreads), 0, stream, true,
                             p);
    }
    return launch_kernel(decode_combine_kernel<D>, dim3((unsigned)pairs), dim3(kCombineThreads), 0, stream, true,
                         p);
}

template <int D, int G>
cudaError_t launch_typed(const DecodeParams &p, cudaStream_t stream, bool early)
{
    using C = Cfg<D, G>;
    static_assert(C::kSmemBytes <= 227 * 1024, "shared memory budget");
    const bool fault = p.debug_drop_copy != 0;
    auto kernel = fault ? decode_partial_kernel<D, G, true> : decode_partial_kernel<D, G, false>;
    // The shared-memory opt-in is per function and device: set it once per device.
    static std::atomic<uint64_t> configured[2]{{0}, {0}};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || (configured[fault].load(std::memory_order_acquire) & bit) == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured[fault].fetch_or(bit, std::memory_order_acq_rel);
    }
    const dim3 grid(p.max_splits, p.num_kv_heads, p.batch);
    e = launch_kernel(kernel, grid, dim3(kThreads), C::kSmemBytes, stream, early, p);
    // plain decode merges here; shared-prefix mode merges after the prefix kernel
    if (e != cudaSuccess || p.max_splits <= 1 || p.request_prefix != nullptr)
        return e;
    return launch_combine_typed<D>(p, stream);
}

}  // namespace

bool decode_supported(int head_dim, int group)
{
    return (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t max_seq_len, int32_t split_tokens, int num_sms, int waves)
{
    DecodePlan plan{};
    const int64_t max_tiles = max_seq_len > 0 ? (max_seq_len + kTileTokens - 1) / kTileTokens : 1;
    int tiles;
    if (split_tokens > 0) {
        tiles = (split_tokens + kTileTokens - 1) / kTileTokens;
    } else {
        // Largest split (fewest partials) that still gives every SM `waves`
        // waves of CTAs at 3 resident CTAs per SM.
        const int64_t target = (int64_t)(num_sms > 0 ? num_sms : 148) * 3 * waves;
        tiles = 128;
        while (tiles > 8 &&
               (int64_t)batch * num_kv_heads * ((max_tiles + tiles - 1) / tiles) < target)
            tiles /= 2;
        // A call this small is bound by launches and latency: one split per request
        // writes the output directly and saves the combine launch.
        if (max_tiles <= 128 && (int64_t)batch * num_kv_heads * max_tiles <= target)
            tiles = 128;
    }
    if (tiles > 128)
        tiles = 128;                             // one page-table entry per lane per warp
    if (tiles < 1)
        tiles = 1;
    plan.tiles_per_split = tiles;
    plan.max_splits = (int32_t)((max_tiles + tiles - 1) / tiles);
    if (plan.max_splits > 1) {
        const size_t rows = (size_t)batch * num_q_heads * plan.max_splits;
        plan.lse_part_bytes = (rows * sizeof(float) + 255) / 256 * 256;
        plan.workspace_bytes = plan.lse_part_bytes + rows * head_dim * sizeof(float);
    }
    return plan;
}

cudaError_t launch_combine(const DecodeParams &p, int head_dim, cudaStream_t stream)
{
    if (head_dim == 128)
        return launch_combine_typed<128>(p, stream);
    if (head_dim == 64)
        return launch_combine_typed<64>(p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeParams &p, int head_dim, int group, cudaStream_t stream, bool early)
{
    if (head_dim == 128) {
        switch (group) {
        case 1: return launch_typed<128, 1>(p, stream, early);
        case 2: return launch_typed<128, 2>(p, stream, early);
        case 4: return launch_typed<128, 4>(p, stream, early);
        case 8: return launch_typed<128, 8>(p, stream, early);
        }
    } else if (head_dim == 64) {
        switch (group) {
        case 1: return launch_typed<64, 1>(p, stream, early);
        case 2: return launch_typed<64, 2>(p, stream, early);
        case 4: return launch_typed<64, 4>(p, stream, early);
        case 8: return launch_typed<64, 8>(p, stream, early);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace rlt
