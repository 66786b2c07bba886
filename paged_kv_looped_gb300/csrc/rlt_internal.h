// Host-side interface between the C-ABI entry points (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "rlt.h"

namespace rlt {

// Tokens per attention tile: one bulk copy of K and one of V per tile.
constexpr int kTileTokens = 16;

// Longest copy-wait limit the timeout test may ask for (rlt_debug_fault_next_decode).
constexpr uint64_t kMaxFaultWaitNs = 1000000000ull;

struct DecodeParams {
    const uint16_t *k_bank;      // bank base of the K pool: [num_pages][Hkv][ps][D]
    const uint16_t *v_bank;
    const uint16_t *q;           // [B][Hq][D]
    const int32_t *page_table;   // [B][max_pages]
    const int32_t *seq_lens;     // [B]
    uint16_t *out;               // [B][Hq][D]
    float *lse_out;              // [B][Hq] or null
    float *lse_part;             // [B][Hq][max_splits], log2 units
    float *o_part;               // [B][Hq][max_splits][D]
    unsigned int *err;
    int64_t num_pages;
    int32_t num_kv_heads;
    int32_t num_q_heads;
    int32_t page_size;
    int32_t max_pages;
    int32_t batch;
    int32_t tiles_per_split;
    int32_t max_splits;
    float qscale;                // softmax scale * log2(e)
    // Shared-prefix (cascade) mode; all zero / null for plain decode.
    const int32_t *request_prefix;  // [B][2]: tokens covered by shared segments, their partial slots
    int32_t prefix_slots;        // partial slots reserved per (b, h) ahead of the split-K slots
    int32_t part_stride;         // partial slots per (b, h): prefix_slots + max_splits
    // Fused append (null: none): request b's K/V at position seq_lens[b] - 1, bf16
    // [B][Hkv][D]; the split-K CTA covering that position stores them to the pool
    // and uses them in place of what it read from there.
    const uint16_t *k_new;
    const uint16_t *v_new;
    // The fault-injection switch of the timeout test (rlt_debug_fault_next_decode): non-zero
    // launches the split-K kernel's fault instance, which leaves the first tile copy of CTA
    // (0, 0, 0)'s warp 0 unissued, so that its wait runs out, and gives every copy wait the
    // limit wait_limit_ns.  Zero in every ordinary call (the waits take the one-second
    // default).
    uint64_t wait_limit_ns;
    int32_t debug_drop_copy;
};

// Tokens per tensor-core tile of the shared-prefix kernel.
constexpr int kPrefixTile = 128;

// Query rows of a tensor-core run are copied into idle TMEM lane quarters: with R
// live rows (members x query group) a run keeps F = 4, 2 or 1 copies of them,
// each copy taking 1/F of every 128-token sub-tile's keys and writing its own
// partial, so that the softmax work of a few rows is spread over all four SM
// sub-partitions.  F follows from the rows of a segment's first (fullest)
// member block; planner and kernel must agree on it.  Four copies only for up to 8
// rows (a private tail at G = 8): measured on GB300, 16 rows (huginn's sessions at
// G = 1) run faster as two copies of half the keys each than as four (25.22 against
// 25.40 us per call), 8 rows slower (longctx 118.0 against 113.8).
__host__ __device__ inline int prefix_replication(int rows)
{
    return rows <= 8 ? 4 : rows <= 64 ? 2 : 1;
}

// Fields of one segment of a prefix plan (rlt_plan_prefix).
enum PrefixSegField { kSegFirstTile = 0, kSegNumTiles, kSegSlotBase, kSegMemberBegin,
                      kSegMemberCount, kSegPageRow, kSegEndToken, kSegWorkBegin, kSegFields };

struct PrefixParams {
    const int32_t *segments;     // [num_segments][kSegFields]
    const int32_t *members;      // query rows (request ids; new-token ids for extend), grouped by segment
    const int32_t *member_limit; // extend: each member's key count (causal limit); null: every key
    int32_t num_rows;            // rows of q: members lie in [0, num_rows)
    int32_t num_segments;
    int32_t chunk_tiles;         // 128-token tiles per CTA
    int32_t work_units;          // (segment, member block, chunk) units per kv head
    int32_t ctas;                // persistent CTAs sharing the num_kv_heads x work_units items
    // Non-zero: the copy warps fetch sub-tiles into L2 kPrefetch ahead of their rings (the call
    // with a split-K rest, whose CTAs hold few sub-tiles each; measured slower when a CTA
    // streams long runs, where the rings already keep the copy bandwidth busy).
    int32_t l2_ahead;
};

// Launch a kernel on `stream`; with `early`, as a programmatic dependent of the kernel
// ahead of it in the stream (it may start before that kernel ends and must call
// pdl_wait before touching what that kernel or any earlier one writes).
template <typename... Exp, typename... Act>
cudaError_t launch_kernel(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool early, Act &&...args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Act &&>(args)...);
}

bool prefix_supported(int head_dim, int group, int page_size);
size_t prefix_smem_bytes(int chunk_tiles, int page_size);
cudaError_t launch_prefix(const DecodeParams &p, const PrefixParams &pp, const void *k_bank,
                          const void *v_bank, int64_t bank_rows, cudaStream_t stream, bool early);

// Split-K plan for one decode call.
struct DecodePlan {
    int32_t tiles_per_split;
    int32_t max_splits;
    size_t workspace_bytes;
    size_t lse_part_bytes;       // offset of o_part inside the workspace
};

// waves: the library's split (split_tokens == 0) is the largest that still gives
// every SM this many waves of 3 CTAs; 8 for plain decode, one for the short
// unshared rests a shared-prefix call leaves, which share the GPU with the
// tensor-core kernel: there each CTA's start-up round trips weigh most, so a
// rest is split only when one wave would leave SMs idle (measured on the huginn
// shape: 30.3 us per call with one wave, 32.3 with three).
constexpr int kPlainWaves = 8, kRestWaves = 1;
DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t max_seq_len, int32_t split_tokens, int num_sms,
                       int waves = kPlainWaves);

bool decode_supported(int head_dim, int group);

// The argument checks of rlt_paged_decode_attn that come before its workspace check, in
// its order (pool and bank, sizes and split, supported shape, pointers and alignment);
// *empty: a batch of 0 requests, nothing to launch.
rlt_status check_decode_args(const rlt_kv_pool *pool, int32_t bank, const void *q, const void *k_new,
                             const void *v_new, int32_t num_q_heads, const int32_t *page_table, int32_t max_pages,
                             const int32_t *seq_lens, int32_t batch, int32_t max_seq_len, float scale,
                             const void *out, int32_t split_tokens, bool *empty);
// early: start as a programmatic dependent of the kernel ahead in the stream (the call's
// RLT_ATTN_EARLY_START).  The combine always starts that way behind the call's own
// partial kernels.
cudaError_t launch_decode(const DecodeParams &p, int head_dim, int group, cudaStream_t stream, bool early);
cudaError_t launch_combine(const DecodeParams &p, int head_dim, cudaStream_t stream);

cudaError_t launch_append(uint16_t *k_bank, uint16_t *v_bank, const uint16_t *k_new,
                          const uint16_t *v_new, const int64_t *out_loc, int32_t n_tokens,
                          int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                          int64_t num_pages, unsigned int *err, cudaStream_t stream);

cudaError_t launch_append_rope(uint16_t *k_bank, uint16_t *v_bank, const uint16_t *k_new,
                               const uint16_t *v_new, const int64_t *positions, const int64_t *out_loc,
                               int32_t n_tokens, int32_t num_kv_heads, int32_t page_size,
                               int32_t head_dim, int64_t num_pages, int32_t rot_dim, double rope_base,
                               const int32_t *request, int32_t *written, int32_t batch,
                               unsigned int *err, cudaStream_t stream);

cudaError_t launch_publishable(const int32_t *written, int32_t num_banks, int32_t batch,
                               int32_t page_size, int32_t *out, cudaStream_t stream);

cudaError_t launch_gather(const uint16_t *k_bank, const uint16_t *v_bank,
                          const int32_t *page_table, int32_t max_pages, const int32_t *seq_lens,
                          int32_t batch, int32_t max_len, uint16_t *k_out, uint16_t *v_out,
                          int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                          int64_t num_pages, unsigned int *err, cudaStream_t stream);

cudaError_t launch_noise(float *out, uint32_t *hash_out, const uint64_t *seeds,
                         const int64_t *positions, int64_t n_rows, int32_t channels,
                         float initializer_range, cudaStream_t stream);

}  // namespace rlt
