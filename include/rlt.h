/*
 * rlt.h - C ABI of the GB300 paged-KV decode path for looped transformers.
 *
 * One shared library (librlt.so, sm_103a) with plain pointers and sizes: no
 * C++ or framework types cross this boundary.  All array arguments of the
 * compute entry points are DEVICE pointers owned by the caller; the library
 * allocates no device memory and keeps no state besides a per-device error
 * word, the fixed scratch array of rlt_paged_decode_attn_noalloc and, once a
 * shared-prefix call needs it, a per-device side stream with two events
 * (rlt_paged_decode_attn_prefix).
 * Every compute call is enqueued on the caller's stream (a cudaStream_t passed
 * as void*; NULL = the legacy default stream), returns without waiting for the
 * GPU, and makes no host/device synchronisation.  Arguments are checked on
 * the host before any launch; a failed check returns a status and launches
 * nothing.  Kernels never trap: a page id or slot that is out of range at run
 * time is skipped and recorded in the device error word
 * (rlt_get_device_error).
 *
 * Debug mode: with RLT_VALIDATE=1 in the environment (read at each call),
 * rlt_kv_append, rlt_paged_decode_attn and rlt_paged_decode_attn_prefix first
 * synchronise the stream, copy the batch's device arrays to the host and check
 * them: append slots inside the pool and distinct; page-table entries in use
 * and lengths in range, and, with a fused append, each request's newest slot
 * on a page no other request maps (rlt_validate_batch's rules).  A violation
 * returns RLT_ERR_OUT_OF_RANGE / RLT_ERR_INVALID_ARG and launches nothing.
 * While the stream is being captured the check is skipped (a capture cannot
 * synchronise).
 *
 * CUDA graphs: every compute call may be recorded by stream capture, so that a
 * whole decode step (every layer-plane bank's append and attention, the noise)
 * is one graph submission, as the pages' engines run decode ([FFM] "Recurrent
 * depth": the decode CUDA graph; vllm-rlt PR #148, decode loops fused into one
 * submission).  Make each kind of call once on the device before capturing it
 * (the first call sets per-device kernel attributes and creates the side
 * stream).  A replay reads the
 * arrays' contents at replay time; shapes, max_seq_len, split_tokens and a
 * shared-prefix plan's sizes are fixed at capture.
 *
 * Sources (page title, section):
 *  [FFM]   "Faster fuzzy minds" (dibbla.space/posts/matrices/fast_subconscious)
 *          - "When scheduler does the work": paged KV cache = a flat pool of
 *            fixed-size slots addressed through page_table[request, position];
 *            two sequences may point at the same physical slots.
 *          - "LOTUS - the one place I opened the scheduler": store_kv scatters
 *            each token's K/V to the physical slots it is handed (out_loc);
 *            handing the same slots again overwrites in place.
 *          - "Recurrent depth - a deep model in a trench coat": L weight layers
 *            looped T times are T*L attention layers; iteration t of layer l
 *            writes KV bank t*L + l; decode attention over the paged pool
 *            treats it as an ordinary deep transformer.
 *  [PR152] vllm-rlt PR #152, "[Huginn] Opt-in prefix caching with
 *          position-keyed recurrent-state noise", Summary para 1 (per-plane
 *          layer map of #147: prelude/coda layers on plane 0 only) and para 2
 *          (latent noise = f(request seed, position, channel) via a stage-wise
 *          SplitMix64-style hash, a 24-bit uniform and an inverse normal CDF
 *          onto a normal with std = initializer_range truncated at +-3 sigma).
 *
 * KV pool layout (this library's convention; the pages leave it open):
 *   k and v are separate bf16 arrays, each
 *       [num_banks][num_pages][num_kv_heads][page_size][head_dim]
 *   so that the page_size rows of one (bank, page, kv head) are one contiguous
 *   page_size*head_dim*2-byte chunk.  Logical position p of request b is at
 *   page page_table[b*max_pages + p/page_size], offset p % page_size, i.e.
 *   slot = page*page_size + offset.
 */
#ifndef RLT_H
#define RLT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef RLT_API
#define RLT_API __attribute__((visibility("default")))
#endif

typedef enum rlt_status {
    RLT_OK = 0,
    RLT_ERR_INVALID_ARG = 1,          /* null pointer, negative size, misaligned buffer */
    RLT_ERR_OUT_OF_RANGE = 2,         /* bank, page, slot or length outside the pool */
    RLT_ERR_UNSUPPORTED = 3,          /* a shape the library has no kernel for */
    RLT_ERR_WORKSPACE_TOO_SMALL = 4,  /* see rlt_paged_decode_workspace_size */
    RLT_ERR_CUDA = 5                  /* the CUDA runtime reported an error */
} rlt_status;

/* Bits of the device error word (rlt_get_device_error). */
#define RLT_DEVERR_BAD_PAGE 1u        /* a page-table entry outside [0, num_pages) was skipped */
#define RLT_DEVERR_BAD_SLOT 2u        /* an append slot >= num_pages*page_size was skipped */
#define RLT_DEVERR_TIMEOUT 4u         /* a copy wait gave up after its time limit */
#define RLT_DEVERR_BAD_LEN 8u         /* a seq_len outside [0, min(max_pages*page_size,
                                         max_seq_len rounded to the split grid)] was clamped */

/*
 * Flags of the attention calls (rlt_paged_decode_attn, rlt_paged_decode_attn_prefix,
 * rlt_paged_extend_attn).
 *
 * RLT_ATTN_EARLY_START: the call's first kernels are launched as programmatic
 * dependents of the kernel ahead of them in the stream (Hopper/Blackwell
 * programmatic dependent launch; under stream capture, programmatic graph edges),
 * so they may be scheduled while that kernel still runs -- as soon as it lets its
 * dependents start, which every kernel of this library does at its start.  Before
 * the work ahead of them has completed they only read the page table, the lengths,
 * the shared-prefix plan and the cached K/V rows of `bank`, and issue the copies of
 * those rows; they read q, k_new and v_new, and write out, lse_out, the workspace
 * and the pool, only after it completed.  So a caller may set the flag when no
 * kernel still running ahead of the call writes the page table, the lengths, the
 * plan or that bank of the pool -- as in a decode step whose page tables are
 * copied in before the step and whose KV append is fused into the attention call
 * (k_new, v_new), where the kernels ahead (projections, an earlier layer's
 * attention) write only q, k_new, v_new.  Not with a separate rlt_kv_append into
 * the same bank right before the call.  Without the flag the first kernels start
 * after all earlier work in the stream; inside a call the combine always starts
 * behind the partial kernels this way (it is this library's own kernel).
 */
#define RLT_ATTN_EARLY_START 1u

/* Element type of a KV pool.  The pages' engines keep K/V in bf16, and so does
 * every kernel here: any other value is refused with RLT_ERR_UNSUPPORTED. */
typedef enum rlt_dtype { RLT_BF16 = 0 } rlt_dtype;

/* A paged KV pool (device memory owned by the caller). */
typedef struct rlt_kv_pool {
    void *k;                /* dtype [num_banks][num_pages][num_kv_heads][page_size][head_dim] */
    void *v;                /* same shape as k */
    int64_t num_pages;      /* physical pages per bank */
    int32_t num_banks;      /* one bank per (layer, plane) the model holds */
    int32_t num_kv_heads;
    int32_t page_size;      /* tokens per page, >= 1 */
    int32_t head_dim;       /* 64 or 128 */
    int32_t dtype;          /* rlt_dtype: RLT_BF16 */
} rlt_kv_pool;

/* Human-readable name of a status code (static string, never NULL). */
RLT_API const char *rlt_status_string(rlt_status status);

/* Library version: major*10000 + minor*100 + patch. */
RLT_API int32_t rlt_version(void);

/*
 * (layer, plane) -> bank map, HOST function ([FFM] "Recurrent depth";
 * [PR152] Summary para 1).  recurrent[l] != 0 marks a looped layer.  Plane 0
 * holds every layer; plane t >= 1 holds only the looped layers.  Banks are
 * numbered plane by plane, layers in order within a plane, so a fully looped
 * stack gets bank t*num_layers + l.  Writes map_out[l*num_planes + t] (bank,
 * or -1 where the plane does not hold the layer) and returns the number of
 * banks, or -RLT_ERR_INVALID_ARG for a null pointer or a size < 1.
 */
RLT_API int32_t rlt_bank_map(const uint8_t *recurrent, int32_t num_layers, int32_t num_planes,
                     int32_t *map_out);

/*
 * One entry of that map, HOST function (same passages): the bank that holds
 * (layer, plane), looked up in map (int32 [num_layers][num_planes], as
 * rlt_bank_map writes it).  Returns -1 where the plane does not hold the layer
 * (a prelude or coda layer at plane >= 1) and for a null map or a layer or
 * plane outside the map.
 */
RLT_API int32_t rlt_bank_index(const int32_t *map, int32_t num_layers, int32_t num_planes, int32_t layer,
                               int32_t plane);

/*
 * KV append = store_kv ([FFM] "LOTUS"): for i < n_tokens with out_loc[i] >= 0,
 * write k_new[i] and v_new[i] (bf16 [n_tokens][num_kv_heads][head_dim], device)
 * to slot out_loc[i] (int64, device) of the given bank.  Negative slots mean
 * "no token" and are skipped.  Slots within one call must be distinct (two
 * writers to one slot race); writing slots of an earlier call again overwrites
 * them in place.  A slot >= num_pages*page_size is skipped and sets
 * RLT_DEVERR_BAD_SLOT.  k_new, v_new and the pool must be 16-byte aligned.
 */
RLT_API rlt_status rlt_kv_append(const rlt_kv_pool *pool, int32_t bank, const void *k_new,
                         const void *v_new, const int64_t *out_loc, int32_t n_tokens,
                         void *stream);

/*
 * KV append with RoPE fused on the keys ([FFM] "Recurrent depth": a token keeps
 * one RoPE position across all T of its banks -- its index in its sequence,
 * never its loop depth -- so every plane's append of the token turns its key
 * by the same angles; [FFM] "LOTUS": store_kv to the handed slots).  As
 * rlt_kv_append, except that each key row is rotated first: for i < rot_dim/2
 * the pair (k[i], k[i + rot_dim/2]) turns by positions[i_token] *
 * rope_base^(-2i/rot_dim) (rotate-half pairing); dims rot_dim.. are stored as
 * given; the result is rounded to bf16 (nearest even).  V rows are stored as
 * given.  The angle is formed and reduced mod 2 pi in fp64, sin/cos and the
 * rotation in fp32: within one bf16 ulp of the exact rotation.
 *   positions  int64 [n_tokens], device: sequence position of each token
 *   rot_dim    even, 2 .. head_dim;  rope_base > 0
 *   written    NULL, or int32 [num_banks][batch] device written-prefix
 *              counters (rlt_publishable_prefix): written[bank][request[i]]
 *              becomes at least positions[i] + 1 for every appended token
 *              (appends come in sequence order); request int32 [n_tokens]
 *              gives each token's request, in [0, batch) (others are skipped
 *              and set RLT_DEVERR_BAD_SLOT).
 */
RLT_API rlt_status rlt_kv_append_rope(const rlt_kv_pool *pool, int32_t bank, const void *k_new,
                                      const void *v_new, const int64_t *positions,
                                      const int64_t *out_loc, int32_t n_tokens, int32_t rot_dim,
                                      double rope_base, const int32_t *request, int32_t *written,
                                      int32_t batch, void *stream);

/*
 * Prefix-cache publication coverage ([PR152] Summary: publication needs a
 * contiguous written prefix in every layer of every plane the model HOLDS --
 * all layers at depth 0, the recurrent layers deeper -- so a partially looped
 * model such as Huginn can publish).  Banks exist exactly for the held
 * (layer, plane) pairs (rlt_bank_map), so out[b] = min over banks of
 * written[bank][b], floored to whole pages of page_size tokens (0 when
 * num_banks == 0).  written int32 [num_banks][batch], out int32 [batch], both
 * device.
 */
RLT_API rlt_status rlt_publishable_prefix(const int32_t *written, int32_t num_banks, int32_t batch,
                                          int32_t page_size, int32_t *out, void *stream);

/*
 * Bytes of device workspace rlt_paged_decode_attn needs for these sizes
 * (split-K partial outputs and log-sum-exps).  split_tokens as passed to
 * rlt_paged_decode_attn (0 = the library's choice).  Returns 0 for invalid
 * sizes.
 */
RLT_API size_t rlt_paged_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t max_seq_len,
                                       int32_t split_tokens);

/*
 * Paged GQA decode attention ([FFM] "When scheduler does the work",
 * "Recurrent depth").  For every request b < batch and query head h:
 *     s_j = scale * <q[b][h], K_j>,  out[b][h] = sum_j softmax(s)_j V_j,
 * over the seq_lens[b] cached tokens j of request b (the token appended this
 * step included), K_j/V_j read from kv head h / (num_q_heads/num_kv_heads)
 * at page page_table[b*max_pages + j/page_size], offset j % page_size, of
 * bank `bank`.
 *   q          bf16 [batch][num_q_heads][head_dim], device
 *   k_new, v_new  NULL (both), or bf16 [batch][num_kv_heads][head_dim], device:
 *              the append fused into this call ([FFM] "When scheduler does the
 *              work": store_kv before attention).  Request b's rows are stored at
 *              its newest position seq_lens[b] - 1 (slot from the page table, as
 *              rlt_kv_append would with that slot) and attended to in the same
 *              call; the split-K CTA that reads that position's tile writes them.
 *              The slot must belong to request b alone (a shared page is read-
 *              only).  A request whose seq_len had to be clamped gets no append.
 *   page_table int32 [batch][max_pages], device; entries past a request's
 *              last page are never read
 *   seq_lens   int32 [batch], device, each in [0, max_seq_len]
 *   max_seq_len host upper bound of seq_lens (sizes the split-K grid)
 *   scale      softmax scale; <= 0 means 1/sqrt(head_dim)
 *   out        bf16 [batch][num_q_heads][head_dim], device
 *   lse_out    fp32 [batch][num_q_heads] natural-log sum of exp(s_j), or NULL
 *   workspace  device scratch of >= rlt_paged_decode_workspace_size() bytes,
 *              16-byte aligned; its contents need no initialisation and are
 *              garbage afterwards.  Calls that overlap on the GPU must not
 *              share one workspace.
 *   split_tokens tokens per split-K chunk, a multiple of 16 up to 2048;
 *              0 = the library's choice for the current device
 *   flags      0 or RLT_ATTN_EARLY_START (any other bit: RLT_ERR_INVALID_ARG)
 * A request with seq_lens[b] == 0 gets out = 0 and lse = -inf.  Supported:
 * head_dim 64 or 128; num_q_heads/num_kv_heads in {1, 2, 4, 8}; page_size a
 * multiple of 16 up to 256.  Page-table entries outside [0, num_pages) are
 * skipped (their tokens count as absent) and set RLT_DEVERR_BAD_PAGE.
 * q, out, the pool and workspace must be 16-byte aligned.
 */
RLT_API rlt_status rlt_paged_decode_attn(const rlt_kv_pool *pool, int32_t bank, const void *q,
                                 const void *k_new, const void *v_new, int32_t num_q_heads, const int32_t *page_table,
                                 int32_t max_pages, const int32_t *seq_lens, int32_t batch,
                                 int32_t max_seq_len, float scale, void *out, float *lse_out,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t split_tokens, uint32_t flags, void *stream);

/*
 * Shared-prefix plan, HOST function ([FFM] "When scheduler does the work":
 * a radix tree makes requests with a common prompt prefix point at the same
 * physical pages).  From host copies of a decode batch's page tables it finds
 * the 128-token tiles that several requests map to identical pages, walking a
 * trie of tiles from position 0, and groups them into segments: runs of tiles
 * shared by one set of requests.  A chain of trie runs whose member set only
 * shrinks (requests leaving one common prompt one after another) is one
 * segment when its members fit one member block: each member carries its key
 * limit, the number of leading tokens it shares, and reads no key past it.
 * Along each request's path the segments' partial slots are numbered from 0.
 *   chunk_tiles     tiles per CTA of the tensor-core prefix kernel (1..32)
 *   query_group     num_q_heads / num_kv_heads of the attention it plans for
 *                   (a CTA holds 128 query rows, so 128 / query_group members)
 *   private_tails   non-zero: also give every request a one-member segment
 *                   for its remaining (unshared) tokens, so that the
 *                   tensor-core kernel covers all of them -- worth it when
 *                   num_q_heads/num_kv_heads >= 4 makes each request's own
 *                   query rows a dense enough contraction
 *   segments        int32 [max_segments][8]: first tile, number of tiles,
 *                   first partial slot, first member entry, member count,
 *                   a member whose page-table row holds the segment's pages
 *                   (the one with the largest limit),
 *                   end token (exclusive; a private tail may end mid-tile),
 *                   first work unit (CTA) of the segment
 *   members         int32 [max_member_entries]: request ids by segment, in
 *                   ascending order of their limits
 *   member_limit    int32 [max_member_entries]: each member's key limit
 *                   (exclusive end token of what it shares in the segment; the
 *                   segment's end token for all members of an unmerged one)
 *   request_prefix  int32 [batch][2]: tokens of request b covered by its
 *                   segments (a multiple of 128 unless a private tail
 *                   covers all of it), partial slots they use
 *   sizes           int32 [7]: segments, member entries, most chunks of one
 *                   segment, most partial slots of one request, most members
 *                   of one segment, most tokens of one request left to the
 *                   split-K kernel, work units (filled even when the
 *                   capacities are short)
 * Returns RLT_ERR_OUT_OF_RANGE when max_segments or max_member_entries is too
 * small (sizes[] says what is needed), RLT_ERR_UNSUPPORTED when page_size
 * neither divides nor is a multiple of 128.
 */
RLT_API rlt_status rlt_plan_prefix(const int32_t *page_table, int32_t max_pages,
                                   const int32_t *seq_lens, int32_t batch, int32_t page_size,
                                   int32_t chunk_tiles, int32_t query_group, int32_t private_tails,
                                   int32_t *segments, int32_t max_segments, int32_t *members,
                                   int32_t *member_limit, int32_t max_member_entries,
                                   int32_t *request_prefix, int32_t *sizes);

/*
 * Work-item size (chunk_tiles) for rlt_plan_prefix / rlt_paged_decode_attn_prefix, HOST
 * function, from the same host page tables and lengths the plan is built from.  The
 * tensor-core kernel gives each of its CTAs a contiguous run of (kv head, segment, member
 * block, chunk) items.  With private_tails it does the whole call, so the call ends with its
 * busiest CTA: the function builds the plan for every chunk of 4..16 tiles, estimates each
 * CTA's busy time (1.55 us per 128-token sub-tile plus 4.7 us per change of run, both measured
 * on GB300) over num_ctas CTAs, and returns the chunk with the smallest maximum (the larger on
 * a tie).  Without private tails a split-K kernel shares the SMs: it returns the largest
 * power of two in 4..16 that still gives every CTA at least 16 items.  Either result is
 * capped at the longest segment.  num_ctas: the tensor-core CTAs (the SM count when the
 * kernel has the GPU to itself).  Returns the chunk (>= 1), or -RLT_ERR_INVALID_ARG /
 * -RLT_ERR_UNSUPPORTED as rlt_plan_prefix would fail.
 */
RLT_API int32_t rlt_choose_chunk_tiles(const int32_t *page_table, int32_t max_pages,
                                       const int32_t *seq_lens, int32_t batch, int32_t page_size,
                                       int32_t query_group, int32_t private_tails,
                                       int32_t num_kv_heads, int32_t num_ctas);

/* Device workspace bytes of rlt_paged_decode_attn_prefix (sizes[5] and sizes[3]
 * of the plan as max_rest_len and max_prefix_slots). */
RLT_API size_t rlt_paged_decode_prefix_workspace_size(int32_t batch, int32_t num_q_heads,
                                                      int32_t num_kv_heads, int32_t head_dim,
                                                      int32_t max_rest_len, int32_t max_prefix_slots,
                                                      int32_t split_tokens);

/*
 * Paged decode attention with shared prefixes read once ("cascade"): the same
 * result as rlt_paged_decode_attn, up to fp32 rounding order.  The plan's
 * arrays (segments, members, member_limit, request_prefix: DEVICE copies of
 * rlt_plan_prefix's output) name the tiles several requests share; each is
 * read from HBM once per kv head and applied to every member's queries by a
 * tcgen05 tensor-core kernel (S = Q K^T, O = P V with the members' query rows
 * as M = 128), the rest of each request goes through the split-K kernel, and
 * a log-sum-exp combine merges the partials.  num_segments, work_units,
 * max_prefix_slots, max_rest_len are sizes[0], [6], [3], [5] of the plan,
 * which must have been built with this call's query group, and chunk_tiles
 * the value it was built with; max_rest_len == 0 (private tails) launches no
 * split-K kernel.  Otherwise the split-K kernel runs at the same time as the
 * tensor-core kernel, on the library's side stream for this device (forked
 * from and joined back to `stream` with events, so stream capture records both
 * branches).  The tensor-core kernel is persistent: max_ctas CTAs (0 = the
 * library's choice: one per SM alone, or the SMs split between the two kernels
 * in proportion to their estimated tokens) share the num_kv_heads x work_units
 * work items in contiguous runs.  k_new / v_new (optional) fuse the append as in
 * rlt_paged_decode_attn: the kernel whose copy covers a request's newest position
 * stores its rows (the split-K kernel for an unshared rest, the tensor-core
 * kernel for a private tail); a newest position inside tiles the request shares,
 * whose slot would be a shared page's, is skipped and sets RLT_DEVERR_BAD_SLOT.
 * Other arguments (flags included) as
 * rlt_paged_decode_attn; the workspace (rlt_paged_decode_prefix_workspace_size
 * bytes) is required.  num_segments == 0 runs rlt_paged_decode_attn.
 * Supported: head_dim 128, num_q_heads/num_kv_heads in {1, 2, 4, 8}, page_size
 * a multiple of 16 dividing or divisible by 128.
 */
RLT_API rlt_status rlt_paged_decode_attn_prefix(
    const rlt_kv_pool *pool, int32_t bank, const void *q, const void *k_new, const void *v_new,
    int32_t num_q_heads,
    const int32_t *page_table, int32_t max_pages, const int32_t *seq_lens, int32_t batch,
    int32_t max_seq_len, const int32_t *segments, const int32_t *members,
    const int32_t *member_limit, const int32_t *request_prefix, int32_t num_segments, int32_t work_units,
    int32_t max_prefix_slots, int32_t chunk_tiles, int32_t max_rest_len, float scale, void *out,
    float *lse_out, void *workspace, size_t workspace_bytes, int32_t split_tokens, int32_t max_ctas,
    uint32_t flags, void *stream);

/*
 * Causal extend (span) attention over the paged pool ([FFM] "LOTUS":
 * re-forwarding a block of positions is one parallel extend-prefill over all
 * of them, their K/V already written -- in place -- to the block's slots;
 * packed prefill is the same call for a whole prompt).  Request b's
 * new_lens[b] new tokens are its last positions; new token i (0-based) sees
 * keys 0 .. seq_lens[b] - new_lens[b] + i.  For every new token and query
 * head h:  out = softmax(scale <q, K>) V over those keys, GQA as in
 * rlt_paged_decode_attn.  q and out are bf16 [num_rows][num_q_heads][D], the
 * new tokens packed request by request; lse_out (nullable) fp32
 * [num_rows][num_q_heads], natural log.
 *
 * rlt_plan_extend (HOST arrays) lays the work out for the tcgen05 kernel of
 * rlt_paged_decode_attn_prefix: one segment per request with new tokens,
 * covering its keys, whose members are its new tokens with their causal
 * limits; each block of 128 / query_group new tokens reads keys only up to its
 * last token's limit.  Outputs: segments [sizes[0]][8], members and
 * member_limit [sizes[1]], row_prefix [num_rows][2] and row_len [num_rows];
 * sizes[0..6] = segments, rows, max chunks, partial slots per row, max
 * members, 0, work units.  Returns RLT_ERR_OUT_OF_RANGE (sizes filled) when
 * the arrays are too small, RLT_ERR_INVALID_ARG for new_lens[b] outside
 * [0, seq_lens[b]].  Same page_size rule as rlt_plan_prefix.
 *
 * rlt_paged_extend_attn takes the plan's arrays as DEVICE copies (plus
 * sizes[0], [6], [3] as num_segments, work_units, max_slots and the
 * chunk_tiles the plan was built with) and a workspace of
 * rlt_paged_extend_workspace_size bytes; page_table is int32 [batch][max_pages]
 * of the requests.  max_ctas as rlt_paged_decode_attn_prefix; flags as
 * rlt_paged_decode_attn (with RLT_ATTN_EARLY_START no kernel still running
 * ahead may write the plan, the page table or the bank).  Supported:
 * head_dim 128, num_q_heads/num_kv_heads in {1, 2, 4, 8}.
 */
RLT_API rlt_status rlt_plan_extend(const int32_t *seq_lens, const int32_t *new_lens, int32_t batch,
                                   int32_t page_size, int32_t chunk_tiles, int32_t query_group,
                                   int32_t *segments, int32_t max_segments, int32_t *members,
                                   int32_t *member_limit, int32_t max_member_entries,
                                   int32_t *row_prefix, int32_t *row_len, int32_t *sizes);

RLT_API size_t rlt_paged_extend_workspace_size(int32_t num_rows, int32_t num_q_heads, int32_t head_dim,
                                               int32_t max_slots);

RLT_API rlt_status rlt_paged_extend_attn(
    const rlt_kv_pool *pool, int32_t bank, const void *q, int32_t num_q_heads, int32_t num_rows,
    const int32_t *page_table, int32_t max_pages, int32_t batch, const int32_t *segments,
    const int32_t *members, const int32_t *member_limit, const int32_t *row_prefix, const int32_t *row_len,
    int32_t num_segments, int32_t work_units, int32_t max_slots, int32_t chunk_tiles, float scale, void *out,
    float *lse_out, void *workspace, size_t workspace_bytes, int32_t max_ctas, uint32_t flags, void *stream);

/* Size of the scratch array rlt_paged_decode_attn_noalloc uses (64 MiB). */
#define RLT_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * rlt_paged_decode_attn without a workspace argument: the same computation,
 * arguments and results as rlt_paged_decode_attn with k_new = v_new = NULL
 * (no fused append; those two arguments are absent), but the split-K partials go
 * to a fixed 64 MiB array inside the library, so the call allocates nothing.
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory at the point of the call, such as
 * plugins whose host framework owns every device allocation, or decode loops
 * that must not risk the device-wide synchronisation a cudaMalloc can cause.
 *   - Each device that loads the library holds the array until the process
 *     exits.  The first call on a device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture.  The address is kept for the life of the process, so this entry
 *     point supports only the device's primary context (the runtime's): after a
 *     cudaDeviceReset, or from another driver context on the same device, it
 *     would hand the kernels a stale address.
 *   - Arguments are checked as rlt_paged_decode_attn checks them, in the same
 *     order, before the scratch size: a bad pool, bank, split or pointer gets
 *     the status rlt_paged_decode_attn would return.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing in it needs to start at zero.  Calls that overlap on the
 *     GPU (other streams, other host threads) race on it: serialise them.
 *   - A shape whose partials need more than RLT_NOALLOC_SCRATCH_BYTES
 *     (rlt_paged_decode_workspace_size) returns RLT_ERR_WORKSPACE_TOO_SMALL
 *     and launches nothing; a larger split_tokens needs less.
 */
RLT_API rlt_status rlt_paged_decode_attn_noalloc(const rlt_kv_pool *pool, int32_t bank,
                                                 const void *q, int32_t num_q_heads,
                                                 const int32_t *page_table, int32_t max_pages,
                                                 const int32_t *seq_lens, int32_t batch,
                                                 int32_t max_seq_len, float scale, void *out,
                                                 float *lse_out, int32_t split_tokens,
                                                 void *stream);

/*
 * Position-keyed latent-state noise ([PR152] Summary para 2).  For each row r
 * (a token) and channel c < channels:
 *     key  = stage(stage(stage(0, seeds[r]), positions[r]), c),
 *            stage(h, x) = mix64((h ^ x) + 0x9E3779B97F4A7C15),
 *            mix64 = the SplitMix64 output function (mod 2^64 arithmetic);
 *     h24  = key >> 40;  u = (h24 + 1/2) / 2^24;
 *     out[r][c] = initializer_range * sqrt(2) * erfinv((2u - 1) * erf(3/sqrt(2)))
 * i.e. the inverse CDF of N(0, initializer_range^2) truncated at +-3 sigma.
 * The value depends only on (seed, position, channel), never on the batch.
 *   out fp32 [n_rows][channels], seeds uint64 [n_rows], positions int64
 *   [n_rows] (absolute token positions), all device.
 */
RLT_API rlt_status rlt_latent_noise_init(float *out, const uint64_t *seeds, const int64_t *positions,
                                 int64_t n_rows, int32_t channels, float initializer_range,
                                 void *stream);

/* The 24-bit uniforms h24 of rlt_latent_noise_init, as uint32 [n_rows][channels]
 * (device); for bit-exact checks of the hash. */
RLT_API rlt_status rlt_noise_hash24(uint32_t *out, const uint64_t *seeds, const int64_t *positions,
                            int64_t n_rows, int32_t channels, void *stream);

/*
 * Page-table gather ([FFM] "When scheduler does the work"): copy the K and V
 * rows of the first seq_lens[b] logical positions of every request, in
 * logical order, into k_out / v_out (bf16 [batch][max_len][num_kv_heads]
 * [head_dim], device).  Rows at positions >= seq_lens[b] are not written.
 * For bit-exact checks of the slot mapping.  seq_lens[b] must be <= max_len.
 */
RLT_API rlt_status rlt_paged_gather(const rlt_kv_pool *pool, int32_t bank, const int32_t *page_table,
                            int32_t max_pages, const int32_t *seq_lens, int32_t batch,
                            int32_t max_len, void *k_out, void *v_out, void *stream);

/*
 * HOST validation of a decode batch before it is handed to the GPU (all
 * arrays are host copies): every page-table entry a request uses lies in
 * [0, num_pages); seq_lens[b] in [0, max_pages*page_size]; every
 * new_slots[b] >= 0 lies in the pool, on the page holding position
 * seq_lens[b]-1 of request b, and no two requests share it; no page holding
 * a new slot appears in another request's page table (shared prefix pages
 * are read-only).  new_slots may be NULL.  Returns RLT_OK or the first
 * violation as RLT_ERR_OUT_OF_RANGE / RLT_ERR_INVALID_ARG.
 */
RLT_API rlt_status rlt_validate_batch(const int32_t *page_table, int32_t max_pages,
                              const int32_t *seq_lens, int32_t batch, const int64_t *new_slots,
                              int64_t num_pages, int32_t page_size);

/*
 * Fault injection for tests of the bounded copy waits; the pages have no
 * counterpart (it exists so that the give-up path can be exercised without a
 * GPU fault).  Arms the next rlt_paged_decode_attn call made by this host
 * thread, once: its split-K kernel gives every copy wait wait_limit_ns (1 ns ..
 * 1 s; the ordinary limit is 1 s) and never issues the first tile copy of warp 0
 * of the CTA for (split 0, kv head 0, request 0), so that wait runs out.  The
 * kernel then records RLT_DEVERR_TIMEOUT, waits (bounded by the same limit) for
 * that warp's copies still in flight, leaves the warp's tiles out of request 0's
 * result for kv head 0's query heads, and returns: nothing faults or hangs, and
 * later calls are unaffected.  RLT_ERR_INVALID_ARG for a limit outside that range.
 */
RLT_API rlt_status rlt_debug_fault_next_decode(uint64_t wait_limit_ns);

/*
 * Read and clear the device error word (RLT_DEVERR_* bits) of the current
 * device.  Synchronises the device.
 */
RLT_API rlt_status rlt_get_device_error(uint32_t *error_bits);

#ifdef __cplusplus
}
#endif

#endif /* RLT_H */
