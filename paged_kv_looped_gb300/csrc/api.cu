// extern "C" entry points of librlt: host-side argument checks, launch
// planning and dispatch to the kernels.  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>
#include <unordered_set>
#include <vector>

#include "rlt.h"
#include "rlt_internal.h"

namespace {

// Per-device error word the kernels OR their RLT_DEVERR_* bits into.
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned int *g_err_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

// Device address of the error word and the SM count of the current device,
// looked up once per device.
rlt_status device_info(unsigned int **err, int *num_sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return RLT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_err_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess)
            return RLT_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return RLT_ERR_CUDA;
        g_num_sms[dev] = sms;
        g_err_ptr[dev] = static_cast<unsigned int *>(p);
    }
    if (err != nullptr)
        *err = g_err_ptr[dev];
    if (num_sms != nullptr)
        *num_sms = g_num_sms[dev];
    return RLT_OK;
}

// A second stream and two events per device: in shared-prefix mode the split-K
// kernel runs beside the tensor-core kernel (fork from the caller's stream, join
// back before the combine).  Created on the first such call on the device.
struct SideStream {
    cudaStream_t stream;
    cudaEvent_t fork, join;
};
SideStream g_side[kMaxDevices];

rlt_status side_stream(SideStream **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return RLT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    SideStream &s = g_side[dev];
    if (s.stream == nullptr) {
        SideStream n{};
        if (cudaStreamCreateWithFlags(&n.stream, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) != cudaSuccess)
            return RLT_ERR_CUDA;
        s = n;
    }
    *out = &s;
    return RLT_OK;
}

int current_sms()
{
    int sms = 0;
    if (device_info(nullptr, &sms) != RLT_OK)
        return 0;
    return sms;
}

rlt_status check_pool(const rlt_kv_pool *pool, int32_t bank)
{
    if (pool == nullptr || pool->k == nullptr || pool->v == nullptr)
        return RLT_ERR_INVALID_ARG;
    if (pool->num_pages < 0 || pool->num_banks < 1 || pool->num_kv_heads < 1 ||
        pool->page_size < 1 || pool->head_dim < 8 || pool->head_dim % 8 != 0)
        return RLT_ERR_INVALID_ARG;
    if (!aligned16(pool->k) || !aligned16(pool->v))
        return RLT_ERR_INVALID_ARG;
    if (pool->dtype != RLT_BF16)
        return RLT_ERR_UNSUPPORTED;
    if (bank < 0 || bank >= pool->num_banks)
        return RLT_ERR_OUT_OF_RANGE;
    return RLT_OK;
}

int64_t bank_elems(const rlt_kv_pool *pool)
{
    return pool->num_pages * pool->num_kv_heads * pool->page_size * (int64_t)pool->head_dim;
}

rlt_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RLT_OK : RLT_ERR_CUDA; }

// rlt_debug_fault_next_decode: copy-wait limit (ns) for the next rlt_paged_decode_attn call of
// this host thread, which also leaves one tile copy unissued; 0 = not armed.
thread_local uint64_t t_fault_wait_ns = 0;

}  // namespace

namespace {

// Debug mode: with RLT_VALIDATE=1 in the environment (read at each call) the compute calls
// synchronise the stream, copy the batch's device arrays to the host and check them
// before launching; a violation fails the call.  Not while the stream is being captured
// (a capture cannot synchronise): there the calls run unchecked.
bool validate_enabled()
{
    const char *v = std::getenv("RLT_VALIDATE");
    return v != nullptr && v[0] == '1' && v[1] == '\0';
}

// Host copies of a batch for validation; false (status set) if the stream is capturing or
// a CUDA call failed.
bool fetch_for_validation(cudaStream_t stream, rlt_status *st)
{
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        *st = RLT_ERR_CUDA;
        return false;
    }
    *st = RLT_OK;
    if (cap != cudaStreamCaptureStatusNone)
        return false;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        *st = RLT_ERR_CUDA;
        return false;
    }
    return true;
}

template <typename T>
bool copy_to_host(std::vector<T> &h, const T *d, size_t n)
{
    h.resize(n);
    return n == 0 || cudaMemcpy(h.data(), d, n * sizeof(T), cudaMemcpyDeviceToHost) == cudaSuccess;
}

// The attention calls' check: page-table entries in use and lengths in range; with a fused
// append, each request's newest slot is derived from its page table and must lie on a page
// no other request maps (shared pages are read-only).
rlt_status validate_attention_batch(const int32_t *page_table, int32_t max_pages, const int32_t *seq_lens,
                                    int32_t batch, int64_t num_pages, int32_t page_size, bool fused,
                                    cudaStream_t stream)
{
    rlt_status st = RLT_OK;
    if (!fetch_for_validation(stream, &st))
        return st;
    std::vector<int32_t> pt, sl;
    if (!copy_to_host(pt, page_table, (size_t)batch * max_pages) || !copy_to_host(sl, seq_lens, (size_t)batch))
        return RLT_ERR_CUDA;
    std::vector<int64_t> slots;
    if (fused) {
        slots.assign((size_t)batch, -1);
        for (int32_t b = 0; b < batch; ++b) {
            const int64_t L = sl[b];
            if (L >= 1 && L <= (int64_t)max_pages * page_size)
                slots[b] = (int64_t)pt[(size_t)b * max_pages + (L - 1) / page_size] * page_size + (L - 1) % page_size;
        }
    }
    return rlt_validate_batch(pt.data(), max_pages, sl.data(), batch, fused ? slots.data() : nullptr, num_pages,
                              page_size);
}

}  // namespace

namespace rlt {

rlt_status check_decode_args(const rlt_kv_pool *pool, int32_t bank, const void *q, const void *k_new,
                             const void *v_new, int32_t num_q_heads, const int32_t *page_table, int32_t max_pages,
                             const int32_t *seq_lens, int32_t batch, int32_t max_seq_len, float scale,
                             const void *out, int32_t split_tokens, bool *empty)
{
    *empty = false;
    rlt_status st = check_pool(pool, bank);
    if (st != RLT_OK)
        return st;
    if (batch < 0 || max_seq_len < 0 || max_pages < 0 || num_q_heads < 1 || split_tokens < 0 ||
        split_tokens % kTileTokens != 0 || split_tokens > 128 * kTileTokens)
        return RLT_ERR_INVALID_ARG;
    if (num_q_heads % pool->num_kv_heads != 0)
        return RLT_ERR_INVALID_ARG;
    const int group = num_q_heads / pool->num_kv_heads;
    if (!decode_supported(pool->head_dim, group) || pool->page_size % kTileTokens != 0)
        return RLT_ERR_UNSUPPORTED;
    if (batch > 65535 || pool->num_kv_heads > 65535)
        return RLT_ERR_UNSUPPORTED;
    if (batch == 0) {
        *empty = true;
        return RLT_OK;
    }
    if (q == nullptr || page_table == nullptr || seq_lens == nullptr || out == nullptr || max_pages < 1)
        return RLT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out))
        return RLT_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || (k_new == nullptr) != (v_new == nullptr) || !aligned16(k_new) ||
        !aligned16(v_new))
        return RLT_ERR_INVALID_ARG;
    return RLT_OK;
}

}  // namespace rlt

extern "C" {

RLT_API const char *rlt_status_string(rlt_status status)
{
    switch (status) {
    case RLT_OK: return "RLT_OK";
    case RLT_ERR_INVALID_ARG: return "RLT_ERR_INVALID_ARG";
    case RLT_ERR_OUT_OF_RANGE: return "RLT_ERR_OUT_OF_RANGE";
    case RLT_ERR_UNSUPPORTED: return "RLT_ERR_UNSUPPORTED";
    case RLT_ERR_WORKSPACE_TOO_SMALL: return "RLT_ERR_WORKSPACE_TOO_SMALL";
    case RLT_ERR_CUDA: return "RLT_ERR_CUDA";
    }
    return "RLT_ERR_UNKNOWN";
}

RLT_API int32_t rlt_version(void) { return 100; }

RLT_API int32_t rlt_bank_map(const uint8_t *recurrent, int32_t num_layers, int32_t num_planes,
                             int32_t *map_out)
{
    if (recurrent == nullptr || map_out == nullptr || num_layers < 1 || num_planes < 1)
        return -RLT_ERR_INVALID_ARG;
    int32_t next = 0;
    for (int32_t t = 0; t < num_planes; ++t)
        for (int32_t l = 0; l < num_layers; ++l)
            map_out[l * num_planes + t] = (t == 0 || recurrent[l] != 0) ? next++ : -1;
    return next;
}

RLT_API int32_t rlt_bank_index(const int32_t *map, int32_t num_layers, int32_t num_planes, int32_t layer,
                               int32_t plane)
{
    if (map == nullptr || layer < 0 || layer >= num_layers || plane < 0 || plane >= num_planes)
        return -1;
    const int32_t bank = map[(int64_t)layer * num_planes + plane];
    return bank >= 0 ? bank : -1;
}

RLT_API rlt_status rlt_kv_append(const rlt_kv_pool *pool, int32_t bank, const void *k_new,
                                 const void *v_new, const int64_t *out_loc, int32_t n_tokens,
                                 void *stream)
{
    rlt_status st = check_pool(pool, bank);
    if (st != RLT_OK)
        return st;
    if (n_tokens < 0)
        return RLT_ERR_INVALID_ARG;
    if (n_tokens == 0)
        return RLT_OK;
    if (k_new == nullptr || v_new == nullptr || out_loc == nullptr)
        return RLT_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || reinterpret_cast<uintptr_t>(out_loc) % 8 != 0)
        return RLT_ERR_INVALID_ARG;
    if (validate_enabled()) {
        std::vector<int64_t> loc;
        if (fetch_for_validation(static_cast<cudaStream_t>(stream), &st)) {
            if (!copy_to_host(loc, out_loc, (size_t)n_tokens))
                return RLT_ERR_CUDA;
            std::unordered_set<int64_t> seen;
            for (const int64_t slot : loc) {
                if (slot < 0)
                    continue;
                if (slot >= pool->num_pages * pool->page_size)
                    return RLT_ERR_OUT_OF_RANGE;
                if (!seen.insert(slot).second)
                    return RLT_ERR_INVALID_ARG;   // two tokens written to one slot
            }
        } else if (st != RLT_OK) {
            return st;
        }
    }
    unsigned int *err = nullptr;
    if ((st = device_info(&err, nullptr)) != RLT_OK)
        return st;
    const int64_t off = bank * bank_elems(pool);
    return from_cuda(rlt::launch_append(
        static_cast<uint16_t *>(pool->k) + off, static_cast<uint16_t *>(pool->v) + off,
        static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new), out_loc,
        n_tokens, pool->num_kv_heads, pool->page_size, pool->head_dim, pool->num_pages, err,
        static_cast<cudaStream_t>(stream)));
}

RLT_API rlt_status rlt_kv_append_rope(const rlt_kv_pool *pool, int32_t bank, const void *k_new,
                                      const void *v_new, const int64_t *positions,
                                      const int64_t *out_loc, int32_t n_tokens, int32_t rot_dim,
                                      double rope_base, const int32_t *request, int32_t *written,
                                      int32_t batch, void *stream)
{
    rlt_status st = check_pool(pool, bank);
    if (st != RLT_OK)
        return st;
    if (n_tokens < 0 || rot_dim < 2 || rot_dim % 2 != 0 || rot_dim > pool->head_dim ||
        !(rope_base > 0.0) || !std::isfinite(rope_base) || (written != nullptr && (request == nullptr || batch < 1)))
        return RLT_ERR_INVALID_ARG;
    if (n_tokens == 0)
        return RLT_OK;
    if (k_new == nullptr || v_new == nullptr || out_loc == nullptr || positions == nullptr)
        return RLT_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || reinterpret_cast<uintptr_t>(out_loc) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(positions) % 8 != 0 ||
        (written != nullptr && (reinterpret_cast<uintptr_t>(written) % 4 != 0 ||
                                reinterpret_cast<uintptr_t>(request) % 4 != 0)))
        return RLT_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    if ((st = device_info(&err, nullptr)) != RLT_OK)
        return st;
    const int64_t off = bank * bank_elems(pool);
    return from_cuda(rlt::launch_append_rope(
        static_cast<uint16_t *>(pool->k) + off, static_cast<uint16_t *>(pool->v) + off,
        static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new), positions, out_loc,
        n_tokens, pool->num_kv_heads, pool->page_size, pool->head_dim, pool->num_pages, rot_dim, rope_base,
        request, written != nullptr ? written + (int64_t)bank * batch : nullptr, batch, err,
        static_cast<cudaStream_t>(stream)));
}

RLT_API rlt_status rlt_publishable_prefix(const int32_t *written, int32_t num_banks, int32_t batch,
                                          int32_t page_size, int32_t *out, void *stream)
{
    if (num_banks < 0 || batch < 0 || page_size < 1 || (batch > 0 && (out == nullptr ||
                                                                       (num_banks > 0 && written == nullptr))))
        return RLT_ERR_INVALID_ARG;
    if (batch == 0)
        return RLT_OK;
    return from_cuda(rlt::launch_publishable(written, num_banks, batch, page_size, out,
                                             static_cast<cudaStream_t>(stream)));
}

RLT_API size_t rlt_paged_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                               int32_t num_kv_heads, int32_t head_dim,
                                               int32_t max_seq_len, int32_t split_tokens)
{
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || max_seq_len < 0 ||
        split_tokens < 0)
        return 0;
    return rlt::plan_decode(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                            split_tokens, current_sms())
        .workspace_bytes;
}

RLT_API rlt_status rlt_paged_decode_attn(const rlt_kv_pool *pool, int32_t bank, const void *q,
                                         const void *k_new, const void *v_new, int32_t num_q_heads, const int32_t *page_table,
                                         int32_t max_pages, const int32_t *seq_lens,
                                         int32_t batch, int32_t max_seq_len, float scale,
                                         void *out, float *lse_out, void *workspace,
                                         size_t workspace_bytes, int32_t split_tokens,
                                         uint32_t flags, void *stream)
{
    if ((flags & ~RLT_ATTN_EARLY_START) != 0)
        return RLT_ERR_INVALID_ARG;
    bool empty = false;
    rlt_status st = rlt::check_decode_args(pool, bank, q, k_new, v_new, num_q_heads, page_table, max_pages,
                                           seq_lens, batch, max_seq_len, scale, out, split_tokens, &empty);
    if (st != RLT_OK || empty)
        return st;
    if (workspace != nullptr && !aligned16(workspace))
        return RLT_ERR_INVALID_ARG;
    const int group = num_q_heads / pool->num_kv_heads;
    if (validate_enabled() &&
        (st = validate_attention_batch(page_table, max_pages, seq_lens, batch, pool->num_pages, pool->page_size,
                                       k_new != nullptr, static_cast<cudaStream_t>(stream))) != RLT_OK)
        return st;

    unsigned int *err = nullptr;
    int sms = 0;
    if ((st = device_info(&err, &sms)) != RLT_OK)
        return st;
    const rlt::DecodePlan plan = rlt::plan_decode(batch, num_q_heads, pool->num_kv_heads,
                                                  pool->head_dim, max_seq_len, split_tokens, sms);
    if (plan.workspace_bytes > 0 && (workspace == nullptr || workspace_bytes < plan.workspace_bytes))
        return RLT_ERR_WORKSPACE_TOO_SMALL;

    rlt::DecodeParams p{};
    const int64_t off = bank * bank_elems(pool);
    p.k_bank = static_cast<const uint16_t *>(pool->k) + off;
    p.v_bank = static_cast<const uint16_t *>(pool->v) + off;
    p.q = static_cast<const uint16_t *>(q);
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.out = static_cast<uint16_t *>(out);
    p.lse_out = lse_out;
    p.lse_part = static_cast<float *>(workspace);
    p.o_part = workspace != nullptr
                   ? reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.lse_part_bytes)
                   : nullptr;
    p.err = err;
    p.num_pages = pool->num_pages;
    p.num_kv_heads = pool->num_kv_heads;
    p.num_q_heads = num_q_heads;
    p.page_size = pool->page_size;
    p.max_pages = max_pages;
    p.batch = batch;
    p.tiles_per_split = plan.tiles_per_split;
    p.max_splits = plan.max_splits;
    p.part_stride = plan.max_splits;
    const double s = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)pool->head_dim);
    p.qscale = (float)(s * 1.4426950408889634);   // log2(e): softmax in base 2
    if (t_fault_wait_ns != 0) {                   // armed by rlt_debug_fault_next_decode
        p.wait_limit_ns = t_fault_wait_ns;
        p.debug_drop_copy = 1;
        t_fault_wait_ns = 0;
    }
    return from_cuda(rlt::launch_decode(p, pool->head_dim, group, static_cast<cudaStream_t>(stream),
                                        (flags & RLT_ATTN_EARLY_START) != 0));
}

// Tensor-core CTAs of a shared-prefix call whose unshared rests run on the split-K kernel at
// the same time: SMs in proportion to the two kernels' tokens (the rest's length is its
// longest, 3/4 of it on average), weighted 9:4 for the tensor-core kernel's lower rate per
// SM on the short runs a split plan leaves it; then as few as keep the same number of items
// on the busiest CTA, so that the items spread evenly (measured on the huginn shape: 96
// items on 72 CTAs 32.0 us per call, on 64 CTAs with 64 items 27.9).
static int tc_share_ctas(int64_t items, int work_units, int chunk_tiles, int32_t batch, int32_t max_rest_len, int sms)
{
    const double pre = (double)work_units * chunk_tiles * rlt::kPrefixTile;
    const double rest = 0.75 * (double)batch * max_rest_len;
    const double share = std::min(1.0, 2.25 * pre / (pre + rest));
    int ctas = std::max(1, std::min(sms - 1, (int)std::ceil(sms * share)));
    if (items > 0) {
        const int64_t per = (items + ctas - 1) / ctas;
        ctas = (int)std::max<int64_t>(1, (items + per - 1) / per);
    }
    return ctas;
}

// Per-CTA costs of the tensor-core kernel measured on GB300 with every SM streaming: one
// 128-token sub-tile in steady state, and the hand-over from one run (kv head, segment,
// member block) to the next.
constexpr double kTcSubTileUs = 1.55;
constexpr double kTcRunUs = 4.7;

RLT_API int32_t rlt_choose_chunk_tiles(const int32_t *page_table, int32_t max_pages,
                                                  const int32_t *seq_lens, int32_t batch,
                                                  int32_t page_size, int32_t query_group,
                                                  int32_t private_tails, int32_t num_kv_heads,
                                                  int32_t num_ctas)
{
    if (batch < 0 || num_kv_heads < 1 || num_ctas < 1 || query_group < 1 || query_group > 128)
        return -RLT_ERR_INVALID_ARG;
    std::vector<int32_t> seg, mem, lim, req(2 * (size_t)std::max(batch, 1));
    int32_t sizes[7] = {0, 0, 0, 0, 0, 0, 0};
    auto plan = [&](int chunk) -> rlt_status {
        size_t seg_cap = 2 * (size_t)batch + 1, mem_cap = 4 * (size_t)batch + 1;
        for (int attempt = 0; attempt < 2; ++attempt) {
            seg.assign(seg_cap * rlt::kSegFields, 0);
            mem.assign(mem_cap, 0);
            lim.assign(mem_cap, 0);
            const rlt_status st = rlt_plan_prefix(page_table, max_pages, seq_lens, batch, page_size, chunk,
                                                  query_group, private_tails, seg.data(), (int32_t)seg_cap,
                                                  mem.data(), lim.data(), (int32_t)mem_cap, req.data(), sizes);
            if (st != RLT_ERR_OUT_OF_RANGE)
                return st;
            seg_cap = std::max(sizes[0], 1);
            mem_cap = std::max(sizes[1], 1);
        }
        return RLT_ERR_OUT_OF_RANGE;
    };
    rlt_status st = plan(1);
    if (st != RLT_OK)
        return -st;
    const int per_block = 128 / query_group;
    int longest = 1;
    int64_t tiles = 0;
    for (int s = 0; s < sizes[0]; ++s) {
        const int32_t *sd = &seg[(size_t)s * rlt::kSegFields];
        longest = std::max(longest, (int)sd[rlt::kSegNumTiles]);
        tiles += (int64_t)sd[rlt::kSegNumTiles] * ((sd[rlt::kSegMemberCount] + per_block - 1) / per_block);
    }
    tiles *= num_kv_heads;
    if (!private_tails) {
        // A split-K kernel shares the SMs (tc_share_ctas gives the tensor-core kernel its
        // CTAs): take the chunk (2..16 tiles, at most the longest segment) that leaves the
        // fewest 128-token sub-tiles on the busiest tensor-core CTA, the larger on a tie
        // (fewer runs, fewer partials).
        int best = std::min(2, longest), best_load = -1;
        for (int chunk = 2; chunk <= std::min(16, longest); ++chunk) {
            if ((st = plan(chunk)) != RLT_OK)
                return -st;
            const int64_t items = (int64_t)num_kv_heads * sizes[6];
            const int ctas = num_ctas > 1 ? tc_share_ctas(items, sizes[6], chunk, batch, sizes[5], num_ctas)
                                          : 1;
            const int64_t load = (items + ctas - 1) / ctas * chunk;
            if (best_load < 0 || load <= best_load) {
                best_load = (int)load;
                best = chunk;
            }
        }
        return std::max(1, best);
    }
    // The tensor-core kernel does the whole call, one CTA per SM, each taking a contiguous
    // run of items: the call ends with the busiest CTA.  Estimate each CTA's busy time from
    // the plan and take the chunk (4..16) with the smallest maximum, the larger on a tie.
    struct Unit {
        int s, mb, tiles;
    };
    int best_chunk = 4;
    double best_cost = -1.0;
    for (int chunk = 4; chunk <= 16; ++chunk) {
        if ((st = plan(chunk)) != RLT_OK)
            return -st;
        std::vector<Unit> units;
        for (int s = 0; s < sizes[0]; ++s) {
            const int32_t *sd = &seg[(size_t)s * rlt::kSegFields];
            const int n = sd[rlt::kSegNumTiles], mc = sd[rlt::kSegMemberCount];
            const int nch = std::max(1, (n + chunk - 1) / chunk);
            for (int mb = 0; mb < (mc + per_block - 1) / per_block; ++mb)
                for (int c = 0; c < nch; ++c)
                    units.push_back({s, mb, std::min(chunk, n - c * chunk)});
        }
        const int64_t n_items = (int64_t)units.size() * num_kv_heads;
        if (n_items == 0)
            continue;
        const int64_t ctas = std::min<int64_t>(num_ctas, n_items);
        double worst = 0.0;
        for (int64_t c = 0; c < ctas; ++c) {
            const int64_t i0 = c * n_items / ctas, i1 = (c + 1) * n_items / ctas;
            int64_t run_key = -1, runs = 0, t = 0;
            for (int64_t i = i0; i < i1; ++i) {
                const Unit &u = units[(size_t)(i % (int64_t)units.size())];
                const int64_t key = ((i / (int64_t)units.size()) * (sizes[0] + 1) + u.s) * 4096 + u.mb;
                t += u.tiles;
                if (key != run_key) {
                    run_key = key;
                    ++runs;
                }
            }
            worst = std::max(worst, t * kTcSubTileUs + runs * kTcRunUs);
        }
        if (best_cost < 0.0 || worst <= best_cost + 1e-9) {
            best_cost = worst;
            best_chunk = chunk;
        }
    }
    return std::min(best_chunk, longest);
}

RLT_API size_t rlt_paged_decode_prefix_workspace_size(int32_t batch, int32_t num_q_heads,
                                                      int32_t num_kv_heads, int32_t head_dim,
                                                      int32_t max_rest_len, int32_t max_prefix_slots,
                                                      int32_t split_tokens)
{
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || max_rest_len < 0 ||
        max_prefix_slots < 0 || split_tokens < 0)
        return 0;
    const rlt::DecodePlan plan = rlt::plan_decode(batch, num_q_heads, num_kv_heads, head_dim,
                                                  max_rest_len, split_tokens, current_sms(), rlt::kRestWaves);
    const size_t rows = (size_t)batch * num_q_heads * (size_t)(max_prefix_slots + plan.max_splits);
    return (rows * sizeof(float) + 255) / 256 * 256 + rows * head_dim * sizeof(float);
}

RLT_API rlt_status rlt_paged_decode_attn_prefix(
    const rlt_kv_pool *pool, int32_t bank, const void *q, const void *k_new, const void *v_new,
    int32_t num_q_heads,
    const int32_t *page_table, int32_t max_pages, const int32_t *seq_lens, int32_t batch,
    int32_t max_seq_len, const int32_t *segments, const int32_t *members,
    const int32_t *member_limit, const int32_t *request_prefix, int32_t num_segments, int32_t work_units,
    int32_t max_prefix_slots, int32_t chunk_tiles, int32_t max_rest_len, float scale, void *out,
    float *lse_out, void *workspace, size_t workspace_bytes, int32_t split_tokens, int32_t max_ctas,
    uint32_t flags, void *stream)
{
    if (max_ctas < 0 || (flags & ~RLT_ATTN_EARLY_START) != 0)
        return RLT_ERR_INVALID_ARG;
    if (num_segments == 0)      // nothing shared: the plain kernel computes the same thing
        return rlt_paged_decode_attn(pool, bank, q, k_new, v_new, num_q_heads, page_table, max_pages, seq_lens,
                                     batch, max_seq_len, scale, out, lse_out, workspace,
                                     workspace_bytes, split_tokens, flags, stream);
    rlt_status st = check_pool(pool, bank);
    if (st != RLT_OK)
        return st;
    if (batch < 0 || max_seq_len < 0 || max_pages < 1 || num_q_heads < 1 || split_tokens < 0 ||
        split_tokens % rlt::kTileTokens != 0 || split_tokens > 128 * rlt::kTileTokens ||
        num_segments < 0 || work_units < 0 || max_prefix_slots < 0 ||
        chunk_tiles < 1 || max_rest_len < 0 || max_rest_len > max_seq_len ||
        num_q_heads % pool->num_kv_heads != 0)
        return RLT_ERR_INVALID_ARG;
    const int group = num_q_heads / pool->num_kv_heads;
    if (!rlt::decode_supported(pool->head_dim, group) || pool->page_size % rlt::kTileTokens != 0 ||
        !rlt::prefix_supported(pool->head_dim, group, pool->page_size) || batch > 65535 ||
        pool->num_kv_heads > 65535)
        return RLT_ERR_UNSUPPORTED;
    if (q == nullptr || page_table == nullptr || seq_lens == nullptr || out == nullptr ||
        segments == nullptr || members == nullptr || member_limit == nullptr || request_prefix == nullptr ||
        workspace == nullptr)
        return RLT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) || !std::isfinite(scale))
        return RLT_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr) || !aligned16(k_new) || !aligned16(v_new))
        return RLT_ERR_INVALID_ARG;
    if (validate_enabled() &&
        (st = validate_attention_batch(page_table, max_pages, seq_lens, batch, pool->num_pages, pool->page_size,
                                       k_new != nullptr, static_cast<cudaStream_t>(stream))) != RLT_OK)
        return st;
    const int64_t bank_rows = pool->num_pages * pool->num_kv_heads * (int64_t)pool->page_size;
    if (bank_rows >= (int64_t(1) << 31))
        return RLT_ERR_UNSUPPORTED;

    unsigned int *err = nullptr;
    int sms = 0;
    if ((st = device_info(&err, &sms)) != RLT_OK)
        return st;
    // the split-K grid covers only what the segments leave: at most max_rest_len tokens
    const rlt::DecodePlan plan = rlt::plan_decode(batch, num_q_heads, pool->num_kv_heads,
                                                  pool->head_dim, max_rest_len, split_tokens, sms, rlt::kRestWaves);
    const int32_t stride = max_prefix_slots + plan.max_splits;
    const size_t rows = (size_t)batch * num_q_heads * stride;
    const size_t lse_bytes = (rows * sizeof(float) + 255) / 256 * 256;
    if (workspace_bytes < lse_bytes + rows * pool->head_dim * sizeof(float))
        return RLT_ERR_WORKSPACE_TOO_SMALL;

    rlt::DecodeParams p{};
    const int64_t off = bank * bank_elems(pool);
    p.k_bank = static_cast<const uint16_t *>(pool->k) + off;
    p.v_bank = static_cast<const uint16_t *>(pool->v) + off;
    p.q = static_cast<const uint16_t *>(q);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.out = static_cast<uint16_t *>(out);
    p.lse_out = lse_out;
    p.lse_part = static_cast<float *>(workspace);
    p.o_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + lse_bytes);
    p.err = err;
    p.num_pages = pool->num_pages;
    p.num_kv_heads = pool->num_kv_heads;
    p.num_q_heads = num_q_heads;
    p.page_size = pool->page_size;
    p.max_pages = max_pages;
    p.batch = batch;
    p.tiles_per_split = plan.tiles_per_split;
    p.max_splits = plan.max_splits;
    const double s = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)pool->head_dim);
    p.qscale = (float)(s * 1.4426950408889634);
    p.request_prefix = request_prefix;
    p.prefix_slots = max_prefix_slots;
    p.part_stride = stride;

    rlt::PrefixParams pp{};
    pp.segments = segments;
    pp.members = members;
    pp.member_limit = member_limit;
    pp.num_rows = batch;
    pp.num_segments = num_segments;
    pp.chunk_tiles = chunk_tiles;
    pp.work_units = work_units;
    const int64_t items = (int64_t)pool->num_kv_heads * work_units;
    int ctas = sms;
    if (max_ctas > 0) {
        ctas = std::min(max_ctas, sms);
    } else if (max_rest_len > 0 && sms > 1) {
        ctas = tc_share_ctas(items, work_units, chunk_tiles, batch, max_rest_len, sms);
    }
    pp.ctas = (int32_t)std::min<int64_t>(ctas, items);
    // L2 prefetch ahead of the copy rings when a split-K rest shares the SMs (measured on the
    // huginn call: 25.25 -> 24.79 us; on the long-context call, whose CTAs stream long runs,
    // 112.9 -> 138.1 us, so not there)
    pp.l2_ahead = max_rest_len > 0 ? 1 : 0;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    // Early start: both partial kernels are programmatic dependents of what precedes the call
    // (under stream capture the fork and the join become programmatic graph edges), and the
    // combine of what they leave.
    const bool early = (flags & RLT_ATTN_EARLY_START) != 0;
    // Fused append: the kernel whose copy covers a request's newest token stores the new
    // rows on the way -- the split-K kernel for an unshared rest, the tensor-core kernel
    // for a private tail -- and flags a newest token inside shared tiles.
    rlt::DecodeParams p_rest = p;
    if (k_new != nullptr) {
        rlt::DecodeParams &q = max_rest_len > 0 ? p_rest : p;
        q.k_new = static_cast<const uint16_t *>(k_new);
        q.v_new = static_cast<const uint16_t *>(v_new);
    }
    if (max_rest_len > 0) {
        SideStream *side = nullptr;
        if ((st = side_stream(&side)) != RLT_OK)
            return st;
        // The tensor-core kernel starts early on the caller's stream (a plain programmatic
        // dependence on the kernel ahead); the split-K rest runs on the side stream with an
        // ordinary, complete dependence on what precedes the call.  Measured on GB300: a kernel
        // started programmatically across the fork starts no earlier than after the kernel ahead
        // completes and keeps the combine from starting early behind it; and with the split-K
        // grid started early its CTAs take every SM the previous call frees, so the tensor-core
        // CTAs (a whole SM each) wait until they drain.
        e = cudaEventRecord(side->fork, cs);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(side->stream, side->fork, 0);
        if (e == cudaSuccess)
            e = rlt::launch_prefix(p, pp, p.k_bank, p.v_bank, bank_rows, cs, early);
        if (e == cudaSuccess)
            e = rlt::launch_decode(p_rest, pool->head_dim, group, side->stream, false);
        if (e == cudaSuccess)
            e = cudaEventRecord(side->join, side->stream);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(cs, side->join, 0);
    } else {
        e = rlt::launch_prefix(p, pp, p.k_bank, p.v_bank, bank_rows, cs, early);
    }
    if (e == cudaSuccess)
        e = rlt::launch_combine(p, pool->head_dim, cs);
    return from_cuda(e);
}

RLT_API size_t rlt_paged_extend_workspace_size(int32_t num_rows, int32_t num_q_heads, int32_t head_dim,
                                               int32_t max_slots)
{
    if (num_rows < 0 || num_q_heads < 1 || head_dim < 1 || max_slots < 0)
        return 0;
    const size_t n = (size_t)num_rows * num_q_heads * max_slots;
    return (n * sizeof(float) + 255) / 256 * 256 + n * head_dim * sizeof(float);
}

RLT_API rlt_status rlt_paged_extend_attn(
    const rlt_kv_pool *pool, int32_t bank, const void *q, int32_t num_q_heads, int32_t num_rows,
    const int32_t *page_table, int32_t max_pages, int32_t batch, const int32_t *segments,
    const int32_t *members, const int32_t *member_limit, const int32_t *row_prefix, const int32_t *row_len,
    int32_t num_segments, int32_t work_units, int32_t max_slots, int32_t chunk_tiles, float scale, void *out,
    float *lse_out, void *workspace, size_t workspace_bytes, int32_t max_ctas, uint32_t flags, void *stream)
{
    rlt_status st = check_pool(pool, bank);
    if (st != RLT_OK)
        return st;
    if (num_rows < 0 || batch < 0 || max_pages < 1 || num_q_heads < 1 || num_segments < 0 || work_units < 0 ||
        max_slots < 0 || chunk_tiles < 1 || max_ctas < 0 || num_q_heads % pool->num_kv_heads != 0 ||
        !std::isfinite(scale) || (flags & ~RLT_ATTN_EARLY_START) != 0)
        return RLT_ERR_INVALID_ARG;
    if (num_rows == 0 || num_segments == 0)
        return RLT_OK;
    const int group = num_q_heads / pool->num_kv_heads;
    if (!rlt::prefix_supported(pool->head_dim, group, pool->page_size) || pool->num_kv_heads > 65535)
        return RLT_ERR_UNSUPPORTED;
    if (q == nullptr || page_table == nullptr || out == nullptr || segments == nullptr || members == nullptr ||
        member_limit == nullptr || row_prefix == nullptr || row_len == nullptr || workspace == nullptr ||
        max_slots < 1)
        return RLT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace))
        return RLT_ERR_INVALID_ARG;
    if (workspace_bytes < rlt_paged_extend_workspace_size(num_rows, num_q_heads, pool->head_dim, max_slots))
        return RLT_ERR_WORKSPACE_TOO_SMALL;
    const int64_t bank_rows = pool->num_pages * pool->num_kv_heads * (int64_t)pool->page_size;
    if (bank_rows >= (int64_t(1) << 31))
        return RLT_ERR_UNSUPPORTED;
    unsigned int *err = nullptr;
    int sms = 0;
    if ((st = device_info(&err, &sms)) != RLT_OK)
        return st;
    const size_t n = (size_t)num_rows * num_q_heads * max_slots;
    rlt::DecodeParams p{};
    const int64_t off = bank * bank_elems(pool);
    p.k_bank = static_cast<const uint16_t *>(pool->k) + off;
    p.v_bank = static_cast<const uint16_t *>(pool->v) + off;
    p.q = static_cast<const uint16_t *>(q);
    p.page_table = page_table;
    p.out = static_cast<uint16_t *>(out);
    p.lse_out = lse_out;
    p.lse_part = static_cast<float *>(workspace);
    p.o_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + (n * sizeof(float) + 255) / 256 * 256);
    p.err = err;
    p.num_pages = pool->num_pages;
    p.num_kv_heads = pool->num_kv_heads;
    p.num_q_heads = num_q_heads;
    p.page_size = pool->page_size;
    p.max_pages = max_pages;
    p.batch = batch;                     // requests: page-table rows
    p.tiles_per_split = 1;
    p.max_splits = 1;
    const double s = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)pool->head_dim);
    p.qscale = (float)(s * 1.4426950408889634);
    p.prefix_slots = max_slots;
    p.part_stride = max_slots;

    rlt::PrefixParams pp{};
    pp.segments = segments;
    pp.members = members;
    pp.member_limit = member_limit;
    pp.num_rows = num_rows;
    pp.num_segments = num_segments;
    pp.chunk_tiles = chunk_tiles;
    pp.work_units = work_units;
    pp.ctas = (int32_t)std::min<int64_t>(max_ctas > 0 ? std::min(max_ctas, sms) : sms,
                                         (int64_t)pool->num_kv_heads * work_units);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = rlt::launch_prefix(p, pp, p.k_bank, p.v_bank, bank_rows, cs,
                                       (flags & RLT_ATTN_EARLY_START) != 0);
    if (e == cudaSuccess) {
        // the merge runs over the new tokens: each row's "request" is its causal prefix
        rlt::DecodeParams pc = p;
        pc.batch = num_rows;
        pc.seq_lens = row_len;
        pc.request_prefix = row_prefix;
        e = rlt::launch_combine(pc, pool->head_dim, cs);
    }
    return from_cuda(e);
}

RLT_API rlt_status rlt_latent_noise_init(float *out, const uint64_t *seeds,
                                         const int64_t *positions, int64_t n_rows,
                                         int32_t channels, float initializer_range, void *stream)
{
    if (n_rows < 0 || channels < 1 || !std::isfinite(initializer_range))
        return RLT_ERR_INVALID_ARG;
    if (n_rows == 0)
        return RLT_OK;
    if (out == nullptr || seeds == nullptr || positions == nullptr)
        return RLT_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(out) % 4 != 0 || reinterpret_cast<uintptr_t>(seeds) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(positions) % 8 != 0)
        return RLT_ERR_INVALID_ARG;
    return from_cuda(rlt::launch_noise(out, nullptr, seeds, positions, n_rows, channels,
                                       initializer_range, static_cast<cudaStream_t>(stream)));
}

RLT_API rlt_status rlt_noise_hash24(uint32_t *out, const uint64_t *seeds, const int64_t *positions,
                                    int64_t n_rows, int32_t channels, void *stream)
{
    if (n_rows < 0 || channels < 1)
        return RLT_ERR_INVALID_ARG;
    if (n_rows == 0)
        return RLT_OK;
    if (out == nullptr || seeds == nullptr || positions == nullptr)
        return RLT_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(out) % 4 != 0 || reinterpret_cast<uintptr_t>(seeds) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(positions) % 8 != 0)
        return RLT_ERR_INVALID_ARG;
    return from_cuda(rlt::launch_noise(nullptr, out, seeds, positions, n_rows, channels, 0.f,
                                       static_cast<cudaStream_t>(stream)));
}

RLT_API rlt_status rlt_paged_gather(const rlt_kv_pool *pool, int32_t bank,
                                    const int32_t *page_table, int32_t max_pages,
                                    const int32_t *seq_lens, int32_t batch, int32_t max_len,
                                    void *k_out, void *v_out, void *stream)
{
    rlt_status st = check_pool(pool, bank);
    if (st != RLT_OK)
        return st;
    if (batch < 0 || max_len < 0 || max_pages < 0)
        return RLT_ERR_INVALID_ARG;
    if (batch == 0 || max_len == 0)
        return RLT_OK;
    if (page_table == nullptr || seq_lens == nullptr || k_out == nullptr || v_out == nullptr ||
        max_pages < 1)
        return RLT_ERR_INVALID_ARG;
    if (!aligned16(k_out) || !aligned16(v_out))
        return RLT_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    if ((st = device_info(&err, nullptr)) != RLT_OK)
        return st;
    const int64_t off = bank * bank_elems(pool);
    return from_cuda(rlt::launch_gather(
        static_cast<const uint16_t *>(pool->k) + off, static_cast<const uint16_t *>(pool->v) + off,
        page_table, max_pages, seq_lens, batch, max_len, static_cast<uint16_t *>(k_out),
        static_cast<uint16_t *>(v_out), pool->num_kv_heads, pool->page_size, pool->head_dim,
        pool->num_pages, err, static_cast<cudaStream_t>(stream)));
}

RLT_API rlt_status rlt_validate_batch(const int32_t *page_table, int32_t max_pages,
                                      const int32_t *seq_lens, int32_t batch,
                                      const int64_t *new_slots, int64_t num_pages,
                                      int32_t page_size)
{
    if (batch < 0 || max_pages < 0 || num_pages < 0 || page_size < 1)
        return RLT_ERR_INVALID_ARG;
    if (batch == 0)
        return RLT_OK;
    if (page_table == nullptr || seq_lens == nullptr)
        return RLT_ERR_INVALID_ARG;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t L = seq_lens[b];
        if (L < 0 || L > (int64_t)max_pages * page_size)
            return RLT_ERR_OUT_OF_RANGE;
        const int64_t n = (L + page_size - 1) / page_size;
        for (int64_t i = 0; i < n; ++i) {
            const int64_t page = page_table[(int64_t)b * max_pages + i];
            if (page < 0 || page >= num_pages)
                return RLT_ERR_OUT_OF_RANGE;
        }
    }
    if (new_slots == nullptr)
        return RLT_OK;
    std::unordered_set<int64_t> slots, write_pages;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t slot = new_slots[b];
        if (slot < 0)
            continue;
        const int64_t L = seq_lens[b];
        if (L < 1 || slot >= num_pages * page_size)
            return RLT_ERR_OUT_OF_RANGE;
        const int64_t last_page = page_table[(int64_t)b * max_pages + (L - 1) / page_size];
        if (slot / page_size != last_page || slot % page_size != (L - 1) % page_size)
            return RLT_ERR_OUT_OF_RANGE;
        if (!slots.insert(slot).second)
            return RLT_ERR_INVALID_ARG;            // two requests append to one slot
        write_pages.insert(last_page);
    }
    // A page that receives a new token must belong to exactly one request.
    std::unordered_set<int64_t> seen_in_request;
    std::unordered_set<int64_t> owned;
    for (int32_t b = 0; b < batch; ++b) {
        seen_in_request.clear();
        const int64_t n = ((int64_t)seq_lens[b] + page_size - 1) / page_size;
        for (int64_t i = 0; i < n; ++i) {
            const int64_t page = page_table[(int64_t)b * max_pages + i];
            if (write_pages.count(page) == 0 || !seen_in_request.insert(page).second)
                continue;
            if (!owned.insert(page).second)
                return RLT_ERR_INVALID_ARG;        // append into a shared (read-only) page
        }
    }
    return RLT_OK;
}

RLT_API rlt_status rlt_debug_fault_next_decode(uint64_t wait_limit_ns)
{
    if (wait_limit_ns == 0 || wait_limit_ns > rlt::kMaxFaultWaitNs)
        return RLT_ERR_INVALID_ARG;
    t_fault_wait_ns = wait_limit_ns;
    return RLT_OK;
}

RLT_API rlt_status rlt_get_device_error(uint32_t *error_bits)
{
    if (error_bits == nullptr)
        return RLT_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return RLT_ERR_CUDA;
    unsigned int *err = nullptr;
    rlt_status st = device_info(&err, nullptr);
    if (st != RLT_OK)
        return st;
    unsigned int v = 0;
    if (cudaMemcpy(&v, err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return RLT_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return RLT_ERR_CUDA;
    *error_bits = v;
    return RLT_OK;
}

}  // extern "C"
