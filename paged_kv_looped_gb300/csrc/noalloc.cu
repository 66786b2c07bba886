// rlt_paged_decode_attn_noalloc: paged decode attention whose split-K scratch
// lives in a fixed array inside this library instead of caller-provided memory.
//
// For callers that cannot allocate device memory when they need attention:
// plugins whose host framework owns every device allocation, and latency-bound
// decode loops where a cudaMalloc (which may synchronise the whole device)
// would stall other streams.  They pass inputs and outputs only.
//
// The array is a file-scope __device__ object, so it exists once per device
// that loads this module and stays until the process exits.  Host code cannot
// use its name as a device address: the address is looked up once per device
// with cudaGetSymbolAddress, with that device current, and handed to the
// kernels.  Nothing in it needs clearing between calls: every partial a call
// reads was written earlier in the same call.  All calls on a device share the
// one array, so calls that overlap on the GPU (different streams, or other
// threads) race on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "rlt.h"
#include "rlt_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RLT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (set-up on the
// first call per device).
rlt_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return RLT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return RLT_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return RLT_OK;
}

}  // namespace

extern "C" RLT_API rlt_status rlt_paged_decode_attn_noalloc(
    const rlt_kv_pool *pool, int32_t bank, const void *q, int32_t num_q_heads,
    const int32_t *page_table, int32_t max_pages, const int32_t *seq_lens, int32_t batch,
    int32_t max_seq_len, float scale, void *out, float *lse_out, int32_t split_tokens, void *stream)
{
    // the same checks, in the same order, as rlt_paged_decode_attn before the scratch size
    bool empty = false;
    const rlt_status arg = rlt::check_decode_args(pool, bank, q, nullptr, nullptr, num_q_heads, page_table,
                                                  max_pages, seq_lens, batch, max_seq_len, scale, out,
                                                  split_tokens, &empty);
    if (arg != RLT_OK || empty)
        return arg;
    const size_t need = rlt_paged_decode_workspace_size(batch, num_q_heads, pool->num_kv_heads,
                                                        pool->head_dim, max_seq_len, split_tokens);
    if (need > (size_t)RLT_NOALLOC_SCRATCH_BYTES)
        return RLT_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    if (need > 0) {
        const rlt_status st = scratch_address(&scratch);
        if (st != RLT_OK)
            return st;
    }
    return rlt_paged_decode_attn(pool, bank, q, nullptr, nullptr, num_q_heads, page_table, max_pages, seq_lens, batch,
                                 max_seq_len, scale, out, lse_out, scratch,
                                 need > 0 ? (size_t)RLT_NOALLOC_SCRATCH_BYTES : 0, split_tokens, 0u,
                                 stream);
}
