// KV append (store_kv scatter) and page-table gather for sm_103a.
//
// "Faster fuzzy minds", "LOTUS": store_kv writes each token's K/V rows to
// whatever physical slots it is handed, so overwrite-in-place is the same call
// with the same slots.  "When scheduler does the work": a token at logical
// position p of request b lives at page page_table[b][p / ps], offset p % ps.
//
// Both kernels move 16-byte vectors, one per thread, with consecutive threads
// on consecutive vectors of a row (D*2 bytes = 8 or 16 vectors), so every row
// is a run of full 32-byte sectors.
#include "rlt_device.cuh"
#include "rlt_internal.h"

namespace rlt {
namespace {

__global__ void __launch_bounds__(256)
    append_kernel(uint4 *__restrict__ k_bank, uint4 *__restrict__ v_bank,
                  const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                  const int64_t *__restrict__ out_loc, int32_t n_tokens, int32_t num_kv_heads,
                  int32_t page_size, int32_t vec_per_row, int64_t num_slots, unsigned int *err)
{
    const int64_t per_token = (int64_t)num_kv_heads * vec_per_row;
    const int64_t total = (int64_t)n_tokens * per_token;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / per_token;
        const int64_t rem = idx - i * per_token;
        const int64_t slot = out_loc[i];
        if (slot < 0)
            continue;                            // no token for this entry
        if (slot >= num_slots) {
            if (rem == 0)
                record_error(err, RLT_DEVERR_BAD_SLOT);
            continue;
        }
        const int64_t g = rem / vec_per_row;
        const int64_t v = rem - g * vec_per_row;
        const int64_t page = slot / page_size;
        const int64_t off = slot - page * page_size;
        const int64_t dst = ((page * num_kv_heads + g) * page_size + off) * vec_per_row + v;
        k_bank[dst] = k_new[idx];
        v_bank[dst] = v_new[idx];
    }
}

__global__ void __launch_bounds__(256)
    gather_kernel(const uint4 *__restrict__ k_bank, const uint4 *__restrict__ v_bank,
                  const int32_t *__restrict__ page_table, int32_t max_pages,
                  const int32_t *__restrict__ seq_lens, int32_t batch, int32_t max_len,
                  uint4 *__restrict__ k_out, uint4 *__restrict__ v_out, int32_t num_kv_heads,
                  int32_t page_size, int32_t vec_per_row, int64_t num_pages, unsigned int *err)
{
    const int64_t per_pos = (int64_t)num_kv_heads * vec_per_row;
    const int64_t per_req = (int64_t)max_len * per_pos;
    const int64_t total = (int64_t)batch * per_req;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = idx / per_req;
        const int64_t rem = idx - b * per_req;
        const int64_t pos = rem / per_pos;
        const int64_t rem2 = rem - pos * per_pos;
        int64_t L = seq_lens[b];
        if (L > (int64_t)max_pages * page_size)
            L = (int64_t)max_pages * page_size;  // never read past the row
        if (pos >= L)
            continue;
        const int64_t page = page_table[b * max_pages + pos / page_size];
        if (page < 0 || page >= num_pages) {
            if (rem2 == 0)
                record_error(err, RLT_DEVERR_BAD_PAGE);
            continue;
        }
        const int64_t g = rem2 / vec_per_row;
        const int64_t v = rem2 - g * vec_per_row;
        const int64_t src =
            ((page * num_kv_heads + g) * page_size + pos % page_size) * vec_per_row + v;
        k_out[idx] = k_bank[src];
        v_out[idx] = v_bank[src];
    }
}

unsigned grid_for(int64_t threads)
{
    const int64_t blocks = (threads + 255) / 256;
    return (unsigned)(blocks < 65536 * 8 ? (blocks > 0 ? blocks : 1) : 65536 * 8);
}

}  // namespace

cudaError_t launch_append(uint16_t *k_bank, uint16_t *v_bank, const uint16_t *k_new,
                          const uint16_t *v_new, const int64_t *out_loc, int32_t n_tokens,
                          int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                          int64_t num_pages, unsigned int *err, cudaStream_t stream)
{
    const int32_t vpr = head_dim / 8;
    const int64_t total = (int64_t)n_tokens * num_kv_heads * vpr;
    append_kernel<<<grid_for(total), 256, 0, stream>>>(
        reinterpret_cast<uint4 *>(k_bank), reinterpret_cast<uint4 *>(v_bank),
        reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), out_loc,
        n_tokens, num_kv_heads, page_size, vpr, num_pages * page_size, err);
    return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t *k_bank, const uint16_t *v_bank,
                          const int32_t *page_table, int32_t max_pages, const int32_t *seq_lens,
                          int32_t batch, int32_t max_len, uint16_t *k_out, uint16_t *v_out,
                          int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                          int64_t num_pages, unsigned int *err, cudaStream_t stream)
{
    const int32_t vpr = head_dim / 8;
    const int64_t total = (int64_t)batch * max_len * num_kv_heads * vpr;
    gather_kernel<<<grid_for(total), 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k_bank), reinterpret_cast<const uint4 *>(v_bank),
        page_table, max_pages, seq_lens, batch, max_len, reinterpret_cast<uint4 *>(k_out),
        reinterpret_cast<uint4 *>(v_out), num_kv_heads, page_size, vpr, num_pages, err);
    return cudaGetLastError();
}

}  // namespace rlt
