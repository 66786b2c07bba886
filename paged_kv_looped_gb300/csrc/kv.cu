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

// ------------------------------------------------------- RoPE + append
//
// "Faster fuzzy minds", "Recurrent depth": a token keeps one RoPE position
// across all T of its banks, so every plane's append of a token rotates its key
// by the same angles: the token's sequence position times the pair frequency
// base^(-2i/rot_dim), pairs (i, i + rot_dim/2).  The angle is formed and
// reduced mod 2 pi in fp64 (positions reach 1e5 and more, where an fp32
// product would be off by ~1e-2 rad); sin/cos and the rotation are fp32, the
// result is rounded to bf16 once.  One warp per (token, kv head).

namespace {

constexpr double kTwoPiHi = 6.283185307179586;          // 2 pi as a double
constexpr double kTwoPiLo = 2.4492935982947064e-16;     // 2 pi minus kTwoPiHi
constexpr double kInvTwoPi = 0.15915494309189535;

__global__ void __launch_bounds__(256)
    append_rope_kernel(uint16_t *__restrict__ k_bank, uint16_t *__restrict__ v_bank,
                       const uint16_t *__restrict__ k_new, const uint16_t *__restrict__ v_new,
                       const int64_t *__restrict__ positions, const int64_t *__restrict__ out_loc,
                       int32_t n_tokens, int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                       int32_t rot_dim, double log2_base, int64_t num_slots,
                       const int32_t *__restrict__ request, int32_t *__restrict__ written, int32_t batch,
                       unsigned int *err)
{
    extern __shared__ double inv_freq[];     // [rot_dim / 2]
    const int half = rot_dim / 2;
    for (int i = threadIdx.x; i < half; i += blockDim.x)
        inv_freq[i] = exp2(-2.0 * i / rot_dim * log2_base);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t items = (int64_t)n_tokens * num_kv_heads;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < items; w += warps) {
        const int64_t i = w / num_kv_heads;
        const int g = (int)(w - i * num_kv_heads);
        const int64_t slot = out_loc[i];
        if (slot < 0)
            continue;                            // no token for this entry
        if (slot >= num_slots) {
            if (lane == 0 && g == 0)
                record_error(err, RLT_DEVERR_BAD_SLOT);
            continue;
        }
        const int64_t pos = positions[i];
        const int64_t page = slot / page_size;
        const int64_t dst = ((page * num_kv_heads + g) * page_size + (slot - page * page_size)) * head_dim;
        const int64_t src = (i * num_kv_heads + g) * head_dim;
        // V: the row as 16-byte vectors
        for (int c = lane; c < head_dim / 8; c += 32)
            reinterpret_cast<uint4 *>(v_bank + dst)[c] = reinterpret_cast<const uint4 *>(v_new + src)[c];
        // K: rotated pairs, then the dims past rot_dim unchanged
        for (int p = lane; p < half; p += 32) {
            double a = (double)pos * inv_freq[p];
            const double k = rint(a * kInvTwoPi);
            a = fma(-k, kTwoPiHi, a);
            a = fma(-k, kTwoPiLo, a);
            float s, c;
            sincosf((float)a, &s, &c);
            const float x = __uint_as_float((uint32_t)k_new[src + p] << 16);
            const float y = __uint_as_float((uint32_t)k_new[src + p + half] << 16);
            k_bank[dst + p] = (uint16_t)bf16_bits(fmaf(x, c, -y * s));
            k_bank[dst + p + half] = (uint16_t)bf16_bits(fmaf(x, s, y * c));
        }
        for (int d = rot_dim + lane; d < head_dim; d += 32)
            k_bank[dst + d] = k_new[src + d];
        if (written != nullptr && g == 0 && lane == 0) {
            const int32_t r = request[i];
            if (r >= 0 && r < batch)
                atomicMax(&written[r], (int32_t)min(pos + 1, (int64_t)INT32_MAX));
            else
                record_error(err, RLT_DEVERR_BAD_SLOT);
        }
    }
}

// out[b] = min over banks of written[bank][b], floored to whole pages (0 with no bank).
__global__ void __launch_bounds__(256)
    publishable_kernel(const int32_t *__restrict__ written, int32_t num_banks, int32_t batch,
                       int32_t page_size, int32_t *__restrict__ out)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch)
        return;
    int32_t m = num_banks > 0 ? INT32_MAX : 0;
    for (int bank = 0; bank < num_banks; ++bank)
        m = min(m, written[(int64_t)bank * batch + b]);
    m = max(m, 0);
    out[b] = m / page_size * page_size;
}

}  // namespace

cudaError_t launch_append_rope(uint16_t *k_bank, uint16_t *v_bank, const uint16_t *k_new,
                               const uint16_t *v_new, const int64_t *positions, const int64_t *out_loc,
                               int32_t n_tokens, int32_t num_kv_heads, int32_t page_size,
                               int32_t head_dim, int64_t num_pages, int32_t rot_dim, double rope_base,
                               const int32_t *request, int32_t *written, int32_t batch,
                               unsigned int *err, cudaStream_t stream)
{
    const int64_t warps = (int64_t)n_tokens * num_kv_heads;
    int64_t blocks = (warps + 7) / 8;
    if (blocks > 65536 * 4)
        blocks = 65536 * 4;
    append_rope_kernel<<<(unsigned)blocks, 256, (rot_dim / 2) * sizeof(double), stream>>>(
        k_bank, v_bank, k_new, v_new, positions, out_loc, n_tokens, num_kv_heads, page_size, head_dim,
        rot_dim, log2(rope_base), num_pages * page_size, request, written, batch, err);
    return cudaGetLastError();
}

cudaError_t launch_publishable(const int32_t *written, int32_t num_banks, int32_t batch,
                               int32_t page_size, int32_t *out, cudaStream_t stream)
{
    publishable_kernel<<<(unsigned)((batch + 255) / 256), 256, 0, stream>>>(written, num_banks, batch,
                                                                              page_size, out);
    return cudaGetLastError();
}

}  // namespace rlt
