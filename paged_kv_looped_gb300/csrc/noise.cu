// Position-keyed latent-state noise for sm_103a.
//
// vllm-rlt PR #152, Summary para 2: the latent state a token starts from depends
// on (request seed, position, channel) only.  SplitMix64 steps fold the three in
// one after another; the top 24 bits of the result pick a uniform cell, and the
// inverse CDF of a normal (std initializer_range) cut off at +-3 sigma turns it
// into the value.  The 64-bit arithmetic is exact mod 2^64 on either side, so
// the 24 bits agree bit for bit with a CPU computation.
//
// One stage and one erfinvf per value, written with coalesced 16-byte stores
// (noise_kernel); the seed and position stages are hashed once per 16 values.
// The work is integer/SFU arithmetic plus a write of 4 bytes per value; the
// per-channel stage is computed on 32-bit halves down to only the 24 bits that
// are kept (stage_top24).
#include "rlt_device.cuh"
#include "rlt_internal.h"

namespace rlt {
namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;   // SplitMix64 increment
constexpr int kChunk = 16;                              // channels per thread

// SplitMix64 output function (Steele, Lea & Flood 2014).
__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Fold key x into state h and advance one SplitMix64 step.
__device__ __forceinline__ uint64_t stage(uint64_t h, uint64_t x)
{
    return mix64((h ^ x) + kGolden);
}

// stage(h, x) >> 40, with 32-bit operations only where the result needs them.  The
// last xor-shift of mix64 (z ^= z >> 31) leaves bits 33..63 unchanged, so the top 24
// bits are those of the second product, and of that product only the high word is
// formed (high half of lo * lo plus the two cross terms, mod 2^32).
__device__ __forceinline__ uint32_t stage_top24(uint64_t h, uint64_t x)
{
    const uint64_t z0 = (h ^ x) + kGolden;
    uint32_t lo = (uint32_t)z0, hi = (uint32_t)(z0 >> 32);
    lo ^= __funnelshift_r(lo, hi, 30);                   // z ^= z >> 30
    hi ^= hi >> 30;
    const uint32_t a_lo = 0x1CE4E5B9u, a_hi = 0xBF58476Du;
    const uint64_t p = (uint64_t)lo * a_lo;              // z *= 0xBF58476D1CE4E5B9
    uint32_t nlo = (uint32_t)p;
    uint32_t nhi = (uint32_t)(p >> 32) + lo * a_hi + hi * a_lo;
    nlo ^= __funnelshift_r(nlo, nhi, 27);                // z ^= z >> 27
    nhi ^= nhi >> 27;
    const uint32_t b_lo = 0x133111EBu, b_hi = 0x94D049BBu;
    const uint32_t top = __umulhi(nlo, b_lo) + nlo * b_hi + nhi * b_lo;   // (z * 0x94D049BB133111EB) >> 32
    return top >> 8;
}

// Truncated-normal value of a 24-bit uniform h24: u = (h24 + 1/2) / 2^24 and
// x = amp * erfinv((2u - 1) * erf(3/sqrt 2)), amp = initializer_range * sqrt 2.
// (2u - 1) * 2^24 = 2*h24 + 1 - 2^24 is an odd integer below 2^24 in magnitude,
// exact in fp32, and so is its scaling by 2^-24.
__device__ __forceinline__ float truncnorm(uint32_t h24, float amp)
{
    const float erf3 = 0.99730020393673981f;             // erf(3 / sqrt(2))
    const float t = (float)((int)(2u * h24 + 1u) - (1 << 24)) * 0x1p-24f;
    return amp * erfinvf(t * erf3);
}

// A warp makes a tile of 512 channels of one row: lane l takes channels
// 128k + 4l .. 128k + 4l + 3 for k = 0..3, so each 16-byte store of the warp
// fills 512 contiguous bytes, and the seed and position stages are hashed once
// per 16 values.
constexpr int kTile = 512;

template <bool kHashOnly>
__global__ void __launch_bounds__(256)
    noise_kernel(float *__restrict__ out, uint32_t *__restrict__ hash_out,
                 const uint64_t *__restrict__ seeds, const int64_t *__restrict__ positions,
                 int64_t n_rows, int32_t channels, int32_t tiles_per_row, float amp, bool vec_ok)
{
    const int lane = threadIdx.x & 31;
    const int64_t total = n_rows * tiles_per_row;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < total; t += warps) {
        const int64_t r = t / tiles_per_row;
        const int32_t cb = (int32_t)(t - r * tiles_per_row) * kTile;
        const uint64_t h_row = stage(stage(0ull, seeds[r]), (uint64_t)positions[r]);
        const int64_t row_base = r * channels;
#pragma unroll
        for (int k = 0; k < kChunk / 4; ++k) {
            const int32_t c0 = cb + k * 128 + lane * 4;
            if (c0 >= channels)
                break;
            uint32_t h24[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                h24[i] = stage_top24(h_row, (uint64_t)(int64_t)(c0 + i));
            const bool full = vec_ok && c0 + 4 <= channels;
            if constexpr (kHashOnly) {
                if (full)
                    *reinterpret_cast<uint4 *>(hash_out + row_base + c0) = make_uint4(h24[0], h24[1], h24[2], h24[3]);
                else
                    for (int i = 0; i < 4 && c0 + i < channels; ++i)
                        hash_out[row_base + c0 + i] = h24[i];
            } else {
                float x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    x[i] = truncnorm(h24[i], amp);
                if (full)
                    *reinterpret_cast<float4 *>(out + row_base + c0) = make_float4(x[0], x[1], x[2], x[3]);
                else
                    for (int i = 0; i < 4 && c0 + i < channels; ++i)
                        out[row_base + c0 + i] = x[i];
            }
        }
    }
}

}  // namespace

cudaError_t launch_noise(float *out, uint32_t *hash_out, const uint64_t *seeds,
                         const int64_t *positions, int64_t n_rows, int32_t channels,
                         float initializer_range, cudaStream_t stream)
{
    const int32_t tiles = (channels + kTile - 1) / kTile;
    const int64_t threads = n_rows * tiles * 32;
    int64_t blocks = (threads + 255) / 256;
    if (blocks > 65536 * 8)
        blocks = 65536 * 8;
    if (blocks < 1)
        blocks = 1;
    const float amp = (float)((double)initializer_range * 1.4142135623730951);
    // 16-byte stores only where every row start is 16-byte aligned
    const void *dst = hash_out != nullptr ? (const void *)hash_out : (const void *)out;
    const bool vec_ok = channels % 4 == 0 && reinterpret_cast<uintptr_t>(dst) % 16 == 0;
    if (hash_out != nullptr)
        noise_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(
            nullptr, hash_out, seeds, positions, n_rows, channels, tiles, amp, vec_ok);
    else
        noise_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(
            out, nullptr, seeds, positions, n_rows, channels, tiles, amp, vec_ok);
    return cudaGetLastError();
}

}  // namespace rlt
