// Position-keyed latent-state noise for sm_103a.
//
// vllm-rlt PR #152, Summary para 2: each token's initial latent state is a
// function of (request seed, position, channel): a stage-wise SplitMix64-style
// hash gives a 24-bit uniform, and an inverse normal CDF maps it onto a normal
// with std = initializer_range truncated at +-3 sigma.  64-bit arithmetic wraps
// mod 2^64 exactly as on the CPU, so the 24 bits are identical everywhere.
//
// One thread makes 8 consecutive channels of one row: the seed and position
// stages are hashed once per thread, then one stage and one erfinvf per value,
// written as two 16-byte stores.  The work is integer/SFU arithmetic plus a
// write of 4 bytes per value.
#include "rlt_device.cuh"
#include "rlt_internal.h"

namespace rlt {
namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;   // SplitMix64 increment
constexpr int kChunk = 8;                               // channels per thread

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

template <bool kHashOnly>
__global__ void __launch_bounds__(256)
    noise_kernel(float *__restrict__ out, uint32_t *__restrict__ hash_out,
                 const uint64_t *__restrict__ seeds, const int64_t *__restrict__ positions,
                 int64_t n_rows, int32_t channels, int32_t chunks_per_row, float amp, bool vec_ok)
{
    const int64_t total = n_rows * chunks_per_row;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = idx / chunks_per_row;
        const int32_t c0 = (int32_t)(idx - r * chunks_per_row) * kChunk;
        const uint64_t h_row = stage(stage(0ull, seeds[r]), (uint64_t)positions[r]);
        uint32_t h24[kChunk];
#pragma unroll
        for (int k = 0; k < kChunk; ++k)
            h24[k] = (uint32_t)(stage(h_row, (uint64_t)(int64_t)(c0 + k)) >> 40);
        const int64_t base = r * channels + c0;
        const bool full = c0 + kChunk <= channels;
        if constexpr (kHashOnly) {
            if (full && vec_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(hash_out + base);
                dst[0] = make_uint4(h24[0], h24[1], h24[2], h24[3]);
                dst[1] = make_uint4(h24[4], h24[5], h24[6], h24[7]);
            } else {
                for (int k = 0; k < kChunk && c0 + k < channels; ++k)
                    hash_out[base + k] = h24[k];
            }
        } else {
            float x[kChunk];
#pragma unroll
            for (int k = 0; k < kChunk; ++k)
                x[k] = truncnorm(h24[k], amp);
            if (full && vec_ok) {
                float4 *dst = reinterpret_cast<float4 *>(out + base);
                dst[0] = make_float4(x[0], x[1], x[2], x[3]);
                dst[1] = make_float4(x[4], x[5], x[6], x[7]);
            } else {
                for (int k = 0; k < kChunk && c0 + k < channels; ++k)
                    out[base + k] = x[k];
            }
        }
    }
}

}  // namespace

cudaError_t launch_noise(float *out, uint32_t *hash_out, const uint64_t *seeds,
                         const int64_t *positions, int64_t n_rows, int32_t channels,
                         float initializer_range, cudaStream_t stream)
{
    const int32_t chunks = (channels + kChunk - 1) / kChunk;
    const int64_t threads = n_rows * chunks;
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
            nullptr, hash_out, seeds, positions, n_rows, channels, chunks, amp, vec_ok);
    else
        noise_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(
            out, nullptr, seeds, positions, n_rows, channels, chunks, amp, vec_ok);
    return cudaGetLastError();
}

}  // namespace rlt
