// Stochastic rounding of fp32 values to bf16, shared by the kernels that offer
// it. Element e (row-major index) of output tensor `tensor` draws the 16-bit
// threshold r = bits 16 (e mod 4) .. 16 (e mod 4) + 15 of output number
// (tensor << 58 | e / 4) of the splitmix64 generator seeded with `seed`
// (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
// 2014: state seed + (n + 1) * golden gamma, then the variant-13 mix). The
// fp32 value is rounded to bf16 by adding r to its 32-bit pattern and dropping
// the low 16 bits: the magnitude is rounded up with probability
// (low 16 bits) / 2^16, so the rounding is unbiased. Infinities stay infinite
// (their low bits are zero, so no carry leaves the pattern) and NaNs are
// truncated: round_bits also keeps an explicit quiet bit; the epilogue's
// branch-free pair form relies on its fp32 inputs coming from additions,
// whose NaN results are the canonical quiet NaN, which truncates to a NaN.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace mmbwd {
namespace sr {

enum : uint32_t { DINP = 0, DWEIGHT = 1, DBIAS = 2, DWTE = 3, DWPE = 4 };

constexpr uint64_t SM64_GAMMA = 0x9E3779B97F4A7C15ull;

// The output function applied to the state seed + (n + 1) * gamma.
__device__ __forceinline__ uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t sm64_out(uint64_t seed, uint64_t n) {
    return sm64_mix(seed + (n + 1) * SM64_GAMMA);
}

__device__ __forceinline__ uint64_t word(uint64_t seed, uint64_t tensor, uint64_t e) {
    return sm64_out(seed, (tensor << 58) | (e >> 2));
}

// State of the word of element e (a multiple of 4): the words of elements
// e + 4 j follow as sm64_mix(state + j * gamma).
__device__ __forceinline__ uint64_t word_state(uint64_t seed, uint64_t tensor, uint64_t e) {
    return seed + (((tensor << 58) | (e >> 2)) + 1) * SM64_GAMMA;
}

__device__ __forceinline__ uint32_t threshold(uint64_t seed, uint64_t tensor, uint64_t e) {
    return static_cast<uint32_t>(word(seed, tensor, e) >> (16 * (e & 3))) & 0xFFFFu;
}

// bf16 bit pattern of x rounded with threshold r.
__device__ __forceinline__ uint32_t round_bits(float x, uint32_t r) {
    const uint32_t b = __float_as_uint(x);
    if ((b & 0x7F800000u) == 0x7F800000u) return (b >> 16) | ((b & 0x007FFFFFu) ? 0x40u : 0u);
    return (b + r) >> 16;
}

__device__ __forceinline__ __nv_bfloat16 from_bits(uint32_t h) {
    __nv_bfloat16_raw raw;
    raw.x = static_cast<unsigned short>(h);
    return __nv_bfloat16(raw);
}

__device__ __forceinline__ __nv_bfloat16 round(float x, uint64_t seed, uint64_t tensor, uint64_t e) {
    return from_bits(round_bits(x, threshold(seed, tensor, e)));
}

}  // namespace sr
}  // namespace mmbwd
