// Device-side helpers shared by the libzr kernels: the SplitMix64 counter
// generator, the h0 partition hash and bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace zr {

// SplitMix64 (Steele, Lea and Flood, "Fast Splittable Pseudorandom Number
// Generators", OOPSLA 2014): output number i of the generator seeded with s is
// the finaliser applied to s + (i + 1) * gamma (mod 2^64).
constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t splitmix_finalise(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t splitmix_output(uint64_t seed, uint64_t i) {
  return splitmix_finalise(seed + (i + 1) * kGamma);
}

// Multiply-high range reduction of a 32-bit value onto [0, n).
__host__ __device__ __forceinline__ uint32_t range_reduce(uint32_t h, uint32_t n) {
  return (uint32_t)(((uint64_t)h * n) >> 32);
}

// Random SkipReduce slice offset for one iteration (SkipReduce section 4.3):
// the high 32 bits of output `step` of SplitMix64(seed), onto [0, n).
__host__ __device__ __forceinline__ int random_offset(uint64_t seed, uint64_t step, int n) {
  return (int)range_reduce((uint32_t)(splitmix_output(seed, step) >> 32), (uint32_t)n);
}

// First-level partition hash h0 (Zen section 3.2, Technique #3): a
// multiply-add-shift universal hash of the 32-bit index, then range reduction
// onto the partitions.
struct H0 {
  uint64_t a, b;
  uint32_t n_parts;
  __host__ __device__ __forceinline__ uint32_t operator()(uint32_t x) const {
    uint32_t h = (uint32_t)((a * (uint64_t)x + b) >> 32);
    return range_reduce(h, n_parts);
  }
};

__host__ __device__ inline H0 make_h0(uint64_t seed, uint32_t n_parts) {
  H0 h;
  h.a = splitmix_output(seed, 0) | 1ull;
  h.b = splitmix_output(seed, 1);
  h.n_parts = n_parts;
  return h;
}

// bf16 <-> fp32.  Widening is exact (bf16 is the top half of a binary32);
// narrowing is the CUDA round-to-nearest-even conversion.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat16 l = __float2bfloat16_rn(lo);
  __nv_bfloat16 h = __float2bfloat16_rn(hi);
  return (uint32_t)__bfloat16_as_ushort(l) | ((uint32_t)__bfloat16_as_ushort(h) << 16);
}

}  // namespace zr
