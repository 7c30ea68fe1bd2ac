// Philox4x64-10 counter-based generator, written from its published
// definition (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of two 64x64->128-bit multiplies whose high
// halves are xored with the other counter words and the round key; the key is
// advanced by the Weyl constants between rounds.  The multipliers and Weyl
// constants are the ones the paper specifies for the 4x64 variant.
#pragma once

#include <stdint.h>

namespace specv {

struct Philox4 {
  uint64_t w[4];
};

__host__ __device__ __forceinline__ void mul_hilo64(uint64_t a, uint64_t b, uint64_t& hi,
                                                    uint64_t& lo) {
#if defined(__CUDA_ARCH__)
  lo = a * b;
  hi = __umul64hi(a, b);
#else
  unsigned __int128 p = (unsigned __int128)a * b;
  lo = (uint64_t)p;
  hi = (uint64_t)(p >> 64);
#endif
}

__host__ __device__ __forceinline__ Philox4 philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2,
                                                          uint64_t c3, uint64_t k0, uint64_t k1) {
  const uint64_t kMul0 = 0xD2E7470EE14C6C93ull;
  const uint64_t kMul1 = 0xCA5A826395121157ull;
  const uint64_t kWeyl0 = 0x9E3779B97F4A7C15ull;  // golden ratio
  const uint64_t kWeyl1 = 0xBB67AE8584CAA73Bull;  // sqrt(3) - 1
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kWeyl0;
      k1 += kWeyl1;
    }
    uint64_t hi0, lo0, hi1, lo1;
    mul_hilo64(kMul0, c0, hi0, lo0);
    mul_hilo64(kMul1, c2, hi1, lo1);
    const uint64_t n0 = hi1 ^ c1 ^ k0;
    const uint64_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return Philox4{{c0, c1, c2, c3}};
}

// Top 24 bits of a word as a uniform in [0, 1) on the 2^-24 grid (exact in fp32).
__host__ __device__ __forceinline__ float u24(uint64_t w) {
  return (float)(uint32_t)(w >> 40) * (1.0f / 16777216.0f);
}

}  // namespace specv
