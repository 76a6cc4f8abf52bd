// Philox4x64-10 counter-based generator on the device.
//
// Written from the definition in J. K. Salmon, M. A. Moraes, R. O. Dror and
// D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11): ten
// rounds, each multiplying counter words 0 and 2 by fixed odd constants,
// keeping both 64-bit halves of the products and mixing them with words 1 and
// 3 and the round key; the key is bumped by two Weyl constants (the golden
// ratio and sqrt(3) - 1, scaled by 2^64) between rounds.
//
// The ISD accept step draws u = top 24 bits * 2^-24 (exact in fp32) from word
// `index % 4` of Philox(counter = (step, request, purpose, index / 4),
// key = (seed, 0)).
#pragma once

#include <stdint.h>

namespace idlm {

constexpr uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ull;
constexpr uint64_t kPhiloxM1 = 0xCA5A826395121157ull;
constexpr uint64_t kPhiloxW0 = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kPhiloxW1 = 0xBB67AE8584CAA73Bull;

enum : uint32_t { kPurposeAccept = 0, kPurposeSample = 1, kPurposePropose = 2 };

struct Philox4 {
  uint64_t w[4];
};

__device__ __forceinline__ Philox4 philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2,
                                                 uint64_t c3, uint64_t k0, uint64_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    const uint64_t hi0 = __umul64hi(kPhiloxM0, c0);
    const uint64_t lo0 = kPhiloxM0 * c0;
    const uint64_t hi1 = __umul64hi(kPhiloxM1, c2);
    const uint64_t lo1 = kPhiloxM1 * c2;
    const uint64_t n0 = hi1 ^ c1 ^ k0;
    const uint64_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  Philox4 out;
  out.w[0] = c0;
  out.w[1] = c1;
  out.w[2] = c2;
  out.w[3] = c3;
  return out;
}

__device__ __forceinline__ float uniform24(uint64_t word) {
  return static_cast<float>(static_cast<uint32_t>(word >> 40)) * (1.0f / 16777216.0f);
}

// Uniform `index` of `purpose` for `request` at `step`.
__device__ __forceinline__ float isd_uniform(uint64_t seed, uint64_t step, uint32_t request,
                                             uint32_t purpose, uint32_t index) {
  const Philox4 b = philox4x64_10(step, request, purpose, index >> 2, seed, 0ull);
  return uniform24(b.w[index & 3]);
}

}  // namespace idlm
