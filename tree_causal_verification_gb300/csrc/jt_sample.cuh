// Device-side draws for temperature-T acceptance: one Gumbel-max sample of
// softmax(x / T) per visited tree node.
//
// "JetSpec++: Foresight Parallel Drafting with Self Refinements" (paperlayer.ai
// summary), App. F.3: with point-mass proposals every committed token is the
// target's own draw; y = argmax_j (x_j / T + G_j) with G_j ~ Gumbel(0, 1) is
// such a draw (lowest j on ties).
//
// Randomness is counter-based, so every draw is fixed by (seed, sequence,
// row, token) and independent of how the vocabulary is split over threads:
//   draw index k = ((b * (B+1) + r) << 32 | j) + 1, r = 0 root row, 1+v node v
//   h = SplitMix64 output k for `seed` (Steele, Lea and Flood, "Fast
//       splittable pseudorandom number generators", OOPSLA 2014: state
//       seed + k * golden gamma through the 64-bit finaliser)
//   U = ((h >> 41) + 1/2) * 2^-23 in (0, 1),  G = -ln(-ln U)
//   key = x * inv_T + G   (binary32 multiply, then add)
// The logarithm is the atanh series ln(m 2^e) = e ln2 + 2 atanh((m-1)/(m+1)),
// m in [sqrt(1/2), sqrt(2)), to the f^9 term, evaluated with one
// correctly rounded binary32 operation per step so the bits do not depend on
// the compiler (checked against the oracle's independent implementation).
#pragma once

#include <stdint.h>

namespace jt {

__device__ __forceinline__ uint64_t splitmix64_output(uint64_t seed, uint64_t k) {
  uint64_t z = seed + k * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float series_ln(float x) {
  const uint32_t u = __float_as_uint(x);
  int e = (int)(u >> 23) - 127;
  float m = __uint_as_float((u & 0x7FFFFFu) | 0x3F800000u);   // [1, 2)
  if (m > 1.41421356f) {
    m = __fmul_rn(m, 0.5f);
    e += 1;
  }
  const float f = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
  const float f2 = __fmul_rn(f, f);
  float p = __fmaf_rn(f2, 1.0f / 9.0f, 1.0f / 7.0f);
  p = __fmaf_rn(p, f2, 0.2f);
  p = __fmaf_rn(p, f2, 1.0f / 3.0f);
  p = __fmaf_rn(p, f2, 1.0f);
  const float lm = __fmul_rn(__fmul_rn(2.0f, f), p);
  return __fmaf_rn((float)e, 0.693147182f, lm);
}

__device__ __forceinline__ float gumbel_noise(uint64_t seed, uint64_t k) {
  const uint64_t h = splitmix64_output(seed, k);
  const float u = __fmul_rn(__fadd_rn((float)(uint32_t)(h >> 41), 0.5f), 1.1920928955078125e-7f);
  return -series_ln(-series_ln(u));
}

// Element transform for the row scans: logit -> Gumbel-max key of the row
// whose draw indices start at `base` = (b * (B+1) + r) << 32.
struct GumbelKeys {
  uint64_t seed, base;
  float inv_t;
  __device__ __forceinline__ float key(float x, uint32_t j) const {
    return __fadd_rn(__fmul_rn(x, inv_t), gumbel_noise(seed, (base | j) + 1));
  }
  __device__ __forceinline__ float4 operator()(float4 x, int j4) const {
    const uint32_t j = 4u * (uint32_t)j4;
    return make_float4(key(x.x, j), key(x.y, j + 1), key(x.z, j + 2), key(x.w, j + 3));
  }
};

}  // namespace jt
