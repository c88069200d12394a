// 2^x on the FMA pipes, for softmax exponentials that should not all go through the MUFU.
//
// Method: range reduction x = i + f with i = floor(x) and f in [0, 1) (exact: x - floor(x)
// loses no bits for |x| < 2^23), then a cubic p(f) ~ 2^f constrained to p(0) = 1 and p(1) = 2,
// so that the result is exact at integers and continuous and monotone across them; its two
// free coefficients were fitted for the smallest maximum relative error on [0, 1]. With the
// fp32 coefficients below the relative error is at most 1.04e-4 (bf16, to which the softmax
// rounds P, steps by 2^-8 relative). The result is p(f) with i added to its exponent field.
// x < -126 gives 0 (the softmax adds nothing there), -inf gives 0, x >= 128 gives +inf.
// Host and device evaluate the same operations in the same order (floor, one subtraction,
// three fused multiply-adds, an integer add), so a host build reproduces device results.
#pragma once

#include <math.h>
#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SSD_EXP2_FN __host__ __device__ __forceinline__
#else
#define SSD_EXP2_FN inline
#endif

namespace ssd {

constexpr float kExp2C1 = 0.69542432f;     // p(f) = 1 + f (C1 + f (C2 + f C3)), C1 + C2 + C3 = 1
constexpr float kExp2C2 = 0.22630768f;
constexpr float kExp2C3 = 0.07826800f;

SSD_EXP2_FN uint32_t exp2_bits(float x) {
#if defined(__CUDA_ARCH__)
  return __float_as_uint(x);
#else
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  return u;
#endif
}

SSD_EXP2_FN float exp2_from_bits(uint32_t u) {
#if defined(__CUDA_ARCH__)
  return __uint_as_float(u);
#else
  float x;
  memcpy(&x, &u, sizeof x);
  return x;
#endif
}

SSD_EXP2_FN float exp2_poly(float x) {
  if (!(x >= -126.f)) return 0.f;          // below the normal range, -inf (and NaN)
  if (x >= 128.f) return INFINITY;
  const float xi = floorf(x);
  const float f = x - xi;                   // exact, in [0, 1)
  const float p = fmaf(fmaf(fmaf(kExp2C3, f, kExp2C2), f, kExp2C1), f, 1.0f);   // in [1, 2]
  const int32_t i = static_cast<int32_t>(xi);
  return exp2_from_bits(exp2_bits(p) + (static_cast<uint32_t>(i) << 23));
}

}  // namespace ssd
