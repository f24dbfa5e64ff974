// softcap_math.cuh -- the tanh softcap s = c * tanh(z / c) and its exp, in
// fp32, as the kernel epilogues evaluate them.
//
// tanh(x) for |x| <= kTanhXmax: x * P(x^2), P the degree-5 minimax (Remez,
// relative error) polynomial fitted by fit_tanh.py (worst relative error
// 3.9e-9 in exact arithmetic, 1.1e-7 evaluated in fp32).
// For |x| > kTanhXmax: tanh(x) = sign(x) * (1 - 2 / (e^{2|x|} + 1)); here
// e^{2|x|} >= 3.5, so the subtraction loses at most two bits.
#pragma once
#include "ptx.cuh"

namespace lmce {

constexpr float kTanhXmax = 0.625f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTanhC0 = 1.0f;
constexpr float kTanhC1 = -0.3333325982093811f;
constexpr float kTanhC2 = 0.13331127166748047f;
constexpr float kTanhC3 = -0.05372106656432152f;
constexpr float kTanhC4 = 0.02059098891913891f;
constexpr float kTanhC5 = -0.005659989081323147f;

// P(u) with coefficients k[0..5] (k = scale * C): Horner in fp32.
__device__ __forceinline__ float tanh_poly_scaled(float u, const float (&k)[6]) {
  float p = fmaf(k[5], u, k[4]);
  p = fmaf(p, u, k[3]);
  p = fmaf(p, u, k[2]);
  p = fmaf(p, u, k[1]);
  p = fmaf(p, u, k[0]);
  return p;
}

__device__ __forceinline__ float tanh_poly(float x) {
  const float u = x * x;
  float p = fmaf(kTanhC5, u, kTanhC4);
  p = fmaf(p, u, kTanhC3);
  p = fmaf(p, u, kTanhC2);
  p = fmaf(p, u, kTanhC1);
  p = fmaf(p, u, kTanhC0);
  return x * p;
}

// tanh for any finite x (and +-inf).
__device__ __forceinline__ float tanh_any(float x) {
  const float ax = fabsf(x);
  if (ax <= kTanhXmax) return tanh_poly(x);
  const float e = ex2_approx(2.0f * kLog2e * ax);  // e^{2|x|}; +inf for large |x|
  const float t = 1.0f - __fdividef(2.0f, e + 1.0f);
  return copysignf(t, x);
}

}  // namespace lmce
