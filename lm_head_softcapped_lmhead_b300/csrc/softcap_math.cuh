// softcap_math.cuh -- the tanh softcap s = c * tanh(z / c) and its exp, in
// fp32, as the kernel epilogues evaluate them.
//
// tanh(x) for |x| <= kTanhXmax: x * P(x^2), P the degree-3 minimax (Remez,
// relative error) polynomial fitted by fit_tanh.py (worst relative error
// 1.0e-8 in exact arithmetic, 1.1e-7 evaluated in fp32).  With c = 30 the
// range covers |z| <= 9, well beyond the logits of a d = 512 head with
// 0.02-scale weights.
// For |x| > kTanhXmax: tanh(x) = sign(x) * (1 - 2 / (e^{2|x|} + 1)); here
// e^{2|x|} >= 1.8, so the subtraction loses at most two bits.
#pragma once
#include "ptx.cuh"

namespace lmce {

constexpr float kTanhXmax = 0.3f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTanhTerms = 4;
constexpr float kTanhC0 = 1.0f;
constexpr float kTanhC1 = -0.33332961797714233f;
constexpr float kTanhC2 = 0.13312597572803497f;
constexpr float kTanhC3 = -0.05022243782877922f;

__device__ __forceinline__ float tanh_poly(float x) {
  const float u = x * x;
  float p = fmaf(kTanhC3, u, kTanhC2);
  p = fmaf(p, u, kTanhC1);
  p = fmaf(p, u, kTanhC0);
  return x * p;
}

// Packed-fp32 (sm_100 FFMA2) evaluation of the same polynomial with the
// scale folded into its coefficients: for z and u = z*z,
//   z * (k0 + k1 u + k2 u^2 + k3 u^3)
// with k_i = s * C_i / c^(2i+1) equals s * tanh_poly(z / c).
__device__ __forceinline__ float2 poly_z2(float2 z, float2 u, const float2 (&k)[kTanhTerms]) {
  float2 p = __ffma2_rn(k[3], u, k[2]);
  p = __ffma2_rn(p, u, k[1]);
  p = __ffma2_rn(p, u, k[0]);
  return __fmul2_rn(z, p);
}

// Coefficients k_i = scale * C_i * inv_c^(2i+1) (host side, in double).
inline void scaled_tanh_coeffs(double scale, double inv_c, float (&k)[kTanhTerms]) {
  const double C[kTanhTerms] = {kTanhC0, kTanhC1, kTanhC2, kTanhC3};
  double f = inv_c;
  for (int i = 0; i < kTanhTerms; ++i) {
    k[i] = static_cast<float>(scale * C[i] * f);
    f *= inv_c * inv_c;
  }
}

// tanh on the SFU (PTX tanh.approx.f32).  Its specified relative error is
// about 2^-11; over |x| <= kTanhXmax it measured at most 9.9e-6 (every float
// in [1e-6, 0.3] on a B300, mean signed error at most 2.2e-6 in any decade
// of x), against 1.1e-7 for tanh_poly.  The backward epilogues use it there,
// with tanh_any for chunks beyond: it keeps their arithmetic off the FMA
// pipe, whose load slows the tensor pipe of the same SM.  The forward
// keeps tanh_poly: with 8 epilogue warps for a 128 x 256 tile per CTA, the
// second SFU operation per logit made it SFU-bound (0.393 -> 0.435 ms at
// N = 65536).
__device__ __forceinline__ float tanh_sfu(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (sm_100 three-input max).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
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
