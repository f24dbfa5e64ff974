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

// The forward + dh pass's epilogue uses a degree-2 fit on the same range (fit_tanh.py,
// DEG = 2: worst relative error 1.2e-6 in exact arithmetic, 1.3e-6 in fp32):
// there s = c tanh(z/c) only enters p = e^{s - lse} and 1 - tanh^2, and an
// error of at most c * 1.3e-6 * 0.3 ~ 1e-5 in s is far below the bf16
// rounding of the gradient tile.  It saves one FFMA2 per logit pair.
constexpr int kTanhTerms2 = 3;
constexpr float kTanh2C0 = 0.9999988675117493f;
constexpr float kTanh2C1 = -0.33310022950172424f;
constexpr float kTanh2C2 = 0.12633946537971497f;

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

// Degree-2 form of poly_z2: z * (k0 + k1 u + k2 u^2).
__device__ __forceinline__ float2 poly2_z2(float2 z, float2 u, const float2 (&k)[kTanhTerms2]) {
  float2 p = __ffma2_rn(k[2], u, k[1]);
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
inline void scaled_tanh2_coeffs(double scale, double inv_c, float (&k)[kTanhTerms2]) {
  const double C[kTanhTerms2] = {kTanh2C0, kTanh2C1, kTanh2C2};
  double f = inv_c;
  for (int i = 0; i < kTanhTerms2; ++i) {
    k[i] = static_cast<float>(scale * C[i] * f);
    f *= inv_c * inv_c;
  }
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
