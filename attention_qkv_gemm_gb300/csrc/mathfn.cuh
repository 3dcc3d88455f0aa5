// mathfn.cuh -- device math used by the epilogues.
#pragma once
#include "ptx.cuh"

namespace tfl {

// Reciprocal on the MUFU unit (approximate, flush-to-zero).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Exact-form GELU, 0.5 x (1 + erf(x / sqrt 2)), with erf from Abramowitz and
// Stegun, Handbook of Mathematical Functions, formula 7.1.26 (Hastings'
// rational approximation): for z >= 0,
//   erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2),
//   t = 1 / (1 + p z),  |error| <= 1.5e-7.
// Written as Phi(x) = 1 - erfc(|x|/sqrt2)/2 for x >= 0 and erfc(|x|/sqrt2)/2
// for x < 0, so the result's absolute error is below 1e-7 |x| (plus the
// MUFU rcp/ex2 rounding, ~2^-22 relative).  Two MUFU operations and about a
// dozen FMA-pipe operations, against roughly thirty for erff.
__device__ __forceinline__ float gelu_as7126(float x) {
  // constants folded: z = |x|/sqrt2, so p z = (p/sqrt2)|x| and -z^2 log2(e) = -(log2(e)/2) x^2;
  // the polynomial carries the factor 1/2 of Phi
  constexpr float p_s = 0.3275911f * 0.7071067811865476f;
  constexpr float h1 = 0.5f * 0.254829592f, h2 = 0.5f * -0.284496736f, h3 = 0.5f * 1.421413741f,
                  h4 = 0.5f * -1.453152027f, h5 = 0.5f * 1.061405429f;
  const float ax = fabsf(x);
  const float t = rcp_approx(fmaf(p_s, ax, 1.0f));
  const float half_erfc = t * fmaf(fmaf(fmaf(fmaf(h5, t, h4), t, h3), t, h2), t, h1) *
                          ex2((x * x) * -0.7213475204444817f);
  return x * (x >= 0.f ? 1.0f - half_erfc : half_erfc);
}

// The same approximation for a packed pair of fp32 values (one 64-bit
// register), with the sign case folded: x Phi(x) = max(x, 0) - |x| erfc(|x|/sqrt2)/2.
// FMA-pipe work runs two lanes per instruction; the two MUFU operations stay
// per value.
__device__ __forceinline__ uint64_t gelu2_as7126(uint64_t x) {
  constexpr float p_s = 0.3275911f * 0.7071067811865476f;
  constexpr float h1 = 0.5f * 0.254829592f, h2 = 0.5f * -0.284496736f, h3 = 0.5f * 1.421413741f,
                  h4 = 0.5f * -1.453152027f, h5 = 0.5f * 1.061405429f;
  float x0, x1;
  f2_unpack(x, x0, x1);
  const uint64_t nax = f2_pack(-fabsf(x0), -fabsf(x1));
  float d0, d1;
  f2_unpack(f2_fma(nax, f2_splat(-p_s), f2_splat(1.0f)), d0, d1);
  const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
  uint64_t poly = f2_fma(f2_splat(h5), t, f2_splat(h4));
  poly = f2_fma(poly, t, f2_splat(h3));
  poly = f2_fma(poly, t, f2_splat(h2));
  poly = f2_fma(poly, t, f2_splat(h1));
  float e0, e1;
  f2_unpack(f2_mul(f2_mul(x, x), f2_splat(-0.7213475204444817f)), e0, e1);
  const uint64_t half_erfc = f2_mul(f2_mul(t, poly), f2_pack(ex2(e0), ex2(e1)));
  return f2_fma(nax, half_erfc, f2_pack(fmaxf(x0, 0.f), fmaxf(x1, 0.f)));
}

// Reference GELU on CUDA's erff (used only by the self-test).
__device__ __forceinline__ float gelu_erff(float x) { return 0.5f * x * (1.0f + erff(x * 0.7071067811865476f)); }

}  // namespace tfl
