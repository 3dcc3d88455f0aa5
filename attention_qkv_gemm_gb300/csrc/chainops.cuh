// chainops.cuh -- row operations of the d_model = 128 epilogues (the fused
// post-attention chain and the whole-stack kernel).
//
// Layout shared by both kernels: 16 epilogue warps, four per TMEM lane
// quarter; warp (quarter q, part p) owns columns [32 p, 32 p + 32) of the
// 32 rows q*32 .. q*32+31, one row per thread.  Row-wide statistics combine
// the four parts through a shared-memory exchange area `red` (four slots of
// 4 x 128 floats) and one named barrier over the 16 warps.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace tfl {
namespace chain {

constexpr int kD = 128;     // d_model
constexpr int kRows = 128;  // rows of a tile
constexpr int kParts = 4;   // 32-column parts of a row
constexpr int kEpi = 16;    // epilogue warps
constexpr int kRedBytes = 4 * kParts * kRows * 4;

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpi) : "memory"); }

// Row mean / rstd of a 128-wide row split over four warps (32 values each).
// Sums run as four packed pairs (eight partial sums) to keep the dependent
// chains short; slots alternate so a fast warp never overwrites partial sums
// a slow one still reads (callers advance `slot` by 2 per exchange).
__device__ __forceinline__ void stats32(const float* t, float eps, float* red, int slot, int part, int r,
                                        float& mean, float& rstd) {
  // This warp's 32 values: their sum and their sum of squares about their own mean;
  // the four partial results of a row then combine in one exchange (Chan, Golub and
  // LeVeque's pairwise update: M2 = sum M2_p + 32 sum (mean_p - mean)^2).
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i & 3] = f2_add(acc[i & 3], f2_pack(t[2 * i], t[2 * i + 1]));
  float s0, s1;
  f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), s0, s1);
  const float sp = s0 + s1;
  const uint64_t mp2 = f2_splat(sp * (1.0f / 32));
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0ull;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t d = f2_sub(f2_pack(t[2 * i], t[2 * i + 1]), mp2);
    acc[i & 3] = f2_fma(d, d, acc[i & 3]);
  }
  f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), s0, s1);
  float* rs = red + slot * kParts * kRows + r;
  float* rq = rs + kParts * kRows;
  rs[part * kRows] = sp;
  rq[part * kRows] = s0 + s1;
  epi_bar();
  const float a0 = rs[0], a1 = rs[kRows], a2 = rs[2 * kRows], a3 = rs[3 * kRows];
  mean = ((a0 + a1) + (a2 + a3)) * (1.0f / kD);
  const float d0 = a0 * (1.0f / 32) - mean, d1 = a1 * (1.0f / 32) - mean, d2 = a2 * (1.0f / 32) - mean,
              d3 = a3 * (1.0f / 32) - mean;
  const float m2 = ((rq[0] + rq[kRows]) + (rq[2 * kRows] + rq[3 * kRows])) +
                   32.0f * ((d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3));
  rstd = rsqrtf(m2 * (1.0f / kD) + eps);
}

// (t - mean) * rstd * g + b for 32 values in place; g, b: this warp's 32 columns.
__device__ __forceinline__ void normalize32(float* t, float mean, float rstd, const float* g, const float* b) {
  const uint64_t m2 = f2_splat(mean), r2 = f2_splat(rstd);
  const float2* g2 = reinterpret_cast<const float2*>(g);
  const float2* b2 = reinterpret_cast<const float2*>(b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 gg = g2[i], bb = b2[i];
    const uint64_t y = f2_fma(f2_mul(f2_sub(f2_pack(t[2 * i], t[2 * i + 1]), m2), r2), f2_pack(gg.x, gg.y),
                              f2_pack(bb.x, bb.y));
    f2_unpack(y, t[2 * i], t[2 * i + 1]);
  }
}

// LayerNorm of a row split over four warps; g, b: gamma / beta of the whole row.
__device__ __forceinline__ void layer_norm32(float* t, float eps, const float* g, const float* b, int c0,
                                             float* red, int& slot, int part, int r) {
  float mean, rstd;
  stats32(t, eps, red, slot, part, r, mean, rstd);
  slot = (slot + 2) & 3;
  normalize32(t, mean, rstd, g + c0, b + c0);
}

// v[i] = v[i] * scale + p[i] for 32 values.
__device__ __forceinline__ void scale_bias32(float* v, float scale, const float* p) {
  const float2* p2 = reinterpret_cast<const float2*>(p);
  const uint64_t s2 = f2_splat(scale);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 q = p2[i];
    f2_unpack(f2_fma(f2_pack(v[2 * i], v[2 * i + 1]), s2, f2_pack(q.x, q.y)), v[2 * i], v[2 * i + 1]);
  }
}

// fp16 hi/lo pairs of v[i] - c for 16 values (the row's mean taken out before the split;
// first value of a pair in the low half): v - c = hi + lo + O(2^-22 |v - c|).
__device__ __forceinline__ void split_centered_pairs16(const float* v, float c, uint32_t* hi, uint32_t* lo) {
  const uint64_t c2 = f2_splat(c);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t x = f2_sub(f2_pack(v[2 * i], v[2 * i + 1]), c2);
    float x0, x1;
    f2_unpack(x, x0, x1);
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    float l0, l1;
    f2_unpack(f2_sub(x, f2_pack(hf.x, hf.y)), l0, l1);
    const __half2 l = __floats2half2_rn(l0, l1);
    hi[i] = *reinterpret_cast<const uint32_t*>(&h);
    lo[i] = *reinterpret_cast<const uint32_t*>(&l);
  }
}

// GELU (A&S 7.1.26 erf) of 32 values x * a + b[i] and their fp16 hi/lo pairs.
__device__ __forceinline__ void gelu_split32(const float* x, float a, const float* b, uint32_t* hi, uint32_t* lo) {
  const uint64_t a2 = f2_splat(a);
  const float2* b2 = reinterpret_cast<const float2*>(b);
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float2 bq = b2[e];
    const uint64_t gl = gelu2_as7126(f2_fma(f2_pack(x[2 * e], x[2 * e + 1]), a2, f2_pack(bq.x, bq.y)));
    float g0, g1;
    f2_unpack(gl, g0, g1);
    const __half2 h = __floats2half2_rn(g0, g1);  // first value in the low half
    const float2 hf = __half22float2(h);
    float l0, l1;
    f2_unpack(f2_sub(gl, f2_pack(hf.x, hf.y)), l0, l1);
    const __half2 l = __floats2half2_rn(l0, l1);
    hi[e] = *reinterpret_cast<const uint32_t*>(&h);
    lo[e] = *reinterpret_cast<const uint32_t*>(&l);
  }
}

__device__ __forceinline__ void tmem_st8_u(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// Write this warp's 32 values (t - c) of a row as fp16 hi/lo pairs into an operand
// area of 128 values per row: hi at col + 16 part + 8 j, lo 64 columns further.
__device__ __forceinline__ void store_split_operand(uint32_t tq_col, const float* t, float c, int part) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t hi[8], lo[8];
    split_centered_pairs16(t + 16 * j, c, hi, lo);
    tmem_st8_u(tq_col + part * 16 + 8 * j, hi);
    tmem_st8_u(tq_col + 64 + part * 16 + 8 * j, lo);
  }
}

}  // namespace chain
}  // namespace tfl
