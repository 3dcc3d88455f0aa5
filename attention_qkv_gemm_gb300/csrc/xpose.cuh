// xpose.cuh -- per-warp transpose stage for coalesced row I/O from
// thread-per-row register data (the tcgen05.ld 32x32b layout: thread = row).
//
// A stage holds the warp's 32 rows of RB bytes (RB = 64 or 128).  Chunk q
// (16 bytes) of row i sits at i*RB + ((q ^ (i % CPR)) << 4), CPR = RB/16, so
// a thread writing its own row and the warp reading 32*16 bytes of whole
// rows per instruction both reach every bank four times (the minimum for 512
// bytes).  Global traffic then moves 512/RB whole rows per warp instruction
// instead of 32 row fragments on 32 different lines.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tfl {

template <int RB>
struct XStage {
  static constexpr int CPR = RB / 16;      // 16-byte chunks per row
  static constexpr int RPI = 32 / CPR;     // rows per warp instruction
  static __device__ __forceinline__ int off(int i, int q) { return i * RB + ((q ^ (i % CPR)) << 4); }

  // Thread `lane` puts its row (CPR x 16 bytes) into the stage.
  static __device__ __forceinline__ void put_row(uint8_t* st, int lane, const uint4* v) {
#pragma unroll
    for (int q = 0; q < CPR; ++q) *reinterpret_cast<uint4*>(st + off(lane, q)) = v[q];
  }
  // The warp stores staged row i to dst + i * pitch for rows whose bit is set in `rows`.
  // All shared reads are issued before the first global store.
  static __device__ __forceinline__ void store_rows(const uint8_t* st, int lane, uint8_t* dst, size_t pitch,
                                                    uint32_t rows) {
    uint4 v[CPR];
#pragma unroll
    for (int k = 0; k < CPR; ++k) v[k] = *reinterpret_cast<const uint4*>(st + off(RPI * k + lane / CPR, lane % CPR));
#pragma unroll
    for (int k = 0; k < CPR; ++k) {
      const int i = RPI * k + lane / CPR;
      if ((rows >> i) & 1u) *reinterpret_cast<uint4*>(dst + (size_t)i * pitch + (lane % CPR) * 16) = v[k];
    }
  }
  // Global half of a staged load: the warp fetches row i of src + i * pitch into
  // registers (zeros where the bit of `rows` is clear); all loads in flight together.
  static __device__ __forceinline__ void fetch_rows(int lane, const uint8_t* src, size_t pitch, uint32_t rows,
                                                    uint4* v) {
#pragma unroll
    for (int k = 0; k < CPR; ++k) {
      const int i = RPI * k + lane / CPR;
      v[k] = ((rows >> i) & 1u) ? *reinterpret_cast<const uint4*>(src + (size_t)i * pitch + (lane % CPR) * 16)
                                : make_uint4(0, 0, 0, 0);
    }
  }
  // Shared half: put fetched rows into the stage.
  static __device__ __forceinline__ void put_fetched(uint8_t* st, int lane, const uint4* v) {
#pragma unroll
    for (int k = 0; k < CPR; ++k) *reinterpret_cast<uint4*>(st + off(RPI * k + lane / CPR, lane % CPR)) = v[k];
  }
  // The warp loads row i from src + i * pitch into the stage (zeros where the bit of `rows` is clear).
  static __device__ __forceinline__ void load_rows(uint8_t* st, int lane, const uint8_t* src, size_t pitch,
                                                   uint32_t rows) {
    uint4 v[CPR];
    fetch_rows(lane, src, pitch, rows, v);
    put_fetched(st, lane, v);
  }
};

// 32 fp32 values -> 8 x 16 bytes.
__device__ __forceinline__ void pack_f32x32(const float* v, uint4* o) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    o[q] = make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                      __float_as_uint(v[4 * q + 3]));
}

// N values (N multiple of 8) -> N/8 x 16 bytes of fp16, times `scale`: the
// values themselves (lo_part = false) or the residuals of their fp16 rounding.
template <int N>
__device__ __forceinline__ void pack_f16(const float* v, uint4* o, bool lo_part, float scale = 1.0f) {
#pragma unroll
  for (int q = 0; q < N / 8; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = v[8 * q + 2 * k] * scale, b = v[8 * q + 2 * k + 1] * scale;
      __half2 h = __floats2half2_rn(a, b);
      if (lo_part) {
        const float2 f = __half22float2(h);
        h = __floats2half2_rn(a - f.x, b - f.y);
      }
      w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    o[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// N values (N multiple of 8) -> N/8 x 16 bytes of bf16, rounded to nearest even.
template <int N>
__device__ __forceinline__ void pack_bf16(const float* v, uint4* o) {
#pragma unroll
  for (int q = 0; q < N / 8; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * q + 2 * k], v[8 * q + 2 * k + 1]);
      w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    o[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---- fp8 operand form: a value v is carried as h = fp16(v), e4m3(h) and e4m3((v - h) 2^11);
// the tensor core multiplies the e4m3 planes (kind::f8f6f4) for the two correction terms of a
// split product, at the scale 2^11 the fp16 product of h with weights pre-scaled by 2^11 shares.
constexpr float kF8LoScale = 2048.0f;

// Two fp32 values as e4m3 (round to nearest even, saturating), a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));  // first source -> high byte
  return r;
}
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

// N values (N multiple of 16) -> the two e4m3 planes of their fp16 rounding, N/16 x 16 bytes each.
template <int N>
__device__ __forceinline__ void pack_f8pair(const float* v, uint4* hi8, uint4* lo8) {
#pragma unroll
  for (int q = 0; q < N / 16; ++q) {
    uint32_t wh[4], wl[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float* x = v + 16 * q + 4 * k;
      float h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __half2float(__float2half_rn(x[i]));
      wh[k] = e4m3x4(h[0], h[1], h[2], h[3]);
      wl[k] = e4m3x4((x[0] - h[0]) * kF8LoScale, (x[1] - h[1]) * kF8LoScale, (x[2] - h[2]) * kF8LoScale,
                     (x[3] - h[3]) * kF8LoScale);
    }
    hi8[q] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    lo8[q] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
}

// Store the two e4m3 planes of N columns (N = 64) of the warp's 32 rows through the stage.
template <int N>
__device__ __forceinline__ void xp_store_f8pair(uint8_t* st, int lane, const float* v, uint8_t* hi_row0,
                                                uint8_t* lo_row0, size_t pitch_bytes, uint32_t rows) {
  using X = XStage<N>;
  uint4 h[N / 16], l[N / 16];
  pack_f8pair<N>(v, h, l);
  X::put_row(st, lane, h);
  __syncwarp();
  X::store_rows(st, lane, hi_row0, pitch_bytes, rows);
  __syncwarp();
  X::put_row(st, lane, l);
  __syncwarp();
  X::store_rows(st, lane, lo_row0, pitch_bytes, rows);
  __syncwarp();
}

// Store N bf16 columns (N = 32 or 64) of the warp's 32 rows through the stage.
template <int N>
__device__ __forceinline__ void xp_store_bf16(uint8_t* st, int lane, const float* v, __nv_bfloat16* row0,
                                              size_t pitch_elems, uint32_t rows) {
  using X = XStage<N * 2>;
  uint4 h[N / 8];
  pack_bf16<N>(v, h);
  X::put_row(st, lane, h);
  __syncwarp();
  X::store_rows(st, lane, reinterpret_cast<uint8_t*>(row0), pitch_elems * 2, rows);
  __syncwarp();
}

// Store N fp16 columns (N = 32 or 64; hi, and lo when given) of the warp's 32 rows through the stage.
template <int N>
__device__ __forceinline__ void xp_store_f16(uint8_t* st, int lane, const float* v, __half* hi_row0, __half* lo_row0,
                                             size_t pitch_elems, uint32_t rows, float scale = 1.0f) {
  using X = XStage<N * 2>;
  uint4 h[N / 8];
  pack_f16<N>(v, h, false, scale);
  X::put_row(st, lane, h);
  __syncwarp();
  X::store_rows(st, lane, reinterpret_cast<uint8_t*>(hi_row0), pitch_elems * 2, rows);
  __syncwarp();
  if (lo_row0 != nullptr) {
    pack_f16<N>(v, h, true, scale);
    X::put_row(st, lane, h);
    __syncwarp();
    X::store_rows(st, lane, reinterpret_cast<uint8_t*>(lo_row0), pitch_elems * 2, rows);
    __syncwarp();
  }
}

// Store 32 fp32 columns of the warp's 32 rows through the stage.
__device__ __forceinline__ void xp_store_f32x32(uint8_t* st, int lane, const float* v, float* row0,
                                                size_t pitch_elems, uint32_t rows) {
  uint4 o[8];
  pack_f32x32(v, o);
  XStage<128>::put_row(st, lane, o);
  __syncwarp();
  XStage<128>::store_rows(st, lane, reinterpret_cast<uint8_t*>(row0), pitch_elems * 4, rows);
  __syncwarp();
}

// Add 32 fp32 columns of the warp's 32 rows, already fetched into `f` by
// XStage<128>::fetch_rows, into v (thread = row) through the stage.
__device__ __forceinline__ void xp_add_fetched_f32x32(uint8_t* st, int lane, float* v, const uint4* f) {
  using X = XStage<128>;
  X::put_fetched(st, lane, f);
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 o = *reinterpret_cast<const uint4*>(st + X::off(lane, q));
    v[4 * q] += __uint_as_float(o.x);
    v[4 * q + 1] += __uint_as_float(o.y);
    v[4 * q + 2] += __uint_as_float(o.z);
    v[4 * q + 3] += __uint_as_float(o.w);
  }
  __syncwarp();
}

// Add 32 fp32 columns of the warp's 32 rows (loaded through the stage; zero where `rows` is clear) into v.
__device__ __forceinline__ void xp_add_f32x32(uint8_t* st, int lane, float* v, const float* row0,
                                              size_t pitch_elems, uint32_t rows) {
  uint4 f[8];
  XStage<128>::fetch_rows(lane, reinterpret_cast<const uint8_t*>(row0), pitch_elems * 4, rows, f);
  xp_add_fetched_f32x32(st, lane, v, f);
}

// 16 fp32 values -> 4 x 16 bytes.
__device__ __forceinline__ void pack_f32x16(const float* v, uint4* o) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    o[q] = make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                      __float_as_uint(v[4 * q + 3]));
}

// Store 16 fp32 columns of the warp's 32 rows through a 2 KB stage.
__device__ __forceinline__ void xp_store_f32x16(uint8_t* st, int lane, const float* v, float* row0,
                                                size_t pitch_elems, uint32_t rows) {
  uint4 o[4];
  pack_f32x16(v, o);
  XStage<64>::put_row(st, lane, o);
  __syncwarp();
  XStage<64>::store_rows(st, lane, reinterpret_cast<uint8_t*>(row0), pitch_elems * 4, rows);
  __syncwarp();
}

// Add 16 fp32 columns of the warp's 32 rows, already fetched into `f` by
// XStage<64>::fetch_rows, into v (thread = row) through a 2 KB stage.
__device__ __forceinline__ void xp_add_fetched_f32x16(uint8_t* st, int lane, float* v, const uint4* f) {
  using X = XStage<64>;
  X::put_fetched(st, lane, f);
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 o = *reinterpret_cast<const uint4*>(st + X::off(lane, q));
    v[4 * q] += __uint_as_float(o.x);
    v[4 * q + 1] += __uint_as_float(o.y);
    v[4 * q + 2] += __uint_as_float(o.z);
    v[4 * q + 3] += __uint_as_float(o.w);
  }
  __syncwarp();
}

}  // namespace tfl
