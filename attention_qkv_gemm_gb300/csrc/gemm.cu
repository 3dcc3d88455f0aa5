// gemm.cu -- persistent tcgen05 GEMM with fused epilogues.
//
// C[M, N] = A[M, K] * W[N, K]^T with fp16 operands and fp32 accumulation in
// tensor memory ("TikTok TechJam 2026 -- Problem 3", section 2.3: fp16
// tensor cores, fp32 accumulate, one rounding at the store).  The four
// epilogues fuse the row-wise work of the forward into the GEMM that
// produces it (section 1.A: add_layernorm_cast, bias_gelu_cast,
// post_attn_chain_tail):
//   EPI_BIAS_F16       QKV projection: c16 = acc + b_qkv (fused QKV, section 2.2)
//   EPI_BIAS_GELU_F16  FFN-in: c16 = GELU_erf(acc + b1)
//   EPI_BIAS_RES_F32   o_proj / FFN-out when d_model > 128: h = acc + b + h
//   EPI_BIAS_RES_ROW   o_proj / FFN-out when d_model == 128: residual add plus
//                      row LayerNorm(s) in fp32, fp16 normed output or the
//                      model tail (final LayerNorm + pad-mask, fp32 out).
//
// Structure (one CTA per SM, persistent over 128 x BN output tiles):
//   warp 0  TMA producer: A and W k-blocks (64 fp16 = 128 B, 128B swizzle)
//           into a STAGES-deep shared-memory ring.
//   warp 1  MMA issuer: 4 tcgen05.mma (K = 16 each) per k-block into one of
//           two TMEM accumulators (double-buffered so the epilogue of tile t
//           overlaps the MMAs of tile t+1).
//   warps 2-5 epilogue: thread = output row (TMEM lane), tcgen05.ld of 32
//           columns at a time, fused math, vectorised global stores.
// Tiles whose 128 rows are all padding (s >= len_b) are skipped entirely;
// the model-tail epilogue writes their zeros without waiting for an MMA.
#include "kernels.h"
#include "ptx.cuh"

namespace tfl {

template <int BN>
struct GemmCfg {
  static constexpr int A_BYTES = kGemmBM * kGemmBK * 2;
  static constexpr int B_BYTES = BN * kGemmBK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (196 * 1024) / STAGE > 8 ? 8 : (196 * 1024) / STAGE;
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE + 256;
};

size_t gemm_smem_bytes(int bn) {
  return bn == 256 ? GemmCfg<256>::SMEM : GemmCfg<128>::SMEM;
}

__device__ __forceinline__ float gelu_erf(float v) { return 0.5f * v * (1.0f + erff(v * 0.7071067811865476f)); }

__device__ __forceinline__ void store_f16x32(__half* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h0 = __floats2half2_rn(v[8 * i + 0], v[8 * i + 1]);
    __half2 h1 = __floats2half2_rn(v[8 * i + 2], v[8 * i + 3]);
    __half2 h2 = __floats2half2_rn(v[8 * i + 4], v[8 * i + 5]);
    __half2 h3 = __floats2half2_rn(v[8 * i + 6], v[8 * i + 7]);
    uint4 u;
    u.x = *reinterpret_cast<uint32_t*>(&h0);
    u.y = *reinterpret_cast<uint32_t*>(&h1);
    u.z = *reinterpret_cast<uint32_t*>(&h2);
    u.w = *reinterpret_cast<uint32_t*>(&h3);
    d[i] = u;
  }
}

// LayerNorm of a thread-owned row of N values in registers: returns mean and rstd.
template <int N>
__device__ __forceinline__ void row_stats(const float* t, float eps, float& mean, float& rstd) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) s += t[i];
  mean = s * (1.0f / N);
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float d = t[i] - mean;
    q = fmaf(d, d, q);
  }
  rstd = rsqrtf(q * (1.0f / N) + eps);
}

template <int BN, int EPI>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs args) {
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* accf = empty + C::STAGES;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* never_flag = abort_flag + 1;  // stays 0: lets the drain waits ignore abort_flag

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *never_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{args.c.status, abort_flag, args.c.timeout_ns};

  const int M = args.c.M, S = args.c.S;
  const int* lengths = args.c.lengths;
  const int num_m = (M + kGemmBM - 1) / kGemmBM, num_n = args.N / BN, num_k = args.K / kGemmBK;
  const int total = num_m * num_n;

  // Producer bookkeeping for the abort path: last parity issued per stage.
  uint32_t issued_mask = 0, issued_par = 0;
  bool mma_issued = false;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int mb = t / num_n, nb = t - mb * num_n;
        if (!rows_live(mb * kGemmBM, min(mb * kGemmBM + kGemmBM, M), S, lengths)) continue;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * C::STAGE;
          mbar_arrive_expect_tx(&full[stage], C::STAGE);
          tma_load_2d(sa, &tmA, &full[stage], kb * kGemmBK, mb * kGemmBM);
          tma_load_2d(sa + C::A_BYTES, &tmB, &full[stage], kb * kGemmBK, nb * BN);
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(128, BN, 0, 0);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int mb = t / num_n;
        if (!rows_live(mb * kGemmBM, min(mb * kGemmBM + kGemmBM, M), S, lengths)) continue;
        if (!wait_bounded(&acce[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_k; ++kb) {
          if (!wait_bounded(&full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)stage * C::STAGE);
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < kGemmBK / 16; ++k) {
            umma_f16(d, sdesc(sa + k * 32, 16, 1024, kSw128), sdesc(sb + k * 32, 16, 1024, kSw128), idesc,
                     (kb | k) != 0);
          }
          mma_issued = true;
          umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&accf[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const int mb = t / num_n, nb = t - mb * num_n;
      const int m = mb * kGemmBM + r;
      if (!rows_live(mb * kGemmBM, min(mb * kGemmBM + kGemmBM, M), S, lengths)) {
        if constexpr (EPI == EPI_BIAS_RES_ROW) {
          if ((args.row.flags & ROW_FINAL) && m < M) {
            float4* o = reinterpret_cast<float4*>(args.row.out32 + (size_t)m * BN);
#pragma unroll
            for (int i = 0; i < BN / 4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        continue;
      }
      if (!wait_bounded(&accf[acc], acc_phase, wc)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const bool in_range = m < M;

      if constexpr (EPI == EPI_BIAS_F16 || EPI == EPI_BIAS_GELU_F16 || EPI == EPI_BIAS_RES_F32) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tb + c * 32, v);
          tmem_wait_ld();
          const int n0 = nb * BN + c * 32;
          if (in_range) {
            const float4* bp = reinterpret_cast<const float4*>(args.bias + n0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 b4 = __ldg(bp + i);
              v[4 * i + 0] += b4.x;
              v[4 * i + 1] += b4.y;
              v[4 * i + 2] += b4.z;
              v[4 * i + 3] += b4.w;
            }
            if constexpr (EPI == EPI_BIAS_GELU_F16) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = gelu_erf(v[i]);
            }
            if constexpr (EPI == EPI_BIAS_RES_F32) {
              float4* hp = reinterpret_cast<float4*>(args.h32 + (size_t)m * args.N + n0);
              if (row_valid(m, S, lengths)) {
                const float4* rp = reinterpret_cast<const float4*>(args.res + (size_t)m * args.N + n0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 r4 = rp[i];
                  v[4 * i + 0] += r4.x;
                  v[4 * i + 1] += r4.y;
                  v[4 * i + 2] += r4.z;
                  v[4 * i + 3] += r4.w;
                }
              }
#pragma unroll
              for (int i = 0; i < 8; ++i) hp[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            } else {
              store_f16x32(args.c16 + (size_t)m * args.N + n0, v);
            }
          }
        }
      } else {
        // EPI_BIAS_RES_ROW: the whole row (BN == N == d_model) is in this thread.
        float t[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(tb + c * 32, t + c * 32);
        tmem_wait_ld();
        if (in_range) {
          const RowOps& ro = args.row;
          const bool valid = row_valid(m, S, lengths);
          const float4* bp = reinterpret_cast<const float4*>(args.bias);
#pragma unroll
          for (int i = 0; i < BN / 4; ++i) {
            const float4 b4 = __ldg(bp + i);
            t[4 * i + 0] += b4.x;
            t[4 * i + 1] += b4.y;
            t[4 * i + 2] += b4.z;
            t[4 * i + 3] += b4.w;
          }
          if (valid) {
            const float4* rp = reinterpret_cast<const float4*>(args.res + (size_t)m * BN);
#pragma unroll
            for (int i = 0; i < BN / 4; ++i) {
              const float4 r4 = rp[i];
              t[4 * i + 0] += r4.x;
              t[4 * i + 1] += r4.y;
              t[4 * i + 2] += r4.z;
              t[4 * i + 3] += r4.w;
            }
          }
          float mean, rstd;
          if (ro.flags & ROW_POST_LN) {
            row_stats<BN>(t, ro.eps, mean, rstd);
#pragma unroll
            for (int i = 0; i < BN; ++i) t[i] = (t[i] - mean) * rstd * __ldg(ro.ga + i) + __ldg(ro.ba + i);
          }
          if (ro.flags & ROW_WRITE_H) {
            float4* hp = reinterpret_cast<float4*>(ro.h32 + (size_t)m * BN);
#pragma unroll
            for (int i = 0; i < BN / 4; ++i) hp[i] = make_float4(t[4 * i], t[4 * i + 1], t[4 * i + 2], t[4 * i + 3]);
          }
          if (ro.flags & (ROW_FINAL | ROW_NORM16)) {
            row_stats<BN>(t, ro.eps, mean, rstd);
            const bool fin = (ro.flags & ROW_FINAL) != 0;
            const float* g = fin ? ro.gf : ro.gb;
            const float* bb = fin ? ro.bf : ro.bb;
#pragma unroll
            for (int i = 0; i < BN; ++i) t[i] = (t[i] - mean) * rstd * __ldg(g + i) + __ldg(bb + i);
            if (fin) {
              float4* op = reinterpret_cast<float4*>(ro.out32 + (size_t)m * BN);
              if (valid) {
#pragma unroll
                for (int i = 0; i < BN / 4; ++i)
                  op[i] = make_float4(t[4 * i], t[4 * i + 1], t[4 * i + 2], t[4 * i + 3]);
              } else {
#pragma unroll
                for (int i = 0; i < BN / 4; ++i) op[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              }
            } else {
#pragma unroll
              for (int c = 0; c < BN / 32; ++c) store_f16x32(ro.n16 + (size_t)m * BN + c * 32, t + c * 32);
            }
          } else if (ro.flags & ROW_CAST16) {
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) store_f16x32(ro.n16 + (size_t)m * BN + c * 32, t + c * 32);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Abort path: let this CTA's in-flight copies and MMAs land before the
    // shared and tensor memory are released (bounded as well).
    const WaitCtl dc{args.c.status, never_flag, 100000000LL};
    if (warp == 0 && lane == 0) {
      for (int s = 0; s < C::STAGES; ++s)
        if (issued_mask & (1u << s)) wait_bounded(&full[s], (issued_par >> s) & 1u, dc);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      umma_commit(drain);
      wait_bounded(drain, 0, dc);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN, int EPI>
static cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int num_sms,
                              cudaStream_t s) {
  auto kern = gemm_kernel<BN, EPI>;
  const size_t smem = GemmCfg<BN>::SMEM;
  const int tiles = ((a.c.M + kGemmBM - 1) / kGemmBM) * (a.N / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, 192, smem, s>>>(ta, tb, a);
  return cudaGetLastError();
}

template <int BN, int EPI>
static cudaError_t prepare_one() {
  return cudaFuncSetAttribute(gemm_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)GemmCfg<BN>::SMEM);
}

cudaError_t prepare_gemm_kernels() {
  cudaError_t e;
  if ((e = prepare_one<128, EPI_BIAS_F16>()) != cudaSuccess) return e;
  if ((e = prepare_one<128, EPI_BIAS_GELU_F16>()) != cudaSuccess) return e;
  if ((e = prepare_one<128, EPI_BIAS_RES_F32>()) != cudaSuccess) return e;
  if ((e = prepare_one<128, EPI_BIAS_RES_ROW>()) != cudaSuccess) return e;
  if ((e = prepare_one<256, EPI_BIAS_F16>()) != cudaSuccess) return e;
  if ((e = prepare_one<256, EPI_BIAS_GELU_F16>()) != cudaSuccess) return e;
  return prepare_one<256, EPI_BIAS_RES_F32>();
}

cudaError_t launch_gemm(int bn, int epi, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                        int num_sms, cudaStream_t s) {
  if (bn == 128) {
    switch (epi) {
      case EPI_BIAS_F16: return launch_one<128, EPI_BIAS_F16>(ta, tb, a, num_sms, s);
      case EPI_BIAS_GELU_F16: return launch_one<128, EPI_BIAS_GELU_F16>(ta, tb, a, num_sms, s);
      case EPI_BIAS_RES_F32: return launch_one<128, EPI_BIAS_RES_F32>(ta, tb, a, num_sms, s);
      case EPI_BIAS_RES_ROW: return launch_one<128, EPI_BIAS_RES_ROW>(ta, tb, a, num_sms, s);
    }
  } else if (bn == 256) {
    switch (epi) {
      case EPI_BIAS_F16: return launch_one<256, EPI_BIAS_F16>(ta, tb, a, num_sms, s);
      case EPI_BIAS_GELU_F16: return launch_one<256, EPI_BIAS_GELU_F16>(ta, tb, a, num_sms, s);
      case EPI_BIAS_RES_F32: return launch_one<256, EPI_BIAS_RES_F32>(ta, tb, a, num_sms, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace tfl
