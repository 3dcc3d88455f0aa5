// gemm.cu -- persistent tcgen05 GEMM with fused epilogues and split-fp16 operands.
//
// C[M, N] = A[M, K] * W[N, K]^T on fp16 tensor cores with fp32 accumulation
// in tensor memory ("TikTok TechJam 2026 -- Problem 3", section 2.3: fp16
// operands, fp32 accumulate, one rounding at the store).
//
// Precision.  One fp16 rounding of every operand is too coarse for the
// graded rule over many seeds ("Transformerkernel", Challenges: a d=32 case
// failed at 0.00208 and the B=10000 case at 0.002074 over 25 trials), so
// operands can be carried as two fp16 terms, x = hi + lo with
// lo = fp16(x - hi):
//   WS  weights split: W * 2^s = W_hi + W_lo (s per matrix keeps W_lo out of
//       the fp16 subnormal range; the epilogue multiplies by 2^-s, exactly).
//   AS  activations split: A = A_hi + A_lo, two fp16 planes in HBM written by
//       the producing kernel.
// Per 16-wide k-step the MMAs A_hi*W_hi (+ A_lo*W_hi) (+ A_hi*W_lo) all
// accumulate into the same fp32 accumulator; A_lo*W_lo (~2^-22) is dropped.
//   F8  fp8 operand form (mode 2, both operands): the two correction terms run
//       on the fp8 tensor path at twice the fp16 rate.  W_hi is stored as fp16
//       times 2^11 (exact), and A and W also as e4m3(hi) and e4m3(lo 2^11);
//       A_hi*(W_hi 2^11) (fp16) + e4m3(A_lo 2^11)*e4m3(W_hi) + e4m3(A_hi)*
//       e4m3(W_lo 2^11) (kind::f8f6f4, K = 32) share one accumulator at the
//       scale 2^(s+11).  The e4m3 rounding of a correction term costs ~2^-4 of
//       a term that is itself ~2^-11 of the product.
//
// Epilogues (the row-wise work of section 1.A fused into the GEMM):
//   EPI_BIAS_F16       QKV projection: c16 = acc + b_qkv
//   EPI_BIAS_GELU_F16  FFN-in: c16 = GELU(acc + b1), exact-erf form (hi [+ lo] planes)
//   EPI_BIAS_RES_F32   o_proj / FFN-out when d_model > 128: h = acc + b + res
//   EPI_BIAS_RES_ROW   o_proj / FFN-out when d_model == 128: residual add and
//                      fp32 row LayerNorm(s): normed fp16 (hi [+ lo]) for the
//                      next sublayer, or the model tail (final LN + mask).
//
// Structure (one CTA per SM, persistent over 128 x BN output tiles):
//   warp 0     TMA producer: k-blocks of 64 (128 B rows, 128B swizzle) of
//              A_hi [A_lo] W_hi [W_lo] into a STAGES-deep ring.
//   warp 1     MMA issuer and TMEM owner; two accumulators so the epilogue
//              of tile t overlaps the MMAs of tile t+1.
//   warps 2-9  epilogue: two warps per TMEM lane quarter (thread = output
//              row), each covering half of the tile's columns.
// Tiles whose 128 rows are all padding are skipped; the model-tail epilogue
// writes their zeros without waiting for an MMA.
#include "kernels.h"
#include "ptx.cuh"
#include "mathfn.cuh"
#include "xpose.cuh"

namespace tfl {

constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;

template <int BN, int AS, int WS, int EPI>
struct GemmCfg {
  static constexpr bool F8 = AS == 2;             // fp8 operand form (then WS == 2 too)
  static constexpr int A_BYTES = kGemmBM * kGemmBK * 2;
  static constexpr int B_BYTES = BN * kGemmBK * 2;
  static constexpr int A8_BYTES = kGemmBM * kGemmBK;  // one e4m3 plane of the k-block (64-byte rows)
  static constexpr int B8_BYTES = BN * kGemmBK;
  // stage: A_hi [A_lo] W_hi [W_lo], or for F8: A_hi A8hi A8lo W_hi W8hi W8lo
  static constexpr int STAGE = F8 ? A_BYTES + 2 * A8_BYTES + B_BYTES + 2 * B8_BYTES
                                  : A_BYTES * (1 + AS) + B_BYTES * (1 + WS);
  // row-statistics exchange, only the row-LayerNorm epilogue has one (the space it
  // frees elsewhere buys the split-operand rings a third stage)
  static constexpr int RED_BYTES = EPI == EPI_BIAS_RES_ROW ? 4 * 2 * kGemmBM * 4 : 0;
  static constexpr int XPOSE_BYTES = kEpiWarps * 32 * 128;  // one 32 x 128 B transpose stage per epilogue warp
  static constexpr int RING_MAX = 232448 - 1024 - RED_BYTES - XPOSE_BYTES - 256;
  static constexpr int STAGES = RING_MAX / STAGE > 8 ? 8 : RING_MAX / STAGE;
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE + RED_BYTES + XPOSE_BYTES + 256;
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T on e4m3 operands (kind::f8f6f4, K = 32); the instruction
// descriptor's A / B format code 0 is e4m3 here, so idesc_f16's encoding serves unchanged.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(1u)
      : "memory");
}

// Row mean / rstd of a row split over the two epilogue warps of a lane quarter.
template <int NH>
__device__ __forceinline__ void row_stats_split(const float* t, float eps, float* red, int slot, int half, int r,
                                                float& mean, float& rstd) {
  constexpr float invN = 1.0f / (2 * NH);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NH; ++i) s += t[i];
  red[(slot * 2 + half) * kGemmBM + r] = s;
  epi_bar();
  mean = (red[(slot * 2 + 0) * kGemmBM + r] + red[(slot * 2 + 1) * kGemmBM + r]) * invN;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NH; ++i) {
    const float d = t[i] - mean;
    q = fmaf(d, d, q);
  }
  red[((slot + 1) * 2 + half) * kGemmBM + r] = q;
  epi_bar();
  rstd = rsqrtf((red[((slot + 1) * 2 + 0) * kGemmBM + r] + red[((slot + 1) * 2 + 1) * kGemmBM + r]) * invN + eps);
}

template <int BN, int EPI, int AS, int WS>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAlo,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBlo,
                const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                const GemmArgs args) {
  using C = GemmCfg<BN, AS, WS, EPI>;
  extern __shared__ uint8_t smem_raw[];
  grid_launch_dependents();  // the next kernel may set itself up meanwhile
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(smem + (size_t)C::STAGES * C::STAGE);
  uint8_t* xpose = smem + (size_t)C::STAGES * C::STAGE + C::RED_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(xpose + C::XPOSE_BYTES);
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
      mbar_init(&acce[a], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *never_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (AS) tma_prefetch_desc(&tmAlo);
    if (WS) tma_prefetch_desc(&tmBlo);
    if (C::F8) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{args.c.status, abort_flag, args.c.timeout_ns};
  grid_wait_prior();  // everything below reads or writes what earlier kernels use

  const int M = args.c.M, S = args.c.S;
  const int* lengths = args.c.lengths;
  const int num_m = (M + kGemmBM - 1) / kGemmBM, num_n = args.N / BN, num_k = args.K / kGemmBK;
  // work item t: live tile t / num_n of the tile list, column block t % num_n
  const int* tile_list = args.c.tiles;
  const int n_live = tile_list[0];
  const int total = n_live * num_n;
  (void)num_m;

  uint32_t issued_mask = 0, issued_par = 0;  // producer: stages with loads in flight (abort path)
  bool mma_issued = false;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int ti = t / num_n, nb = t - ti * num_n;
        const int mb = tile_list[2 + ti];
        for (int kb = 0; kb < num_k; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * C::STAGE;
          mbar_arrive_expect_tx(&full[stage], C::STAGE);
          tma_load_2d(sa, &tmA, &full[stage], kb * kGemmBK, mb * kGemmBM);
          if constexpr (C::F8) {
            tma_load_2d(sa + C::A_BYTES, &tmAlo, &full[stage], kb * kGemmBK, mb * kGemmBM);
            tma_load_2d(sa + C::A_BYTES + C::A8_BYTES, &tmA2, &full[stage], kb * kGemmBK, mb * kGemmBM);
            uint8_t* sb = sa + C::A_BYTES + 2 * C::A8_BYTES;
            tma_load_2d(sb, &tmB, &full[stage], kb * kGemmBK, nb * BN);
            tma_load_2d(sb + C::B_BYTES, &tmBlo, &full[stage], kb * kGemmBK, nb * BN);
            tma_load_2d(sb + C::B_BYTES + C::B8_BYTES, &tmB2, &full[stage], kb * kGemmBK, nb * BN);
          } else {
            if (AS) tma_load_2d(sa + C::A_BYTES, &tmAlo, &full[stage], kb * kGemmBK, mb * kGemmBM);
            uint8_t* sb = sa + C::A_BYTES * (1 + AS);
            tma_load_2d(sb, &tmB, &full[stage], kb * kGemmBK, nb * BN);
            if (WS) tma_load_2d(sb + C::B_BYTES, &tmBlo, &full[stage], kb * kGemmBK, nb * BN);
          }
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
          if constexpr (C::F8) {
            // fp16 A_hi * W_hi 2^11, then the e4m3 corrections (64-byte rows, 64B swizzle)
            const uint32_t sa8h = sa + C::A_BYTES, sa8l = sa8h + C::A8_BYTES;
            const uint32_t sb = sa8l + C::A8_BYTES;
            const uint32_t sb8h = sb + C::B_BYTES, sb8l = sb8h + C::B8_BYTES;
#pragma unroll
            for (int k = 0; k < kGemmBK / 16; ++k)
              umma_f16(d, sdesc(sa + k * 32, 16, 1024, kSw128), sdesc(sb + k * 32, 16, 1024, kSw128), idesc,
                       (kb | k) != 0);
#pragma unroll
            for (int k = 0; k < kGemmBK / 32; ++k) {
              umma_f8(d, sdesc(sa8l + k * 32, 16, 512, kSw64), sdesc(sb8h + k * 32, 16, 512, kSw64), idesc);
              umma_f8(d, sdesc(sa8h + k * 32, 16, 512, kSw64), sdesc(sb8l + k * 32, 16, 512, kSw64), idesc);
            }
          } else {
            const uint32_t sal = sa + C::A_BYTES;
            const uint32_t sb = sa + C::A_BYTES * (1 + AS);
            const uint32_t sbl = sb + C::B_BYTES;
#pragma unroll
            for (int k = 0; k < kGemmBK / 16; ++k) {
              const uint64_t ah = sdesc(sa + k * 32, 16, 1024, kSw128);
              const uint64_t bh = sdesc(sb + k * 32, 16, 1024, kSw128);
              umma_f16(d, ah, bh, idesc, (kb | k) != 0);
              if (AS) umma_f16(d, sdesc(sal + k * 32, 16, 1024, kSw128), bh, idesc, 1u);
              if (WS) umma_f16(d, ah, sdesc(sbl + k * 32, 16, 1024, kSw128), idesc, 1u);
            }
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
    // ------------------------------------------------------------ epilogue (8 warps)
    constexpr int NH = BN / 2;  // columns per epilogue warp
    const int q = warp & 3;     // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;
    const int c0 = half * NH;   // first tile column of this warp
    uint8_t* st = xpose + (warp - 2) * 4096;
    const float sc = args.acc_scale;
    WaitCtl ewc = wc;
    ewc.early_exit = false;  // the epilogue warps meet at a named barrier: leave only on their own bound
    int acc = 0;
    uint32_t acc_phase = 0;
    // the final row epilogue also zeroes the all-padding tiles, listed after the live ones
    bool zero_dead = false;
    if constexpr (EPI == EPI_BIAS_RES_ROW) zero_dead = (args.row.flags & ROW_FINAL) != 0;
    const int all_work = (zero_dead ? tile_list[1] : n_live) * num_n;
    for (int t = blockIdx.x; t < all_work; t += gridDim.x) {
      const int ti = t / num_n, nb = t - ti * num_n;
      const int mb = tile_list[2 + ti];
      const int m0w = mb * kGemmBM + q * 32;  // first row of this warp's 32 rows
      const int m = m0w + lane;
      const uint32_t in_rows = __ballot_sync(0xffffffffu, m < M);
      const uint32_t valid_rows = __ballot_sync(0xffffffffu, m < M && row_valid(m, S, lengths));
      if (ti >= n_live) {
        if constexpr (EPI == EPI_BIAS_RES_ROW) {
          if (args.row.flags & ROW_FINAL) {
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
            for (int c = 0; c < NH / 32; ++c) {
              const size_t off = (size_t)m0w * BN + c0 + c * 32;
              if (args.row.outbf)
                xp_store_bf16<32>(st, lane, z, args.row.outbf + off, BN, in_rows);
              else
                xp_store_f32x32(st, lane, z, args.row.out32 + off, BN, in_rows);
            }
          }
        }
        continue;
      }
      uint4 pre[8];  // EPI_BIAS_RES_ROW: first 32 residual columns, fetched before the wait
      if constexpr (EPI == EPI_BIAS_RES_ROW)
        XStage<128>::fetch_rows(lane, reinterpret_cast<const uint8_t*>(args.res + (size_t)m0w * BN + c0), BN * 4,
                                valid_rows, pre);
      if (!wait_bounded(&accf[acc], acc_phase, ewc)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c0);

      if constexpr (EPI == EPI_BIAS_F16 || EPI == EPI_BIAS_GELU_F16) {
#pragma unroll 1
        for (int g = 0; g < NH / 64; ++g) {
          float v[64];
          tmem_ld32(tb + g * 64, v);
          tmem_ld32(tb + g * 64 + 32, v + 32);
          tmem_wait_ld();
          const int n0 = nb * BN + c0 + g * 64;
          const float4* bp = reinterpret_cast<const float4*>(args.bias + n0);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 b4 = __ldg(bp + i);
            v[4 * i + 0] = fmaf(v[4 * i + 0], sc, b4.x);
            v[4 * i + 1] = fmaf(v[4 * i + 1], sc, b4.y);
            v[4 * i + 2] = fmaf(v[4 * i + 2], sc, b4.z);
            v[4 * i + 3] = fmaf(v[4 * i + 3], sc, b4.w);
          }
          if constexpr (EPI == EPI_BIAS_GELU_F16) {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = gelu_as7126(v[i]);
          } else {
            // q, k, v of padding rows are written as exact zeros, so attention can take
            // whole key blocks (a zero probability times a zero value row) whatever the
            // padding positions of the input held
            if (!((valid_rows >> lane) & 1u)) {
#pragma unroll
              for (int i = 0; i < 64; ++i) v[i] = 0.f;
            }
          }
          const size_t off = (size_t)m0w * args.N + n0;
          xp_store_f16<64>(st, lane, v, args.c16 + off, args.c16lo ? args.c16lo + off : nullptr, args.N, in_rows);
          // the fp8 operand form of the output for the next GEMM (GELU output)
          if (args.c8hi) xp_store_f8pair<64>(st, lane, v, args.c8hi + off, args.c8lo + off, args.N, in_rows);
        }
      } else if constexpr (EPI == EPI_BIAS_RES_F32) {
#pragma unroll 1
        for (int c = 0; c < NH / 32; ++c) {
          float v[32];
          tmem_ld32(tb + c * 32, v);
          tmem_wait_ld();
          const int n0 = nb * BN + c0 + c * 32;
          const float4* bp = reinterpret_cast<const float4*>(args.bias + n0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 b4 = __ldg(bp + i);
            v[4 * i + 0] = fmaf(v[4 * i + 0], sc, b4.x);
            v[4 * i + 1] = fmaf(v[4 * i + 1], sc, b4.y);
            v[4 * i + 2] = fmaf(v[4 * i + 2], sc, b4.z);
            v[4 * i + 3] = fmaf(v[4 * i + 3], sc, b4.w);
          }
          const size_t off = (size_t)m0w * args.N + n0;
          xp_add_f32x32(st, lane, v, args.res + off, args.N, valid_rows);
          xp_store_f32x32(st, lane, v, args.h32 + off, args.N, in_rows);
        }
      } else {
        // EPI_BIAS_RES_ROW: BN == N == d_model; this thread owns half of row m.
        float tv[NH];
#pragma unroll
        for (int c = 0; c < NH / 32; ++c) tmem_ld32(tb + c * 32, tv + c * 32);
        tmem_wait_ld();
        const RowOps& ro = args.row;
        const bool valid = (valid_rows >> lane) & 1u;
        const int r = q * 32 + lane;
        {
          const float4* bp = reinterpret_cast<const float4*>(args.bias + c0);
#pragma unroll
          for (int i = 0; i < NH / 4; ++i) {
            const float4 b4 = __ldg(bp + i);
            tv[4 * i + 0] = fmaf(tv[4 * i + 0], sc, b4.x);
            tv[4 * i + 1] = fmaf(tv[4 * i + 1], sc, b4.y);
            tv[4 * i + 2] = fmaf(tv[4 * i + 2], sc, b4.z);
            tv[4 * i + 3] = fmaf(tv[4 * i + 3], sc, b4.w);
          }
        }
        xp_add_fetched_f32x32(st, lane, tv, pre);
#pragma unroll
        for (int c = 1; c < NH / 32; ++c)
          xp_add_f32x32(st, lane, tv + c * 32, args.res + (size_t)m0w * BN + c0 + c * 32, BN, valid_rows);
        float mean, rstd;
        int slot = 0;
        if (ro.flags & ROW_POST_LN) {
          row_stats_split<NH>(tv, ro.eps, red, slot, half, r, mean, rstd);
          slot += 2;
#pragma unroll
          for (int i = 0; i < NH; ++i)
            tv[i] = (tv[i] - mean) * rstd * __ldg(ro.ga + c0 + i) + __ldg(ro.ba + c0 + i);
        }
        if (ro.flags & ROW_WRITE_H) {
#pragma unroll
          for (int c = 0; c < NH / 32; ++c)
            xp_store_f32x32(st, lane, tv + c * 32, ro.h32 + (size_t)m0w * BN + c0 + c * 32, BN, in_rows);
        }
        if (ro.flags & (ROW_FINAL | ROW_NORM16)) {
          row_stats_split<NH>(tv, ro.eps, red, slot, half, r, mean, rstd);
          const bool fin = (ro.flags & ROW_FINAL) != 0;
          const float* g = fin ? ro.gf : ro.gb;
          const float* bb = fin ? ro.bf : ro.bb;
#pragma unroll
          for (int i = 0; i < NH; ++i) {
            const float y = (tv[i] - mean) * rstd * __ldg(g + c0 + i) + __ldg(bb + c0 + i);
            tv[i] = (fin && !valid) ? 0.f : y;
          }
          if (fin) {
#pragma unroll
            for (int c = 0; c < NH / 32; ++c) {
              const size_t off = (size_t)m0w * BN + c0 + c * 32;
              if (ro.outbf)
                xp_store_bf16<32>(st, lane, tv + c * 32, ro.outbf + off, BN, in_rows);
              else
                xp_store_f32x32(st, lane, tv + c * 32, ro.out32 + off, BN, in_rows);
            }
          } else {
#pragma unroll
            for (int c = 0; c < NH / 64; ++c) {
              const size_t off = (size_t)m0w * BN + c0 + c * 64;
              xp_store_f16<64>(st, lane, tv + c * 64, ro.n16 + off, ro.n16lo ? ro.n16lo + off : nullptr, BN, in_rows);
            }
          }
        } else if (ro.flags & ROW_CAST16) {
#pragma unroll
          for (int c = 0; c < NH / 64; ++c) {
            const size_t off = (size_t)m0w * BN + c0 + c * 64;
            xp_store_f16<64>(st, lane, tv + c * 64, ro.n16 + off, ro.n16lo ? ro.n16lo + off : nullptr, BN, in_rows);
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

template <int BN, int EPI, int AS, int WS>
static cudaError_t launch_one(const GemmMaps& mp, const GemmArgs& a, int num_sms, cudaStream_t s) {
  using C = GemmCfg<BN, AS, WS, EPI>;
  const int tiles = ((a.c.M + kGemmBM - 1) / kGemmBM) * (a.N / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  return launch_dependent(gemm_kernel<BN, EPI, AS, WS>, grid, kGemmThreads, C::SMEM, s, mp.a, mp.alo, mp.b, mp.blo,
                          mp.a2, mp.b2, a);
}

template <int BN, int EPI, int AS, int WS>
static cudaError_t prepare_one() {
  return cudaFuncSetAttribute(gemm_kernel<BN, EPI, AS, WS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)GemmCfg<BN, AS, WS, EPI>::SMEM);
}

// Every (BN, EPI) pair the planner uses, at the three fp16 operand modes (AS, WS) = (0,0),
// (0,1), (1,1); and the pairs that run in the fp8 operand form (2,2) above d_model 128.
#define TFL_GEMM_VARIANTS(X)                                                                       \
  X(128, EPI_BIAS_F16) X(256, EPI_BIAS_F16) X(128, EPI_BIAS_GELU_F16) X(256, EPI_BIAS_GELU_F16) \
  X(128, EPI_BIAS_RES_F32) X(256, EPI_BIAS_RES_F32) X(128, EPI_BIAS_RES_ROW)
#define TFL_GEMM_F8_VARIANTS(X)                                                                    \
  X(128, EPI_BIAS_F16) X(256, EPI_BIAS_F16) X(128, EPI_BIAS_GELU_F16) X(256, EPI_BIAS_GELU_F16) \
  X(128, EPI_BIAS_RES_F32)

cudaError_t prepare_gemm_kernels() {
  cudaError_t e = cudaSuccess;
#define TFL_PREP(BN, EPI)                                 \
  if (e == cudaSuccess) e = prepare_one<BN, EPI, 0, 0>(); \
  if (e == cudaSuccess) e = prepare_one<BN, EPI, 0, 1>(); \
  if (e == cudaSuccess) e = prepare_one<BN, EPI, 1, 1>();
  TFL_GEMM_VARIANTS(TFL_PREP)
#undef TFL_PREP
#define TFL_PREP_F8(BN, EPI) \
  if (e == cudaSuccess) e = prepare_one<BN, EPI, 2, 2>();
  TFL_GEMM_F8_VARIANTS(TFL_PREP_F8)
#undef TFL_PREP_F8
  return e;
}

cudaError_t launch_gemm(int bn, int epi, int as, int ws, const GemmMaps& mp, const GemmArgs& a, int num_sms,
                        cudaStream_t s) {
  if ((as && !ws) || ((as == 2) != (ws == 2))) return cudaErrorInvalidValue;
  if (as == 2) {
#define TFL_LAUNCH_F8(BN, EPI) \
  if (bn == BN && epi == EPI) return launch_one<BN, EPI, 2, 2>(mp, a, num_sms, s);
    TFL_GEMM_F8_VARIANTS(TFL_LAUNCH_F8)
#undef TFL_LAUNCH_F8
    return cudaErrorInvalidValue;
  }
#define TFL_LAUNCH(BN, EPI)                                      \
  if (bn == BN && epi == EPI) {                                  \
    if (as) return launch_one<BN, EPI, 1, 1>(mp, a, num_sms, s); \
    if (ws) return launch_one<BN, EPI, 0, 1>(mp, a, num_sms, s); \
    return launch_one<BN, EPI, 0, 0>(mp, a, num_sms, s);         \
  }
  TFL_GEMM_VARIANTS(TFL_LAUNCH)
#undef TFL_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace tfl
