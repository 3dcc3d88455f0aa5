// stack.cu -- the whole L-layer forward in one persistent kernel for
// sequences of at most 128 tokens at d_model 128, head_dim 32: one sequence
// is one 128-row tile, and its residual stream stays in tensor memory from
// the input to the output.  Per layer and tile:
//
//   E1  N = LN1(h) as fp16 hi/lo pairs (pre-LN: LN1's affine folded into
//       W_qkv, the operand is h - mean, rstd applied to the products);
//       R = h * 2^so (the o_proj accumulator starts as the residual)
//   QKV k, v, q = N W_qkv^T (+ bias) into two accumulators in turn; k and v
//       go to shared memory as fp16 tiles (padding rows as zeros), q to
//       tensor memory as fp16 pairs -- the [tokens, 3 d_model] buffer never
//       exists ("TikTok TechJam 2026 -- Problem 3", section 1.A: a fused
//       QKV + attention step for short sequences)
//   ATT per head: S = Q K^T over all 128 keys (no online rescale: the whole
//       row is one block), the row max from a four-warp exchange,
//       P = exp2(S log2(e)/sqrt(hd) - max) in fp16 over S, O = P V and the
//       row sum l = P 1 on the tensor core; O / l as fp16 pairs
//   CHAIN R += O Wo^T; t = R 2^-so + bo; LN2; FFN in 128-wide d_ff chunks
//       with GELU (A&S 7.1.26) kept on chip; R accumulates FFN-out onto
//       t 2^s2; h = R 2^-s2 + b2 is the next layer's input (no HBM traffic)
//   after the last layer: out = LN_f(h), padding rows zero.
// HBM sees x once, the output once and the (L2-resident) weights.
//
// Roles (19 warps, one CTA per SM, persistent over sequences): warp 0 TMA
// producer of the weight ring (128 x 128 blocks, hi and lo planes), warp 1
// MMA issuer for QKV, attention, o_proj and FFN-out (and TMEM owner), warp
// 18 MMA issuer for FFN-in, warps 2-17 epilogue (four per TMEM lane quarter,
// 32 columns each; for head_dim 32 a warp's columns are one head).
// Tensor memory (512 columns):
//   [0,128) R (residual / o_proj / FFN-out accumulator, fp32)
//   [128,256) N hi/lo (QKV operand), then Q pairs [128,192) and
//             O pairs + row sums l_h [192,256), then N2 hi/lo (FFN-in operand)
//   [256,384) k, then q accumulator, then S / P of one head, then G (FFN-in)
//   [384,512) v accumulator, then O_h (fp32, 32 columns per head), then GP hi/lo
#include "kernels.h"
#include "ptx.cuh"
#include "mathfn.cuh"
#include "xpose.cuh"
#include "chainops.cuh"

namespace tfl {

namespace {

using namespace chain;

constexpr int kFC = 128;            // d_ff chunk
constexpr int kUnit = 64 * 1024;    // ring unit: a 128 x 128 weight block, hi + lo planes
constexpr int kHalf = 16 * 1024;    // one 64-column (K) half of a plane
constexpr int kRing = 2;
constexpr int kFfn1Warp = 2 + kEpi;
constexpr int kThreads = 32 * (kFfn1Warp + 1);
constexpr int kHD = 32;             // head_dim
constexpr int kH = kD / kHD;        // heads
constexpr int kKVTile = 128 * kHD * 2;  // one head's K (or V): 128 rows x 64 B, 64-byte swizzle
constexpr int kOnesBytes = 16 * 128;
// Parameter vectors staged in shared memory once per CTA (floats): the final LayerNorm's
// gamma / beta, then per layer [bq | bk | bv] (384), bo (128), b1 (d_ff), b2 (128) and, for
// post-LN, LN1 / LN2 gamma and beta (4 x 128), for as many layers as fit; the epilogue reads
// the others from global memory.
constexpr int kPrmCap = 5632;
constexpr size_t kSmem =
    1024 + (size_t)kRing * kUnit + 2 * (size_t)kH * kKVTile + kOnesBytes + kRedBytes + (size_t)kPrmCap * 4 + 512;

constexpr uint32_t kColR = 0, kColN = 128, kColQ = 128, kColOP = 192, kColA = 256, kColB = 384;

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st4_u(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

// One row (32 fp16 values, 64 bytes) of a head's K or V tile, in the 64-byte
// swizzled K-major layout the MMA descriptors describe (16-byte chunk c of row r
// at r * 64 + ((c ^ ((r >> 1) & 3)) << 4)).
__device__ __forceinline__ void put_kv_row(uint8_t* tile, int r, const float* v) {
  uint4 pk[4];
  pack_f16<32>(v, pk, false, 1.0f);
#pragma unroll
  for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(tile + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) = pk[c];
}

// 32 fp32 values from global memory (one thread's 32 columns of a row).
__device__ __forceinline__ void load_row32(const float* p, float* v) {
  const float4* p4 = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 f = __ldg(p4 + i);
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
}

__device__ __forceinline__ void load_row32_bf16(const __nv_bfloat16* p, float* v) {
  const uint4* p4 = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = __ldg(p4 + i);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[k]));
      v[8 * i + 2 * k] = f.x;
      v[8 * i + 2 * k + 1] = f.y;
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    stack_kernel(const __grid_constant__ StackMaps maps, const __grid_constant__ StackArgs args) {
  extern __shared__ uint8_t smem_raw[];
  grid_launch_dependents();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* sK = ring + (size_t)kRing * kUnit;
  uint8_t* sV = sK + (size_t)kH * kKVTile;
  uint8_t* sOnes = sV + (size_t)kH * kKVTile;
  float* red = reinterpret_cast<float*>(sOnes + kOnesBytes);
  float* prm = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(red) + kRedBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(prm + kPrmCap);
  uint64_t* r_full = bars + 0;     // [kRing]
  uint64_t* r_empty = bars + 2;    // [kRing]
  uint64_t* n_ready = bars + 4;    // epilogue -> A: N and R written
  uint64_t* acc_k = bars + 5;      // A -> epilogue
  uint64_t* acc_v = bars + 6;
  uint64_t* k_read = bars + 7;     // epilogue -> A: the k accumulator is free
  uint64_t* acc_q = bars + 8;
  uint64_t* kv_ready = bars + 9;   // epilogue -> A: K and V tiles in shared memory
  uint64_t* q_ready = bars + 10;   // epilogue -> A: Q pairs in tensor memory
  uint64_t* s_full = bars + 11;    // A -> epilogue: S of the current head
  uint64_t* p_full = bars + 12;    // epilogue -> A: P written over S
  uint64_t* pv_done = bars + 13;   // [kH] A -> epilogue: O_h and l_h complete
  uint64_t* o_ready = bars + 17;   // epilogue -> A: O pairs written
  uint64_t* acc_full = bars + 18;  // A -> epilogue: o_proj done
  uint64_t* acc_read = bars + 19;  // epilogue -> B: N2 written
  uint64_t* g_full = bars + 20;    // B -> epilogue
  uint64_t* g_read = bars + 21;    // epilogue -> B
  uint64_t* gp_ready = bars + 22;  // epilogue -> A
  uint64_t* gp_free = bars + 23;   // A -> epilogue
  uint64_t* out_full = bars + 24;  // A -> epilogue: FFN-out done
  uint64_t* drain = bars + 25;     // [2] abort path
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 27);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* never_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kOnesBytes / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sOnes)[i] = 0x3C003C00u;
  fence_async_smem();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], 1);
    }
    for (uint64_t* b : {acc_k, acc_v, acc_q, s_full, acc_full, g_full, gp_free, out_full}) mbar_init(b, 1);
    for (int h = 0; h < kH; ++h) mbar_init(&pv_done[h], 1);
    for (uint64_t* b : {n_ready, k_read, kv_ready, q_ready, p_full, o_ready, acc_read, g_read, gp_ready})
      mbar_init(b, kEpi);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    *never_flag = 0;
    fence_barrier_init();
  }
  // parameter staging (weights and vectors are written at create time, before any kernel
  // of this stream, so this needs no dependent-launch wait); every thread issues all of its
  // loads before any store: one global-memory round trip
  const int prm_stride = 640 + args.F + (args.post_ln ? 4 * kD : 0);
  const int prm_layers = min(args.L, (kPrmCap - 2 * kD) / prm_stride);
  {
    const int n = 2 * kD + prm_layers * prm_stride;
    constexpr int kPer = (kPrmCap + kThreads - 1) / kThreads;
    auto source = [&](int i) -> const float* {
      if (i < kD) return args.lnf_g + i;
      if (i < 2 * kD) return args.lnf_b + (i - kD);
      const int j = i - 2 * kD, l = j / prm_stride;
      int o = j - l * prm_stride;
      const StackLayerArgs& P = args.layer[l];
      if (o < 3 * kD) return P.bqkv + o;
      if ((o -= 3 * kD) < kD) return P.bo + o;
      if ((o -= kD) < args.F) return P.b1 + o;
      if ((o -= args.F) < kD) return P.b2 + o;
      o -= kD;
      const int w = o / kD;
      const float* ln = w == 0 ? P.ln1_g : w == 1 ? P.ln1_b : w == 2 ? P.ln2_g : P.ln2_b;
      return ln + (o - w * kD);
    };
    float pv[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kThreads;
      pv[k] = i < n ? __ldg(source(i)) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kThreads;
      if (i < n) prm[i] = pv[k];
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{args.c.status, abort_flag, args.c.timeout_ns};
  grid_wait_prior();

  const int S = args.c.S, B = args.B, L = args.L;
  const int nch = args.F / kFC;
  // lengths outside [0, S] are clamped (seq_len) and reported through the status word
  if (warp == 0 && args.c.lengths != nullptr) {
    bool bad = false;
    for (int b = blockIdx.x + lane * gridDim.x; b < B; b += 32 * gridDim.x) {
      const int l = args.c.lengths[b];
      bad |= (l < 0) || (l > S);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(args.c.status, TFL_DEV_BAD_LENGTHS);
  }
  const int units = 4 + 2 * nch;  // ring units per tile and layer: Wk, Wv, Wq, Wo, W1 / W2 chunks
  const int* lengths = args.c.lengths;
  auto idx_w1 = [&](int k) { return 3 + (k == 0 ? 1 : (k == 1 ? 2 : 2 * k)); };
  auto idx_w2 = [&](int c) { return 3 + (c <= nch - 2 ? 3 + 2 * c : 2 * nch); };

  uint32_t issued_mask = 0, issued_par = 0;
  bool mma_issued = false;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0;
      bool ok = true;
      auto block = [&](const CUtensorMap* hi, const CUtensorMap* lo, int x, int y) -> bool {
        if (!wait_bounded(&r_empty[rs], rph ^ 1u, wc)) return false;
        uint8_t* d = ring + (size_t)rs * kUnit;
        mbar_arrive_expect_tx(&r_full[rs], kUnit);
        tma_load_2d(d, hi, &r_full[rs], x, y);
        tma_load_2d(d + kHalf, hi, &r_full[rs], x + 64, y);
        tma_load_2d(d + 2 * kHalf, lo, &r_full[rs], x, y);
        tma_load_2d(d + 3 * kHalf, lo, &r_full[rs], x + 64, y);
        issued_mask |= 1u << rs;
        issued_par = (issued_par & ~(1u << rs)) | (rph << rs);
        if (++rs == kRing) {
          rs = 0;
          rph ^= 1u;
        }
        return true;
      };
      for (int b = blockIdx.x; b < B && ok; b += gridDim.x) {
        if (seq_len(lengths, b, S) == 0) continue;
        const int rot = b % nch;
        for (int l = 0; l < L && ok; ++l) {
          const CUtensorMap *wq = &maps.wqkv[l], *wql = &maps.wqkv_lo[l];
          ok = block(wq, wql, 0, 128) && block(wq, wql, 0, 256) && block(wq, wql, 0, 0) &&
               block(&maps.wo[l], &maps.wo_lo[l], 0, 0);
          auto w1 = [&](int c) { return block(&maps.w1[l], &maps.w1_lo[l], 0, ((c + rot) % nch) * kFC); };
          auto w2 = [&](int c) { return block(&maps.w2[l], &maps.w2_lo[l], ((c + rot) % nch) * kFC, 0); };
          if (ok) ok = w1(0);
          if (ok && nch > 1) ok = w1(1);
          for (int c = 0; c < nch && ok; ++c) {
            ok = w2(c);
            if (ok && c + 2 < nch) ok = w1(c + 2);
          }
        }
      }
    }
  } else if (warp == 1 || warp == kFfn1Warp) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t id128 = idesc_f16(128, 128, 0, 0);
      auto take = [&](uint32_t g) -> uint32_t {
        if (!wait_bounded(&r_full[g % kRing], (g / kRing) & 1u, wc)) return 0;
        tc_fence_after();
        return smem_u32(ring + (size_t)(g % kRing) * kUnit);
      };
      auto give = [&](uint32_t g) { umma_commit(&r_empty[g % kRing]); };
      auto kdesc = [](uint32_t p, int kk) { return sdesc(p + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024, kSw128); };
      // d (+)= (a hi, lo pairs at col, col + 64) x (block u hi, lo)^T, 128 x 128 x 128
      auto split_mma = [&](uint32_t d, uint32_t a, uint32_t u, bool acc) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bh = kdesc(u, kk), bl = kdesc(u + 2 * kHalf, kk);
          const uint32_t ah = a + kk * 8, al = ah + 64;
          umma_f16_ts(d, ah, bh, id128, (acc || kk > 0) ? 1u : 0u);
          umma_f16_ts(d, al, bh, id128, 1u);
          umma_f16_ts(d, ah, bl, id128, 1u);
        }
      };
      bool ok = true;
      uint32_t seq = 0;  // tile-layers issued by this CTA
      if (warp == 1) {
        constexpr uint32_t id_s = idesc_f16(128, 128, 0, 0);
        constexpr uint32_t id_pv = idesc_f16(128, kHD, 0, 1);
        constexpr uint32_t id_l = idesc_f16(128, 16, 0, 0);
        const uint64_t ones_d = sdesc(smem_u32(sOnes), 16, 1024, kSw128);
        uint32_t ph_n = 0, ph_kr = 0, ph_kv = 0, ph_q = 0, ph_p = 0, ph_o = 0, ph_gp = 0;
        for (int b = blockIdx.x; b < B && ok; b += gridDim.x) {
          if (seq_len(lengths, b, S) == 0) continue;
          for (int l = 0; l < L && ok; ++l, ++seq) {
            const uint32_t g0 = seq * units;
            if (!wait_bounded(n_ready, ph_n, wc)) { ok = false; break; }
            ph_n ^= 1u;
            tc_fence_after();
            // k and v into the two accumulators, then q once k has been drained
            uint32_t u = take(g0 + 0);
            if (!u) { ok = false; break; }
            split_mma(tmem_base + kColA, tmem_base + kColN, u, false);
            mma_issued = true;
            give(g0 + 0);
            umma_commit(acc_k);
            if (!(u = take(g0 + 1))) { ok = false; break; }
            split_mma(tmem_base + kColB, tmem_base + kColN, u, false);
            give(g0 + 1);
            umma_commit(acc_v);
            if (!wait_bounded(k_read, ph_kr, wc)) { ok = false; break; }
            ph_kr ^= 1u;
            tc_fence_after();
            if (!(u = take(g0 + 2))) { ok = false; break; }
            split_mma(tmem_base + kColA, tmem_base + kColN, u, false);
            give(g0 + 2);
            umma_commit(acc_q);
            if (!wait_bounded(kv_ready, ph_kv, wc) || !wait_bounded(q_ready, ph_q, wc)) { ok = false; break; }
            ph_kv ^= 1u;
            ph_q ^= 1u;
            tc_fence_after();
            // attention, one head at a time: S = Q K^T; then O = P V, l = P 1 with P over S.
            // S of head h + 1 overwrites P of head h: issued after P V of head h.
            for (int h = 0; h < kH && ok; ++h) {
              const uint64_t kd = sdesc(smem_u32(sK + h * kKVTile), 16, 512, kSw64);
#pragma unroll
              for (int kk = 0; kk < kHD / 16; ++kk)
                umma_f16_ts(tmem_base + kColA, tmem_base + kColQ + 16 * h + 8 * kk, kd + (uint32_t)((kk * 32) >> 4),
                            id_s, kk > 0 ? 1u : 0u);
              umma_commit(s_full);
              if (!wait_bounded(p_full, ph_p, wc)) { ok = false; break; }
              ph_p ^= 1u;
              tc_fence_after();
              const uint64_t vd = sdesc(smem_u32(sV + h * kKVTile), 128 * 64, 512, kSw64);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_f16_ts(tmem_base + kColB + kHD * h, tmem_base + kColA + 8 * kk,
                            vd + (uint32_t)((kk * 16 * 64) >> 4), id_pv, kk > 0 ? 1u : 0u);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_f16_ts(tmem_base + kColOP + 16 * h, tmem_base + kColA + 8 * kk, ones_d, id_l, kk > 0 ? 1u : 0u);
              umma_commit(&pv_done[h]);
            }
            if (!ok) break;
            // o_proj onto the residual: R += O Wo^T (O pairs from TMEM, Wo hi and lo)
            if (!wait_bounded(o_ready, ph_o, wc)) { ok = false; break; }
            ph_o ^= 1u;
            tc_fence_after();
            if (!(u = take(g0 + 3))) { ok = false; break; }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t a = tmem_base + kColOP + kk * 8;
              umma_f16_ts(tmem_base + kColR, a, kdesc(u, kk), id128, 1u);
              umma_f16_ts(tmem_base + kColR, a, kdesc(u + 2 * kHalf, kk), id128, 1u);
            }
            give(g0 + 3);
            umma_commit(acc_full);
            // FFN-out of each chunk onto t 2^s2 in R, once its GELU output is in TMEM
            for (int c = 0; c < nch; ++c) {
              if (!wait_bounded(gp_ready, ph_gp, wc)) { ok = false; break; }
              ph_gp ^= 1u;
              tc_fence_after();
              const uint32_t g = g0 + idx_w2(c);
              if (!(u = take(g))) { ok = false; break; }
              split_mma(tmem_base + kColR, tmem_base + kColB, u, true);
              give(g);
              umma_commit(gp_free);
            }
            if (!ok) break;
            umma_commit(out_full);
          }
        }
      } else {
        uint32_t ph_ar = 0, ph_gr = 0;
        for (int b = blockIdx.x; b < B && ok; b += gridDim.x) {
          if (seq_len(lengths, b, S) == 0) continue;
          for (int l = 0; l < L && ok; ++l, ++seq) {
            const uint32_t g0 = seq * units;
            if (!wait_bounded(acc_read, ph_ar, wc)) { ok = false; break; }
            ph_ar ^= 1u;
            tc_fence_after();
            for (int c = 0; c < nch; ++c) {
              if (c > 0) {  // G is reused once the epilogue has read the previous chunk
                if (!wait_bounded(g_read, ph_gr, wc)) { ok = false; break; }
                ph_gr ^= 1u;
                tc_fence_after();
              }
              const uint32_t g = g0 + idx_w1(c);
              const uint32_t u = take(g);
              if (!u) { ok = false; break; }
              split_mma(tmem_base + kColA, tmem_base + kColN, u, false);
              mma_issued = true;
              give(g);
              umma_commit(g_full);
            }
            if (!ok) break;
            // the epilogue's read of the last chunk (keeps this barrier's phases paired)
            if (!wait_bounded(g_read, ph_gr, wc)) { ok = false; break; }
            ph_gr ^= 1u;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (16 warps)
    const int q = warp & 3;
    const int part = (warp - 2) >> 2;
    const int c0 = part * 32;
    const int r = q * 32 + lane;  // the row: position in the sequence
    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16);
    WaitCtl ewc = wc;
    ewc.early_exit = false;  // the epilogue warps meet at a named barrier: leave only on their own bound
    uint32_t ph_k = 0, ph_v = 0, ph_qa = 0, ph_s = 0, ph_pv = 0, ph_af = 0, ph_g = 0, ph_gf = 0, ph_of = 0;
    bool gp_written = false;
    int slot = 0;
    const float eps = args.eps, sl2 = args.scale_log2;
    uint8_t* st = sK + (warp - 2) * 2048;  // output stage (the K tiles are dead by then)
    bool ok = true;
    for (int b = blockIdx.x; b < B && ok; b += gridDim.x) {
      const int len = seq_len(lengths, b, S);
      const bool in_seq = r < S;
      const uint32_t in_rows = __ballot_sync(0xffffffffu, in_seq);
      const size_t row0 = (size_t)b * S + q * 32;  // first row of this warp
      float tv[32];
      if (len == 0) {  // an empty sequence: zero output
#pragma unroll
        for (int i = 0; i < 32; ++i) tv[i] = 0.f;
      } else {
        if (in_seq && r < len) {
          if (args.xbf)
            load_row32_bf16(args.xbf + (row0 + lane) * kD + c0, tv);
          else
            load_row32(args.x + (row0 + lane) * kD + c0, tv);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) tv[i] = 0.f;
        }
        for (int l = 0; l < L; ++l) {
          const StackLayerArgs& P = args.layer[l];
          // the layer's vectors: shared-memory copies when staged (offset within the layer's
          // block), else global memory
          const bool st_l = l < prm_layers;
          auto vec = [&](int off, const float* g) -> const float* {
            return st_l ? prm + 2 * kD + l * prm_stride + off : g;
          };
          // ---- E1: the layer's QKV operand and the residual accumulator
          float mean = 0.f, rstd = 1.f;
          if (!args.post_ln) {
            stats32(tv, eps, red, slot, part, r, mean, rstd);
            slot = (slot + 2) & 3;
          }
          store_split_operand(tq + kColN, tv, mean, part);
          {
            float rv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) rv[i] = tv[i] * P.inv_scale_o;
            tmem_st32(tq + kColR + c0, rv);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(n_ready);
          const float aq = rstd * P.scale_qkv;
          // ---- E2: k and v (this warp's 32 columns are head `part`), padding rows as zeros
          float v[32];
          if (!wait_bounded(acc_k, ph_k, ewc)) { ok = false; break; }
          ph_k ^= 1u;
          tc_fence_after();
          tmem_ld32(tq + kColA + c0, v);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(k_read);
          scale_bias32(v, aq, vec(0, P.bqkv) + kD + c0);
          if (r >= len) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
          put_kv_row(sK + part * kKVTile, r, v);
          if (!wait_bounded(acc_v, ph_v, ewc)) { ok = false; break; }
          ph_v ^= 1u;
          tc_fence_after();
          tmem_ld32(tq + kColB + c0, v);
          tmem_wait_ld();
          scale_bias32(v, aq, vec(0, P.bqkv) + 2 * kD + c0);
          if (r >= len) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
          put_kv_row(sV + part * kKVTile, r, v);
          fence_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(kv_ready);
          // ---- E3: q as fp16 pairs in TMEM
          if (!wait_bounded(acc_q, ph_qa, ewc)) { ok = false; break; }
          ph_qa ^= 1u;
          tc_fence_after();
          tmem_ld32(tq + kColA + c0, v);
          tmem_wait_ld();
          scale_bias32(v, aq, vec(0, P.bqkv) + c0);
          {
            uint32_t pq[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const __half2 h2 = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
              pq[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            tmem_st16_u(tq + kColQ + 16 * part, pq);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(q_ready);
          // ---- ATT: softmax of each head over its 128 keys; this warp holds keys c0 .. c0+31
          for (int h = 0; h < kH; ++h) {
            if (!wait_bounded(s_full, ph_s, ewc)) { ok = false; break; }
            ph_s ^= 1u;
            tc_fence_after();
            tmem_ld32(tq + kColA + c0, v);
            tmem_wait_ld();
            // key j = c0 + e is visible to query r iff j < len and (not causal or j <= r)
            const int lim = args.causal ? min(len - 1, r) : len - 1;
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              v[e] = (c0 + e <= lim) ? v[e] : -INFINITY;
              mx = fmaxf(mx, v[e]);
            }
            float* rs = red + slot * kParts * kRows + r;
            rs[part * kRows] = mx;
            epi_bar();
            mx = fmaxf(fmaxf(rs[0], rs[kRows]), fmaxf(rs[2 * kRows], rs[3 * kRows]));
            slot = (slot + 2) & 3;
            const float mref = mx == -INFINITY ? 0.f : mx * sl2;
            const uint64_t s2 = f2_splat(sl2), nm = f2_splat(-mref);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(v[2 * e], v[2 * e + 1]), s2, nm), x0, x1);
              const __half2 hp = __floats2half2_rn(ex2(x0), ex2(x1));  // first key in the low half
              pk[e] = *reinterpret_cast<const uint32_t*>(&hp);
            }
            // every warp has read its S columns (the exchange above), so P may go over them
            tmem_st16_u(tq + kColA + 16 * part, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
          }
          if (!ok) break;
          // O / l of each head as fp16 pairs: this warp takes head h's columns 8 part .. +7,
          // reading l from the first of the four columns it then overwrites
          for (int h = 0; h < kH; ++h) {
            if (!wait_bounded(&pv_done[h], ph_pv, ewc)) { ok = false; break; }
            tc_fence_after();
            float o[8];
            tmem_ld8(tq + kColB + kHD * h + 8 * part, o);
            const float lsum = tmem_ld1(tq + kColOP + 16 * h + 4 * part);
            const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
            uint32_t po[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 h2 = __floats2half2_rn(o[2 * e] * inv, o[2 * e + 1] * inv);
              po[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            tmem_st4_u(tq + kColOP + 16 * h + 4 * part, po);
          }
          if (!ok) break;
          ph_pv ^= 1u;
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_ready);
          // ---- CHAIN phase 1: t = R 2^-so + bo (post-LN: LN1(t)); R <- t 2^s2; N2
          if (!wait_bounded(acc_full, ph_af, ewc)) { ok = false; break; }
          ph_af ^= 1u;
          tc_fence_after();
          tmem_ld32(tq + kColR + c0, tv);
          tmem_wait_ld();
          scale_bias32(tv, P.scale_o, vec(3 * kD, P.bo) + c0);
          if (args.post_ln) layer_norm32(tv, eps, vec(5 * kD + args.F, P.ln1_g), vec(6 * kD + args.F, P.ln1_b), c0, red, slot, part, r);
          {
            float rv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) rv[i] = tv[i] * P.inv_scale_2;
            tmem_st32(tq + kColR + c0, rv);
          }
          float a1 = P.scale_1, mean2 = 0.f;
          if (!args.post_ln) {
            float rstd2;
            stats32(tv, eps, red, slot, part, r, mean2, rstd2);
            slot = (slot + 2) & 3;
            a1 = rstd2 * P.scale_1;
          }
          store_split_operand(tq + kColN, tv, mean2, part);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_read);
          // ---- CHAIN phase 2: GELU of each FFN-in chunk as hi/lo pairs
          for (int c = 0; c < nch; ++c) {
            if (!wait_bounded(g_full, ph_g, ewc)) { ok = false; break; }
            ph_g ^= 1u;
            tc_fence_after();
            float gv[32];
            tmem_ld32(tq + kColA + c0, gv);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(g_read);
            uint32_t hi[16], lo[16];
            gelu_split32(gv, a1, vec(4 * kD, P.b1) + ((c + b) % nch) * kFC + c0, hi, lo);
            if (gp_written) {  // GP is free once FFN-out of the previous chunk has read it
              if (!wait_bounded(gp_free, ph_gf, ewc)) { ok = false; break; }
              ph_gf ^= 1u;
              tc_fence_after();
            }
            tmem_st16_u(tq + kColB + part * 16, hi);
            tmem_st16_u(tq + kColB + 64 + part * 16, lo);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(gp_ready);
            gp_written = true;
          }
          if (!ok) break;
          // ---- CHAIN phase 3: h = R 2^-s2 + b2 (post-LN: LN2(h)), the next layer's input
          if (!wait_bounded(out_full, ph_of, ewc)) { ok = false; break; }
          ph_of ^= 1u;
          tc_fence_after();
          tmem_ld32(tq + kColR + c0, tv);
          tmem_wait_ld();
          scale_bias32(tv, P.scale_2, vec(4 * kD + args.F, P.b2) + c0);
          if (args.post_ln) layer_norm32(tv, eps, vec(7 * kD + args.F, P.ln2_g), vec(8 * kD + args.F, P.ln2_b), c0, red, slot, part, r);
        }
        if (!ok) break;
        // ---- tail: final LayerNorm, padding rows zero
        layer_norm32(tv, eps, prm, prm + kD, c0, red, slot, part, r);
        if (r >= len) {
#pragma unroll
          for (int i = 0; i < 32; ++i) tv[i] = 0.f;
        }
      }
      if (args.outbf) {
        xp_store_bf16<32>(st, lane, tv, args.outbf + row0 * kD + c0, kD, in_rows);
      } else {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          xp_store_f32x16(st, lane, tv + 16 * hh, args.out32 + row0 * kD + c0 + 16 * hh, kD, in_rows);
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    const WaitCtl dc{args.c.status, never_flag, 100000000LL};
    if (warp == 0 && lane == 0)
      for (int s = 0; s < kRing; ++s)
        if (issued_mask & (1u << s)) wait_bounded(&r_full[s], (issued_par >> s) & 1u, dc);
    if ((warp == 1 || warp == kFfn1Warp) && lane == 0 && mma_issued) {
      uint64_t* db = &drain[warp == 1 ? 0 : 1];
      umma_commit(db);
      wait_bounded(db, 0, dc);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

cudaError_t prepare_stack_kernel() {
  return cudaFuncSetAttribute(stack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
}

cudaError_t launch_stack(const StackMaps& mp, const StackArgs& a, int num_sms, cudaStream_t s) {
  if (a.F % kFC != 0 || a.F < kFC || a.L < 1 || a.L > kStackMaxLayers || a.c.S > 128) return cudaErrorInvalidValue;
  const int grid = a.B < num_sms ? a.B : num_sms;
  if (grid <= 0) return cudaSuccess;
  return launch_dependent(stack_kernel, grid, kThreads, kSmem, s, mp, a);
}

}  // namespace tfl
