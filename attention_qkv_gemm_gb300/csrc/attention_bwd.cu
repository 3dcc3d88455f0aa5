// attention_bwd.cu -- flash attention backward on tcgen05 tensor cores.
//
// Gradients of O = softmax(Q K^T / sqrt(hd) + mask) V for one head, given the
// output gradient dO, the output O and the row log-sum-exp the forward kept
// ("Training throughput baseline", Fused attention: the backward runs as two
// kernels, one complete inside a query tile (dQ) and one inside a key tile
// (dK, dV), both rebuilding the probabilities from the stored log-sum-exp, with
// the softmax row sum D_i = dO_i . O_i taken from the output gradient and the
// output; no atomics):
//   P_ij  = 2^(S_ij log2(e)/sqrt(hd) - lse2_i)          (lse2 in log2 units)
//   dP    = dO V^T,   dS_ij = P_ij (dP_ij - D_i)
//   dQ    = dS K / sqrt(hd)      dK = dS^T Q / sqrt(hd)      dV = P^T dO
// Masks: key j of sequence b exists iff j < len_b; with causal, query i sees
// key j iff j <= i.  Query rows at or past len_b are padding: their dO is
// ignored (dQ = 0 there) and they add nothing to dK and dV.  A 64-row step no mask
// touches for any row of an elementwise warp (all but the ones at len_b or across the
// diagonal) takes a body without the per-pair test.
//
// One kernel template serves both directions.  A CTA owns 128 resident rows
// (queries for dQ, keys for dK/dV) and streams 64-row tiles of the other side:
//   dQ : resident Q, dO;   streamed K_j, V_j;  S = Q K_j^T, dP = dO V_j^T,
//        dQ += dS K_j
//   dKV: resident K, V;    streamed Q_j, dO_j; S^T = K Q_j^T, dP^T = V dO_j^T,
//        dV += P^T dO_j, dK += dS^T Q_j
// Thread = TMEM lane = resident row; the elementwise step turns S and dP into
// P and dS as fp16 pairs written over S and dP, which the next MMAs read as A
// operands from tensor memory.  Warps: 0 MMA issuer and TMEM owner, 1 TMA
// producer, 2-5 elementwise and output.  Work items (b, h, 128-row block) are
// dealt round-robin, heaviest first under causal.  dQ double-buffers S in tensor
// memory (it has room beside dP and one accumulator): the next step's S, and its dP
// once the elementwise warps hold the current dP in registers, are computed while
// those warps work, so the tensor core no longer waits for each step's elementwise
// pass.  dK/dV fills tensor memory with S, dP and two accumulators and runs each step
// after the previous one's elementwise pass.
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace tfl {

namespace {

template <int HD, int MODE>
struct BwdCfg {
  static constexpr int BM = 128;                 // resident rows
  static constexpr int BN = 64;                  // streamed rows per step
  static constexpr int ROWB = HD * 2;            // bytes per row (one swizzle atom: HD <= 64)
  static constexpr uint32_t SWZ = ROWB == 64 ? kSw64 : kSw128;
  static constexpr int RES = BM * ROWB;          // one resident tile
  static constexpr int STEP = BN * ROWB;         // one streamed tile
  // stages of streamed tile pairs: dQ pipelines the next step's S and dP under the current
  // step's elementwise work, so a stage frees one step later there
  static constexpr int NST = MODE == 0 ? 3 : 2;
  // tensor memory: dQ keeps two S buffers (step parity) beside dP and the accumulator;
  // dK/dV holds S, dP and two accumulators
  static constexpr int S_COL = 0, DP_COL = MODE == 0 ? 128 : 64, ACC_COL = MODE == 0 ? 192 : 128;
  static constexpr int TMEM_COLS = 256;
  static constexpr int STAGE_F = MODE == 1 ? 2 * 2 * BN : 0;  // lse2 / D of the step's queries, two buffers
  static constexpr size_t SMEM = 1024 + 2 * (size_t)RES + (size_t)NST * 2 * STEP + STAGE_F * 4 + 256;
};

struct BwdItem {
  int b, h, blk, len;
};

// Work item i (heaviest first under causal): dQ takes the last query blocks first,
// dK/dV the first key blocks (they see the most queries).  False when the block is
// all padding.
template <int MODE>
__device__ __forceinline__ bool bwd_item(int i, const AttnBwdArgs& a, int nblk, BwdItem& it) {
  const int bh = a.B * a.H;
  const int r = i / bh, j = i - r * bh;
  it.blk = MODE == 0 ? nblk - 1 - r : r;
  it.b = j / a.H;
  it.h = j - it.b * a.H;
  it.len = seq_len(a.c.lengths, it.b, a.c.S);
  return it.blk * 128 < it.len;
}

// The streamed 64-row steps of an item: dQ -- key sub-blocks [0, kend);
// dK/dV -- query sub-blocks from the first query that can see the block to len.
template <int MODE>
__device__ __forceinline__ void bwd_steps(const BwdItem& it, int causal, int& s0, int& s1) {
  if (MODE == 0) {
    const int kend = causal ? min((it.blk + 1) * 128, it.len) : it.len;
    s0 = 0;
    s1 = (kend + 63) / 64;
  } else {
    s0 = causal ? it.blk * 2 : 0;
    s1 = (it.len + 63) / 64;
  }
}

__device__ __forceinline__ void elem_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

}  // namespace

template <int HD, int MODE>
__global__ void __launch_bounds__(192, 2)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmDO,
                    const AttnBwdArgs args) {
  using C = BwdCfg<HD, MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA1 = smem;                 // dQ: Q    dKV: K
  uint8_t* sA2 = sA1 + C::RES;         // dQ: dO   dKV: V
  uint8_t* sB = sA2 + C::RES;          // stages: [B1 | B2]  (dQ: K_j, V_j; dKV: Q_j, dO_j)
  float* stagef = reinterpret_cast<float*>(sB + (size_t)C::NST * 2 * C::STEP);
  uint64_t* bars = reinterpret_cast<uint64_t*>(stagef + C::STAGE_F);
  uint64_t* res_full = bars + 0;
  uint64_t* res_empty = bars + 1;
  uint64_t* s_full = bars + 2;
  uint64_t* x_full = bars + 3;
  uint64_t* acc_full = bars + 4;
  uint64_t* acc_empty = bars + 5;
  uint64_t* drain = bars + 6;
  uint64_t* dp_read = bars + 7;           // dQ: elementwise -> MMA, the step's dP is in registers
  uint64_t* b_full = bars + 8;            // [NST]
  uint64_t* b_empty = b_full + C::NST;    // [NST]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b_empty + C::NST);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* never_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(res_full, 1);
    mbar_init(res_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(x_full, 4);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    mbar_init(dp_read, 4);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    *abort_flag = 0;
    *never_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{args.c.status, abort_flag, args.c.timeout_ns};

  const int S = args.c.S, D = args.H * HD;
  const int nblk = (S + 127) / 128;
  const int items = args.B * args.H * nblk;
  uint32_t issued_mask = 0, issued_par = 0;
  bool res_issued = false;
  uint32_t res_par = 0;
  bool mma_issued = false;

  if (warp == 1) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQKV);
      tma_prefetch_desc(&tmDO);
      int st = 0;
      uint32_t sph = 0, rph = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
        BwdItem it;
        if (!bwd_item<MODE>(i, args, nblk, it)) continue;
        int s0, s1;
        bwd_steps<MODE>(it, args.causal, s0, s1);
        // resident tiles (two 64-row boxes each), once the previous item's MMAs are done with them
        if (!wait_bounded(res_empty, rph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(res_full, 2 * C::RES);
        const int r0 = it.blk * 128;
        for (int hh = 0; hh < 2; ++hh) {
          if (MODE == 0) {
            tma_load_3d(sA1 + hh * C::STEP, &tmQKV, res_full, it.h * HD, r0 + 64 * hh, it.b);
            tma_load_3d(sA2 + hh * C::STEP, &tmDO, res_full, it.h * HD, r0 + 64 * hh, it.b);
          } else {
            tma_load_3d(sA1 + hh * C::STEP, &tmQKV, res_full, D + it.h * HD, r0 + 64 * hh, it.b);
            tma_load_3d(sA2 + hh * C::STEP, &tmQKV, res_full, 2 * D + it.h * HD, r0 + 64 * hh, it.b);
          }
        }
        res_issued = true;
        res_par = rph;
        rph ^= 1u;
        for (int s = s0; s < s1; ++s) {
          if (!wait_bounded(&b_empty[st], sph ^ 1u, wc)) {
            ok = false;
            break;
          }
          uint8_t* b1 = sB + (size_t)st * 2 * C::STEP;
          mbar_arrive_expect_tx(&b_full[st], 2 * C::STEP);
          if (MODE == 0) {
            tma_load_3d(b1, &tmQKV, &b_full[st], D + it.h * HD, 64 * s, it.b);
            tma_load_3d(b1 + C::STEP, &tmQKV, &b_full[st], 2 * D + it.h * HD, 64 * s, it.b);
          } else {
            tma_load_3d(b1, &tmQKV, &b_full[st], it.h * HD, 64 * s, it.b);
            tma_load_3d(b1 + C::STEP, &tmDO, &b_full[st], it.h * HD, 64 * s, it.b);
          }
          issued_mask |= 1u << st;
          issued_par = (issued_par & ~(1u << st)) | (sph << st);
          if (++st == C::NST) {
            st = 0;
            sph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16(128, 64, 0, 0);
      constexpr uint32_t id_acc = idesc_f16(128, HD, 0, 1);
      const uint32_t a1 = smem_u32(sA1), a2 = smem_u32(sA2);
      int st = 0;
      uint32_t sph = 0, rph = 0, xph = 0, aph = 0, dph = 0;
      bool first_item = true, ok = true;
      for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
        BwdItem it;
        if (!bwd_item<MODE>(i, args, nblk, it)) continue;
        int s0, s1;
        bwd_steps<MODE>(it, args.causal, s0, s1);
        if (!wait_bounded(res_full, rph, wc)) break;
        rph ^= 1u;
        if (!first_item) {  // the accumulators were read out for the previous item
          if (!wait_bounded(acc_empty, aph, wc)) break;
          aph ^= 1u;
        }
        tc_fence_after();
        if constexpr (MODE == 0) {
          // dQ, pipelined: S of step s goes to S buffer (s - s0) & 1 as soon as its tiles are
          // in (that buffer last held dS of step s - 2, read by the dQ MMAs issued before);
          // dP of step s once the elementwise warps have dP of step s - 1 in registers.  The
          // next step's S and dP thus compute while the elementwise warps work on the current
          // one.  Step s is released to them (s_full) only after x_full of step s - 1 is seen,
          // so neither barrier runs more than one phase ahead of its waiter; then dQ += dS K
          // of step s - 1.
          int prev_st = 0;  // stage of step s - 1
          for (int s = s0; s <= s1 && ok; ++s) {
            int cur_st = st;
            if (s < s1) {
              if (!wait_bounded(&b_full[st], sph, wc)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t b1 = smem_u32(sB + (size_t)st * 2 * C::STEP), b2 = b1 + C::STEP;
              const uint64_t ad1 = sdesc(a1, 16, 8 * C::ROWB, C::SWZ), ad2 = sdesc(a2, 16, 8 * C::ROWB, C::SWZ);
              const uint64_t bd1 = sdesc(b1, 16, 8 * C::ROWB, C::SWZ), bd2 = sdesc(b2, 16, 8 * C::ROWB, C::SWZ);
              const uint32_t s_col = C::S_COL + 64 * ((s - s0) & 1);
#pragma unroll
              for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (uint32_t)((kk * 32) >> 4);
                umma_f16(tmem_base + s_col, ad1 + off, bd1 + off, id_s, kk > 0 ? 1u : 0u);
              }
              if (s > s0) {
                if (!wait_bounded(dp_read, dph, wc)) {
                  ok = false;
                  break;
                }
                dph ^= 1u;
                tc_fence_after();
              }
#pragma unroll
              for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (uint32_t)((kk * 32) >> 4);
                umma_f16(tmem_base + C::DP_COL, ad2 + off, bd2 + off, id_s, kk > 0 ? 1u : 0u);
              }
              mma_issued = true;
              if (++st == C::NST) {
                st = 0;
                sph ^= 1u;
              }
            } else if (s > s0) {
              // the last step's dP read (every step's dp_read phase is consumed once)
              if (!wait_bounded(dp_read, dph, wc)) {
                ok = false;
                break;
              }
              dph ^= 1u;
            }
            if (s > s0) {
              if (!wait_bounded(x_full, xph, wc)) {
                ok = false;
                break;
              }
              xph ^= 1u;
              tc_fence_after();
            }
            if (s < s1) umma_commit(s_full);
            if (s > s0) {
              const uint64_t bd1 = sdesc(smem_u32(sB + (size_t)prev_st * 2 * C::STEP), C::STEP, 8 * C::ROWB, C::SWZ);
              const uint32_t ds_col = C::S_COL + 64 * ((s - 1 - s0) & 1);
              const bool acc0 = s - 1 > s0;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t off = (uint32_t)((kk * 16 * C::ROWB) >> 4);
                umma_f16_ts(tmem_base + C::ACC_COL, tmem_base + ds_col + 8 * kk, bd1 + off, id_acc,
                            (acc0 || kk > 0) ? 1u : 0u);
              }
              umma_commit(&b_empty[prev_st]);
            }
            prev_st = cur_st;
          }
        } else {
        int pst = 0;  // stage of the step whose second half (accumulating MMAs) is pending
        for (int s = s0; s <= s1 && ok; ++s) {
          if (s < s1) {
            // S and dP of step s; for s > s0 the accumulating MMAs of step s - 1 are issued
            // first below, so these overwrite its P / dS only after they have been read
            if (!wait_bounded(&b_full[st], sph, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (s > s0) {
            if (!wait_bounded(x_full, xph, wc)) {
              ok = false;
              break;
            }
            xph ^= 1u;
            tc_fence_after();
            const uint32_t pb1 = smem_u32(sB + (size_t)pst * 2 * C::STEP);
            const uint32_t pb2 = pb1 + C::STEP;
            const uint64_t bd1 = sdesc(pb1, C::STEP, 8 * C::ROWB, C::SWZ);
            const uint64_t bd2 = sdesc(pb2, C::STEP, 8 * C::ROWB, C::SWZ);
            const bool acc0 = s - 1 > s0;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t off = (uint32_t)((kk * 16 * C::ROWB) >> 4);
              if (MODE == 0) {
                umma_f16_ts(tmem_base + C::ACC_COL, tmem_base + C::S_COL + 8 * kk, bd1 + off, id_acc,
                            (acc0 || kk > 0) ? 1u : 0u);
              } else {
                umma_f16_ts(tmem_base + C::ACC_COL, tmem_base + C::S_COL + 8 * kk, bd2 + off, id_acc,
                            (acc0 || kk > 0) ? 1u : 0u);
                umma_f16_ts(tmem_base + C::ACC_COL + HD, tmem_base + C::DP_COL + 8 * kk, bd1 + off, id_acc,
                            (acc0 || kk > 0) ? 1u : 0u);
              }
            }
            umma_commit(&b_empty[pst]);
          }
          if (s < s1) {
            const uint32_t b1 = smem_u32(sB + (size_t)st * 2 * C::STEP), b2 = b1 + C::STEP;
            const uint64_t ad1 = sdesc(a1, 16, 8 * C::ROWB, C::SWZ), ad2 = sdesc(a2, 16, 8 * C::ROWB, C::SWZ);
            const uint64_t bd1 = sdesc(b1, 16, 8 * C::ROWB, C::SWZ), bd2 = sdesc(b2, 16, 8 * C::ROWB, C::SWZ);
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
              const uint32_t off = (uint32_t)((kk * 32) >> 4);
              umma_f16(tmem_base + C::S_COL, ad1 + off, bd1 + off, id_s, kk > 0 ? 1u : 0u);
              umma_f16(tmem_base + C::DP_COL, ad2 + off, bd2 + off, id_s, kk > 0 ? 1u : 0u);
            }
            mma_issued = true;
            umma_commit(s_full);
            pst = st;
            if (++st == C::NST) {
              st = 0;
              sph ^= 1u;
            }
          }
        }
        }
        if (!ok) break;
        umma_commit(res_empty);
        umma_commit(acc_full);
        first_item = false;
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise + output (warps 2-5)
    const int q = warp & 3;
    const int t = threadIdx.x - 64;  // 0..127
    const int r = q * 32 + lane;     // resident row == TMEM lane
    const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16);
    const float sl2 = args.scale_log2;
    // dK/dV's elementwise warps meet at a named barrier each step: they leave only on their own
    // bound, never on another waiter's abort, so that all four leave at the same point
    WaitCtl ewc = wc;
    ewc.early_exit = MODE == 0;
    uint32_t sph = 0, aph = 0;
    int sbuf = 0;
    for (int i = blockIdx.x; i < items; i += gridDim.x) {
      BwdItem it;
      if (!bwd_item<MODE>(i, args, nblk, it)) continue;
      int s0, s1;
      bwd_steps<MODE>(it, args.causal, s0, s1);
      const int row = it.blk * 128 + r;             // resident position (query for dQ, key for dK/dV)
      const size_t bhS = ((size_t)it.b * args.H + it.h) * S;
      float lse_r = 0.f, d_r = 0.f;
      if (MODE == 0 && row < it.len) {
        lse_r = args.lse[bhS + row];
        d_r = args.delta[bhS + row];
      }
      bool ok = true;
      for (int s = s0; s < s1; ++s) {
        const int c0 = 64 * s;  // first streamed position of the step
        float* sf = stagef + sbuf * 2 * 64;
        if (MODE == 1) {  // the step's queries: lse2 and D (0 past len)
          const int qi = c0 + (t & 63);
          const float v = qi < it.len ? (t < 64 ? args.lse[bhS + qi] : args.delta[bhS + qi]) : 0.f;
          sf[t] = v;
          elem_bar();
        }
        if (!wait_bounded(s_full, sph, ewc)) {
          ok = false;
          break;
        }
        sph ^= 1u;
        tc_fence_after();
        // A step no mask touches for any of this warp's rows (every row and column inside
        // len_b and, under causal, every pair on the allowed side) skips the per-pair test.
        const int wr0 = it.blk * 128 + q * 32;  // this warp's first resident row
        const bool unmasked = wr0 + 31 < it.len && c0 + 63 < it.len &&
                              (!args.causal || (MODE == 0 ? c0 + 63 <= wr0 : wr0 + 31 <= c0));
        // P and dS of 32 columns of the step (half 0 or 1) from S and dP in registers
        auto ew_half = [&](auto full_tag, int half, const float* sv, const float* dv, uint32_t* pp, uint32_t* dd) {
          constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
          for (int e0 = 0; e0 < 32; e0 += 8) {
            // the 8 columns' log-sum-exp and row sums: per-thread constants for dQ (row =
            // query), per column from the step's shared staging for dK/dV (row = key)
            float lse8[8], d8[8];
            if (MODE == 0) {
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                lse8[k] = lse_r;
                d8[k] = d_r;
              }
            } else {
              const float4* l4 = reinterpret_cast<const float4*>(sf + 32 * half + e0);
              const float4* d4 = reinterpret_cast<const float4*>(sf + 64 + 32 * half + e0);
              const float4 la = l4[0], lb = l4[1], da = d4[0], db = d4[1];
              lse8[0] = la.x; lse8[1] = la.y; lse8[2] = la.z; lse8[3] = la.w;
              lse8[4] = lb.x; lse8[5] = lb.y; lse8[6] = lb.z; lse8[7] = lb.w;
              d8[0] = da.x; d8[1] = da.y; d8[2] = da.z; d8[3] = da.w;
              d8[4] = db.x; d8[5] = db.y; d8[6] = db.z; d8[7] = db.w;
            }
#pragma unroll
            for (int e = e0; e < e0 + 8; e += 2) {
              float p2[2], ds2[2];
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int col = c0 + 32 * half + e + k;  // streamed position
                bool allowed = true;
                if constexpr (!FULL)
                  allowed = MODE == 0 ? (row < it.len && col < it.len && (!args.causal || col <= row))
                                      : (row < it.len && col < it.len && (!args.causal || row <= col));
                const float p = allowed ? ex2(fmaf(sv[e + k], sl2, -lse8[e - e0 + k])) : 0.f;
                p2[k] = p;
                ds2[k] = p * (dv[e + k] - d8[e - e0 + k]);
              }
              const __half2 hp = __floats2half2_rn(p2[0], p2[1]);
              const __half2 hd = __floats2half2_rn(ds2[0], ds2[1]);
              pp[e / 2] = *reinterpret_cast<const uint32_t*>(&hp);
              dd[e / 2] = *reinterpret_cast<const uint32_t*>(&hd);
            }
          }
        };
        auto step = [&](auto full_tag) {
          if constexpr (MODE == 0) {
            // dQ: the whole dP and the first half of S come in together; once dP is in
            // registers the MMA thread may compute the next step's dP, and the next step's
            // S already goes to the other S buffer.  dS is written over this step's S.
            const uint32_t s_buf = t_row + C::S_COL + 64 * ((s - s0) & 1);
            float sv[32], dv[32], dn[32];
            uint32_t pp[16], dd[16];
            tmem_ld32(s_buf, sv);
            tmem_ld32(t_row + C::DP_COL, dv);
            tmem_ld32(t_row + C::DP_COL + 32, dn);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dp_read);
            ew_half(full_tag, 0, sv, dv, pp, dd);
            tmem_st16_u(s_buf, dd);  // dS over S, columns 0-31 of the step
            tmem_ld32(s_buf + 32, sv);
            tmem_wait_ld();
            ew_half(full_tag, 1, sv, dn, pp, dd);
            tmem_st16_u(s_buf + 16, dd);
          } else {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              float sv[32], dv[32];
              tmem_ld32(t_row + C::S_COL + 32 * half, sv);
              tmem_ld32(t_row + C::DP_COL + 32 * half, dv);
              tmem_wait_ld();
              uint32_t pp[16], dd[16];
              ew_half(full_tag, half, sv, dv, pp, dd);
              tmem_st16_u(t_row + C::S_COL + 16 * half, pp);   // P^T over S^T
              tmem_st16_u(t_row + C::DP_COL + 16 * half, dd);  // dS^T over dP^T
            }
          }
        };
        if (unmasked)
          step(std::true_type{});
        else
          step(std::false_type{});
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(x_full);
        sbuf ^= 1;
      }
      if (!ok) break;
      // ---- accumulators out: fp32 rows of dqkv (rows past len stay as the caller cleared them)
      if (!wait_bounded(acc_full, aph, ewc)) break;
      aph ^= 1u;
      tc_fence_after();
      const float inv_sqrt = args.inv_sqrt_hd;
#pragma unroll 1
      for (int which = 0; which < (MODE == 0 ? 1 : 2); ++which) {
        // dQ: cols h*HD (scaled); dK/dV: dV at 2D + h*HD (acc 0), dK at D + h*HD (acc 1, scaled)
        const float sc = (MODE == 1 && which == 0) ? 1.0f : inv_sqrt;
        const int col0 = MODE == 0 ? it.h * HD : (which == 0 ? 2 * D : D) + it.h * HD;
        float* dst = args.dqkv + ((size_t)it.b * S + row) * (3 * D) + col0;
#pragma unroll 1
        for (int c = 0; c < HD; c += 32) {
          float v[32];
          tmem_ld32(t_row + C::ACC_COL + which * HD + c, v);
          tmem_wait_ld();
          if (row < it.len) {
            float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              d4[k] = make_float4(v[4 * k] * sc, v[4 * k + 1] * sc, v[4 * k + 2] * sc, v[4 * k + 3] * sc);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    const WaitCtl dc{args.c.status, never_flag, 100000000LL};
    if (warp == 1 && lane == 0) {
      if (res_issued) wait_bounded(res_full, res_par, dc);
      for (int s = 0; s < C::NST; ++s)
        if (issued_mask & (1u << s)) wait_bounded(&b_full[s], (issued_par >> s) & 1u, dc);
    }
    if (warp == 0 && lane == 0 && mma_issued) {
      umma_commit(drain);
      wait_bounded(drain, 0, dc);
    }
    __syncthreads();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// D[b, h, i] = dO_i . O_i over the head's columns, for i < len_b (0 past it).
__global__ void attn_bwd_delta_kernel(const __half* dout, const __half* o, float* delta, int B, int S, int H, int hd,
                                      const int* lengths) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // (b, i, h), h fastest
  if (idx >= (size_t)B * S * H) return;
  const int h = (int)(idx % H);
  const size_t bi = idx / H;
  const int b = (int)(bi / S), i = (int)(bi % S);
  float acc = 0.f;
  if (i < seq_len(lengths, b, S)) {
    const size_t off = bi * (size_t)H * hd + (size_t)h * hd;
    const uint4* a = reinterpret_cast<const uint4*>(dout + off);
    const uint4* c = reinterpret_cast<const uint4*>(o + off);
    for (int k = 0; k < hd / 8; ++k) {
      const uint4 x = a[k], y = c[k];
      const __half2* xh = reinterpret_cast<const __half2*>(&x);
      const __half2* yh = reinterpret_cast<const __half2*>(&y);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xf = __half22float2(xh[e]), yf = __half22float2(yh[e]);
        acc = fmaf(xf.x, yf.x, fmaf(xf.y, yf.y, acc));
      }
    }
  }
  delta[((size_t)b * H + h) * S + i] = acc;
}

template <int HD, int MODE>
static cudaError_t launch_bwd_one(const CUtensorMap& tqkv, const CUtensorMap& tdo, const AttnBwdArgs& a, int num_sms,
                                  cudaStream_t s) {
  using C = BwdCfg<HD, MODE>;
  const int items = a.B * a.H * ((a.c.S + 127) / 128);
  const int cap = 2 * num_sms;  // two CTAs per SM (256 TMEM columns, ~66-100 KB shared memory each)
  const int grid = items < cap ? items : cap;
  if (grid <= 0) return cudaSuccess;
  attn_bwd_kernel<HD, MODE><<<grid, 192, C::SMEM, s>>>(tqkv, tdo, a);
  return cudaGetLastError();
}

cudaError_t prepare_attention_bwd_kernels() {
  cudaError_t e = cudaSuccess;
  auto set = [&](auto kern, size_t bytes) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  };
  set(attn_bwd_kernel<32, 0>, BwdCfg<32, 0>::SMEM);
  set(attn_bwd_kernel<32, 1>, BwdCfg<32, 1>::SMEM);
  set(attn_bwd_kernel<64, 0>, BwdCfg<64, 0>::SMEM);
  set(attn_bwd_kernel<64, 1>, BwdCfg<64, 1>::SMEM);
  return e;
}

cudaError_t launch_attention_bwd(int hd, const CUtensorMap& tqkv, const CUtensorMap& tdo, const AttnBwdArgs& a,
                                 const __half* dout, const __half* o, int num_sms, cudaStream_t s) {
  const size_t n = (size_t)a.B * a.c.S * a.H;
  attn_bwd_delta_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(dout, o, a.delta, a.B, a.c.S, a.H, hd,
                                                                    a.c.lengths);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  switch (hd) {
    case 32:
      if ((e = launch_bwd_one<32, 0>(tqkv, tdo, a, num_sms, s)) != cudaSuccess) return e;
      return launch_bwd_one<32, 1>(tqkv, tdo, a, num_sms, s);
    case 64:
      if ((e = launch_bwd_one<64, 0>(tqkv, tdo, a, num_sms, s)) != cudaSuccess) return e;
      return launch_bwd_one<64, 1>(tqkv, tdo, a, num_sms, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tfl
