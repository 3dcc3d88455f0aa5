// attention.cu -- flash attention forward on tcgen05 tensor cores.
//
// Per (sequence b, head h, block of 128 queries) the kernel computes
// O = softmax(Q K^T / sqrt(hd) + mask) V without materialising the score
// matrix ("TikTok TechJam 2026 -- Problem 3", section 2.1):
//   * S = Q K_j^T for one key block at a time goes to tensor memory (fp32).
//   * Online softmax in fp32, one query row per thread (the row's TMEM lane):
//     running max m, running sum l, O rescaled by exp(m_old - m_new)
//     (section 2.1, the running-max recurrence).  The rescale is lazy: the
//     reference max only moves when the row max grew by more than 8 in log2
//     units, so P <= 2^8 and O is touched rarely; O / l is exact either way.
//   * P = exp2(S * log2(e)/sqrt(hd) - m) in fp16 goes to tensor memory (two
//     values per column) and O += P V_j takes its A operand from there
//     (tcgen05.mma with A in TMEM), so only V is read from shared memory.
//   * Causal: key blocks above the diagonal are never loaded (block skipping,
//     section 1.C); the mask is applied only on the diagonal block; the key
//     mask is not applied at all, because for a valid query i every key j <= i
//     is valid (section 2.1, "the mask trick").
//   * Key padding (non-causal): only the block holding len_b is masked.
//   * Query blocks past len_b are skipped; their output rows are never read
//     for a valid token.
// q, k, v are strided views of the fused QKV output [B, S, 3D] (section 1.A,
// head-split copies removed); O is written straight into [B, S, H*hd].
//
// Warp roles: warps 0-3 softmax + output (thread = query row), warp 4 TMA
// producer (Q once per work item, K/V blocks into an NST-deep ring), warp 5
// MMA issuer and TMEM owner.  Persistent CTAs claim work items from a global
// atomic counter, heaviest first (causal: the last query blocks have the most
// keys); the producer publishes each claimed item to the other warps through
// a small shared-memory ring.
//
// Softmax fast path: for key blocks after the first, P is computed in one
// pass over S with the running max as the exponent reference while the block
// max is tracked; only when a row's max grew by more than 2^8 does its warp
// redo the block with the two-pass path (block max, rescale O, exponentials).
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "xpose.cuh"

namespace tfl {

template <int HD>
struct AttnCfg {
  static constexpr int BM = kAttnBM;
  static constexpr int BN = attn_block_n(HD);      // keys per block
  static constexpr int ATOM_C = HD < 64 ? HD : 64;  // head-dim columns per TMA box / swizzle atom
  static constexpr int NATOM = HD / ATOM_C;
  static constexpr int ROWB = ATOM_C * 2;           // bytes of one row inside an atom
  static constexpr uint32_t SWZ = ROWB == 64 ? kSw64 : kSw128;
  static constexpr int Q_BYTES = BM * HD * 2;
  static constexpr int KV_BYTES = BN * HD * 2;      // one K (or V) block
  static constexpr int XP_BYTES = 4 * 32 * 128;     // output transpose stage, one per softmax warp
  static constexpr int NST = HD == 32 ? 4 : 2;
  static constexpr int CTAS_PER_SM = HD <= 64 ? 2 : 1;
  // tensor memory: S [0, BN), P (fp16 pairs) [BN, BN + BN/2), O from O_COL
  static constexpr int P_COL = BN;
  static constexpr int O_COL = HD <= 64 ? 192 : 256;
  static constexpr int TMEM_COLS = O_COL + HD <= 256 ? 256 : 512;
  static constexpr size_t SMEM = 1024 + Q_BYTES + (size_t)NST * 2 * KV_BYTES + XP_BYTES + 384;
};

size_t attn_smem_bytes(int hd) {
  switch (hd) {
    case 32: return AttnCfg<32>::SMEM;
    case 64: return AttnCfg<64>::SMEM;
    case 256: return AttnCfg<256>::SMEM;
  }
  return 0;
}

struct Item {
  int b, h, qb, len, nkb;
};

constexpr int kItemRing = 4;

// Work item i (heaviest first) -> (b, h, query block); false if the block is all padding.
__device__ __forceinline__ bool decode_item(int i, const AttnArgs& a, int nqb, int bn, Item& it) {
  const int bh_count = a.B * a.H;
  const int qr = i / bh_count, bh = i - qr * bh_count;
  it.qb = nqb - 1 - qr;
  it.b = bh / a.H;
  it.h = bh - it.b * a.H;
  it.len = seq_len(a.c.lengths, it.b, a.c.S);
  if (it.qb * kAttnBM >= it.len) return false;
  const int kend = a.causal ? min((it.qb + 1) * kAttnBM, it.len) : it.len;
  it.nkb = (kend + bn - 1) / bn;
  return true;
}

template <int HD>
__global__ void __launch_bounds__(192, AttnCfg<HD>::CTAS_PER_SM)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                const AttnArgs args) {
  using C = AttnCfg<HD>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::Q_BYTES;
  uint8_t* sV = sK + (size_t)C::NST * C::KV_BYTES;
  uint8_t* sX = sV + (size_t)C::NST * C::KV_BYTES;  // output transpose stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(sX + C::XP_BYTES);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* s_full = bars + 2;
  uint64_t* p_full = bars + 3;
  uint64_t* o_full = bars + 4;
  uint64_t* o_empty = bars + 5;
  uint64_t* drain = bars + 6;
  uint64_t* kv_full = bars + 7;
  uint64_t* kv_empty = kv_full + C::NST;
  uint64_t* it_full = kv_empty + C::NST;
  uint64_t* it_empty = it_full + kItemRing;
  int* it_slot = reinterpret_cast<int*>(it_empty + kItemRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(it_slot + kItemRing);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* never_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(o_full, 1);
    mbar_init(o_empty, 4);
    mbar_init(drain, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(&it_full[s], 1);
      mbar_init(&it_empty[s], 5);  // the MMA warp and the four softmax warps
    }
    *abort_flag = 0;
    *never_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmKV);
  }
  if (warp == 5) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{args.c.status, abort_flag, args.c.timeout_ns};

  const int S = args.c.S, D = args.D;
  const int nqb = (S + kAttnBM - 1) / kAttnBM;
  const int items = args.B * args.H * nqb;

  uint32_t issued_mask = 0, issued_par = 0;  // producer: stages with loads in flight (abort path)
  bool q_issued = false;
  uint32_t q_par = 0;
  bool mma_issued = false;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer + scheduler
    if (lane == 0) {
      int st = 0, ik = 0;
      uint32_t kvph = 0, qph = 0, itph = 0;
      bool ok = true;
      while (ok) {
        // claim the next work item that holds a valid query (heaviest first)
        int i;
        Item it;
        do {
          i = atomicAdd(args.counter, 1);
        } while (i < items && !decode_item(i, args, nqb, BN, it));
        if (i >= items) i = -1;
        if (!wait_bounded(&it_empty[ik], itph ^ 1u, wc)) break;
        it_slot[ik] = i;
        mbar_arrive(&it_full[ik]);
        if (++ik == kItemRing) {
          ik = 0;
          itph ^= 1u;
        }
        if (i < 0) break;
        if (!wait_bounded(q_empty, qph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
        for (int a = 0; a < C::NATOM; ++a)
          tma_load_3d(sQ + a * (kAttnBM * C::ROWB), &tmQ, q_full, it.h * HD + a * C::ATOM_C, it.qb * kAttnBM, it.b);
        q_issued = true;
        q_par = qph;
        qph ^= 1u;
        for (int j = 0; j < it.nkb; ++j) {
          if (!wait_bounded(&kv_empty[st], kvph ^ 1u, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&kv_full[st], 2 * C::KV_BYTES);
          uint8_t* k = sK + (size_t)st * C::KV_BYTES;
          uint8_t* v = sV + (size_t)st * C::KV_BYTES;
#pragma unroll
          for (int a = 0; a < C::NATOM; ++a) {
            tma_load_3d(k + a * (BN * C::ROWB), &tmKV, &kv_full[st], D + it.h * HD + a * C::ATOM_C, j * BN, it.b);
            tma_load_3d(v + a * (BN * C::ROWB), &tmKV, &kv_full[st], 2 * D + it.h * HD + a * C::ATOM_C, j * BN,
                        it.b);
          }
          issued_mask |= 1u << st;
          issued_par = (issued_par & ~(1u << st)) | (kvph << st);
          if (++st == C::NST) {
            st = 0;
            kvph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    constexpr uint32_t idesc_qk = idesc_f16(128, BN, 0, 0);
    constexpr uint32_t idesc_pv = idesc_f16(128, HD, 0, 1);
    const uint32_t d_s = tmem_base;
    const uint32_t d_o = tmem_base + C::O_COL;
    int st = 0, ik = 0;
    uint32_t kvph = 0, qph = 0, pph = 0, oeph = 0, itph = 0;
    bool first_item = true, ok = true;
    const uint32_t t_p = tmem_base + C::P_COL;
    auto issue_pv = [&](int pst, bool accumulate) {
      const uint32_t sv = smem_u32(sV + (size_t)pst * C::KV_BYTES);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t bd = sdesc(sv + kk * 16 * C::ROWB, BN * C::ROWB, 8 * C::ROWB, C::SWZ);
        umma_f16_ts(d_o, t_p + kk * 8, bd, idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
      }
    };
    while (ok) {
      if (!wait_bounded(&it_full[ik], itph, wc)) break;
      const int i = it_slot[ik];
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[ik]);
      if (++ik == kItemRing) {
        ik = 0;
        itph ^= 1u;
      }
      if (i < 0) break;
      Item it;
      decode_item(i, args, nqb, BN, it);
      if (!wait_bounded(q_full, qph, wc)) break;
      qph ^= 1u;
      tc_fence_after();
      bool need_oe = !first_item;
      int prev_st = 0;
      for (int j = 0; j < it.nkb; ++j) {
        if (!wait_bounded(&kv_full[st], kvph, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Keys at or past len_b in this block: clear their V rows so stale
        // workspace contents can never reach O through a zero probability.
        const int vrow0 = it.len - j * BN;
        if (vrow0 < BN) {
          uint8_t* v = sV + (size_t)st * C::KV_BYTES;
          for (int rr = max(vrow0, 0) + lane; rr < BN; rr += 32) {
#pragma unroll
            for (int a = 0; a < C::NATOM; ++a) {
              uint4* row = reinterpret_cast<uint4*>(v + a * (BN * C::ROWB) + rr * C::ROWB);
#pragma unroll
              for (int c = 0; c < C::ROWB / 16; ++c) row[c] = make_uint4(0, 0, 0, 0);
            }
          }
          fence_async_smem();
          __syncwarp();
        }
        if (j > 0) {
          if (!wait_bounded(p_full, pph, wc)) {
            ok = false;
            break;
          }
          pph ^= 1u;
          if (need_oe) {
            if (!wait_bounded(o_empty, oeph, wc)) {
              ok = false;
              break;
            }
            oeph ^= 1u;
            need_oe = false;
          }
          tc_fence_after();
          if (lane == 0) {
            issue_pv(prev_st, j - 1 > 0);
            umma_commit(&kv_empty[prev_st]);
          }
        }
        if (lane == 0) {
          const uint32_t sq = smem_u32(sQ), sk = smem_u32(sK + (size_t)st * C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const int a = kk / (C::ATOM_C / 16), w = kk % (C::ATOM_C / 16);
            const uint64_t ad = sdesc(sq + a * (kAttnBM * C::ROWB) + w * 32, 16, 8 * C::ROWB, C::SWZ);
            const uint64_t bd = sdesc(sk + a * (BN * C::ROWB) + w * 32, 16, 8 * C::ROWB, C::SWZ);
            umma_f16(d_s, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_issued = true;
          umma_commit(s_full);
          if (j == it.nkb - 1) umma_commit(q_empty);
        }
        __syncwarp();
        prev_st = st;
        if (++st == C::NST) {
          st = 0;
          kvph ^= 1u;
        }
      }
      if (!ok) break;
      if (!wait_bounded(p_full, pph, wc)) break;
      pph ^= 1u;
      if (need_oe) {
        if (!wait_bounded(o_empty, oeph, wc)) break;
        oeph ^= 1u;
      }
      tc_fence_after();
      if (lane == 0) {
        issue_pv(prev_st, it.nkb > 1);
        umma_commit(&kv_empty[prev_st]);
        umma_commit(o_full);
      }
      __syncwarp();
      first_item = false;
    }
  } else {
    // ------------------------------------------------------------ softmax + output (warps 0-3)
    const int r = warp * 32 + lane;  // query row within the block == TMEM lane
    const uint32_t t_s = tmem_base + ((uint32_t)(warp * 32) << 16);
    const uint32_t t_o = t_s + C::O_COL;
    const uint32_t t_p = t_s + C::P_COL;
    const float sl2 = args.scale_log2;
    uint32_t sph = 0, oph = 0, itph = 0;
    int ik = 0;
    uint8_t* xst = sX + warp * 4096;

    // exponentials of one 64-key group against reference mref, packed as fp16
    // pairs into this row's 32 P columns of group g; returns the group's sum in
    // four partials and its max.  MASKED: keys past kmax get p = 0 and no max.
    auto exp_group = [&](auto masked, const float* sv, int g, int kbase, int kmax, float mref, float* ls,
                         float* bm) {
      constexpr bool MASKED = decltype(masked)::value;
      uint32_t pk[32];
#pragma unroll
      for (int e2 = 0; e2 < 32; ++e2) {
        float p2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int idx = 2 * e2 + u;
          const float v = sv[idx];
          if constexpr (MASKED) {
            const bool ok2 = kbase + idx <= kmax;
            bm[idx & 3] = ok2 ? fmaxf(bm[idx & 3], v) : bm[idx & 3];
            p2[u] = ok2 ? ex2(fmaf(v, sl2, -mref)) : 0.f;
          } else {
            bm[idx & 3] = fmaxf(bm[idx & 3], v);
            p2[u] = ex2(fmaf(v, sl2, -mref));
          }
          ls[idx & 3] += p2[u];
        }
        const __half2 hp = __floats2half2_rn(p2[0], p2[1]);  // first key in the low half
        pk[e2] = *reinterpret_cast<const uint32_t*>(&hp);
      }
      tmem_st32_u(t_p + g * 32, pk);
    };
    // one pass over S against reference mref: P into TMEM, partial sums and maxima
    auto exp_block = [&](bool need_mask, int k0, int kmax, float mref, float* ls, float* bm) {
#pragma unroll
      for (int g = 0; g < BN / 64; ++g) {
        float sv[64];
        tmem_ld32(t_s + g * 64, sv);
        tmem_ld32(t_s + g * 64 + 32, sv + 32);
        tmem_wait_ld();
        if (need_mask)
          exp_group(std::true_type{}, sv, g, k0 + g * 64, kmax, mref, ls, bm);
        else
          exp_group(std::false_type{}, sv, g, k0 + g * 64, kmax, mref, ls, bm);
      }
    };

    while (true) {
      if (!wait_bounded(&it_full[ik], itph, wc)) break;
      const int i = it_slot[ik];
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[ik]);
      if (++ik == kItemRing) {
        ik = 0;
        itph ^= 1u;
      }
      if (i < 0) break;
      Item it;
      decode_item(i, args, nqb, BN, it);
      const int qpos = it.qb * kAttnBM + r;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < it.nkb; ++j) {
        if (!wait_bounded(s_full, sph, wc)) {
          ok = false;
          break;
        }
        sph ^= 1u;
        tc_fence_after();
        const int k0 = j * BN;
        const bool need_mask = args.causal ? (k0 + BN - 1 > it.qb * kAttnBM) : (k0 + BN > it.len);
        const int kmax = args.causal ? qpos : it.len - 1;  // last allowed key when masking
        bool slow = (j == 0);
        if (!slow) {
          // fast path: exponentials against the running max, block max tracked alongside
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
          float bm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          exp_block(need_mask, k0, kmax, m_run, ls, bm);
          const float bmax = fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3]));
          slow = __any_sync(0xffffffffu, bmax * sl2 > m_run + 8.0f);
          if (!slow) l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        if (slow) {
          // pass 1: block max
          float bm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
          for (int g = 0; g < BN / 64; ++g) {
            float sv[64];
            tmem_ld32(t_s + g * 64, sv);
            tmem_ld32(t_s + g * 64 + 32, sv + 32);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 64; ++e) {
              const bool ok2 = !need_mask || (k0 + g * 64 + e <= kmax);
              bm[e & 3] = ok2 ? fmaxf(bm[e & 3], sv[e]) : bm[e & 3];
            }
          }
          const float bmax = fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3]));
          const float m_new = fmaxf(m_run, bmax * sl2);
          const bool resc = m_new > m_run + 8.0f;
          if (j > 0 && __any_sync(0xffffffffu, resc)) {
            // O holds PV of every earlier block (s_full(j) was committed after PV(j-1)).
            const float alpha = resc ? ex2(m_run - m_new) : 1.0f;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
              float o[32];
              tmem_ld32(t_o + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_st32(t_o + c * 32, o);
            }
            tmem_wait_st();
            l_run *= alpha;
          }
          if (resc) m_run = m_new;
          const float mref = (m_run == -INFINITY) ? 0.f : m_run;
          // pass 2: exponentials
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
          float bm2[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          exp_block(need_mask, k0, kmax, mref, ls, bm2);
          l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) break;
      if (!wait_bounded(o_full, oph, wc)) break;
      oph ^= 1u;
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
      const int q0 = it.qb * kAttnBM + warp * 32;  // first query row of this warp
      const uint32_t rows = __ballot_sync(0xffffffffu, qpos < S);
      __half* orow0 = args.o16 + ((size_t)it.b * S + q0) * D + it.h * HD;
      if constexpr (HD == 32) {
        float o[32];
        tmem_ld32(t_o, o);
        tmem_wait_ld();
        xp_store_f16<32>(xst, lane, o, orow0, nullptr, D, rows, inv);
      } else {
#pragma unroll 1
        for (int c = 0; c < HD / 64; ++c) {
          float o[64];
          tmem_ld32(t_o + c * 64, o);
          tmem_ld32(t_o + c * 64 + 32, o + 32);
          tmem_wait_ld();
          xp_store_f16<64>(xst, lane, o, orow0 + c * 64, nullptr, D, rows, inv);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    const WaitCtl dc{args.c.status, never_flag, 100000000LL};
    if (warp == 4 && lane == 0) {
      if (q_issued) wait_bounded(q_full, q_par, dc);
      for (int s = 0; s < C::NST; ++s)
        if (issued_mask & (1u << s)) wait_bounded(&kv_full[s], (issued_par >> s) & 1u, dc);
    }
    if (warp == 5 && lane == 0 && mma_issued) {
      umma_commit(drain);
      wait_bounded(drain, 0, dc);
    }
    __syncthreads();
  }
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int HD>
static cudaError_t launch_attn_hd(const CUtensorMap& tq, const CUtensorMap& tkv, const AttnArgs& a, int num_sms,
                                  cudaStream_t s) {
  using C = AttnCfg<HD>;
  auto kern = attn_kernel<HD>;
  const int items = a.B * a.H * ((a.c.S + kAttnBM - 1) / kAttnBM);
  const int cap = num_sms * C::CTAS_PER_SM;
  const int grid = items < cap ? items : cap;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, 192, C::SMEM, s>>>(tq, tkv, a);
  return cudaGetLastError();
}

cudaError_t prepare_attention_kernels() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attn_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)AttnCfg<32>::SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)AttnCfg<64>::SMEM)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(attn_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)AttnCfg<256>::SMEM);
}

cudaError_t launch_attention(int hd, const CUtensorMap& tq, const CUtensorMap& tkv, const AttnArgs& a,
                             int num_sms, cudaStream_t s) {
  switch (hd) {
    case 32: return launch_attn_hd<32>(tq, tkv, a, num_sms, s);
    case 64: return launch_attn_hd<64>(tq, tkv, a, num_sms, s);
    case 256: return launch_attn_hd<256>(tq, tkv, a, num_sms, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tfl
