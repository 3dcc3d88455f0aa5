// attention.cu -- flash attention forward on tcgen05 tensor cores.
//
// Per (sequence b, head h, block of 128 queries) the kernel computes
// O = softmax(Q K^T / sqrt(hd) + mask) V without materialising the score
// matrix ("TikTok TechJam 2026 -- Problem 3", section 2.1):
//   * Keys are taken in sub-blocks of 64.  S = Q K_u^T of sub-block u goes to
//     tensor memory (fp32), in one of three buffers; the softmax writes P of u
//     (fp16) over the S it read.  Two threads issue the MMAs: one Q K^T, one
//     P V.  Once the softmax warps have written P of sub-block u (p_full), the
//     P V thread issues P V of u; once that is done (pv_done), the Q K^T thread
//     issues Q K^T of u + 3 into the same buffer, which runs while the softmax
//     works on u + 1 and u + 2.  One issuing thread for both products was the
//     bottleneck: each tcgen05 instruction holds its thread for tens of cycles,
//     and 8 MMAs and their commits a sub-block took longer than the softmax.
//   * A warp's sub-blocks that no mask touches (all but the last one or two
//     of an item) run a body without any mask logic; the masked ones take a
//     general body.
//   * Online softmax in fp32, one query row per thread (the row's TMEM lane):
//     running max m, running sum l, O rescaled by exp(m_old - m_new)
//     (section 2.1, the running-max recurrence).  The row max of a sub-block
//     is taken from registers (four independent max chains) before its
//     exponentials, and the rescale is
//     lazy: the reference max only moves when the row max grew by more than 8
//     in log2 units, so P <= 2^8 and O is touched rarely; O / l is exact
//     either way.
//   * P = exp2(S * log2(e)/sqrt(hd) - m) in fp16 goes to tensor memory (two
//     values per column, double-buffered) and O += P V_u takes its A operand
//     from there (tcgen05.mma with A in TMEM), so only V is read from shared
//     memory.
//   * Causal: key blocks above the diagonal are never loaded (block skipping,
//     section 1.C); a warp whose 32 rows lie entirely below a sub-block skips
//     it, and only sub-blocks crossing the diagonal are masked per key; the
//     key mask is not applied at all, because for a valid query i every key
//     j <= i is valid (section 2.1, "the mask trick").
//   * Key padding (non-causal): only the sub-block holding len_b is masked.
//   * Query blocks past len_b are skipped; their output rows are never read
//     for a valid token.
// q, k, v are strided views of the fused QKV output [B, S, 3D] (section 1.A,
// head-split copies removed); O is written straight into [B, S, H*hd].
//
// Warp roles: warp 0 P V issuer and TMEM owner, warp 1 TMA producer (Q once
// per work item, K/V blocks into an NST-deep ring), warp 2 Q K^T issuer, warp 3
// idle, warps 4-7 softmax + output (thread = query row of TMEM lane quarter
// warp % 4; the four warps form the second warpgroup, which at two CTAs per SM
// takes registers from the first with setmaxnreg).  Persistent CTAs claim work items from a global
// atomic counter, heaviest first (causal: the last query blocks have the most
// keys); the producer publishes each claimed item to the other warps through
// a small shared-memory ring.
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
  // Q tiles: two at head_dim <= 64, so the next work item's Q loads while the
  // current item runs (its load would otherwise wait for the last QK^T)
  static constexpr int NQ = HD <= 64 ? 2 : 1;
  static constexpr int KV_BYTES = BN * HD * 2;      // one K (or V) block
  static constexpr int XPW = HD == 64 ? 2048 : 4096;  // output transpose stage per softmax warp
  static constexpr int XP_BYTES = 4 * XPW;
  static constexpr int NST = HD == 32 ? 4 : 2;
  static constexpr int CTAS_PER_SM = HD <= 64 ? 2 : 1;
  // Keys are taken 64 at a time (a sub-block; a K/V stage holds BN / 64 of
  // them).  Tensor memory: S[b] (fp32) at 64 b for three sub-block buffers b
  // (sub-block g uses buffer g mod 3), P (fp16 pairs) written over the first 32
  // columns of its own S, O from O_COL.
  static constexpr int SUB = 64;
  static constexpr int SUBS = BN / SUB;
  static constexpr int S_COL = 0;
  static constexpr int NSB = 3;  // S buffers (P is written over the S it came from)
  static constexpr int O_COL = HD <= 64 ? 192 : 256;
  static constexpr int TMEM_COLS = O_COL + HD <= 256 ? 256 : 512;
  static constexpr size_t SMEM = 1024 + (size_t)NQ * Q_BYTES + (size_t)NST * 2 * KV_BYTES + XP_BYTES + 384;
};

size_t attn_smem_bytes(int hd) {
  switch (hd) {
    case 32: return AttnCfg<32>::SMEM;
    case 64: return AttnCfg<64>::SMEM;
    case 256: return AttnCfg<256>::SMEM;
  }
  return 0;
}

// mbarrier arrive by the threads whose predicate is set, as a predicated instruction
// (no branch)
__device__ __forceinline__ void mbar_arrive_pred(uint64_t* bar, bool p) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t@q mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(
          smem_u32(bar)),
      "r"((uint32_t)p)
      : "memory");
}

struct Item {
  int b, h, qb, len, nkb;
};

constexpr int kItemRing = 4;
// Warps: 0 issues P V (and owns tensor memory), 1 loads, 2 issues Q K^T, 3 idles, 4-7 softmax
constexpr int kAttnThreads = 256;

// Work item i -> (b, h, query block); false if the block is all padding.  The
// (b, h) pairs are taken in groups of args.group; within a group the last (the
// heaviest, under causal) query blocks of every pair come first, so each group,
// and the launch, ends on light items.  One group (the default) is plain
// heaviest-first.  Groups matter once the keys and values of all sequences no
// longer fit in L2: the CTAs running at any moment then work on the few
// sequences of one group and share their keys and values through L2, instead
// of each streaming its own sequence's prefix from HBM once per query block.
__device__ __forceinline__ bool decode_item(int i, const AttnArgs& a, int nqb, int bn, Item& it) {
  const int bh_count = a.B * a.H;
  const int G = (a.group > 0 && a.group < bh_count) ? a.group : bh_count;
  const int grp = i / (G * nqb);                 // every group before this one is full
  const int gsize = min(G, bh_count - grp * G);  // pairs in this group
  const int j = i - grp * G * nqb;
  const int qr = j / gsize;
  const int bh = grp * G + (j - qr * gsize);
  it.qb = nqb - 1 - qr;
  it.b = bh / a.H;
  it.h = bh - it.b * a.H;
  it.len = seq_len(a.c.lengths, it.b, a.c.S);
  if (it.qb * kAttnBM >= it.len) return false;
  const int kend = a.causal ? min((it.qb + 1) * kAttnBM, it.len) : it.len;
  it.nkb = (kend + bn - 1) / bn;
  return true;
}

// How a warp's rows meet a sub-block's keys (see the softmax loop).
enum SubMode { kFull = 0, kNone = 1, kTriLo = 2, kTriHi = 3, kKeyPad = 4 };

// Sub-blocks of 64 keys an item visits: keys [0, kend) with kend the last
// allowed key + 1 (causal: the block's last query; otherwise len_b).
__device__ __forceinline__ int item_subblocks(const Item& it, int causal) {
  const int kend = causal ? min((it.qb + 1) * kAttnBM, it.len) : it.len;
  return (kend + 63) / 64;
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, AttnCfg<HD>::CTAS_PER_SM)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                const AttnArgs args) {
  using C = AttnCfg<HD>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  grid_launch_dependents();  // the next kernel may set itself up meanwhile
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::NQ * C::Q_BYTES;
  uint8_t* sV = sK + (size_t)C::NST * C::KV_BYTES;
  uint8_t* sX = sV + (size_t)C::NST * C::KV_BYTES;  // output transpose stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(sX + C::XP_BYTES);
  uint64_t* q_full = bars + 0;   // [NQ] (bars 0 and 1)
  uint64_t* q_empty = bars + 2;  // [NQ] (bars 2 and 3)
  uint64_t* o_full = bars + 4;
  uint64_t* o_empty = bars + 5;
  uint64_t* drain = bars + 6;     // abort path: the P V issuer's MMAs are done
  uint64_t* s_full = bars + 7;   // [3] Q K^T issuer -> softmax: S[b] computed
  uint64_t* p_full = bars + 10;  // [3] softmax -> P V issuer: P written over S[b]
  uint64_t* pv_done = bars + 13; // [3] P V issuer -> Q K^T issuer, softmax: P V of buffer b done
  uint64_t* drain_qk = bars + 16; // abort path: the Q K^T issuer's MMAs are done
  uint64_t* kv_full = bars + 17;
  uint64_t* kv_empty = kv_full + C::NST;
  uint64_t* it_full = kv_empty + C::NST;
  uint64_t* it_empty = it_full + kItemRing;
  int* it_slot = reinterpret_cast<int*>(it_empty + kItemRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(it_slot + kItemRing);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* never_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < C::NQ; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
    }
    for (int b = 0; b < C::NSB; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, 4);
    mbar_init(drain, 1);
    mbar_init(drain_qk, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(&it_full[s], 1);
      mbar_init(&it_empty[s], 6);  // the two MMA issuers and the four softmax warps
    }
    *abort_flag = 0;
    *never_flag = 0;
    fence_barrier_init();
  }
  // Two MMA issuers: one thread issuing both products of every sub-block (4 + 4 MMAs
  // and their commits, each tcgen05 instruction holding the thread for tens of cycles)
  // took longer per sub-block than the softmax, which then waited for S.
  constexpr int kMmaWarp = 0, kProdWarp = 1, kQkWarp = 2;
  if (warp == kProdWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmKV);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtl wc{args.c.status, abort_flag, args.c.timeout_ns};
  grid_wait_prior();  // everything below reads or writes what earlier kernels use

  const int S = args.c.S, D = args.D;
  const int nqb = (S + kAttnBM - 1) / kAttnBM;
  const int items = args.B * args.H * nqb;

  uint32_t issued_mask = 0, issued_par = 0;  // producer: stages with loads in flight (abort path)
  uint32_t q_issued = 0, q_par = 0;  // producer: Q buffers with loads in flight, and their parities
  bool mma_issued = false;

  // Two CTAs of 256 threads launch with 128 registers a thread: warpgroup 0 (issuers,
  // loader, one idle warp) hands registers to the softmax warpgroup, 4 x 32 x 64 +
  // 4 x 32 x 192 = 256 x 128.  Each warpgroup changes its count at one point, at the top
  // of its branch.
  if (warp < 4) {
  if constexpr (C::CTAS_PER_SM == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 64;\n" ::: "memory");
  if (warp == kProdWarp) {
    // ------------------------------------------------------------ TMA producer + scheduler
    if (lane == 0) {
      int st = 0, ik = 0;
      uint32_t kvph = 0, qph = 0, itph = 0;  // qph: parity bit per Q buffer
      int qb_i = 0;                          // Q buffer of the next item
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
        const uint32_t qpar = (qph >> qb_i) & 1u;
        if (!wait_bounded(&q_empty[qb_i], qpar ^ 1u, wc)) break;
        mbar_arrive_expect_tx(&q_full[qb_i], C::Q_BYTES);
        uint8_t* sq = sQ + (size_t)qb_i * C::Q_BYTES;
#pragma unroll
        for (int a = 0; a < C::NATOM; ++a)
          tma_load_3d(sq + a * (kAttnBM * C::ROWB), &tmQ, &q_full[qb_i], it.h * HD + a * C::ATOM_C, it.qb * kAttnBM,
                      it.b);
        q_issued |= 1u << qb_i;
        q_par = (q_par & ~(1u << qb_i)) | (qpar << qb_i);
        qph ^= 1u << qb_i;
        if (++qb_i == C::NQ) qb_i = 0;
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
  } else if (warp == kMmaWarp || warp == kQkWarp) {
   if (lane == 0) {
    // ------------------------------------------------------------ MMA issuers (one thread each)
    // Warp 2 issues S = Q K^T of every sub-block, warp 0 O += P V.  Both follow the item
    // ring and number the sub-blocks of all items this CTA runs (sub-block g uses buffer
    // g mod 3, phase g / 3 of its barriers).  P V of g reads the P the softmax wrote over
    // S[g mod 3] (p_full); Q K^T of g writes S[g mod 3] once P V of g - 3 has read the
    // buffer (pv_done), which also means the softmax is done with it.
    // Key rows at or past len_b hold exact zeros (the QKV producers write padding rows
    // as zeros; rows past S are zero-filled by the TMA), so whole key blocks are used.
    const bool is_qk = warp == kQkWarp;
    constexpr uint32_t idesc_qk = idesc_f16(128, C::SUB, 0, 0);
    constexpr uint32_t idesc_pv = idesc_f16(128, HD, 0, 1);
    const uint32_t d_o = tmem_base + C::O_COL;
    int st = 0, ik = 0;  // stage of the next sub-block
    uint32_t kvph = 0, qph = 0, oeph = 0, itph = 0;  // qph: parity bit per Q buffer
    int qb_i = 0;    // Q buffer of the current item
    uint32_t g = 0;  // sub-blocks of all earlier items
    bool first_item = true, ok = true;
    // Operand descriptors: built once; a buffer / stage / half only moves the
    // start-address field (shared-memory byte offset / 16, which stays below 2^14).
    const uint64_t qd0 = sdesc(smem_u32(sQ), 16, 8 * C::ROWB, C::SWZ);
    const uint64_t kd0 = sdesc(smem_u32(sK), 16, 8 * C::ROWB, C::SWZ);
    const uint64_t vd0 = sdesc(smem_u32(sV), BN * C::ROWB, 8 * C::ROWB, C::SWZ);
    // S[b] = Q K^T for the keys of half h of stage s
    auto issue_qk = [&](int s, int h, uint32_t b) {
      const uint64_t ad0 = qd0 + (uint32_t)((qb_i * C::Q_BYTES) >> 4);
      const uint64_t bd0 = kd0 + (uint32_t)((s * C::KV_BYTES + h * C::SUB * C::ROWB) >> 4);
      const uint32_t d = tmem_base + C::S_COL + b * C::SUB;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const int a = kk / (C::ATOM_C / 16), w = kk % (C::ATOM_C / 16);
        const uint64_t ad = ad0 + (uint32_t)((a * (kAttnBM * C::ROWB) + w * 32) >> 4);
        const uint64_t bd = bd0 + (uint32_t)((a * (BN * C::ROWB) + w * 32) >> 4);
        if (kk == 0)
          umma_f16_k<0>(d, ad, bd, idesc_qk);
        else
          umma_f16_k<1>(d, ad, bd, idesc_qk);
      }
    };
    // O += P[b] V for the keys of half h of stage s (P from tensor memory)
    auto issue_pv = [&](int s, int h, uint32_t b, bool accumulate) {
      const uint64_t bd0 = vd0 + (uint32_t)((s * C::KV_BYTES + h * C::SUB * C::ROWB) >> 4);
      const uint32_t pa = tmem_base + C::S_COL + b * C::SUB;
#pragma unroll
      for (int kk = 0; kk < C::SUB / 16; ++kk) {
        const uint64_t bd = bd0 + (uint32_t)((kk * 16 * C::ROWB) >> 4);
        if (kk == 0)
          umma_f16_ts(d_o, pa, bd, idesc_pv, accumulate ? 1u : 0u);
        else
          umma_f16_ts_k<1>(d_o, pa + kk * 8, bd, idesc_pv);
      }
    };
    while (ok) {
      if (!wait_bounded(&it_full[ik], itph, wc)) break;
      const int i = it_slot[ik];
      mbar_arrive(&it_empty[ik]);
      if (++ik == kItemRing) {
        ik = 0;
        itph ^= 1u;
      }
      if (i < 0) break;
      Item it;
      decode_item(i, args, nqb, BN, it);
      const int nsub = item_subblocks(it, args.causal);
      if (is_qk) {
        if (!wait_bounded(&q_full[qb_i], (qph >> qb_i) & 1u, wc)) break;
        qph ^= 1u << qb_i;
      }
      for (int u = 0; u < nsub; ++u) {
        const uint32_t gg = g + u, b = gg % 3u, ph = (gg / 3u) & 1u;
        const int h = u % C::SUBS;
        const bool stage_done = h == C::SUBS - 1 || u == nsub - 1;
        if (is_qk) {
          // S[b] last held S and P of sub-block gg - 3, which P V has read
          if (gg >= 3 && !wait_bounded(&pv_done[b], ph ^ 1u, wc)) {
            ok = false;
            break;
          }
        } else {
          if (!wait_bounded(&p_full[b], ph, wc)) {
            ok = false;
            break;
          }
          if (u == 0 && !first_item) {
            if (!wait_bounded(o_empty, oeph, wc)) {
              ok = false;
              break;
            }
            oeph ^= 1u;
          }
        }
        if (h == 0) {
          if (!wait_bounded(&kv_full[st], kvph, wc)) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        mma_issued = true;
        if (is_qk) {
          issue_qk(st, h, b);
          umma_commit(&s_full[b]);
          if (u == nsub - 1) umma_commit(&q_empty[qb_i]);
        } else {
          issue_pv(st, h, b, u > 0);
          umma_commit(&pv_done[b]);
          // P V of the stage's last sub-block comes after the softmax read S of both, so
          // the Q K^T products that read its keys are done too
          if (stage_done) umma_commit(&kv_empty[st]);
          if (u == nsub - 1) umma_commit(o_full);
        }
        if (stage_done) {
          if (++st == C::NST) {
            st = 0;
            kvph ^= 1u;
          }
        }
      }
      if (!ok) break;
      g += nsub;
      first_item = false;
      if (++qb_i == C::NQ) qb_i = 0;
    }
   }
  }
  } else {
    if constexpr (C::CTAS_PER_SM == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 192;\n" ::: "memory");
    // ------------------------------------------------------------ softmax + output (warps 4-7)
    const int q = warp & 3;          // TMEM lane quarter of this warp
    const int r = q * 32 + lane;     // query row within the block == TMEM lane
    const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16);
    const uint32_t t_o = t_row + C::O_COL;
    const float sl2 = args.scale_log2;
    uint32_t oph = 0, itph = 0, g = 0;
    int ik = 0;
    uint8_t* xst = sX + (warp - 4) * C::XPW;

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
      const int nsub = item_subblocks(it, args.causal);
      const int qpos = it.qb * kAttnBM + r;
      const int wq0 = it.qb * kAttnBM + q * 32;          // first query row of this warp
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      // How this warp's 32 rows meet the 64 keys of sub-block u.  Causal: with
      // d = (first row of the warp) - k0, d >= 63 is unmasked, d <= -32 is
      // entirely above the diagonal (P = 0, nothing computed), and d = 0 / 32
      // (the only other values: query blocks are 128-row and sub-blocks
      // 64-key aligned) mask one 32-key half triangularly.  Key padding
      // masks the keys at or past len_b, the same for every row.
      auto mode_of = [&](int u) -> int {
        const int k0 = u * C::SUB;
        if (args.causal) {
          const int d = wq0 - k0;
          return d >= C::SUB - 1 ? kFull : d <= -32 ? kNone : d == 0 ? kTriLo : kTriHi;
        }
        return k0 + C::SUB > it.len ? kKeyPad : kFull;
      };
      // Sub-blocks [0, nfull) are unmasked for every row of this warp (all but
      // the last one or two): they take a body with no mask logic.
      int nfull;
      if (args.causal) {
        const int t = wq0 - (C::SUB - 1);
        nfull = t < 0 ? 0 : t / C::SUB + 1;
      } else {
        nfull = it.len / C::SUB;
      }
      nfull = min(nfull, nsub);
      float sv[C::SUB];
      // S of sub-block gg from tensor memory (the columns that can be non-zero),
      // once its QK^T has completed; the caller waits for the load
      auto load_s = [&](uint32_t gg, int mode) -> bool {
        if (!wait_bounded(&s_full[gg % 3u], (gg / 3u) & 1u, wc)) return false;
        tc_fence_after();
        const uint32_t t_s = t_row + C::S_COL + (gg % 3u) * C::SUB;
        if (mode != kNone) {
          tmem_ld32(t_s, sv);
          if (mode != kTriLo) tmem_ld32(t_s + 32, sv + 32);
        }
        return true;
      };
      auto body = [&](auto full_tag, int u) -> bool {
        constexpr bool FULL = decltype(full_tag)::value;
        const uint32_t b = g % 3u;
        const int k0 = u * C::SUB;
        const int mode = FULL ? kFull : mode_of(u);
        uint32_t pk[C::SUB / 2];
        if (!load_s(g, mode)) return false;
        if (!FULL && mode == kNone) {
#pragma unroll
          for (int e = 0; e < C::SUB / 2; ++e) pk[e] = 0u;
        } else {
          tmem_wait_ld();
          if constexpr (!FULL) {
            if (mode == kTriLo) {
#pragma unroll
              for (int e = 0; e < 32; ++e) sv[e] = e <= lane ? sv[e] : -INFINITY;
            } else if (mode == kTriHi) {
#pragma unroll
              for (int e = 0; e < 32; ++e) sv[32 + e] = e <= lane ? sv[32 + e] : -INFINITY;
            } else if (mode == kKeyPad) {
              const int lim = it.len - 1 - k0;
#pragma unroll
              for (int e = 0; e < C::SUB; ++e) sv[e] = e <= lim ? sv[e] : -INFINITY;
            }
          }
          const bool half = !FULL && mode == kTriLo;  // only the first 32 keys can be non-zero
          // block maximum in four independent chains (short dependent paths)
          float bm0 = -INFINITY, bm1 = -INFINITY, bm2 = -INFINITY, bm3 = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            bm0 = fmax3(bm0, sv[e], sv[e + 1]);
            bm1 = fmax3(bm1, sv[e + 2], sv[e + 3]);
            bm2 = fmax3(bm2, sv[e + 4], sv[e + 5]);
            bm3 = fmax3(bm3, sv[e + 6], sv[e + 7]);
          }
          if (!half) {
#pragma unroll
            for (int e = 32; e < C::SUB; e += 8) {
              bm0 = fmax3(bm0, sv[e], sv[e + 1]);
              bm1 = fmax3(bm1, sv[e + 2], sv[e + 3]);
              bm2 = fmax3(bm2, sv[e + 4], sv[e + 5]);
              bm3 = fmax3(bm3, sv[e + 6], sv[e + 7]);
            }
          }
          const float m_new = fmaxf(m_run, fmaxf(fmax3(bm0, bm1, bm2), bm3) * sl2);
          const bool resc = m_new > m_run + 8.0f;
          if (__any_sync(0xffffffffu, resc)) {
            if (u > 0) {
              // O must hold P V of every earlier sub-block of this item before it is rescaled
              const uint32_t gp = g - 1;
              if (!wait_bounded(&pv_done[gp % 3u], (gp / 3u) & 1u, wc)) return false;
              tc_fence_after();
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
          }
          // p = 2^(s * scale * log2(e) - m): pairs of scores scaled in one
          // packed FMA, partial sums kept as four packed pairs
          const float mref = (m_run == -INFINITY) ? 0.f : m_run;
          const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mref, -mref);
          uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
          auto exp_pairs = [&](int e2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sv[2 * e2], sv[2 * e2 + 1]), sl2x2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            acc[e2 & 3] = f2_add(acc[e2 & 3], f2_pack(p0, p1));
            const __half2 hp = __floats2half2_rn(p0, p1);  // first key in the low half
            pk[e2] = *reinterpret_cast<const uint32_t*>(&hp);
          };
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) exp_pairs(e2);
          if (!half) {
#pragma unroll
            for (int e2 = 16; e2 < C::SUB / 2; ++e2) exp_pairs(e2);
          } else {
#pragma unroll
            for (int e2 = 16; e2 < C::SUB / 2; ++e2) pk[e2] = 0u;
          }
          float a0, a1;
          f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
          l_run += a0 + a1;
        }
        // P over the first 32 columns of this sub-block's S (read above)
        tmem_st32_u(t_row + C::S_COL + b * C::SUB, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        mbar_arrive_pred(&p_full[b], lane == 0);
        return true;
      };
      int u = 0;
      for (; ok && u < nfull; ++u, ++g) ok = body(std::true_type{}, u);
      for (; ok && u < nsub; ++u, ++g) ok = body(std::false_type{}, u);
      if (!ok) break;
      if (!wait_bounded(o_full, oph, wc)) break;
      oph ^= 1u;
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
      // the row's log-sum-exp for a backward pass: log2 sum_j 2^(s_j log2(e)/sqrt(hd)) = m + log2 l
      if (args.lse != nullptr && qpos < it.len)
        args.lse[((size_t)it.b * args.H + it.h) * S + qpos] = m_run + __log2f(l_run);
      const int q0 = it.qb * kAttnBM + q * 32;  // first query row of this warp
      const uint32_t rows = __ballot_sync(0xffffffffu, qpos < S);
      __half* orow0 = args.o16 + ((size_t)it.b * S + q0) * D + it.h * HD;
      if constexpr (HD <= 64) {
#pragma unroll 1
        for (int c = 0; c < HD; c += 32) {
          float o[32];
          tmem_ld32(t_o + c, o);
          tmem_wait_ld();
          xp_store_f16<32>(xst, lane, o, orow0 + c, nullptr, D, rows, inv);
        }
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
    if (warp == kProdWarp && lane == 0) {
      for (int b = 0; b < C::NQ; ++b)
        if (q_issued & (1u << b)) wait_bounded(&q_full[b], (q_par >> b) & 1u, dc);
      for (int s = 0; s < C::NST; ++s)
        if (issued_mask & (1u << s)) wait_bounded(&kv_full[s], (issued_par >> s) & 1u, dc);
    }
    if ((warp == kMmaWarp || warp == kQkWarp) && lane == 0 && mma_issued) {
      uint64_t* dr = warp == kMmaWarp ? drain : drain_qk;
      umma_commit(dr);
      wait_bounded(dr, 0, dc);
    }
    __syncthreads();
  }
  if (warp == kMmaWarp) {
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
  return launch_dependent(kern, grid, kAttnThreads, C::SMEM, s, tq, tkv, a);
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
