// postchain.cu -- the whole post-attention chain of one layer in one kernel
// (d_model = 128): o_proj + bias + residual (+ LayerNorm) -> LayerNorm ->
// FFN-in + bias + GELU -> FFN-out + bias + residual -> LayerNorm of the next
// layer, or the model tail.
//
// This is the post_attn_chain / post_attn_chain_tail fusion of "TikTok
// TechJam 2026 -- Problem 3", section 1.A, rebuilt for tcgen05: the pages
// keep all three weights resident in shared memory, which only fits at
// d_model = d_ff = 128; here the weights stream through a shared-memory ring
// from L2 while every activation operand stays on chip in tensor memory, so
// d_ff = 512 (and the fp16 hi/lo operand splits) fit as well.  Per 128-row tile:
//
//   A1  = O Wo^T                    O: TMA tile in SMEM;  Wo hi/lo: ring
//   t   = A1 * 2^-s + bo + res      (registers, fp32; post-LN: LN1(t))
//   N2  = LN2(t) as fp16 hi/lo pairs, written to TMEM        (pre-LN)
//   per 128-wide chunk c of d_ff:
//     G_c   = N2 W1_c^T             A from TMEM (hi, lo), W1_c hi/lo: ring
//     GP_c  = GELU(G_c * 2^-s + b1_c) as fp16 hi/lo pairs, to TMEM
//     OUT  += GP_c W2_c^T           A from TMEM (hi, lo), W2_c hi/lo: ring;
//                                   OUT starts as t * 2^s (written by the epilogue)
//   t2  = OUT * 2^-s + b2 -> residual / next LayerNorm / tail  (HBM)
//
// The GELU output never leaves the SM: per token it saves the d_ff-wide
// round trip (2 * 2 * d_ff bytes written and read with split planes) and the
// normed-row round trip of the unfused path.
//
// Weight streaming: every tile re-reads the layer's weights from L2 through
// a two-slot ring of 128 x 128 blocks (hi and lo planes, 64 KB).  Tile t walks
// the d_ff chunks starting at chunk t mod (d_ff/128), so CTAs running at the
// same time read different weight blocks instead of all hitting the same L2
// lines (the FFN-out sum order differs per tile but is fixed for a shape).
//
// Pipelining: the d_ff chunks are 128 wide, so every MMA is M = N = 128 (a
// 64-wide N runs the tensor core at about half rate).  G and GP are single
// buffers: the epilogue releases G as soon as it has read it, so FFN-in of
// chunk c+1 runs on the tensor core while chunk c's GELU is being computed,
// and FFN-out of chunk c runs while the epilogue reads G of chunk c+1.
// FFN-out accumulates onto t, which the epilogue writes into the
// accumulator columns (scaled by 2^s2) after the o_proj epilogue.
//
// Roles: warp 0 TMA producer, warp 1 o_proj / FFN-out MMA issuer + TMEM
// owner, warp 18 FFN-in MMA issuer, warps 2-17
// epilogue (four warps per TMEM lane quarter; each owns 32 of the 128 columns
// of its 32 rows, so four warps per scheduler hide each other's latencies).  Tensor memory (512 columns):
//   [0,128) A1 / t / OUT   [128,192) N2 hi  [192,256) N2 lo
//   [256,384) G (fp32)     [384,448) GP hi  [448,512) GP lo
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "mathfn.cuh"
#include "xpose.cuh"
#include "chainops.cuh"

namespace tfl {

namespace {

using namespace chain;  // kD, kEpi, kParts, kRedBytes and the row operations

constexpr int kFC = 128;            // d_ff chunk
constexpr int kUnit = 64 * 1024;    // one ring unit: a 128 x 128 weight block, hi + lo planes
constexpr int kHalf = 16 * 1024;    // one 64-column (K) half of a plane: 128 rows x 128 B
constexpr int kRing = 2;
constexpr int kFfn1Warp = 2 + kEpi;  // the FFN-in MMA issuer (scheduler 2; o_proj / FFN-out issue from warp 1)
constexpr int kThreads = 32 * (kFfn1Warp + 1);
constexpr int kOBytes = kGemmBM * kD * 2;
constexpr int kXpWarp = 2048;       // per-warp transpose stage: 32 rows x 64 B
constexpr int kXpBytes = kEpi * kXpWarp;
// parameter vectors staged in shared memory once per CTA (floats):
// bo, b2, ln1 g/b, ln2 g/b, next-layer ln1 g/b, final ln g/b (128 each), then b1 (d_ff <= kMaxF)
constexpr int kMaxF = 2048;
constexpr int kPBo = 0, kPB2 = 128, kPLn1g = 256, kPLn1b = 384, kPLn2g = 512, kPLn2b = 640, kPLnng = 768,
              kPLnnb = 896, kPLnfg = 1024, kPLnfb = 1152, kPB1 = 1280;
constexpr int kPBqkv = kPB1 + kMaxF;  // next layer's [bq | bk | bv] (fuse_qkv)
constexpr int kParamBytes = (kPBqkv + 3 * kD) * 4;
constexpr size_t kSmem = 1024 + kOBytes + (size_t)kRing * kUnit + kXpBytes + kRedBytes + kParamBytes + 512;

constexpr uint32_t kColA1 = 0, kColN2 = 128, kColG = 256, kColGP = 384;  // GP: hi [384,448), lo [448,512)

}  // namespace

// One warp's 32 rows x 64 bytes (v: this thread's row, four 16-byte pieces) into
// its stage in the 64-byte-swizzled order of a SWIZZLE_64B map, then stored by
// TMA at (x, y).  The stage is reused only after the previous store has read it.
__device__ __forceinline__ void stage_tma_store(uint8_t* st, int lane, const uint4* v, const CUtensorMap* m, int x,
                                                int y) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(st + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = v[c];
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(m, st, x, y);
    bulk_commit();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    postchain_kernel(const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmWo,
                     const __grid_constant__ CUtensorMap tmWoLo, const __grid_constant__ CUtensorMap tmW1,
                     const __grid_constant__ CUtensorMap tmW1Lo, const __grid_constant__ CUtensorMap tmW2,
                     const __grid_constant__ CUtensorMap tmW2Lo, const __grid_constant__ CUtensorMap tmWq,
                     const __grid_constant__ CUtensorMap tmWqLo, const __grid_constant__ CUtensorMap tmH32St,
                     const __grid_constant__ CUtensorMap tmQkvSt, const ChainArgs args) {
  extern __shared__ uint8_t smem_raw[];
  grid_launch_dependents();  // the next kernel may set itself up meanwhile
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sO = smem;
  uint8_t* ring = sO + kOBytes;
  uint8_t* xpose = ring + (size_t)kRing * kUnit;
  float* red = reinterpret_cast<float*>(xpose + kXpBytes);
  float* prm = red + kRedBytes / 4;
  uint64_t* bars = reinterpret_cast<uint64_t*>(prm + kParamBytes / 4);
  uint64_t* o_full = bars + 0;
  uint64_t* o_free = bars + 1;
  uint64_t* acc_full = bars + 2;
  uint64_t* acc_read = bars + 3;
  uint64_t* out_full = bars + 4;
  uint64_t* out_read = bars + 5;
  uint64_t* drain = bars + 6;      // [2]: one per MMA issuer (abort path)
  uint64_t* g_full = bars + 8;
  uint64_t* gp_ready = bars + 9;
  uint64_t* gp_free = bars + 10;
  uint64_t* g_read = bars + 11;
  uint64_t* n_ready = bars + 12;   // fuse_qkv: the next layer's normed rows are in TMEM
  uint64_t* qkv_full = bars + 13;  // [3] fuse_qkv: the q, k, v accumulators are complete
  uint64_t* r_full = bars + 16;    // [kRing]
  uint64_t* r_empty = r_full + kRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(r_empty + kRing);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* never_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(o_full, 1);
    mbar_init(o_free, 1);
    mbar_init(acc_full, 1);
    mbar_init(acc_read, kEpi);
    mbar_init(out_full, 1);
    mbar_init(out_read, kEpi);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(g_full, 1);
    mbar_init(gp_ready, kEpi);
    mbar_init(gp_free, 1);
    mbar_init(g_read, kEpi);
    mbar_init(n_ready, kEpi);
    for (int j = 0; j < 3; ++j) mbar_init(&qkv_full[j], 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], 1);
    }
    *abort_flag = 0;
    *never_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmO);
    tma_prefetch_desc(&tmWo);
    tma_prefetch_desc(&tmWoLo);
    tma_prefetch_desc(&tmW1);
    tma_prefetch_desc(&tmW1Lo);
    tma_prefetch_desc(&tmW2);
    tma_prefetch_desc(&tmW2Lo);
    if (args.fuse_qkv) {
      tma_prefetch_desc(&tmWq);
      tma_prefetch_desc(&tmWqLo);
    }
  }
  {
    // every thread issues all of its loads before any store, so the staging costs
    // one global-memory round trip rather than one per loop iteration
    const float* src[10] = {args.bo,    args.b2,    args.ln1_g, args.ln1_b, args.ln2_g,
                            args.ln2_b, args.lnn_g, args.lnn_b, args.lnf_g, args.lnf_b};
    constexpr int kPrm = kParamBytes / 4, kPer = (kPrm + kThreads - 1) / kThreads;
    auto source = [&](int i) -> const float* {
      if (i < kPB1) return src[i / kD] ? src[i / kD] + (i % kD) : nullptr;
      if (i < kPBqkv) return i - kPB1 < args.F ? args.b1 + (i - kPB1) : nullptr;
      return args.fuse_qkv ? args.bqkv + (i - kPBqkv) : nullptr;
    };
    float pv[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kThreads;
      const float* a = i < kPrm ? source(i) : nullptr;
      pv[k] = a ? __ldg(a) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kThreads;
      if (i < kPrm) prm[i] = pv[k];
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{args.c.status, abort_flag, args.c.timeout_ns};
  grid_wait_prior();  // everything below reads or writes what earlier kernels use

  const int M = args.c.M, S = args.c.S;
  const int* lengths = args.c.lengths;
  // tiles from the list: the live ones, then (last layer only) the all-padding
  // ones, whose output rows the epilogue zeroes
  const int* tile_list = args.c.tiles;
  const int n_live = tile_list[0];
  const int n_work = args.last ? tile_list[1] : n_live;
  const int nch = args.F / kFC;

  uint32_t issued_mask = 0, issued_par = 0;  // producer: ring stages in flight (abort path)
  bool o_issued = false;
  uint32_t o_par = 0;
  bool mma_issued = false;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0, oph = 0;
      bool ok = true;
      auto unit = [&](auto&& load) -> bool {
        if (!wait_bounded(&r_empty[rs], rph ^ 1u, wc)) return false;
        mbar_arrive_expect_tx(&r_full[rs], kUnit);
        load(ring + (size_t)rs * kUnit, &r_full[rs]);
        issued_mask |= 1u << rs;
        issued_par = (issued_par & ~(1u << rs)) | (rph << rs);
        if (++rs == kRing) {
          rs = 0;
          rph ^= 1u;
        }
        return true;
      };
      int rot = 0;  // this tile's chunk rotation (see the header)
      // a 128 x 128 block of a weight: hi plane (two 64-column halves), then lo
      auto w1 = [&](int c) {
        const int f0 = ((c + rot) % nch) * kFC;
        return unit([&](uint8_t* d, uint64_t* b) {
          tma_load_2d(d, &tmW1, b, 0, f0);
          tma_load_2d(d + kHalf, &tmW1, b, 64, f0);
          tma_load_2d(d + 2 * kHalf, &tmW1Lo, b, 0, f0);
          tma_load_2d(d + 3 * kHalf, &tmW1Lo, b, 64, f0);
        });
      };
      auto w2 = [&](int c) {
        const int f0 = ((c + rot) % nch) * kFC;
        return unit([&](uint8_t* d, uint64_t* b) {
          tma_load_2d(d, &tmW2, b, f0, 0);
          tma_load_2d(d + kHalf, &tmW2, b, f0 + 64, 0);
          tma_load_2d(d + 2 * kHalf, &tmW2Lo, b, f0, 0);
          tma_load_2d(d + 3 * kHalf, &tmW2Lo, b, f0 + 64, 0);
        });
      };
      for (int ti = blockIdx.x; ti < n_live && ok; ti += gridDim.x) {
        const int t = tile_list[2 + ti];
        rot = t % nch;
        if (!wait_bounded(o_free, oph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(o_full, kOBytes);
        tma_load_2d(sO, &tmO, o_full, 0, t * kGemmBM);
        tma_load_2d(sO + kOBytes / 2, &tmO, o_full, 64, t * kGemmBM);
        o_issued = true;
        o_par = oph;
        oph ^= 1u;
        // the order the MMA warp consumes them: Wo, FFN-in 0 and 1, then FFN-out c / FFN-in c+2
        ok = unit([&](uint8_t* d, uint64_t* b) {
          tma_load_2d(d, &tmWo, b, 0, 0);
          tma_load_2d(d + kHalf, &tmWo, b, 64, 0);
          tma_load_2d(d + 2 * kHalf, &tmWoLo, b, 0, 0);
          tma_load_2d(d + 3 * kHalf, &tmWoLo, b, 64, 0);
        });
        if (ok) ok = w1(0);
        if (ok && nch > 1) ok = w1(1);
        for (int c = 0; c < nch && ok; ++c) {
          ok = w2(c);
          if (ok && c + 2 < nch) ok = w1(c + 2);
        }
        // fuse_qkv: the next layer's W_qkv, one 128-row block (q, k, v) per unit
        for (int j = 0; j < 3 && ok && args.fuse_qkv; ++j)
          ok = unit([&](uint8_t* d, uint64_t* b) {
            tma_load_2d(d, &tmWq, b, 0, 128 * j);
            tma_load_2d(d + kHalf, &tmWq, b, 64, 128 * j);
            tma_load_2d(d + 2 * kHalf, &tmWqLo, b, 0, 128 * j);
            tma_load_2d(d + 3 * kHalf, &tmWqLo, b, 64, 128 * j);
          });
      }
    }
  } else if (warp == 1 || warp == kFfn1Warp) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads on different schedulers issue the MMAs, so neither starves
    // behind the epilogue warps sharing its scheduler: warp 1 o_proj and
    // FFN-out (accumulator A1 / OUT), warp kFfn1Warp FFN-in (accumulator G).
    // Both walk the producer's ring sequence by unit index: per tile Wo,
    // W1_0, W1_1, then W2_c, W1_(c+2) for each chunk c.
    if (lane == 0) {
      constexpr uint32_t id128 = idesc_f16(128, 128, 0, 0);
      const uint32_t tA1 = tmem_base + kColA1;
      const int units = 1 + 2 * nch + (args.fuse_qkv ? 3 : 0);  // ring units per tile
      auto idx_w1 = [&](int k) { return k == 0 ? 1 : (k == 1 ? 2 : 2 * k); };
      auto idx_w2 = [&](int c) { return c <= nch - 2 ? 3 + 2 * c : 2 * nch; };
      // wait for ring unit g (counted over all tiles of this CTA); returns its smem address
      auto take = [&](uint32_t g) -> uint32_t {
        if (!wait_bounded(&r_full[g % kRing], (g / kRing) & 1u, wc)) return 0;
        tc_fence_after();
        return smem_u32(ring + (size_t)(g % kRing) * kUnit);
      };
      auto give = [&](uint32_t g) { umma_commit(&r_empty[g % kRing]); };
      // k-step kk of a 128 x 128 ring block (plane base p): 16 columns of one 64-column half
      auto kdesc = [](uint32_t p, int kk) { return sdesc(p + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024, kSw128); };
      bool ok = true;
      uint32_t tile_seq = 0;
      if (warp == 1) {
        uint32_t oph = 0, orph = 0, gpr = 0, nrph = 0, qbph = 0;
        for (int ti = blockIdx.x; ti < n_live && ok; ti += gridDim.x, ++tile_seq) {
          const uint32_t g0 = tile_seq * units;
          // o_proj into A1 (free once the previous tile's epilogue read OUT)
          if (tile_seq > 0) {
            if (!wait_bounded(out_read, orph, wc)) break;
            orph ^= 1u;
          }
          if (!wait_bounded(o_full, oph, wc)) break;
          oph ^= 1u;
          tc_fence_after();
          {
            const uint32_t u = take(g0);
            if (!u) break;
            const uint32_t so = smem_u32(sO);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t a = sdesc(so + (kk >> 2) * (kOBytes / 2) + (kk & 3) * 32, 16, 1024, kSw128);
              umma_f16(tA1, a, kdesc(u, kk), id128, kk > 0 ? 1u : 0u);
              umma_f16(tA1, a, kdesc(u + 2 * kHalf, kk), id128, 1u);
            }
            mma_issued = true;
            give(g0);
          }
          umma_commit(o_free);
          umma_commit(acc_full);
          // FFN-out of chunk c once its GELU output is in TMEM:
          // OUT += GP_c (hi, lo in TMEM) * W2_c^T (hi, lo), onto t (written by the epilogue)
          for (int c = 0; c < nch; ++c) {
            if (!wait_bounded(gp_ready, gpr, wc)) {
              ok = false;
              break;
            }
            gpr ^= 1u;
            tc_fence_after();
            const uint32_t g = g0 + idx_w2(c);
            const uint32_t u = take(g);
            if (!u) {
              ok = false;
              break;
            }
            const uint32_t gp = tmem_base + kColGP;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t bh = kdesc(u, kk), bl = kdesc(u + 2 * kHalf, kk);
              const uint32_t ah = gp + kk * 8, al = gp + 64 + kk * 8;
              umma_f16_ts(tA1, ah, bh, id128, 1u);
              umma_f16_ts(tA1, al, bh, id128, 1u);
              umma_f16_ts(tA1, ah, bl, id128, 1u);
            }
            give(g);
            umma_commit(gp_free);
          }
          if (!ok) break;
          umma_commit(out_full);
          if (args.fuse_qkv) {
            // the next layer's [q | k | v] = N W_qkv^T into [128, 512), N (hi, lo pairs per
            // 32-column part) in [0, 128).
            // This thread's o_proj of the next tile, which rewrites [0, 128), issues after these.
            if (!wait_bounded(n_ready, nrph, wc)) break;
            nrph ^= 1u;
            tc_fence_after();
            for (int j = 0; j < 3 && ok; ++j) {
              const uint32_t g = g0 + 1 + 2 * nch + j;
              const uint32_t u = take(g);
              if (!u) {
                ok = false;
                break;
              }
              const uint32_t d = tmem_base + 128 + 128 * j;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bh = kdesc(u, kk), bl = kdesc(u + 2 * kHalf, kk);
                // k-step kk: values 16 kk .. +15, written by epilogue part kk / 2
                const uint32_t ah = tmem_base + 32 * (kk >> 1) + 8 * (kk & 1), al = ah + 16;
                umma_f16_ts(d, ah, bh, id128, kk > 0 ? 1u : 0u);
                umma_f16_ts(d, al, bh, id128, 1u);
                umma_f16_ts(d, ah, bl, id128, 1u);
              }
              give(g);
              // the epilogue drains q while k and v are computed
              umma_commit(&qkv_full[j]);
            }
            if (!ok) break;
            // the next tile's o_proj overwrites N: let these MMAs finish reading it first
            if (!wait_bounded(&qkv_full[2], qbph, wc)) break;
            qbph ^= 1u;
          }
        }
      } else {
        uint32_t arph = 0, grd = 0;
        // FFN-in chunk k: G = N2 (hi, lo in TMEM) * W1_k^T (hi, lo)
        auto ffn1 = [&](uint32_t g0, int k) -> bool {
          const uint32_t g = g0 + idx_w1(k);
          const uint32_t u = take(g);
          if (!u) return false;
          const uint32_t d = tmem_base + kColG;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bh = kdesc(u, kk), bl = kdesc(u + 2 * kHalf, kk);
            const uint32_t ah = tmem_base + kColN2 + kk * 8, al = ah + 64;
            umma_f16_ts(d, ah, bh, id128, kk > 0 ? 1u : 0u);
            umma_f16_ts(d, al, bh, id128, 1u);
            umma_f16_ts(d, ah, bl, id128, 1u);
          }
          mma_issued = true;
          give(g);
          umma_commit(g_full);
          return true;
        };
        for (int ti = blockIdx.x; ti < n_live && ok; ti += gridDim.x, ++tile_seq) {
          const uint32_t g0 = tile_seq * units;
          // N2 of this tile is in TMEM (the previous tile's last G read was awaited below)
          if (!wait_bounded(acc_read, arph, wc)) break;
          arph ^= 1u;
          tc_fence_after();
          if (!ffn1(g0, 0)) break;
          for (int c = 0; c < nch; ++c) {
            // FFN-in of chunk c+1 reuses G as soon as the epilogue has read chunk c
            if (!wait_bounded(g_read, grd, wc)) {
              ok = false;
              break;
            }
            grd ^= 1u;
            tc_fence_after();
            if (c + 1 < nch && !ffn1(g0, c + 1)) {
              ok = false;
              break;
            }
          }
        }
      }
    }
  } else if (warp >= 2 && warp < 2 + kEpi) {
    // ------------------------------------------------------------ epilogue (16 warps)
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int part = (warp - 2) >> 2;   // which 32 of the 128 columns it owns
    const int c0 = part * 32;
    const int r = q * 32 + lane;
    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16);
    uint8_t* st = xpose + (warp - 2) * kXpWarp;
    WaitCtl ewc = wc;
    ewc.early_exit = false;  // the epilogue warps meet at a named barrier: leave only on their own bound
    uint32_t afph = 0, ofph = 0, gfph = 0, gffph = 0, qfph = 0;
    bool gp_written = false;  // GP holds an earlier chunk that FFN-out must have consumed before a rewrite
    int slot = 0;
    const float eps = args.eps;
    int t_next = (int)blockIdx.x < n_work ? tile_list[2 + blockIdx.x] : 0;  // loaded one tile ahead
    for (int ti = blockIdx.x; ti < n_work; ti += gridDim.x) {
      const int t = t_next;
      if (ti + (int)gridDim.x < n_work) t_next = tile_list[2 + ti + gridDim.x];
      const int m0w = t * kGemmBM + q * 32;
      const int m = m0w + lane;
      const uint32_t in_rows = __ballot_sync(0xffffffffu, m < M);
      if (args.fuse_qkv) {  // the stage's last tensor store must have read it
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
      if (ti >= n_live) {  // all-padding tile (last layer only): zero output rows
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
        if (args.outbf) {
          xp_store_bf16<32>(st, lane, z, args.outbf + (size_t)m0w * kD + c0, kD, in_rows);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            xp_store_f32x16(st, lane, z, args.out32 + (size_t)m0w * kD + c0 + 16 * h, kD, in_rows);
        }
        continue;
      }
      // ---- phase 1: t = o_proj + bias + residual (post-LN: LN1 of it).  t goes
      // back into the accumulator columns, scaled by 2^s2, and FFN-out then
      // accumulates onto it, so t is not held in registers through the FFN.
      // this warp's 32 residual columns, fetched before the accumulator wait; padding
      // rows are fetched too (finite values whose results no valid token reads)
      uint4 res0[4], res1[4];
      XStage<64>::fetch_rows(lane, reinterpret_cast<const uint8_t*>(args.res + (size_t)m0w * kD + c0), kD * 4,
                             in_rows, res0);
      XStage<64>::fetch_rows(lane, reinterpret_cast<const uint8_t*>(args.res + (size_t)m0w * kD + c0 + 16), kD * 4,
                             in_rows, res1);
      if (!wait_bounded(acc_full, afph, ewc)) break;
      afph ^= 1u;
      tc_fence_after();
      // FFN-in: GELU input = acc * a1 + b1 (pre-LN: a1 = rstd 2^-s, the row's mean taken
      // out of the operand before the product; post-LN: a1 = 2^-s)
      float a1 = args.scale_1;
      {
        float tv[32];
        tmem_ld32(tq + kColA1 + c0, tv);
        tmem_wait_ld();
        scale_bias32(tv, args.scale_o, prm + kPBo + c0);
        xp_add_fetched_f32x16(st, lane, tv, res0);
        xp_add_fetched_f32x16(st, lane, tv + 16, res1);
        if (args.post_ln) layer_norm32(tv, eps, prm + kPLn1g, prm + kPLn1b, c0, red, slot, part, r);
        // t * 2^s2 into the accumulator columns (exact: a power of two), then t back
#pragma unroll
        for (int i = 0; i < 32; ++i) tv[i] *= args.inv_scale_2;
        tmem_st32(tq + kColA1 + c0, tv);
        tmem_wait_st();
#pragma unroll
        for (int i = 0; i < 32; ++i) tv[i] *= args.scale_2;
        // the FFN's input as fp16 hi/lo pairs in TMEM.  Pre-LN, LN2's affine is folded
        // into W1 and the operand is t - mean (centred before the split, so its size is
        // the row's spread, not its offset); rstd enters the GELU input.  Post-LN the FFN
        // reads t itself.
        float mean = 0.f;
        if (!args.post_ln) {
          float rstd;
          stats32(tv, eps, red, slot, part, r, mean, rstd);
          slot = (slot + 2) & 3;
          a1 = rstd * args.scale_1;
        }
        store_split_operand(tq + kColN2, tv, mean, part);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_read);
      }
      // pull the next tile's residual rows into L2 while this tile's FFN runs
      if (ti + (int)gridDim.x < n_live) {
        const int mn = t_next * kGemmBM + q * 32 + lane;
        if (mn < M) prefetch_l2(args.res + (size_t)mn * kD + c0);
      }
      // ---- phase 2: GELU of each FFN-in chunk, back into TMEM as hi/lo pairs
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        if (!wait_bounded(g_full, gfph, ewc)) {
          ok = false;
          break;
        }
        gfph ^= 1u;
        tc_fence_after();
        float gv[32];  // this warp's 32 of the chunk's 128 columns
        tmem_ld32(tq + kColG + c0, gv);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(g_read);
        const int f0 = ((c + t) % nch) * kFC + c0;
        // GELU and fp16 hi/lo split of the 32 values in registers, then into GP once
        // FFN-out of the previous chunk has read it (the GELU overlaps that MMA)
        uint32_t hi[16], lo[16];
        gelu_split32(gv, a1, prm + kPB1 + f0, hi, lo);
        if (gp_written) {  // GP is free once FFN-out of the previous chunk has read it
          if (!wait_bounded(gp_free, gffph, ewc)) {
            ok = false;
            break;
          }
          gffph ^= 1u;
          tc_fence_after();
        }
        tmem_st16_u(tq + kColGP + part * 16, hi);
        tmem_st16_u(tq + kColGP + 64 + part * 16, lo);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(gp_ready);
        gp_written = true;
      }
      if (!ok) break;
      // ---- phase 3: t2 = (t 2^s2 + FFN-out) 2^-s2 + bias, then the next LayerNorm or the tail
      if (!wait_bounded(out_full, ofph, ewc)) break;
      ofph ^= 1u;
      tc_fence_after();
      float tv[32];
      tmem_ld32(tq + kColA1 + c0, tv);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(out_read);
      scale_bias32(tv, args.scale_2, prm + kPB2 + c0);
      if (args.post_ln) layer_norm32(tv, eps, prm + kPLn2g, prm + kPLn2b, c0, red, slot, part, r);
      if (!args.last && args.fuse_qkv) {
        // the next layer's QKV input as fp16 hi/lo pairs into this warp's own 32 OUT
        // columns of [0, 128) (values c0 + 16 j .. +15: hi at 32 part + 8 j, lo 16
        // further), so no other warp's OUT read is overtaken.  Pre-LN, the next LN1's
        // affine is folded into W_qkv and the operand is t2 - mean (rstd enters the
        // drains below); post-LN, t2 is the normalised residual already.
        float aq = args.scale_qkv, mean = 0.f;
        if (!args.post_ln) {
          float rstd;
          stats32(tv, eps, red, slot, part, r, mean, rstd);
          slot = (slot + 2) & 3;
          aq = rstd * args.scale_qkv;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t hi[8], lo[8];
          split_centered_pairs16(tv + 16 * j, mean, hi, lo);
          tmem_st8_u(tq + 32 * part + 8 * j, hi);
          tmem_st8_u(tq + 32 * part + 16 + 8 * j, lo);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(n_ready);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint4 pk[4];
          pack_f32x16(tv + 16 * h, pk);
          stage_tma_store(st, lane, pk, &tmH32St, c0 + 16 * h, m0w);
        }
        // qkv = acc 2^-s + b, fp16, this warp's 32 columns of each of q, k, v; padding rows
        // as exact zeros (attention takes whole key blocks: zero probability times zero value)
        const bool valid = m < M && row_valid(m, S, lengths);
        bool qkv_ok = true;
#pragma unroll 1
        for (int j = 0; j < 3; ++j) {
          if (!wait_bounded(&qkv_full[j], qfph, ewc)) {
            qkv_ok = false;
            break;
          }
          tc_fence_after();
          float qv[32];
          tmem_ld32(tq + 128 + 128 * j + c0, qv);
          tmem_wait_ld();
          scale_bias32(qv, aq, prm + kPBqkv + 128 * j + c0);
          if (!valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) qv[i] = 0.f;
          }
          uint4 pk[4];
          pack_f16<32>(qv, pk, false, 1.0f);
          stage_tma_store(st, lane, pk, &tmQkvSt, 128 * j + c0, m0w);
        }
        if (!qkv_ok) break;
        qfph ^= 1u;
      } else if (!args.last) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          xp_store_f32x16(st, lane, tv + 16 * h, args.h32 + (size_t)m0w * kD + c0 + 16 * h, kD, in_rows);
        if (!args.post_ln) layer_norm32(tv, eps, prm + kPLnng, prm + kPLnnb, c0, red, slot, part, r);
        const size_t off = (size_t)m0w * kD + c0;
        xp_store_f16<32>(st, lane, tv, args.n16 + off, args.n16lo + off, kD, in_rows);
      } else {
        layer_norm32(tv, eps, prm + kPLnfg, prm + kPLnfb, c0, red, slot, part, r);
        const bool valid = m < M && row_valid(m, S, lengths);
#pragma unroll
        for (int i = 0; i < 32; ++i) tv[i] = valid ? tv[i] : 0.f;
        if (args.outbf) {
          xp_store_bf16<32>(st, lane, tv, args.outbf + (size_t)m0w * kD + c0, kD, in_rows);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            xp_store_f32x16(st, lane, tv + 16 * h, args.out32 + (size_t)m0w * kD + c0 + 16 * h, kD, in_rows);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  if (warp >= 2 && warp < 2 + kEpi && lane == 0) bulk_wait<0>();  // tensor stores complete
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    const WaitCtl dc{args.c.status, never_flag, 100000000LL};
    if (warp == 0 && lane == 0) {
      if (o_issued) wait_bounded(o_full, o_par, dc);
      for (int s = 0; s < kRing; ++s)
        if (issued_mask & (1u << s)) wait_bounded(&r_full[s], (issued_par >> s) & 1u, dc);
    }
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

cudaError_t prepare_postchain_kernel() {
  return cudaFuncSetAttribute(postchain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
}

cudaError_t launch_postchain(const ChainMaps& mp, const ChainArgs& a, int num_sms, cudaStream_t s) {
  if (a.F % kFC != 0 || a.F < kFC || a.F > kMaxF) return cudaErrorInvalidValue;
  const int tiles = (a.c.M + kGemmBM - 1) / kGemmBM;
  const int grid = tiles < num_sms ? tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  return launch_dependent(postchain_kernel, grid, kThreads, kSmem, s, mp.o, mp.wo, mp.wo_lo, mp.w1, mp.w1_lo, mp.w2,
                          mp.w2_lo, mp.wqkv, mp.wqkv_lo, mp.h32_st, mp.qkv_st, a);
}

}  // namespace tfl
