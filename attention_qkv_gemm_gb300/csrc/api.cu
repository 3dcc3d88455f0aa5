// api.cu -- the C ABI (include/tfl.h) and the runtime behind it: shape
// validation, weight packing, workspace carve-up, TMA descriptors, the
// per-forward launch sequence and its CUDA-graph capture.
//
// Launch sequence of one forward ("TikTok TechJam 2026 -- Problem 3",
// sections 1.A and 1.B; 5 or 7 kernels per layer, replayed as one graph):
//   [length check] [layer-0 input LayerNorm, no residual copy]
//   per layer: QKV GEMM (+bias) -> flash attention -> o_proj GEMM (+bias
//   +residual, LayerNorm fused when d_model = 128) -> FFN-in GEMM (+bias
//   +GELU) -> FFN-out GEMM (+bias +residual, then LayerNorm of the next
//   layer, or the model tail on the last layer).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <string>
#include <mutex>
#include <vector>

#include "tfl.h"
#include "kernels.h"

using namespace tfl;

namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(TFL_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define TFL_CUDA(call, what)                         \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D fp16 map over a row-major [rows, cols] matrix, box {64, box_rows}, 128B swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D e4m3 (byte) map over a row-major [rows, cols] plane, box {64, box_rows}: 64-byte rows,
// 64B swizzle (the fp8 operand planes of a 64-wide GEMM k-block).
bool make_map_2d_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D fp16 map over qkv [B, S, 3D]: box {atom_cols, box_rows, 1}.
bool make_map_qkv(CUtensorMap* m, const void* base, uint64_t B, uint64_t S, uint64_t C3, uint32_t atom_cols,
                  uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {C3, S, B};
  cuuint64_t strides[2] = {C3 * 2, S * C3 * 2};
  cuuint32_t box[3] = {atom_cols, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = atom_cols * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map for 32-row tile stores of 64-byte row pieces (fp16: 32 columns, fp32: 16)
// over a row-major [rows, cols] matrix, 64-byte swizzle.
bool make_map_store64(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, bool f32) {
  auto enc = get_encode();
  if (!enc) return false;
  const uint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {(cuuint32_t)(64 / es), 32};
  cuuint32_t ess[2] = {1, 1};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, ess, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// One packed weight matrix: fp16 hi (and lo) parts of W * 2^s, and the 2^-s the GEMM applies.
// In the fp8 operand form (f8) hi holds fp16(W 2^s) 2^11 and the lo storage [N, K] fp16 holds
// the two e4m3 planes [N, K] bytes each (hi, then lo times 2^11); the GEMM applies 2^-(s+11).
struct PackedW {
  __half* hi = nullptr;
  __half* lo = nullptr;
  float acc_scale = 1.f;
  bool f8 = false;
  size_t elems = 0;
  CUtensorMap tm_hi{}, tm_lo{}, tm_lo2{};
  uint8_t* f8hi() const { return reinterpret_cast<uint8_t*>(lo); }
  uint8_t* f8lo() const { return reinterpret_cast<uint8_t*>(lo) + elems; }
};

struct LayerDev {
  PackedW wqkv, wo, w1, w2;
  float *bqkv, *bo, *b1, *b2, *ln1_g, *ln1_b, *ln2_g, *ln2_b;
};

struct GraphEntry {
  int causal;
  int bf16;
  const void* x;
  const void* len;
  void* out;
  cudaGraphExec_t exec;
};

struct WsLayout {
  size_t h32, n16, n16lo, qkv16, o16, g16, g16lo, status, sched, total;
};

// Ints before the tile list in the scheduling area.
inline size_t tile_list_offset(int n_layers) { return align_up((size_t)n_layers, 32); }

// precision 2 adds the lo planes of the GEMM activations (normed rows, GELU output); in the fp8
// operand form the same bytes hold their two e4m3 planes.
WsLayout ws_layout(const tfl_shape& s, int precision) {
  const size_t M = (size_t)s.B * s.S, D = s.d_model, F = s.d_ff;
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 1024);
    return o;
  };
  w.h32 = take(M * D * 4);
  w.n16 = take(M * D * 2);
  w.n16lo = precision == 2 ? take(M * D * 2) : 0;
  w.qkv16 = take(M * 3 * D * 2);
  w.o16 = take(M * D * 2);
  w.g16 = take(M * F * 2);
  w.g16lo = precision == 2 ? take(M * F * 2) : 0;
  w.status = take(256);
  // attention work counters (one per layer), then the tile list
  w.sched = take((size_t)(tile_list_offset(s.n_layers) + 2 + (M + kGemmBM - 1) / kGemmBM) * sizeof(int));
  w.total = off;
  return w;
}

// The fused post-attention chain serves d_model = 128, d_ff <= 2048 at precision 2.
bool use_chain(int D, int F, int precision) { return D == 128 && F <= 2048 && precision == 2; }

// The whole-stack kernel: one sequence per 128-row tile, head_dim 32, the chain's limits.
bool use_stack(const tfl_shape& s, const tfl_options& o) {
  return o.whole_stack && use_chain(s.d_model, s.d_ff, o.precision) && s.S <= 128 && s.n_heads == 4 &&
         s.n_layers <= kStackMaxLayers;
}

// Output tile width: 256 when N allows it, except with split activations (the
// four operand tiles of a 256-wide stage leave room for only two stages).
// GEMM tile width.  A 256-wide tile issues half the MMA instructions per FLOP of a 128-wide
// one, and MMA issue is what holds these GEMMs below the tensor peak; with split activations
// (then two 96 KB ring stages) that pays for the QKV and FFN-in GEMMs above d_model 128
// (N = 3 d_model, d_ff) but not for FFN-out (N = d_model: too few tile rounds on small
// batches, no gain on large ones).  At d_model 128 the fused chain and the whole-stack kernel
// share the 128-row weight maps.
int gemm_bn(int N, int split_act, bool wide_split) {
  return (N % 256 == 0 && (!split_act || wide_split)) ? 256 : 128;
}

}  // namespace

struct tfl_handle {
  tfl_shape shape{};
  tfl_options opt{};
  int device = 0, num_sms = 0;
  int M = 0, D = 0, H = 0, hd = 0, F = 0, L = 0;
  // pre-LN fused chain: W1 carries LN2's affine, and W_qkv of layers >= 1 carries
  // LN1's (layer 0's QKV GEMM reads rows the input LayerNorm already normalised);
  // the whole-stack kernel normalises layer 0's input itself, so there W_qkv of
  // every layer carries LN1's affine
  bool fold = false;
  bool stack = false;
  void* wmem = nullptr;
  void* ws = nullptr;
  WsLayout lay{};
  std::vector<LayerDev> layers;
  float *lnf_g = nullptr, *lnf_b = nullptr;
  float* h32 = nullptr;
  __half *n16 = nullptr, *qkv16 = nullptr, *o16 = nullptr, *g16 = nullptr;
  __half *n16lo = nullptr, *g16lo = nullptr;  // precision 2 only
  // fp8 operand form of the d_model > 128 split GEMMs (QKV, FFN-in, FFN-out): the lo planes'
  // storage holds the two e4m3 planes of the normed rows / GELU output instead
  bool f8 = false;
  int* status = nullptr;
  int* sched = nullptr;
  CUtensorMap tm_n16{}, tm_n16lo{}, tm_o16{}, tm_g16{}, tm_g16lo{}, tm_q{}, tm_kv{};
  CUtensorMap tm_n8hi{}, tm_n8lo{}, tm_g8hi{}, tm_g8lo{};
  uint8_t* n8hi() const { return f8 ? reinterpret_cast<uint8_t*>(n16lo) : nullptr; }
  uint8_t* n8lo() const { return f8 ? reinterpret_cast<uint8_t*>(n16lo) + (size_t)M * D : nullptr; }
  uint8_t* g8hi() const { return f8 ? reinterpret_cast<uint8_t*>(g16lo) : nullptr; }
  uint8_t* g8lo() const { return f8 ? reinterpret_cast<uint8_t*>(g16lo) + (size_t)M * F : nullptr; }
  __half* n16lo_fp16() const { return f8 ? nullptr : n16lo; }  // the fp16 lo plane, when that form is used
  __half* g16lo_fp16() const { return f8 ? nullptr : g16lo; }
  std::vector<GraphEntry> graphs;
  float *hx_dev = nullptr, *hout_dev = nullptr;
  int* hlen_dev = nullptr;
  cudaStream_t cap_stream = nullptr;  // graphs are captured here (the legacy stream cannot be captured)
  // tfl_forward_streamed: two device buffers each for x, out and lengths of one slice;
  // copy-in, compute and copy-out streams; per-slice lengths staged in pinned memory
  float *sx_dev[2] = {}, *sout_dev[2] = {};
  int* slen_dev[2] = {};
  int* slen_pin = nullptr;
  size_t slen_cap = 0;
  cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {}, ev_staged = nullptr;
  bool staged_pending = false;
};

namespace {
// The fused chain (d_model 128) also computes the next layer's QKV projection in its tail.
bool chain_fuses_qkv(const tfl_handle* h) { return use_chain(h->D, h->F, h->opt.precision); }

// Tensor maps of the activation planes the GEMMs and attention read (rebuilt whenever the
// planes move).  Without a lo plane the lo maps repeat the hi ones (never read).
bool make_activation_maps(tfl_handle* h) {
  const uint64_t M = (uint64_t)h->M;
  const int D = h->D, F = h->F;
  const int atom = h->hd < 64 ? h->hd : 64;
  bool ok = make_map_2d(&h->tm_n16, h->n16, M, D, kGemmBM) && make_map_2d(&h->tm_o16, h->o16, M, D, kGemmBM) &&
            make_map_2d(&h->tm_g16, h->g16, M, F, kGemmBM) &&
            make_map_qkv(&h->tm_q, h->qkv16, h->shape.B, h->shape.S, 3 * D, atom, kAttnBM) &&
            make_map_qkv(&h->tm_kv, h->qkv16, h->shape.B, h->shape.S, 3 * D, atom, attn_block_n(h->hd));
  h->tm_n16lo = h->tm_n8hi = h->tm_n8lo = h->tm_n16;
  h->tm_g16lo = h->tm_g8hi = h->tm_g8lo = h->tm_g16;
  if (ok && h->f8)
    ok = make_map_2d_u8(&h->tm_n8hi, h->n8hi(), M, D, kGemmBM) && make_map_2d_u8(&h->tm_n8lo, h->n8lo(), M, D, kGemmBM) &&
         make_map_2d_u8(&h->tm_g8hi, h->g8hi(), M, F, kGemmBM) && make_map_2d_u8(&h->tm_g8lo, h->g8lo(), M, F, kGemmBM);
  else if (ok) {
    if (h->n16lo) ok = make_map_2d(&h->tm_n16lo, h->n16lo, M, D, kGemmBM);
    if (ok && h->g16lo) ok = make_map_2d(&h->tm_g16lo, h->g16lo, M, F, kGemmBM);
  }
  return ok;
}
}  // namespace

namespace {

int check_shape(const tfl_shape* s) {
  if (!s) return fail(TFL_ERR_INVALID_ARG, "shape is NULL");
  if (s->B < 1 || s->S < 1 || s->d_model < 1 || s->n_heads < 1 || s->d_ff < 1 || s->n_layers < 1)
    return fail(TFL_ERR_INVALID_ARG, "every shape field must be >= 1");
  if (s->norm_placement != 0 && s->norm_placement != 1)
    return fail(TFL_ERR_INVALID_ARG, "norm_placement must be 0 (pre-LN) or 1 (post-LN)");
  if (s->d_model % s->n_heads != 0) return fail(TFL_ERR_INVALID_ARG, "n_heads must divide d_model");
  const int hd = s->d_model / s->n_heads;
  if (s->d_model % 128 != 0 || !(s->d_model / 128 == 1 || s->d_model / 128 == 2 || s->d_model / 128 == 4 ||
                                 s->d_model / 128 == 8))
    return fail(TFL_ERR_UNSUPPORTED, "d_model must be 128, 256, 512 or 1024");
  if (s->d_ff % 128 != 0) return fail(TFL_ERR_UNSUPPORTED, "d_ff must be a multiple of 128");
  if (!(hd == 32 || hd == 64 || hd == 256)) return fail(TFL_ERR_UNSUPPORTED, "head_dim must be 32, 64 or 256");
  if ((int64_t)s->B * s->S >= (int64_t)1 << 31) return fail(TFL_ERR_UNSUPPORTED, "B*S must be < 2^31");
  return TFL_OK;
}

// Copy a float32 tensor from host or device memory into a device scratch buffer.
int stage_f32(const float* src, size_t n, float* tmp, const char* name) {
  if (!src) return fail(TFL_ERR_INVALID_ARG, std::string("weight pointer ") + name + " is NULL");
  TFL_CUDA(cudaMemcpy(tmp, src, n * sizeof(float), cudaMemcpyDefault), name);
  return TFL_OK;
}

// Pack `count` float32 matrices (consecutive rows of one GEMM operand) into
// hi (and lo) fp16 parts of W * 2^s, s chosen from the largest |w| so that
// the lo parts sit well inside the normal fp16 range.
int pack_staged(const float* tmp, size_t off, unsigned* dmax, PackedW& w, bool split, const char* name,
                bool f8 = false) {
  TFL_CUDA(cudaMemset(dmax, 0, sizeof(unsigned)), name);
  TFL_CUDA(launch_absmax(tmp, off, dmax, 0), name);
  unsigned bits = 0;
  TFL_CUDA(cudaMemcpy(&bits, dmax, sizeof(unsigned), cudaMemcpyDeviceToHost), name);
  float amax;
  std::memcpy(&amax, &bits, sizeof(float));
  if (!std::isfinite(amax)) return fail(TFL_ERR_INVALID_ARG, std::string("non-finite value in weight ") + name);
  int s = 0;
  if (amax > 0.f) {
    s = 4 - (int)std::ceil(std::log2((double)amax));  // largest |W * 2^s| in (8, 16]
    s = s < -24 ? -24 : (s > 24 ? 24 : s);
  }
  const float scale = std::ldexp(1.0f, s);
  w.acc_scale = std::ldexp(1.0f, -s);
  w.f8 = f8 && split;
  w.elems = off;
  if (w.f8) {
    w.acc_scale = std::ldexp(1.0f, -s - 11);
    TFL_CUDA(launch_split_f8(tmp, w.hi, w.f8hi(), w.f8lo(), off, scale, 0), name);
  } else {
    TFL_CUDA(launch_split_f16(tmp, w.hi, split ? w.lo : nullptr, off, scale, 0), name);
  }
  TFL_CUDA(cudaDeviceSynchronize(), name);
  return TFL_OK;
}

// Stage `count` float32 matrices (consecutive rows of one GEMM operand) into tmp.
int stage_weights(const float* const* src, const size_t* n, int count, float* tmp, size_t* total,
                  const char* name) {
  size_t off = 0;
  for (int i = 0; i < count; ++i) {
    const int rc = stage_f32(src[i], n[i], tmp + off, name);
    if (rc) return rc;
    off += n[i];
  }
  *total = off;
  return TFL_OK;
}

int pack_weights(const float* const* src, const size_t* n, int count, float* tmp, unsigned* dmax, PackedW& w,
                 bool split, const char* name, bool f8 = false) {
  size_t total = 0;
  const int rc = stage_weights(src, n, count, tmp, &total, name);
  return rc ? rc : pack_staged(tmp, total, dmax, w, split, name, f8);
}

int copy_f32(const float* src, size_t n, float* dst, const char* name) {
  if (!src) return fail(TFL_ERR_INVALID_ARG, std::string("weight pointer ") + name + " is NULL");
  TFL_CUDA(cudaMemcpy(dst, src, n * sizeof(float), cudaMemcpyDefault), name);
  return TFL_OK;
}

struct Rec {
  bool on = false;
  std::vector<cudaEvent_t>* ev = nullptr;
  std::vector<int>* kinds = nullptr;
};

cudaError_t rec_mark(const Rec& r, cudaStream_t s, int kind) {
  if (!r.on) return cudaSuccess;
  cudaEvent_t e;
  cudaError_t err = cudaEventCreate(&e);
  if (err != cudaSuccess) return err;
  r.ev->push_back(e);
  if (kind) r.kinds->push_back(kind);
  return cudaEventRecord(e, s);
}

// Enqueue the whole forward on `st`.
// Host memory the device can address directly (pinned and mapped; with unified
// addressing its device pointer is the host pointer).
bool host_resident(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost && a.devicePointer != nullptr;
}

// bf16 = 1: x and out hold bf16 model-dtype rows (the pointers are reinterpreted).
int enqueue(tfl_handle* h, const float* x, const int32_t* lengths, int causal, float* out, cudaStream_t st,
            const Rec& rec, int bf16 = 0) {
  // x in host memory (read over the host link) or in bf16: the input row kernel also
  // writes it into the fp32 residual buffer, which is then the first layer's residual
  const bool x_host = bf16 || host_resident(x);
  const __nv_bfloat16* xbf = bf16 ? reinterpret_cast<const __nv_bfloat16*>(x) : nullptr;
  __nv_bfloat16* outbf = bf16 ? reinterpret_cast<__nv_bfloat16*>(out) : nullptr;
  const bool pre = h->shape.norm_placement == 0;
  const int prec = h->opt.precision;
  const int ws = prec >= 1 ? 1 : 0;  // weights carry lo parts
  const int as = prec == 2 ? 1 : 0;  // normed rows and GELU output carry lo planes
  Common c;
  c.M = h->M;
  c.S = h->shape.S;
  c.lengths = lengths;
  c.status = h->status;
  c.timeout_ns = h->opt.wait_timeout_ns;
  int* tiles = h->sched + tile_list_offset(h->L);
  c.tiles = tiles;
  const float eps = h->opt.ln_eps;
  const int D = h->D, F = h->F, L = h->L;
  auto maps = [](const CUtensorMap& a, const CUtensorMap& alo, const PackedW& w) {
    GemmMaps m;
    m.a = m.a2 = a;
    m.alo = alo;
    m.b = m.b2 = w.tm_hi;
    m.blo = w.tm_lo;
    return m;
  };
  // the GEMMs above d_model 128 that read split activations (QKV, FFN-in, FFN-out): the fp8
  // operand form (mode 2) when the handle uses it, else the fp16 lo planes
  const int as_x = h->f8 ? 2 : as, ws_x = h->f8 ? 2 : ws;
  auto maps_x = [&](const CUtensorMap& a, const CUtensorMap& alo, const CUtensorMap& a8hi, const CUtensorMap& a8lo,
                    const PackedW& w) {
    GemmMaps m = maps(a, alo, w);
    if (h->f8) {
      m.alo = a8hi;
      m.a2 = a8lo;
      m.b2 = w.tm_lo2;
    }
    return m;
  };

  if (h->stack) {  // one launch: the kernel checks the lengths itself and needs no tile list
    StackArgs sa;
    sa.c = c;
    sa.B = h->shape.B;
    sa.F = F;
    sa.L = L;
    sa.causal = causal;
    sa.post_ln = pre ? 0 : 1;
    sa.eps = eps;
    sa.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)h->hd));
    sa.x = bf16 ? nullptr : x;
    sa.xbf = xbf;
    sa.out32 = bf16 ? nullptr : out;
    sa.outbf = outbf;
    sa.lnf_g = h->lnf_g;
    sa.lnf_b = h->lnf_b;
    StackMaps sm;
    for (int l = 0; l < L; ++l) {
      const LayerDev& ly = h->layers[l];
      StackLayerArgs& la = sa.layer[l];
      la.scale_qkv = ly.wqkv.acc_scale;
      la.scale_o = ly.wo.acc_scale;
      la.inv_scale_o = 1.0f / ly.wo.acc_scale;  // exact: powers of two
      la.scale_1 = ly.w1.acc_scale;
      la.scale_2 = ly.w2.acc_scale;
      la.inv_scale_2 = 1.0f / ly.w2.acc_scale;
      la.bqkv = ly.bqkv;
      la.bo = ly.bo;
      la.b1 = ly.b1;
      la.b2 = ly.b2;
      la.ln1_g = ly.ln1_g;
      la.ln1_b = ly.ln1_b;
      la.ln2_g = ly.ln2_g;
      la.ln2_b = ly.ln2_b;
      sm.wqkv[l] = ly.wqkv.tm_hi;
      sm.wqkv_lo[l] = ly.wqkv.tm_lo;
      sm.wo[l] = ly.wo.tm_hi;
      sm.wo_lo[l] = ly.wo.tm_lo;
      sm.w1[l] = ly.w1.tm_hi;
      sm.w1_lo[l] = ly.w1.tm_lo;
      sm.w2[l] = ly.w2.tm_hi;
      sm.w2_lo[l] = ly.w2.tm_lo;
    }
    TFL_CUDA(rec_mark(rec, st, 0), "event");
    TFL_CUDA(launch_stack(sm, sa, h->num_sms, st), "whole-stack kernel");
    TFL_CUDA(rec_mark(rec, st, TFL_KIND_STACK), "event");
    return TFL_OK;
  }

  TFL_CUDA(cudaMemsetAsync(h->sched, 0, (size_t)L * sizeof(int), st), "work counter reset");
  TFL_CUDA(launch_prepare(lengths, h->shape.B, h->shape.S, h->M, h->status, tiles, st), "preparation launch");

  TFL_CUDA(rec_mark(rec, st, 0), "event");
  {
    RowArgs ra;
    ra.c = c;
    ra.D = D;
    ra.in32 = bf16 ? nullptr : x;
    ra.inbf = xbf;
    ra.row.eps = eps;
    ra.row.n16 = h->n16;
    ra.row.n16lo = h->n16lo_fp16();
    ra.row.n8hi = h->n8hi();
    ra.row.n8lo = h->n8lo();
    if (pre) {
      ra.row.flags = ROW_NORM16;
      ra.row.gb = h->layers[0].ln1_g;
      ra.row.bb = h->layers[0].ln1_b;
    } else {
      ra.row.flags = ROW_CAST16;
    }
    if (x_host) {
      ra.row.flags |= ROW_WRITE_H;
      ra.row.h32 = h->h32;
    }
    TFL_CUDA(launch_rows(ra, st), "input row kernel launch");
  }
  TFL_CUDA(rec_mark(rec, st, TFL_KIND_ROWNORM), "event");

  for (int l = 0; l < L; ++l) {
    const LayerDev& ly = h->layers[l];
    const bool last = l == L - 1;
    // QKV projection: [q | k | v] = normed [Wq; Wk; Wv]^T + b (from layer 1 on, the fused
    // chain of the previous layer computes it in its tail)
    if (!(l > 0 && chain_fuses_qkv(h))) {
      GemmArgs g;
      g.c = c;
      g.N = 3 * D;
      g.K = D;
      g.acc_scale = ly.wqkv.acc_scale;
      g.bias = ly.bqkv;
      g.c16 = h->qkv16;
      TFL_CUDA(launch_gemm(gemm_bn(3 * D, as, D > 128), EPI_BIAS_F16, as_x, ws_x,
                           maps_x(h->tm_n16, h->tm_n16lo, h->tm_n8hi, h->tm_n8lo, ly.wqkv), g, h->num_sms, st),
               "qkv gemm");
      TFL_CUDA(rec_mark(rec, st, TFL_KIND_GEMM_QKV), "event");
    }
    // attention
    {
      AttnArgs a;
      a.c = c;
      a.B = h->shape.B;
      a.H = h->H;
      a.D = D;
      a.causal = causal;
      a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)h->hd));
      a.o16 = h->o16;
      a.counter = h->sched + l;
      // work-order groups of (b, h) pairs whose keys and values (fp16) fit in 48 MB of L2
      const double kv_pair = 4.0 * (double)h->shape.S * h->hd;
      const double fit = 48.0 * 1024 * 1024 / kv_pair;
      a.group = fit >= (double)h->shape.B * h->H ? 0 : (fit < 1.0 ? 1 : (int)fit);
      TFL_CUDA(launch_attention(h->hd, h->tm_q, h->tm_kv, a, h->num_sms, st), "attention");
      TFL_CUDA(rec_mark(rec, st, TFL_KIND_ATTENTION), "event");
    }
    if (use_chain(D, F, prec)) {
      // o_proj .. FFN-out .. next LayerNorm in one kernel
      ChainArgs ca;
      ca.c = c;
      ca.F = F;
      ca.eps = eps;
      ca.post_ln = pre ? 0 : 1;
      ca.last = last ? 1 : 0;
      ca.scale_o = ly.wo.acc_scale;
      ca.scale_1 = ly.w1.acc_scale;
      ca.scale_2 = ly.w2.acc_scale;
      ca.inv_scale_2 = 1.0f / ly.w2.acc_scale;  // exact: acc_scale is a power of two
      ca.bo = ly.bo;
      ca.b1 = ly.b1;
      ca.b2 = ly.b2;
      ca.ln1_g = ly.ln1_g;
      ca.ln1_b = ly.ln1_b;
      ca.ln2_g = ly.ln2_g;
      ca.ln2_b = ly.ln2_b;
      if (!last) {
        ca.lnn_g = h->layers[l + 1].ln1_g;
        ca.lnn_b = h->layers[l + 1].ln1_b;
      }
      ca.lnf_g = h->lnf_g;
      ca.lnf_b = h->lnf_b;
      ca.res = (l == 0 && !x_host) ? x : h->h32;
      ca.h32 = h->h32;
      ca.n16 = h->n16;
      ca.n16lo = h->n16lo;
      ca.out32 = bf16 ? nullptr : out;
      ca.outbf = outbf;
      ChainMaps cm;
      if (!last && chain_fuses_qkv(h)) {
        const LayerDev& nx = h->layers[l + 1];
        ca.fuse_qkv = 1;
        ca.scale_qkv = nx.wqkv.acc_scale;
        ca.bqkv = nx.bqkv;
        ca.qkv16 = h->qkv16;
        cm.wqkv = nx.wqkv.tm_hi;  // 128-row boxes at d_model 128
        cm.wqkv_lo = nx.wqkv.tm_lo;
        if (!make_map_store64(&cm.h32_st, h->h32, (uint64_t)h->M, h->D, true) ||
            !make_map_store64(&cm.qkv_st, h->qkv16, (uint64_t)h->M, 3 * h->D, false))
          return fail(TFL_ERR_CUDA, "chain store tensor map encoding failed");
      } else {
        cm.wqkv = ly.wqkv.tm_hi;  // unused
        cm.wqkv_lo = ly.wqkv.tm_lo;
        cm.h32_st = h->tm_o16;  // unused
        cm.qkv_st = h->tm_o16;
      }
      cm.o = h->tm_o16;
      cm.wo = ly.wo.tm_hi;
      cm.wo_lo = ly.wo.tm_lo;
      cm.w1 = ly.w1.tm_hi;  // 128-row boxes at d_model 128
      cm.w1_lo = ly.w1.tm_lo;
      cm.w2 = ly.w2.tm_hi;
      cm.w2_lo = ly.w2.tm_lo;
      TFL_CUDA(launch_postchain(cm, ca, h->num_sms, st), "post-attention chain");
      TFL_CUDA(rec_mark(rec, st, TFL_KIND_POSTCHAIN), "event");
      continue;
    }
    // o_proj + bias + residual (+ LayerNorm); the attention output has no lo plane
    {
      GemmArgs g;
      g.c = c;
      g.N = D;
      g.K = D;
      g.acc_scale = ly.wo.acc_scale;
      g.bias = ly.bo;
      g.res = (l == 0 && !x_host) ? x : h->h32;
      RowOps ro;
      ro.eps = eps;
      ro.h32 = h->h32;
      ro.n16 = h->n16;
      ro.n16lo = h->n16lo_fp16();
      ro.n8hi = h->n8hi();
      ro.n8lo = h->n8lo();
      if (pre) {
        ro.flags = ROW_NORM16;
        ro.gb = ly.ln2_g;
        ro.bb = ly.ln2_b;
      } else {
        ro.flags = ROW_POST_LN | ROW_WRITE_H | ROW_CAST16;
        ro.ga = ly.ln1_g;
        ro.ba = ly.ln1_b;
      }
      const GemmMaps mp = maps(h->tm_o16, h->tm_o16, ly.wo);
      if (D == 128) {
        ro.flags |= ROW_WRITE_H;
        g.row = ro;
        TFL_CUDA(launch_gemm(128, EPI_BIAS_RES_ROW, 0, ws, mp, g, h->num_sms, st), "o_proj gemm");
        TFL_CUDA(rec_mark(rec, st, TFL_KIND_GEMM_OPROJ), "event");
      } else {
        g.h32 = h->h32;
        TFL_CUDA(launch_gemm(gemm_bn(D, 0, false), EPI_BIAS_RES_F32, 0, ws, mp, g, h->num_sms, st), "o_proj gemm");
        TFL_CUDA(rec_mark(rec, st, TFL_KIND_GEMM_OPROJ), "event");
        RowArgs ra;
        ra.c = c;
        ra.D = D;
        ra.in32 = h->h32;
        ra.row = ro;
        TFL_CUDA(launch_rows(ra, st), "row kernel");
        TFL_CUDA(rec_mark(rec, st, TFL_KIND_ROWNORM), "event");
      }
    }
    // FFN-in + bias + GELU
    {
      GemmArgs g;
      g.c = c;
      g.N = F;
      g.K = D;
      g.acc_scale = ly.w1.acc_scale;
      g.bias = ly.b1;
      g.c16 = h->g16;
      g.c16lo = h->g16lo_fp16();
      g.c8hi = h->g8hi();
      g.c8lo = h->g8lo();
      TFL_CUDA(launch_gemm(gemm_bn(F, as, D > 128), EPI_BIAS_GELU_F16, as_x, ws_x,
                           maps_x(h->tm_n16, h->tm_n16lo, h->tm_n8hi, h->tm_n8lo, ly.w1), g, h->num_sms, st),
               "ffn1 gemm");
      TFL_CUDA(rec_mark(rec, st, TFL_KIND_GEMM_FFN1), "event");
    }
    // FFN-out + bias + residual (+ next LayerNorm or the tail)
    {
      GemmArgs g;
      g.c = c;
      g.N = D;
      g.K = F;
      g.acc_scale = ly.w2.acc_scale;
      g.bias = ly.b2;
      g.res = h->h32;
      RowOps ro;
      ro.eps = eps;
      ro.h32 = h->h32;
      ro.n16 = h->n16;
      ro.n16lo = h->n16lo_fp16();
      ro.n8hi = h->n8hi();
      ro.n8lo = h->n8lo();
      ro.out32 = bf16 ? nullptr : out;
      ro.outbf = outbf;
      if (!pre) {
        ro.flags |= ROW_POST_LN;
        ro.ga = ly.ln2_g;
        ro.ba = ly.ln2_b;
      }
      if (last) {
        ro.flags |= ROW_FINAL;
        ro.gf = h->lnf_g;
        ro.bf = h->lnf_b;
      } else if (pre) {
        ro.flags |= ROW_NORM16;
        ro.gb = h->layers[l + 1].ln1_g;
        ro.bb = h->layers[l + 1].ln1_b;
      } else {
        ro.flags |= ROW_WRITE_H | ROW_CAST16;
      }
      const GemmMaps mp = maps_x(h->tm_g16, h->tm_g16lo, h->tm_g8hi, h->tm_g8lo, ly.w2);
      if (D == 128) {
        if (pre && !last) ro.flags |= ROW_WRITE_H;
        g.row = ro;
        TFL_CUDA(launch_gemm(128, EPI_BIAS_RES_ROW, as, ws, mp, g, h->num_sms, st), "ffn2 gemm");
        TFL_CUDA(rec_mark(rec, st, TFL_KIND_GEMM_FFN2), "event");
      } else {
        g.h32 = h->h32;
        TFL_CUDA(launch_gemm(gemm_bn(D, as, false), EPI_BIAS_RES_F32, as_x, ws_x, mp, g, h->num_sms, st), "ffn2 gemm");
        TFL_CUDA(rec_mark(rec, st, TFL_KIND_GEMM_FFN2), "event");
        RowArgs ra;
        ra.c = c;
        ra.D = D;
        ra.in32 = h->h32;
        ra.row = ro;
        TFL_CUDA(launch_rows(ra, st), "row kernel");
        TFL_CUDA(rec_mark(rec, st, TFL_KIND_ROWNORM), "event");
      }
    }
  }
  return TFL_OK;
}

}  // namespace

extern "C" {

int tfl_default_options(tfl_options* o) {
  if (!o) return fail(TFL_ERR_INVALID_ARG, "options is NULL");
  o->precision = 2;
  o->ln_eps = 1e-5f;
  o->wait_timeout_ns = 2000000000LL;
  o->max_workspace_bytes = 0;
  o->use_graph = 1;
  o->whole_stack = 1;
  o->fp8_corrections = 1;
  return TFL_OK;
}

size_t tfl_workspace_bytes(const tfl_shape* s) {
  if (check_shape(s) != TFL_OK) return 0;
  return ws_layout(*s, 2).total;
}

const char* tfl_last_error(void) { return g_err.c_str(); }

int tfl_launch_count(const tfl_handle* h, int causal) {
  (void)causal;
  if (!h) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  if (h->stack) return 1;                           // the whole-stack kernel (it checks the lengths)
  if (chain_fuses_qkv(h)) return 2 + 1 + 2 * h->L;  // layer 0's QKV GEMM, then attention + chain per layer
  const int per_layer = use_chain(h->D, h->F, h->opt.precision) ? 3 : (h->D == 128 ? 5 : 7);
  return 2 + per_layer * h->L;
}

int tfl_create(const tfl_shape* shape, const tfl_weights* w, const tfl_options* opt, tfl_handle** out) {
  g_err.clear();
  if (!out) return fail(TFL_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!w || !w->layers) return fail(TFL_ERR_INVALID_ARG, "weights are NULL");
  if (w->n_layers != shape->n_layers) return fail(TFL_ERR_INVALID_ARG, "weights.n_layers != shape.n_layers");
  tfl_options o;
  tfl_default_options(&o);
  if (opt) o = *opt;
  if (o.precision < 0 || o.precision > 2) return fail(TFL_ERR_INVALID_ARG, "precision must be 0, 1 or 2");
  if (o.fp8_corrections != 0 && o.fp8_corrections != 1)
    return fail(TFL_ERR_INVALID_ARG, "fp8_corrections must be 0 or 1");
  if (!(o.ln_eps > 0.f)) return fail(TFL_ERR_INVALID_ARG, "ln_eps must be > 0");
  if (o.wait_timeout_ns <= 0) o.wait_timeout_ns = 2000000000LL;

  int dev = 0;
  TFL_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  cudaDeviceProp prop;
  TFL_CUDA(cudaGetDeviceProperties(&prop, dev), "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(TFL_ERR_UNSUPPORTED, "device is sm_" + std::to_string(prop.major) + std::to_string(prop.minor) +
                                         "; this library is built for sm_103a (GB300)");
  if (!get_encode()) return fail(TFL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  TFL_CUDA(prepare_gemm_kernels(), "gemm kernel attributes");
  TFL_CUDA(prepare_attention_kernels(), "attention kernel attributes");
  TFL_CUDA(prepare_postchain_kernel(), "chain kernel attributes");
  TFL_CUDA(prepare_stack_kernel(), "whole-stack kernel attributes");

  const int D = shape->d_model, F = shape->d_ff, L = shape->n_layers;
  const WsLayout lay = ws_layout(*shape, o.precision);
  const bool wsplit = o.precision >= 1;
  // weights block: per layer (1 or 2) x (3D*D + D*D + F*D + D*F) halves, 3D + D + F + D + 4D floats; + final LN
  const size_t wl_half = (wsplit ? 2 : 1) * ((size_t)3 * D * D + (size_t)D * D + 2 * (size_t)F * D);
  const size_t wl_float = (size_t)3 * D + D + F + D + 4 * (size_t)D;
  const size_t per_layer = align_up(wl_half * 2, 1024) + align_up(wl_float * 4, 1024);
  const size_t wbytes = per_layer * L + align_up((size_t)2 * D * 4, 1024);
  if (o.max_workspace_bytes > 0 && (int64_t)(lay.total + wbytes) > o.max_workspace_bytes)
    return fail(TFL_ERR_OOM, "workspace + weights (" + std::to_string(lay.total + wbytes) +
                                 " bytes) exceed max_workspace_bytes");

  tfl_handle* h = new tfl_handle();
  h->shape = *shape;
  h->opt = o;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->M = shape->B * shape->S;
  h->D = D;
  h->H = shape->n_heads;
  h->hd = D / shape->n_heads;
  h->F = F;
  h->L = L;
  h->lay = lay;
  h->fold = use_chain(D, F, o.precision) && shape->norm_placement == 0;
  h->stack = use_stack(*shape, o);
  // above d_model 128 the split GEMMs (QKV, FFN-in, FFN-out) take the fp8 operand form
  h->f8 = D > 128 && o.precision == 2 && o.fp8_corrections != 0;
  auto bail = [&](int code) {
    tfl_destroy(h);
    return code;
  };

  cudaError_t e = cudaMalloc(&h->ws, lay.total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(TFL_ERR_OOM, "workspace allocation of " + std::to_string(lay.total) + " bytes failed"));
  }
  e = cudaMalloc(&h->wmem, wbytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(TFL_ERR_OOM, "weight allocation failed"));
  }
  if ((e = cudaMemset(h->ws, 0, lay.total)) != cudaSuccess) return bail(cuda_fail(e, "workspace memset"));
  if ((e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking)) != cudaSuccess)
    return bail(cuda_fail(e, "capture stream"));
  uint8_t* wsb = static_cast<uint8_t*>(h->ws);
  h->h32 = reinterpret_cast<float*>(wsb + lay.h32);
  h->n16 = reinterpret_cast<__half*>(wsb + lay.n16);
  h->qkv16 = reinterpret_cast<__half*>(wsb + lay.qkv16);
  h->o16 = reinterpret_cast<__half*>(wsb + lay.o16);
  h->g16 = reinterpret_cast<__half*>(wsb + lay.g16);
  if (o.precision == 2) {
    h->n16lo = reinterpret_cast<__half*>(wsb + lay.n16lo);
    h->g16lo = reinterpret_cast<__half*>(wsb + lay.g16lo);
  }
  h->status = reinterpret_cast<int*>(wsb + lay.status);
  h->sched = reinterpret_cast<int*>(wsb + lay.sched);

  float* tmp = nullptr;
  if ((e = cudaMalloc(&tmp, (size_t)D * (F > 3 * D ? F : 3 * D) * sizeof(float) + 256)) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(TFL_ERR_OOM, "staging allocation failed"));
  }
  unsigned* dmax = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(tmp) +
                                               (size_t)D * (F > 3 * D ? F : 3 * D) * sizeof(float));
  uint8_t* wp = static_cast<uint8_t*>(h->wmem);
  h->layers.resize(L);
  for (int l = 0; l < L && rc == TFL_OK; ++l) {
    const tfl_layer_weights& src = w->layers[l];
    LayerDev& d = h->layers[l];
    uint8_t* base = wp + per_layer * l;
    __half* hp = reinterpret_cast<__half*>(base);
    auto carve = [&](PackedW& pw, size_t n) {
      pw.hi = hp;
      hp += n;
      if (wsplit) {
        pw.lo = hp;
        hp += n;
      }
    };
    carve(d.wqkv, (size_t)3 * D * D);
    carve(d.wo, (size_t)D * D);
    carve(d.w1, (size_t)F * D);
    carve(d.w2, (size_t)F * D);
    float* fb = reinterpret_cast<float*>(base + align_up(wl_half * 2, 1024));
    d.bqkv = fb;
    d.bo = d.bqkv + 3 * D;
    d.b1 = d.bo + D;
    d.b2 = d.b1 + F;
    d.ln1_g = d.b2 + D;
    d.ln1_b = d.ln1_g + D;
    d.ln2_g = d.ln1_b + D;
    d.ln2_b = d.ln2_g + D;
    const size_t DD = (size_t)D * D, FD = (size_t)F * D;
    if (!rc) rc = copy_f32(src.bq, D, d.bqkv, "bq");
    if (!rc) rc = copy_f32(src.bk, D, d.bqkv + D, "bk");
    if (!rc) rc = copy_f32(src.bv, D, d.bqkv + 2 * D, "bv");
    if (!rc) rc = copy_f32(src.bo, D, d.bo, "bo");
    if (!rc) rc = copy_f32(src.b1, F, d.b1, "b1");
    if (!rc) rc = copy_f32(src.b2, D, d.b2, "b2");
    if (!rc) rc = copy_f32(src.ln1_g, D, d.ln1_g, "ln1_g");
    if (!rc) rc = copy_f32(src.ln1_b, D, d.ln1_b, "ln1_b");
    if (!rc) rc = copy_f32(src.ln2_g, D, d.ln2_g, "ln2_g");
    if (!rc) rc = copy_f32(src.ln2_b, D, d.ln2_b, "ln2_b");
    {
      const float* qkv[3] = {src.wq, src.wk, src.wv};
      const size_t nq[3] = {DD, DD, DD};
      size_t n = 0;
      if (!rc) rc = stage_weights(qkv, nq, 3, tmp, &n, "wq/wk/wv");
      if (!rc && h->fold && (l > 0 || h->stack) &&
          launch_fold_ln(tmp, 3 * D, D, d.ln1_g, d.ln1_b, d.bqkv, 0) != cudaSuccess)
        rc = fail(TFL_ERR_CUDA, "LayerNorm fold of W_qkv failed");
      if (!rc) rc = pack_staged(tmp, n, dmax, d.wqkv, wsplit, "wq/wk/wv", h->f8);
    }
    if (!rc) rc = pack_weights(&src.wo, &DD, 1, tmp, dmax, d.wo, wsplit, "wo");
    {
      size_t n = 0;
      if (!rc) rc = stage_weights(&src.w1, &FD, 1, tmp, &n, "w1");
      if (!rc && h->fold && launch_fold_ln(tmp, F, D, d.ln2_g, d.ln2_b, d.b1, 0) != cudaSuccess)
        rc = fail(TFL_ERR_CUDA, "LayerNorm fold of W1 failed");
      if (!rc) rc = pack_staged(tmp, n, dmax, d.w1, wsplit, "w1", h->f8);
    }
    if (!rc) rc = pack_weights(&src.w2, &FD, 1, tmp, dmax, d.w2, wsplit, "w2", h->f8);
    if (!rc) {
      auto maps = [&](PackedW& pw, uint64_t rows, uint64_t cols, uint32_t box_rows) {
        bool ok = make_map_2d(&pw.tm_hi, pw.hi, rows, cols, box_rows);
        pw.tm_lo = pw.tm_lo2 = pw.tm_hi;
        if (ok && pw.f8)
          ok = make_map_2d_u8(&pw.tm_lo, pw.f8hi(), rows, cols, box_rows) &&
               make_map_2d_u8(&pw.tm_lo2, pw.f8lo(), rows, cols, box_rows);
        else if (ok && pw.lo)
          ok = make_map_2d(&pw.tm_lo, pw.lo, rows, cols, box_rows);
        return ok;
      };
      const int aw = o.precision == 2;
      bool ok = maps(d.wqkv, 3 * D, D, gemm_bn(3 * D, aw, D > 128)) && maps(d.wo, D, D, D == 128 ? 128 : gemm_bn(D, 0, false)) &&
                maps(d.w1, F, D, gemm_bn(F, aw, D > 128)) && maps(d.w2, D, F, D == 128 ? 128 : gemm_bn(D, aw, false));
      if (!ok) rc = fail(TFL_ERR_CUDA, "weight tensor map encoding failed");
    }
  }
  cudaFree(tmp);
  if (rc) return bail(rc);
  float* lnf = reinterpret_cast<float*>(wp + per_layer * L);
  h->lnf_g = lnf;
  h->lnf_b = lnf + D;
  if ((rc = copy_f32(w->lnf_g, D, h->lnf_g, "lnf_g")) != TFL_OK) return bail(rc);
  if ((rc = copy_f32(w->lnf_b, D, h->lnf_b, "lnf_b")) != TFL_OK) return bail(rc);

  if (!make_activation_maps(h)) return bail(fail(TFL_ERR_CUDA, "activation tensor map encoding failed"));
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return bail(cuda_fail(e, "create"));
  *out = h;
  return TFL_OK;
}

static int run_forward(tfl_handle* h, const float* x, const int32_t* lengths, int causal, float* out,
                       cudaStream_t st, int bf16 = 0) {
  if (!h->opt.use_graph) return enqueue(h, x, lengths, causal, out, st, Rec{}, bf16);
  for (auto& g : h->graphs)
    if (g.causal == causal && g.bf16 == bf16 && g.x == x && g.len == lengths && g.out == out) {
      TFL_CUDA(cudaGraphLaunch(g.exec, st), "cudaGraphLaunch");
      return TFL_OK;
    }
  cudaGraph_t graph = nullptr;
  cudaStream_t cs = h->cap_stream;
  TFL_CUDA(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal), "cudaStreamBeginCapture");
  int rc = enqueue(h, x, lengths, causal, out, cs, Rec{}, bf16);
  cudaError_t e = cudaStreamEndCapture(cs, &graph);
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphInstantiate");
  if (h->graphs.size() >= 8) {
    cudaGraphExecDestroy(h->graphs.front().exec);
    h->graphs.erase(h->graphs.begin());
  }
  h->graphs.push_back(GraphEntry{causal, bf16, x, lengths, out, exec});
  TFL_CUDA(cudaGraphLaunch(exec, st), "cudaGraphLaunch");
  return TFL_OK;
}

int tfl_forward(tfl_handle* h, const float* x, const int32_t* lengths, int causal, float* out, tfl_stream stream) {
  g_err.clear();
  if (!h) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  if (!x || !out) return fail(TFL_ERR_INVALID_ARG, "x and out must be non-NULL device pointers");
  if (causal != 0 && causal != 1) return fail(TFL_ERR_INVALID_ARG, "causal must be 0 or 1");
  const size_t bytes = (size_t)h->M * h->D * sizeof(float);
  const uint8_t *xb = reinterpret_cast<const uint8_t*>(x), *ob = reinterpret_cast<const uint8_t*>(out);
  if (xb < ob + bytes && ob < xb + bytes) return fail(TFL_ERR_INVALID_ARG, "out overlaps x");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(TFL_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  return run_forward(h, x, lengths, causal, out, static_cast<cudaStream_t>(stream));
}

int tfl_forward_bf16(tfl_handle* h, const void* x, const int32_t* lengths, int causal, void* out,
                     tfl_stream stream) {
  g_err.clear();
  if (!h) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  if (!x || !out) return fail(TFL_ERR_INVALID_ARG, "x and out must be non-NULL device pointers");
  if (causal != 0 && causal != 1) return fail(TFL_ERR_INVALID_ARG, "causal must be 0 or 1");
  const size_t bytes = (size_t)h->M * h->D * 2;
  const uint8_t *xb = static_cast<const uint8_t*>(x), *ob = static_cast<const uint8_t*>(out);
  if (xb < ob + bytes && ob < xb + bytes) return fail(TFL_ERR_INVALID_ARG, "out overlaps x");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(TFL_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  return run_forward(h, static_cast<const float*>(x), lengths, causal, static_cast<float*>(out),
                     static_cast<cudaStream_t>(stream), 1);
}

int tfl_status(tfl_handle* h, tfl_stream stream) {
  if (!h) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TFL_CUDA(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  int v = 0;
  TFL_CUDA(cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost), "status read");
  if (v) TFL_CUDA(cudaMemset(h->status, 0, sizeof(int)), "status clear");
  if (v & TFL_DEV_TIMEOUT) return fail(TFL_ERR_DEVICE_TIMEOUT, "a device-side wait ran out of time");
  if (v & TFL_DEV_BAD_LENGTHS) return fail(TFL_ERR_BAD_LENGTHS, "a length was outside [0, S] and was clamped");
  return TFL_OK;
}

int tfl_forward_host(tfl_handle* h, const float* x_host, const int32_t* lengths_host, int causal, float* out_host,
                     tfl_stream stream) {
  g_err.clear();
  if (!h) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  if (!x_host || !out_host) return fail(TFL_ERR_INVALID_ARG, "x and out must be non-NULL host pointers");
  const size_t bytes = (size_t)h->M * h->D * sizeof(float);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Pinned, mapped host buffers: the kernels read x and write out across the host
  // link themselves (no staging copies); only the lengths are copied to the device.
  if (host_resident(x_host) && host_resident(out_host) &&
      !((reinterpret_cast<uintptr_t>(x_host) | reinterpret_cast<uintptr_t>(out_host)) & 15)) {
    const uint8_t *xb = reinterpret_cast<const uint8_t*>(x_host), *ob = reinterpret_cast<const uint8_t*>(out_host);
    if (xb < ob + bytes && ob < xb + bytes) return fail(TFL_ERR_INVALID_ARG, "out overlaps x");
    if (lengths_host && !h->hlen_dev && cudaMalloc(&h->hlen_dev, (size_t)h->shape.B * sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return fail(TFL_ERR_OOM, "lengths buffer for tfl_forward_host");
    }
    if (lengths_host)
      TFL_CUDA(cudaMemcpyAsync(h->hlen_dev, lengths_host, (size_t)h->shape.B * sizeof(int), cudaMemcpyHostToDevice, st),
               "lengths upload");
    cudaPointerAttributes ax{}, ao{};
    TFL_CUDA(cudaPointerGetAttributes(&ax, x_host), "x attributes");
    TFL_CUDA(cudaPointerGetAttributes(&ao, out_host), "out attributes");
    const int rc = run_forward(h, static_cast<const float*>(ax.devicePointer), lengths_host ? h->hlen_dev : nullptr,
                               causal, static_cast<float*>(ao.devicePointer), st);
    if (rc) return rc;
    return tfl_status(h, stream);
  }
  if (!h->hx_dev) {
    if (cudaMalloc(&h->hx_dev, bytes) != cudaSuccess || cudaMalloc(&h->hout_dev, bytes) != cudaSuccess ||
        cudaMalloc(&h->hlen_dev, (size_t)h->shape.B * sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return fail(TFL_ERR_OOM, "staging buffers for tfl_forward_host");
    }
  }
  TFL_CUDA(cudaMemcpyAsync(h->hx_dev, x_host, bytes, cudaMemcpyHostToDevice, st), "x upload");
  if (lengths_host)
    TFL_CUDA(cudaMemcpyAsync(h->hlen_dev, lengths_host, (size_t)h->shape.B * sizeof(int), cudaMemcpyHostToDevice, st),
             "lengths upload");
  int rc = run_forward(h, h->hx_dev, lengths_host ? h->hlen_dev : nullptr, causal, h->hout_dev, st);
  if (rc) return rc;
  TFL_CUDA(cudaMemcpyAsync(out_host, h->hout_dev, bytes, cudaMemcpyDeviceToHost, st), "out download");
  return tfl_status(h, stream);
}

namespace {
// Pinned (page-locked) host memory: allocated or registered with the CUDA runtime.
bool host_pinned(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

int streamed_setup(tfl_handle* h, size_t n_slices) {
  const size_t slice = (size_t)h->M * h->D * sizeof(float);
  if (!h->s_in) {
    for (cudaStream_t* st : {&h->s_in, &h->s_comp, &h->s_out})
      TFL_CUDA(cudaStreamCreateWithFlags(st, cudaStreamNonBlocking), "streamed: stream");
    TFL_CUDA(cudaEventCreateWithFlags(&h->ev_start, cudaEventDisableTiming), "streamed: event");
    TFL_CUDA(cudaEventCreateWithFlags(&h->ev_staged, cudaEventDisableTiming), "streamed: event");
    for (int i = 0; i < 2; ++i) {
      TFL_CUDA(cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming), "streamed: event");
      TFL_CUDA(cudaEventCreateWithFlags(&h->ev_comp[i], cudaEventDisableTiming), "streamed: event");
      TFL_CUDA(cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming), "streamed: event");
    }
  }
  for (int i = 0; i < 2; ++i) {
    if (h->sx_dev[i]) continue;
    if (cudaMalloc(&h->sx_dev[i], slice) != cudaSuccess || cudaMalloc(&h->sout_dev[i], slice) != cudaSuccess ||
        cudaMalloc(&h->slen_dev[i], (size_t)h->shape.B * sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return fail(TFL_ERR_OOM, "slice buffers for tfl_forward_streamed");
    }
  }
  const size_t need = n_slices * (size_t)h->shape.B;
  if (need > h->slen_cap) {
    if (h->slen_pin) cudaFreeHost(h->slen_pin);
    h->slen_pin = nullptr;
    h->slen_cap = 0;
    if (cudaHostAlloc(reinterpret_cast<void**>(&h->slen_pin), need * sizeof(int), cudaHostAllocDefault) !=
        cudaSuccess) {
      cudaGetLastError();
      return fail(TFL_ERR_OOM, "pinned lengths staging for tfl_forward_streamed");
    }
    h->slen_cap = need;
  }
  return TFL_OK;
}
}  // namespace

int tfl_forward_streamed(tfl_handle* h, const float* x_host, const int32_t* lengths_host, int64_t n_seq, int causal,
                         float* out_host, tfl_stream stream) {
  g_err.clear();
  if (!h) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  if (!x_host || !out_host) return fail(TFL_ERR_INVALID_ARG, "x and out must be non-NULL host pointers");
  if (n_seq < 1) return fail(TFL_ERR_INVALID_ARG, "n_seq must be >= 1");
  if (causal != 0 && causal != 1) return fail(TFL_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!host_pinned(x_host) || !host_pinned(out_host))
    return fail(TFL_ERR_INVALID_ARG, "x and out must be pinned host memory (cudaHostAlloc / cudaHostRegister)");
  const int B = h->shape.B, S = h->shape.S;
  const size_t seq_elems = (size_t)S * h->D;
  const size_t total = (size_t)n_seq * seq_elems * sizeof(float);
  const uint8_t *xb = reinterpret_cast<const uint8_t*>(x_host), *ob = reinterpret_cast<const uint8_t*>(out_host);
  if (xb < ob + total && ob < xb + total) return fail(TFL_ERR_INVALID_ARG, "out overlaps x");
  if (lengths_host)
    for (int64_t b = 0; b < n_seq; ++b)
      if (lengths_host[b] < 0 || lengths_host[b] > S) return fail(TFL_ERR_INVALID_ARG, "a length is outside [0, S]");
  const size_t n_slices = (size_t)((n_seq + B - 1) / B);
  // the staging area of the previous call must no longer be read by its copies
  if (h->staged_pending) TFL_CUDA(cudaEventSynchronize(h->ev_staged), "streamed: previous call");
  h->staged_pending = false;
  int rc = streamed_setup(h, n_slices);
  if (rc) return rc;
  // per-slice lengths; sequences past n_seq in the last slice get length 0 (output zero, never copied back)
  for (size_t k = 0; k < n_slices; ++k)
    for (int j = 0; j < B; ++j) {
      const int64_t b = (int64_t)k * B + j;
      h->slen_pin[k * B + j] = b < n_seq ? (lengths_host ? lengths_host[b] : S) : 0;
    }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TFL_CUDA(cudaEventRecord(h->ev_start, st), "streamed: start");
  for (cudaStream_t s2 : {h->s_in, h->s_comp, h->s_out})
    TFL_CUDA(cudaStreamWaitEvent(s2, h->ev_start, 0), "streamed: start wait");
  for (size_t k = 0; k < n_slices; ++k) {
    const int i = (int)(k & 1);
    const int64_t nk = std::min<int64_t>(B, n_seq - (int64_t)k * B);
    const size_t off = k * (size_t)B * seq_elems;
    const size_t bytes = (size_t)nk * seq_elems * sizeof(float);
    // copy-in: buffer i was last read by the forward of slice k - 2
    if (k >= 2) TFL_CUDA(cudaStreamWaitEvent(h->s_in, h->ev_comp[i], 0), "streamed: wait");
    TFL_CUDA(cudaMemcpyAsync(h->sx_dev[i], x_host + off, bytes, cudaMemcpyHostToDevice, h->s_in), "streamed: x in");
    TFL_CUDA(cudaMemcpyAsync(h->slen_dev[i], h->slen_pin + k * B, (size_t)B * sizeof(int), cudaMemcpyHostToDevice,
                             h->s_in),
             "streamed: lengths in");
    TFL_CUDA(cudaEventRecord(h->ev_in[i], h->s_in), "streamed: event");
    // compute: out buffer i was last read by the copy-out of slice k - 2
    TFL_CUDA(cudaStreamWaitEvent(h->s_comp, h->ev_in[i], 0), "streamed: wait");
    if (k >= 2) TFL_CUDA(cudaStreamWaitEvent(h->s_comp, h->ev_out[i], 0), "streamed: wait");
    rc = run_forward(h, h->sx_dev[i], h->slen_dev[i], causal, h->sout_dev[i], h->s_comp);
    if (rc) return rc;
    TFL_CUDA(cudaEventRecord(h->ev_comp[i], h->s_comp), "streamed: event");
    // copy-out
    TFL_CUDA(cudaStreamWaitEvent(h->s_out, h->ev_comp[i], 0), "streamed: wait");
    TFL_CUDA(cudaMemcpyAsync(out_host + off, h->sout_dev[i], bytes, cudaMemcpyDeviceToHost, h->s_out),
             "streamed: out");
    TFL_CUDA(cudaEventRecord(h->ev_out[i], h->s_out), "streamed: event");
  }
  // every copy-in precedes its forward, every forward its copy-out: the last copy-out ends the batch
  TFL_CUDA(cudaEventRecord(h->ev_staged, h->s_out), "streamed: event");
  h->staged_pending = true;
  TFL_CUDA(cudaStreamWaitEvent(st, h->ev_staged, 0), "streamed: end wait");
  return TFL_OK;
}

int tfl_profile_forward(tfl_handle* h, const float* x, const int32_t* lengths, int causal, float* out,
                        tfl_stream stream, float* kernel_ms, int32_t* kernel_kind, int32_t cap, int32_t* n) {
  g_err.clear();
  if (!h || !x || !out || !n) return fail(TFL_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<cudaEvent_t> ev;
  std::vector<int> kinds;
  Rec r;
  r.on = true;
  r.ev = &ev;
  r.kinds = &kinds;
  int rc = enqueue(h, x, lengths, causal, out, st, r);
  cudaError_t e = cudaStreamSynchronize(st);
  if (!rc && e != cudaSuccess) rc = cuda_fail(e, "profile sync");
  const int cnt = (int)kinds.size();
  *n = cnt;
  for (int i = 0; i < cnt && i < cap && !rc; ++i) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, ev[i], ev[i + 1]);
    if (kernel_ms) kernel_ms[i] = ms;
    if (kernel_kind) kernel_kind[i] = kinds[i];
  }
  for (auto e2 : ev) cudaEventDestroy(e2);
  return rc;
}

void tfl_destroy(tfl_handle* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);
  for (int i = 0; i < 2; ++i) {
    if (h->sx_dev[i]) cudaFree(h->sx_dev[i]);
    if (h->sout_dev[i]) cudaFree(h->sout_dev[i]);
    if (h->slen_dev[i]) cudaFree(h->slen_dev[i]);
    if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
    if (h->ev_comp[i]) cudaEventDestroy(h->ev_comp[i]);
    if (h->ev_out[i]) cudaEventDestroy(h->ev_out[i]);
  }
  if (h->slen_pin) cudaFreeHost(h->slen_pin);
  if (h->ev_start) cudaEventDestroy(h->ev_start);
  if (h->ev_staged) cudaEventDestroy(h->ev_staged);
  for (cudaStream_t st : {h->s_in, h->s_comp, h->s_out})
    if (st) cudaStreamDestroy(st);
  if (h->ws) cudaFree(h->ws);
  if (h->wmem) cudaFree(h->wmem);
  if (h->hx_dev) cudaFree(h->hx_dev);
  if (h->hout_dev) cudaFree(h->hout_dev);
  if (h->hlen_dev) cudaFree(h->hlen_dev);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  delete h;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free forward: every intermediate of the forward (residual, normed
// rows, qkv, attention output, FFN activations, attention work counters) lives
// in this file-scope device array instead of the handle's workspace.  It is
// created with the library's device code, so every GPU that loads the library
// holds it until the process exits; calls on one device share it.
static constexpr size_t kNoallocScratchBytes = (size_t)32 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {
// Device address of g_noalloc_scratch per device (host code cannot use the
// symbol itself: on the host it names a stand-in, not device memory).
std::mutex g_noalloc_mu;
void* g_noalloc_base[128] = {};
}  // namespace

extern "C" {

int tfl_forward_noalloc(tfl_handle* h, const float* x, const int32_t* lengths, int causal, float* out,
                        tfl_stream stream) {
  g_err.clear();
  if (!h) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  if (!x || !out) return fail(TFL_ERR_INVALID_ARG, "x and out must be non-NULL device pointers");
  if (causal != 0 && causal != 1) return fail(TFL_ERR_INVALID_ARG, "causal must be 0 or 1");
  const size_t bytes = (size_t)h->M * h->D * sizeof(float);
  const uint8_t *xb = reinterpret_cast<const uint8_t*>(x), *ob = reinterpret_cast<const uint8_t*>(out);
  if (xb < ob + bytes && ob < xb + bytes) return fail(TFL_ERR_INVALID_ARG, "out overlaps x");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(TFL_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  const WsLayout lay = ws_layout(h->shape, h->opt.precision);
  if (lay.total > kNoallocScratchBytes)
    return fail(TFL_ERR_UNSUPPORTED, "tfl_forward_noalloc: this shape needs " + std::to_string(lay.total) +
                                         " bytes of scratch, more than its fixed " +
                                         std::to_string(kNoallocScratchBytes) + "-byte device array");
  int dev = 0;
  TFL_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != h->device) return fail(TFL_ERR_INVALID_ARG, "the current device is not the handle's device");
  if (dev < 0 || dev >= 128) return fail(TFL_ERR_UNSUPPORTED, "device ordinal above 127");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_base[dev]) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
      g_noalloc_base[dev] = p;
    }
    base = g_noalloc_base[dev];
  }

  // Point this call's intermediates at the scratch (the handle keeps its own
  // weights and status word), run the launch sequence eagerly, then restore.
  uint8_t* sb = static_cast<uint8_t*>(base);
  struct Intermediates {
    float* h32;
    __half *n16, *n16lo, *qkv16, *o16, *g16, *g16lo;
    int* sched;
    CUtensorMap tm_n16, tm_n16lo, tm_o16, tm_g16, tm_g16lo, tm_q, tm_kv, tm_n8hi, tm_n8lo, tm_g8hi, tm_g8lo;
  };
  const Intermediates saved{h->h32,       h->n16,     h->n16lo,   h->qkv16,   h->o16,    h->g16,
                            h->g16lo,     h->sched,   h->tm_n16,  h->tm_n16lo, h->tm_o16, h->tm_g16,
                            h->tm_g16lo,  h->tm_q,    h->tm_kv,   h->tm_n8hi, h->tm_n8lo, h->tm_g8hi,
                            h->tm_g8lo};
  auto restore = [&]() {
    h->h32 = saved.h32;
    h->n16 = saved.n16;
    h->n16lo = saved.n16lo;
    h->qkv16 = saved.qkv16;
    h->o16 = saved.o16;
    h->g16 = saved.g16;
    h->g16lo = saved.g16lo;
    h->sched = saved.sched;
    h->tm_n16 = saved.tm_n16;
    h->tm_n16lo = saved.tm_n16lo;
    h->tm_o16 = saved.tm_o16;
    h->tm_g16 = saved.tm_g16;
    h->tm_g16lo = saved.tm_g16lo;
    h->tm_q = saved.tm_q;
    h->tm_kv = saved.tm_kv;
    h->tm_n8hi = saved.tm_n8hi;
    h->tm_n8lo = saved.tm_n8lo;
    h->tm_g8hi = saved.tm_g8hi;
    h->tm_g8lo = saved.tm_g8lo;
  };
  h->h32 = reinterpret_cast<float*>(sb + lay.h32);
  h->n16 = reinterpret_cast<__half*>(sb + lay.n16);
  h->n16lo = h->opt.precision == 2 ? reinterpret_cast<__half*>(sb + lay.n16lo) : nullptr;
  h->qkv16 = reinterpret_cast<__half*>(sb + lay.qkv16);
  h->o16 = reinterpret_cast<__half*>(sb + lay.o16);
  h->g16 = reinterpret_cast<__half*>(sb + lay.g16);
  h->g16lo = h->opt.precision == 2 ? reinterpret_cast<__half*>(sb + lay.g16lo) : nullptr;
  h->sched = reinterpret_cast<int*>(sb + lay.sched);  // zeroed by the launch sequence itself
  if (!make_activation_maps(h)) {
    restore();
    return fail(TFL_ERR_CUDA, "scratch tensor map encoding failed");
  }
  // The array keeps whatever the last call left, from any handle, shape or precision.
  // Some rows of it are read without being written first (rows of a 128-row tile that
  // lies wholly in padding, read as keys past len_b and multiplied by a zero
  // probability): clear the part this call uses, so that stale bytes can never decode
  // as Inf or NaN there.
  cudaError_t ce = cudaMemsetAsync(base, 0, lay.total, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) {
    restore();
    return cuda_fail(ce, "scratch clear");
  }
  const int rc = enqueue(h, x, lengths, causal, out, static_cast<cudaStream_t>(stream), Rec{});
  restore();
  return rc;
}

int tfl_selftest_gelu(int32_t n, float* max_abs_diff, tfl_stream stream) {
  g_err.clear();
  if (n < 2 || !max_abs_diff) return fail(TFL_ERR_INVALID_ARG, "n must be >= 2 and max_abs_diff non-NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* d = nullptr;
  TFL_CUDA(cudaMalloc(&d, sizeof(unsigned)), "selftest alloc");
  cudaError_t e = cudaMemsetAsync(d, 0, sizeof(unsigned), st);
  if (e == cudaSuccess) e = launch_gelu_selftest(n, d, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  unsigned bits = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&bits, d, sizeof(unsigned), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) return cuda_fail(e, "gelu selftest");
  std::memcpy(max_abs_diff, &bits, sizeof(float));
  return TFL_OK;
}

int tfl_probe_wait_timeout(int64_t timeout_ns, tfl_stream stream) {
  g_err.clear();
  if (timeout_ns <= 0) return fail(TFL_ERR_INVALID_ARG, "timeout must be > 0");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = nullptr;
  TFL_CUDA(cudaMalloc(&status, sizeof(int)), "probe alloc");
  cudaMemset(status, 0, sizeof(int));
  cudaError_t e = launch_probe_wait(status, timeout_ns, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  int v = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(status);
  if (e != cudaSuccess) return cuda_fail(e, "probe");
  if (v & TFL_DEV_TIMEOUT) return fail(TFL_ERR_DEVICE_TIMEOUT, "probe wait ran out as expected");
  return TFL_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Attention on its own (forward with the row log-sum-exp, backward).
struct tfl_attn {
  int B = 0, S = 0, H = 0, hd = 0;
  int device = 0, num_sms = 0;
  int* scratch = nullptr;  // [0] status word, [1] work counter (256 bytes), then delta
  float* delta = nullptr;  // [B, H, S]
  int64_t timeout_ns = 2000000000LL;
};

extern "C" {

int tfl_attn_create(int32_t B, int32_t S, int32_t n_heads, int32_t head_dim, tfl_attn** out) {
  g_err.clear();
  if (!out) return fail(TFL_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (B < 1 || S < 1 || n_heads < 1) return fail(TFL_ERR_INVALID_ARG, "B, S and n_heads must be >= 1");
  if (head_dim != 32 && head_dim != 64) return fail(TFL_ERR_UNSUPPORTED, "head_dim must be 32 or 64");
  if ((int64_t)B * S * 3 * n_heads * head_dim >= ((int64_t)1 << 31))
    return fail(TFL_ERR_UNSUPPORTED, "B * S * 3 * n_heads * head_dim must be < 2^31");
  int dev = 0;
  TFL_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  cudaDeviceProp prop;
  TFL_CUDA(cudaGetDeviceProperties(&prop, dev), "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(TFL_ERR_UNSUPPORTED, "device is sm_" + std::to_string(prop.major) + std::to_string(prop.minor) +
                                         "; this library is built for sm_103a (GB300)");
  if (!get_encode()) return fail(TFL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  TFL_CUDA(prepare_attention_kernels(), "attention kernel attributes");
  TFL_CUDA(prepare_attention_bwd_kernels(), "attention backward kernel attributes");
  tfl_attn* a = new tfl_attn();
  a->B = B;
  a->S = S;
  a->H = n_heads;
  a->hd = head_dim;
  a->device = dev;
  a->num_sms = prop.multiProcessorCount;
  const size_t bytes = 256 + (size_t)B * n_heads * S * sizeof(float);
  if (cudaMalloc(&a->scratch, bytes) != cudaSuccess) {
    cudaGetLastError();
    delete a;
    return fail(TFL_ERR_OOM, "attention scratch allocation failed");
  }
  a->delta = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(a->scratch) + 256);
  if (cudaMemset(a->scratch, 0, 256) != cudaSuccess) {
    cudaFree(a->scratch);
    delete a;
    return fail(TFL_ERR_CUDA, "attention scratch clear failed");
  }
  *out = a;
  return TFL_OK;
}

int tfl_attn_forward(tfl_attn* a, const void* qkv, const int32_t* lengths, int causal, void* o, float* lse,
                     tfl_stream stream) {
  g_err.clear();
  if (!a) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  if (!qkv || !o || !lse) return fail(TFL_ERR_INVALID_ARG, "qkv, o and lse must be non-NULL device pointers");
  if (causal != 0 && causal != 1) return fail(TFL_ERR_INVALID_ARG, "causal must be 0 or 1");
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(lse)) & 15)
    return fail(TFL_ERR_INVALID_ARG, "qkv, o and lse must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int D = a->H * a->hd, atom = a->hd < 64 ? a->hd : 64;
  CUtensorMap tq, tkv;
  if (!make_map_qkv(&tq, qkv, a->B, a->S, 3 * D, atom, kAttnBM) ||
      !make_map_qkv(&tkv, qkv, a->B, a->S, 3 * D, atom, attn_block_n(a->hd)))
    return fail(TFL_ERR_CUDA, "attention tensor map encoding failed");
  TFL_CUDA(cudaMemsetAsync(a->scratch + 1, 0, sizeof(int), st), "work counter reset");
  AttnArgs args;
  args.c.M = a->B * a->S;
  args.c.S = a->S;
  args.c.lengths = lengths;
  args.c.status = a->scratch;
  args.c.timeout_ns = a->timeout_ns;
  args.B = a->B;
  args.H = a->H;
  args.D = D;
  args.causal = causal;
  args.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a->hd));
  args.o16 = static_cast<__half*>(o);
  args.counter = a->scratch + 1;
  const double fit = 48.0 * 1024 * 1024 / (4.0 * (double)a->S * a->hd);
  args.group = fit >= (double)a->B * a->H ? 0 : (fit < 1.0 ? 1 : (int)fit);
  args.lse = lse;
  TFL_CUDA(launch_prepare(lengths, a->B, a->S, a->B * a->S, a->scratch, nullptr, st), "length check");
  TFL_CUDA(launch_attention(a->hd, tq, tkv, args, a->num_sms, st), "attention");
  return TFL_OK;
}

int tfl_attn_backward(tfl_attn* a, const void* qkv, const void* o, const void* dout, const float* lse,
                      const int32_t* lengths, int causal, float* dqkv, tfl_stream stream) {
  g_err.clear();
  if (!a) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  if (!qkv || !o || !dout || !lse || !dqkv) return fail(TFL_ERR_INVALID_ARG, "NULL device pointer");
  if (causal != 0 && causal != 1) return fail(TFL_ERR_INVALID_ARG, "causal must be 0 or 1");
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dout) |
       reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(dqkv)) & 15)
    return fail(TFL_ERR_INVALID_ARG, "all buffers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int D = a->H * a->hd;
  CUtensorMap tqkv, tdo;
  if (!make_map_qkv(&tqkv, qkv, a->B, a->S, 3 * D, a->hd, 64) || !make_map_qkv(&tdo, dout, a->B, a->S, D, a->hd, 64))
    return fail(TFL_ERR_CUDA, "attention backward tensor map encoding failed");
  TFL_CUDA(cudaMemsetAsync(dqkv, 0, (size_t)a->B * a->S * 3 * D * sizeof(float), st), "dqkv clear");
  AttnBwdArgs args;
  args.c.M = a->B * a->S;
  args.c.S = a->S;
  args.c.lengths = lengths;
  args.c.status = a->scratch;
  args.c.timeout_ns = a->timeout_ns;
  args.B = a->B;
  args.H = a->H;
  args.causal = causal;
  args.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a->hd));
  args.inv_sqrt_hd = (float)(1.0 / std::sqrt((double)a->hd));
  args.lse = lse;
  args.delta = a->delta;
  args.dqkv = dqkv;
  TFL_CUDA(launch_prepare(lengths, a->B, a->S, a->B * a->S, a->scratch, nullptr, st), "length check");
  TFL_CUDA(launch_attention_bwd(a->hd, tqkv, tdo, args, static_cast<const __half*>(dout),
                                static_cast<const __half*>(o), a->num_sms, st),
           "attention backward");
  return TFL_OK;
}

int tfl_attn_status(tfl_attn* a, tfl_stream stream) {
  if (!a) return fail(TFL_ERR_INVALID_ARG, "handle is NULL");
  TFL_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "cudaStreamSynchronize");
  int v = 0;
  TFL_CUDA(cudaMemcpy(&v, a->scratch, sizeof(int), cudaMemcpyDeviceToHost), "status read");
  if (v) TFL_CUDA(cudaMemset(a->scratch, 0, sizeof(int)), "status clear");
  if (v & TFL_DEV_TIMEOUT) return fail(TFL_ERR_DEVICE_TIMEOUT, "a device-side wait ran out of time");
  if (v & TFL_DEV_BAD_LENGTHS) return fail(TFL_ERR_BAD_LENGTHS, "a length was outside [0, S] and was clamped");
  return TFL_OK;
}

void tfl_attn_destroy(tfl_attn* a) {
  if (!a) return;
  cudaDeviceSynchronize();
  if (a->scratch) cudaFree(a->scratch);
  delete a;
}

}  // extern "C"
