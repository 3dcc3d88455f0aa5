// kernels.h -- argument blocks and host launchers of the forward's kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

// Bits of the device status word (OR-ed by kernels, read by tfl_status).
#define TFL_DEV_TIMEOUT 1
#define TFL_DEV_BAD_LENGTHS 2

namespace tfl {

// Row-epilogue operations (GEMM epilogue with BN == d_model, and the
// standalone row kernel).  Starting from the fp32 row t:
//   POST_LN     t = LN(t; ga, ba)                     (post-LN residual norm)
//   WRITE_H     h32[row] = t                          (residual stream)
//   FINAL       out32[row] = valid ? LN(t; gf, bf) : 0 (model tail)
//   NORM16      n16[row] = fp16(LN(t; gb, bb))        (pre-LN sublayer input)
//   CAST16      n16[row] = fp16(t)                    (post-LN sublayer input)
enum RowFlags : int {
  ROW_POST_LN = 1,
  ROW_WRITE_H = 2,
  ROW_FINAL = 4,
  ROW_NORM16 = 8,
  ROW_CAST16 = 16,
};

struct RowOps {
  int flags = 0;
  float eps = 1e-5f;
  const float *ga = nullptr, *ba = nullptr;  // POST_LN affine
  const float *gb = nullptr, *bb = nullptr;  // NORM16 affine
  const float *gf = nullptr, *bf = nullptr;  // FINAL affine
  float* h32 = nullptr;                      // [M, D]
  __half* n16 = nullptr;                     // [M, D] fp16 (hi part when split)
  __half* n16lo = nullptr;                   // [M, D] fp16 residual plane, or null
  // fp8 operand form (instead of n16lo): e4m3 of the fp16 value and e4m3 of its
  // rounding residual times 2^11, [M, D] bytes each
  uint8_t* n8hi = nullptr;
  uint8_t* n8lo = nullptr;
  float* out32 = nullptr;                    // [M, D]
  __nv_bfloat16* outbf = nullptr;            // [M, D] bf16 model output instead of out32 (FINAL)
};

struct Common {
  int M = 0;                       // B * S rows
  int S = 0;
  const int* lengths = nullptr;    // device [B] or null
  int* status = nullptr;           // device status word
  int64_t timeout_ns = 2000000000LL;
  // 128-row tiles in processing order, written once per forward by the
  // preparation kernel: [0] tiles holding a valid row, [1] all tiles, then the
  // live tiles ascending followed by the dead ones ascending
  const int* tiles = nullptr;
};

// GEMM: C[M, N] = A[M, K] (fp16, K-major) * W[N, K]^T (fp16, K-major), fp32 accumulate.
enum GemmEpi : int {
  EPI_BIAS_F16 = 0,       // c16 = acc + bias
  EPI_BIAS_GELU_F16 = 1,  // c16 = GELU(acc + bias)
  EPI_BIAS_RES_F32 = 2,   // h32 = acc + bias + (valid ? res : 0)
  EPI_BIAS_RES_ROW = 3,   // t = acc + bias + (valid ? res : 0), then RowOps (N == BN == d_model)
};

struct GemmArgs {
  Common c;
  int N = 0, K = 0;
  float acc_scale = 1.f;         // 2^-s undoing the weight pre-scale
  const float* bias = nullptr;   // [N]
  __half* c16 = nullptr;         // [M, N] for the fp16 epilogues
  __half* c16lo = nullptr;       // [M, N] residual plane (split activations), or null
  uint8_t* c8hi = nullptr;       // fp8 operand form of c16 (instead of c16lo): e4m3(c16) and
  uint8_t* c8lo = nullptr;       //   e4m3(residual * 2^11), [M, N] bytes each
  const float* res = nullptr;    // [M, N] residual for the fp32 epilogues (may alias h32)
  float* h32 = nullptr;          // EPI_BIAS_RES_F32 output
  RowOps row;                    // EPI_BIAS_RES_ROW
};

struct AttnArgs {
  Common c;
  int B = 0, H = 0, D = 0;
  int causal = 0;
  float scale_log2 = 0.f;        // log2(e) / sqrt(head_dim)
  __half* o16 = nullptr;         // [M, D]
  int* counter = nullptr;        // work-item counter, zero before the launch
  int group = 0;                 // (b, h) pairs per work-order group (see decode_item); 0: one group
  float* lse = nullptr;          // [B, H, S] row log-sum-exp in log2 units (rows < len_b), or null
};

// Attention backward (head_dim 32 or 64): qkv [B, S, 3 H hd] fp16, dO [B, S, H hd] fp16.
struct AttnBwdArgs {
  Common c;
  int B = 0, H = 0, causal = 0;
  float scale_log2 = 0.f;        // log2(e) / sqrt(head_dim)
  float inv_sqrt_hd = 0.f;
  const float* lse = nullptr;    // [B, H, S] from the forward, log2 units
  float* delta = nullptr;        // [B, H, S] dO_i . O_i, written by the first kernel
  float* dqkv = nullptr;         // [B, S, 3 H hd] fp32; rows past len_b are left untouched
};
cudaError_t prepare_attention_bwd_kernels();
// D = rowsum(dO O), then the dQ kernel and the dK / dV kernel.
cudaError_t launch_attention_bwd(int hd, const CUtensorMap& tqkv, const CUtensorMap& tdo, const AttnBwdArgs& a,
                                 const __half* dout, const __half* o, int num_sms, cudaStream_t s);

struct RowArgs {
  Common c;
  int D = 0;
  const float* in32 = nullptr;   // [M, D] fp32 input rows (x or h32)
  const __nv_bfloat16* inbf = nullptr;  // [M, D] bf16 input rows instead of in32
  RowOps row;
};

// One-time kernel attributes (dynamic shared memory opt-in); call before any capture.
cudaError_t prepare_gemm_kernels();
cudaError_t prepare_attention_kernels();
cudaError_t prepare_postchain_kernel();

// Fused post-attention chain (d_model = 128): o_proj + residual (+LN) -> LN ->
// FFN-in + GELU -> FFN-out + residual -> next LN / tail.  Operands split as
// at precision 2 (weights hi/lo; normed rows and GELU output hi/lo in TMEM).
struct ChainArgs {
  Common c;
  int F = 0;
  float eps = 1e-5f;
  int post_ln = 0;  // 1: h = LN1(h + attn), h = LN2(h + FFN)
  int last = 0;     // 1: write the model tail (final LN + pad-mask) to out32
  float scale_o = 1.f, scale_1 = 1.f, scale_2 = 1.f;  // weight pre-scales undone
  float inv_scale_2 = 1.f;                            // 1 / scale_2 (a power of two)
  // Pre-LN: the LayerNorm affines that feed FFN-in and the next layer's QKV are
  // folded into those weights (b1, bqkv are the folded biases), so
  // LN(t) W^T + b = rstd ((t - mean) W'^T) + b' with W' = W diag(gamma), b' = b + W beta.
  const float *bo = nullptr, *b1 = nullptr, *b2 = nullptr;
  const float *ln1_g = nullptr, *ln1_b = nullptr, *ln2_g = nullptr, *ln2_b = nullptr;
  const float *lnn_g = nullptr, *lnn_b = nullptr;  // next layer's LN1 (pre-LN, not last)
  const float *lnf_g = nullptr, *lnf_b = nullptr;  // final LN (last)
  const float* res = nullptr;                      // residual in: x (layer 0) or h32
  float* h32 = nullptr;                            // residual out (not last)
  __half *n16 = nullptr, *n16lo = nullptr;         // next layer's QKV input, hi/lo (not last, not fused)
  float* out32 = nullptr;                          // model output (last)
  __nv_bfloat16* outbf = nullptr;                  // bf16 model output instead of out32 (last)
  // fuse_qkv (not last): the next layer's QKV projection runs in the tail on its
  // normed rows, writing qkv16 directly (n16 is not written)
  int fuse_qkv = 0;
  float scale_qkv = 1.f;                           // next layer's W_qkv pre-scale undone
  const float* bqkv = nullptr;                     // next layer's [bq | bk | bv]
  __half* qkv16 = nullptr;                         // [M, 3 * 128]
};

struct ChainMaps {
  CUtensorMap o, wo, wo_lo, w1, w1_lo, w2, w2_lo;
  CUtensorMap wqkv, wqkv_lo;  // next layer's W_qkv (fuse_qkv)
  // fuse_qkv: stores of the residual h32 [M, D] fp32 and q, k, v [M, 3D] fp16,
  // box 64 B x 32 rows, 64-byte swizzle
  CUtensorMap h32_st, qkv_st;
};

// Whole-stack kernel (d_model 128, head_dim 32, S <= 128): every layer of the
// forward in one launch, one sequence per 128-row tile, the residual kept in
// tensor memory.  Operands split as at precision 2.
constexpr int kStackMaxLayers = 8;
struct StackLayerArgs {
  float scale_qkv = 1.f, scale_o = 1.f, scale_1 = 1.f, scale_2 = 1.f;  // weight pre-scales undone
  float inv_scale_o = 1.f, inv_scale_2 = 1.f;                          // their inverses (powers of two)
  // pre-LN: LN1's affine folded into W_qkv (bqkv folded), LN2's into W1 (b1 folded)
  const float *bqkv = nullptr, *bo = nullptr, *b1 = nullptr, *b2 = nullptr;
  const float *ln1_g = nullptr, *ln1_b = nullptr, *ln2_g = nullptr, *ln2_b = nullptr;  // post-LN
};
struct StackArgs {
  Common c;
  int B = 0, F = 0, L = 0, causal = 0, post_ln = 0;
  float eps = 1e-5f;
  float scale_log2 = 0.f;                      // log2(e) / sqrt(head_dim)
  const float* x = nullptr;                    // [B, S, 128] fp32 input, or
  const __nv_bfloat16* xbf = nullptr;          // bf16 input
  float* out32 = nullptr;                      // [B, S, 128] fp32 output, or
  __nv_bfloat16* outbf = nullptr;              // bf16 output
  const float *lnf_g = nullptr, *lnf_b = nullptr;
  StackLayerArgs layer[kStackMaxLayers];
};
struct StackMaps {
  CUtensorMap wqkv[kStackMaxLayers], wqkv_lo[kStackMaxLayers], wo[kStackMaxLayers], wo_lo[kStackMaxLayers];
  CUtensorMap w1[kStackMaxLayers], w1_lo[kStackMaxLayers], w2[kStackMaxLayers], w2_lo[kStackMaxLayers];
};
cudaError_t prepare_stack_kernel();
cudaError_t launch_stack(const StackMaps& mp, const StackArgs& a, int num_sms, cudaStream_t s);

// TMA descriptors of one GEMM: A (and its lo plane), W (and its lo part).
// Operand maps.  Split fp16 form: a / alo, b / blo are the hi / lo planes.  fp8 operand form
// (operand mode 2): a, b the fp16 hi planes (b pre-scaled by 2^11), alo / blo the e4m3 copies
// of the hi planes, a2 / b2 the e4m3 residual planes (times 2^11).
struct GemmMaps {
  CUtensorMap a, alo, b, blo, a2, b2;
};

// Launch with programmatic dependent launch allowed (the kernel waits on the
// device for the previous kernel of the stream before using its results).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launchers (return cudaError_t of the launch).
// as / ws: 1 = A / W carries an fp16 lo plane (as requires ws); 2 = both in the fp8 operand
// form (as == 2 requires ws == 2).
cudaError_t launch_gemm(int bn, int epi, int as, int ws, const GemmMaps& mp, const GemmArgs& a, int num_sms,
                        cudaStream_t s);
cudaError_t launch_attention(int hd, const CUtensorMap& tq, const CUtensorMap& tkv, const AttnArgs& a,
                             int num_sms, cudaStream_t s);
cudaError_t launch_rows(const RowArgs& a, cudaStream_t s);
cudaError_t launch_postchain(const ChainMaps& mp, const ChainArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_gelu_selftest(int n, unsigned* out, cudaStream_t s);
// Checks the lengths (TFL_DEV_BAD_LENGTHS) and writes the tile list of Common::tiles (tiles may be null).
cudaError_t launch_prepare(const int* lengths, int B, int S, int M, int* status, int* tiles, cudaStream_t s);
cudaError_t launch_f32_to_f16(const float* src, __half* dst, size_t n, cudaStream_t s);
cudaError_t launch_absmax(const float* src, size_t n, unsigned* out, cudaStream_t s);
// In place: w [rows, cols] <- w * gamma (per column), bias += w beta.
cudaError_t launch_fold_ln(float* w, int rows, int cols, const float* gamma, const float* beta, float* bias,
                           cudaStream_t s);
cudaError_t launch_split_f16(const float* src, __half* hi, __half* lo, size_t n, float scale, cudaStream_t s);
// fp8 operand form of x * scale: hi16 = fp16(x s) 2^11 (exact), hi8 = e4m3(fp16(x s)),
// lo8 = e4m3((x s - fp16(x s)) 2^11).
cudaError_t launch_split_f8(const float* src, __half* hi16, uint8_t* hi8, uint8_t* lo8, size_t n, float scale,
                            cudaStream_t s);
cudaError_t launch_probe_wait(int* status, int64_t timeout_ns, cudaStream_t s);

// Tile sizes shared by the host planner and the kernels.
constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;
constexpr int kAttnBM = 128;
__host__ __device__ constexpr int attn_block_n(int hd) { return hd >= 128 ? 64 : 128; }
size_t attn_smem_bytes(int hd);

}  // namespace tfl
