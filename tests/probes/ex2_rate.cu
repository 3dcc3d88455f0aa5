// ex2_rate.cu -- measures the per-SM throughput of ex2.approx.ftz.f32 (the
// exponential of the attention softmax) and, for comparison, of
// ex2.approx.f16x2 and of fp32 FMA, in operations per clock per SM.
// The attention kernel's roofline peak is this ex2 rate x SMs x SM clock.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o ex2_rate ex2_rate.cu && ./ex2_rate
// (tests/test_gpu_ex2_rate.py builds and runs it)
//
// Each thread runs 8 independent dependency chains; one CTA per SM; the
// clock64 interval around the loop gives the rate.
#include <cstdio>

template <int K>
__global__ void rate_kernel(float* out, long long* cycles, int iters) {
  float v[8];
  for (int i = 0; i < 8; ++i) v[i] = -0.001f * (threadIdx.x + i);
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (K == 0) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(v[i]));
      if (K == 1) asm volatile("{.reg .b32 h; mov.b32 h, %0; ex2.approx.f16x2 h, h; mov.b32 %0, h;}" : "+f"(v[i]));
      if (K == 2) asm volatile("fma.rn.f32 %0, %0, 0f3F7FFFFF, 0f3A83126F;" : "+f"(v[i]));
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
  for (int i = 0; i < 8; ++i) s += v[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  float* out;
  long long* cyc;
  if (cudaMalloc(&out, (size_t)sms * 1024 * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&cyc, (size_t)sms * sizeof(long long)) != cudaSuccess) {
    printf("allocation failed\n");
    return 1;
  }
  const char* names[] = {"ex2.approx.f32 (results)", "ex2.approx.f16x2 (instr)", "fma.rn.f32"};
  for (int k = 0; k < 3; ++k) {
    for (int warps : {8, 32}) {
      const int iters = 2000;
      auto f = k == 0 ? rate_kernel<0> : k == 1 ? rate_kernel<1> : rate_kernel<2>;
      f<<<sms, warps * 32>>>(out, cyc, 10);
      f<<<sms, warps * 32>>>(out, cyc, iters);
      const cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) {
        printf("error: %s\n", cudaGetErrorString(e));
        return 1;
      }
      long long c[1024];
      cudaMemcpy(c, cyc, (size_t)sms * sizeof(long long), cudaMemcpyDeviceToHost);
      double avg = 0;
      for (int i = 0; i < sms; ++i) avg += (double)c[i];
      avg /= sms;
      printf("%-26s %2d warps/SM: %6.2f per clock per SM\n", names[k], warps, (double)warps * 32 * iters * 8 / avg);
    }
  }
  return 0;
}
