// Per-SM throughput of the instructions the softmax of the FLARE++ kernels is
// made of: exp2 on the special-function unit (fp32, bf16x2, f16x2), fp32 FMA,
// packed f32x2 FMA, 3-input fp32 max, the fp32 -> bf16x2 rounding pack and
// the byte permute, and exp2 issued together with each of the last two (to
// see whether they share a pipe). One CTA per SM, 16 independent
// dependency chains per thread, clock64 around the loop. Prints lane-
// operations per clock per SM; these set the exp2 roofline the benchmark
// reports against.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

template <int KIND>
__global__ void rate_kernel(float* out, int iters, long long* cycles) {
  float a[16], c[16];
  uint32_t b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = -0.001f * (threadIdx.x + i);
    c[i] = -0.002f * (threadIdx.x + i);
    b[i] = 0x3c003c00u + i;
  }
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (KIND == 0) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(a[i]));
      if (KIND == 1) asm volatile("ex2.approx.ftz.bf16x2 %0, %0;" : "+r"(b[i]));
      if (KIND == 2) asm volatile("ex2.approx.f16x2 %0, %0;" : "+r"(b[i]));
      if (KIND == 3) asm volatile("fma.rn.f32 %0, %0, %0, %0;" : "+f"(a[i]));
      if (KIND == 4) {
        uint64_t v = (static_cast<uint64_t>(__float_as_uint(a[i])) << 32) | __float_as_uint(a[i]);
        asm volatile("fma.rn.f32x2 %0, %0, %0, %0;" : "+l"(v));
        a[i] = __uint_as_float(static_cast<uint32_t>(v));
      }
      if (KIND == 5) asm volatile("max.f32 %0, %0, %1, %0;" : "+f"(a[i]) : "f"(a[(i + 1) & 15]));
      if (KIND == 6 || KIND == 8)
        asm volatile("{\n\t.reg .b32 t;\n\tcvt.rn.bf16x2.f32 t, %0, %0;\n\tmov.b32 %0, t;\n\t}" : "+f"(a[i]));
      if (KIND == 7 || KIND == 9) asm volatile("prmt.b32 %0, %0, %1, 0x7632;" : "+r"(b[i]) : "r"(b[(i + 1) & 15]));
      if (KIND == 8) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(c[i]));
      if (KIND == 9) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(a[i]));
    }
  }
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) s += a[i] + c[i] + __uint_as_float(b[i]);
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int KIND>
void run(const char* name, int sms, float* out, long long* cyc) {
  const int iters = 4096, threads = 512;
  rate_kernel<KIND><<<sms, threads>>>(out, iters, cyc);  // warm-up
  cudaDeviceSynchronize();
  rate_kernel<KIND><<<sms, threads>>>(out, iters, cyc);
  cudaDeviceSynchronize();
  long long c = 0;
  cudaMemcpy(&c, cyc, sizeof(c), cudaMemcpyDeviceToHost);
  const double lane_instr = static_cast<double>(iters) * 16 * threads;
  // the mixed kinds issue two instructions per chain step: pairs per clock
  printf("%-12s %7.2f instructions x lanes per clock per SM%s\n", name, lane_instr / c,
         KIND >= 8 ? " (pairs)" : "");
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  float* out = nullptr;
  long long* cyc = nullptr;
  cudaMalloc(&out, sms * 512 * sizeof(float));
  cudaMalloc(&cyc, sms * sizeof(long long));
  run<0>("ex2.f32", sms, out, cyc);
  run<1>("ex2.bf16x2", sms, out, cyc);
  run<2>("ex2.f16x2", sms, out, cyc);
  run<3>("fma.f32", sms, out, cyc);
  run<4>("fma.f32x2", sms, out, cyc);
  run<5>("max3.f32", sms, out, cyc);
  run<6>("cvt.bf16x2", sms, out, cyc);
  run<7>("prmt", sms, out, cyc);
  run<8>("ex2+cvt", sms, out, cyc);
  run<9>("ex2+prmt", sms, out, cyc);
  const cudaError_t e = cudaGetLastError();
  printf("SMs %d, status %s\n", sms, cudaGetErrorString(e));
  cudaFree(out);
  cudaFree(cyc);
  return e == cudaSuccess ? 0 : 1;
}
