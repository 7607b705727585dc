// Instruction fetch of straight-line code: one warp per SM runs N independent
// FMAs (N x 16 bytes of code, no loop) three times per launch, three launches;
// the time of each pass shows how fast code that is executed once per launch
// is fetched, and whether it stays cached from one launch to the next.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o straight_line_fetch straight_line_fetch.cu
#include <cstdio>
#include <cuda_runtime.h>
template <int N>
__global__ void k(float *out, unsigned long long *t, int reps) {
  float a0 = threadIdx.x, a1 = a0 + 1, a2 = a0 + 2, a3 = a0 + 3, a4 = a0 + 4, a5 = a0 + 5, a6 = a0 + 6, a7 = a0 + 7;
  const float m = 1.0001f, c = 0.5f;
  for (int r = 0; r < reps; ++r) {
    unsigned long long t0, t1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
#pragma unroll
    for (int i = 0; i < N / 8; ++i) {
      asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a0) : "f"(m), "f"(c));
      asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a1) : "f"(m), "f"(c));
      asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a2) : "f"(m), "f"(c));
      asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a3) : "f"(m), "f"(c));
      asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a4) : "f"(m), "f"(c));
      asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a5) : "f"(m), "f"(c));
      asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a6) : "f"(m), "f"(c));
      asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a7) : "f"(m), "f"(c));
    }
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (threadIdx.x == 0 && r < 4) t[blockIdx.x * 4 + r] = t1 - t0;
  }
  out[blockIdx.x * blockDim.x + threadIdx.x] = a0 + a1 + a2 + a3 + a4 + a5 + a6 + a7;
}
template <int N>
void run(float *out, unsigned long long *t, unsigned long long *h, int blocks) {
  for (int launch = 0; launch < 3; ++launch) {
    k<N><<<blocks, 32>>>(out, t, 3);
    cudaDeviceSynchronize();
    cudaMemcpy(h, t, blocks * 4 * 8, cudaMemcpyDeviceToHost);
    double s[3] = {0, 0, 0};
    for (int b = 0; b < blocks; ++b)
      for (int r = 0; r < 3; ++r) s[r] += h[b * 4 + r];
    printf("N=%5d instr (%6d B code) launch %d: pass0 %.3f us  pass1 %.3f us  pass2 %.3f us  (mean over %d CTAs)\n", N,
           N * 16, launch, s[0] / blocks / 1e3, s[1] / blocks / 1e3, s[2] / blocks / 1e3, blocks);
  }
}
int main() {
  const int blocks = 152;
  float *out;
  unsigned long long *t, *h = new unsigned long long[blocks * 4];
  cudaMalloc(&out, blocks * 32 * 4);
  cudaMalloc(&t, blocks * 4 * 8);
  cudaMemset(t, 0, blocks * 4 * 8);
  run<512>(out, t, h, blocks);
  run<2048>(out, t, h, blocks);
  run<4096>(out, t, h, blocks);
  run<4096>(out, t, h, 1);
  cudaError_t e = cudaGetLastError();
  printf("status %s\n", cudaGetErrorString(e));
  return e == cudaSuccess ? 0 : 1;
}
