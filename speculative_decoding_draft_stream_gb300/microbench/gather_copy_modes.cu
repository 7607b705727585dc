// Throughput per SM of gathering W_head rows (rows of 4096 bf16, ids sorted
// like an I_t of 3072 ids out of 128256) into shared memory, by copy method:
//   mode 0/1  16-byte cp.async (LDGSTS) by 4 or 8 warps, each warp
//             instruction four 128-byte rows, into the 128-byte-swizzled
//             operand layout of the tcgen05 tiles (6, 8 or 12 16 KB stages);
//   mode 2    TMA tile::gather4 (four rows of 128 bytes per instruction, box
//             one row high, 128-byte swizzle) into rows 0-3 of each 1024-byte
//             swizzle atom, so every destination stays 1024-byte aligned;
//   mode 3    untiled bulk copies of 1 KB (one row's k slice);
//   mode 4    untiled bulk copies of 128 bytes (the LDGSTS layout, one row
//             chunk per copy).
// Every CTA moves 208 KB; a consumer thread releases each stage as it lands.
// The rows are L2-resident (the launch is repeated three times and the last
// is reported).  Every mbarrier wait is bounded; a timeout is counted and
// makes the program exit 1.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o gather_copy_modes gather_copy_modes.cu
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <vector>
#include <algorithm>
#include <cuda.h>
#include <cuda_runtime.h>
constexpr int V = 128256, H = 4096;
constexpr int kThreads = 384;
constexpr int kStage = 16384;
constexpr int kMaxStages = 13;
__device__ uint32_t g_err;
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtime() { unsigned long long t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }
__device__ __forceinline__ void mbar_init(uint32_t b, uint32_t c) { asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(c) : "memory"); }
__device__ __forceinline__ bool mbar_wait(uint32_t b, uint32_t par) {
  for (long long i = 0; i < (1ll << 24); ++i) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }" : "=r"(ok) : "r"(b), "r"(par) : "memory");
    if (ok) return true;
  }
  atomicOr(&g_err, 1u);
  return false;
}
__device__ __forceinline__ void mbar_arrive(uint32_t b) { asm volatile("{ .reg .b64 s; mbarrier.arrive.shared::cta.b64 s, [%0]; }" ::"r"(b) : "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t b, uint32_t bytes) { asm volatile("{ .reg .b64 s; mbarrier.arrive.expect_tx.shared::cta.b64 s, [%0], %1; }" ::"r"(b), "r"(bytes) : "memory"); }

// mode 0/1: LDGSTS by warps 4..11 (stages: 8 or 12); mode 2: gather4 into rows 0-3 of each 8-row atom;
// mode 3: 1D bulk copies of 1 KB; mode 4: 1D bulk copies of 128 B (same layout as mode 0)
template <int MODE, int GW = 8>
__global__ void __launch_bounds__(kThreads, 1) gbw(const __grid_constant__ CUtensorMap tm, const uint16_t *W, const int *rows, int nrows, int nstages, int total_stages, unsigned long long *t) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) unsigned long long bars[2 * kMaxStages];
  __shared__ int s_rows[256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_u32(sm);
  const uint32_t full = smem_u32(&bars[0]), empty = smem_u32(&bars[kMaxStages]);
  for (int i = tid; i < 256; i += kThreads) s_rows[i] = rows[(blockIdx.x * 256 + i) % nrows];
  if (tid == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(full + 8 * s, (MODE <= 1) ? GW * 32 : 1);
      mbar_init(empty + 8 * s, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const unsigned long long t0 = gtime();
  if (MODE <= 1) {
    if (warp >= 4 && warp < 4 + GW) {
      const int p = tid - 128, wl = p >> 5, c = lane & 7;
      for (int g = 0; g < total_stages; ++g) {
        const int s = g % nstages;
        if (g >= nstages && !mbar_wait(empty + 8 * s, ((g / nstages) - 1) & 1)) break;
        const uint32_t A = base + s * kStage;
        const int col = g * 64 + c * 8;  // K-chunk g
#pragma unroll
        for (int rg = 0; rg < 32 / GW; ++rg) {
          const int row = (rg * GW + wl) * 4 + (lane >> 3);
          const uint16_t *src = W + (size_t)s_rows[row] * H + col;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(A + row * 128 + ((c ^ (row & 7)) << 4)), "l"(src) : "memory");
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(full + 8 * s) : "memory");
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (tid == 0) {
    for (int g = 0; g < total_stages; ++g) {
      const int s = g % nstages;
      if (g >= nstages && !mbar_wait(empty + 8 * s, ((g / nstages) - 1) & 1)) break;
      const uint32_t A = base + s * kStage;
      if (MODE == 2) {  // 64 real rows: K-chunk g/2, rows 64*(g&1) .. +64, four per 1024-byte atom
        mbar_expect_tx(full + 8 * s, 64 * 128);
        const int kc = g >> 1, r0 = 64 * (g & 1);
        for (int a = 0; a < 16; ++a) {
          const int *r = s_rows + r0 + 4 * a;
          asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
                       ::"r"(A + 1024 * a), "l"(reinterpret_cast<uint64_t>(&tm)), "r"(kc * 64), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(full + 8 * s) : "memory");
        }
      } else if (MODE == 3) {  // 16 rows x 1 KB (K-slice of 512 at 512 * (g % 8))
        mbar_expect_tx(full + 8 * s, 16 * 1024);
        for (int q = 0; q < 16; ++q) {
          const uint16_t *src = W + (size_t)s_rows[(g * 16 + q) % 256] * H + 512 * (g % 8);
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 1024, [%2];" ::"r"(A + 1024 * q), "l"(src), "r"(full + 8 * s) : "memory");
        }
      } else {  // MODE 4: 128 rows x 128 B of K-chunk g
        mbar_expect_tx(full + 8 * s, 128 * 128);
        for (int q = 0; q < 128; ++q) {
          const uint16_t *src = W + (size_t)s_rows[q] * H + g * 64;
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 128, [%2];" ::"r"(A + 128 * q), "l"(src), "r"(full + 8 * s) : "memory");
        }
      }
    }
  }
  if (tid == 32) {  // consumer
    for (int g = 0; g < total_stages; ++g) {
      const int s = g % nstages;
      if (!mbar_wait(full + 8 * s, (g / nstages) & 1)) break;
      mbar_arrive(empty + 8 * s);
    }
    t[blockIdx.x * 2] = t0;
    t[blockIdx.x * 2 + 1] = gtime();
  }
  __syncthreads();
}

typedef CUresult (*EncFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *, const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int MODE, int GW = 8>
void run(const char *name, const CUtensorMap &tm, const uint16_t *W, const int *rows, int nrows, int nstages, int total_stages, int real_bytes_per_stage, int blocks, unsigned long long *t) {
  const int smem = nstages * kStage + 1024;
  cudaFuncSetAttribute(gbw<MODE, GW>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  std::vector<unsigned long long> h(blocks * 2);
  for (int rep = 0; rep < 3; ++rep) {
    gbw<MODE, GW><<<blocks, kThreads, smem>>>(tm, W, rows, nrows, nstages, total_stages, t);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("%s: %s\n", name, cudaGetErrorString(e)); exit(1); }
  }
  cudaMemcpy(h.data(), t, blocks * 16, cudaMemcpyDeviceToHost);
  double sum = 0, mx = 0;
  unsigned long long t0 = ~0ull, t1 = 0;
  for (int b = 0; b < blocks; ++b) {
    const double d = (h[2 * b + 1] - h[2 * b]) * 1e-3;
    sum += d; mx = std::max(mx, d);
    t0 = std::min(t0, h[2 * b]); t1 = std::max(t1, h[2 * b + 1]);
  }
  const double bytes = (double)real_bytes_per_stage * total_stages;
  printf("%-34s CTAs %3d: %6.1f KB/CTA  mean %.2f us  max %.2f us  -> %.1f GB/s per SM, aggregate %.2f TB/s\n", name, blocks, bytes / 1024,
         sum / blocks, mx, bytes / (sum / blocks) / 1e3, bytes * blocks / ((t1 - t0) * 1e-9) / 1e12);
}

int main() {
  uint16_t *W; int *rows; unsigned long long *t;
  cudaMalloc(&W, (size_t)V * H * 2);
  cudaMemset(W, 0, (size_t)V * H * 2);
  std::vector<int> r(3072);
  srand(7);
  std::vector<int> all(V);
  for (int i = 0; i < V; ++i) all[i] = i;
  for (int i = 0; i < 3072; ++i) { int j = i + rand() % (V - i); std::swap(all[i], all[j]); }
  for (int i = 0; i < 3072; ++i) r[i] = all[i];
  std::sort(r.begin(), r.end());
  cudaMalloc(&rows, 3072 * 4);
  cudaMemcpy(rows, r.data(), 3072 * 4, cudaMemcpyHostToDevice);
  cudaMalloc(&t, 152 * 16);
  void *fn = nullptr; cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  CUtensorMap tm;
  cuuint64_t dims[2] = {H, V}, strides[1] = {H * 2};
  cuuint32_t box[2] = {64, 1}, estr[2] = {1, 1};
  CUresult cr = ((EncFn)fn)(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) { printf("encode failed %d\n", (int)cr); return 1; }
  for (int blocks : {120}) {
    run<0, 4>("LDGSTS 4 warps, 6 stages", tm, W, rows, 3072, 6, 13, 16384, blocks, t);
    run<0, 4>("LDGSTS 4 warps, 8 stages", tm, W, rows, 3072, 8, 13, 16384, blocks, t);
    run<0, 8>("LDGSTS 8 warps, 6 stages", tm, W, rows, 3072, 6, 13, 16384, blocks, t);
    run<0>("LDGSTS 8 warps, 8 stages", tm, W, rows, 3072, 8, 13, 16384, blocks, t);
    run<1>("LDGSTS 8 warps, 12 stages", tm, W, rows, 3072, 12, 13, 16384, blocks, t);
    run<2>("TMA gather4 (half atoms), 13 st", tm, W, rows, 3072, 13, 26, 8192, blocks, t);
    run<3>("bulk 1 KB rows, 12 stages", tm, W, rows, 3072, 12, 13, 16384, blocks, t);
    run<4>("bulk 128 B chunks, 12 stages", tm, W, rows, 3072, 12, 13, 16384, blocks, t);
  }
  unsigned int err = 0;
  cudaMemcpyFromSymbol(&err, g_err, 4);
  printf("wait timeouts: %u\n", err);
  return err ? 1 : 0;
}
