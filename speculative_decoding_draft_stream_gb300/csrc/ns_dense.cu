// Dense LM head on the 5th-generation tensor cores: logits = hidden ·
// W_head[0:rows, :]ᵀ for every row (the full vocabulary, or a static
// sub-head made of its first rows), MicroSpec §3.1 Eq. 1 without the
// restriction to I_t.  It is the comparator of the sub-head step.
//
// The rows are contiguous, so each 128-row tile is loaded with tiled TMA
// loads (128 rows x 64 k per stage, 128-byte swizzle) and there is no gather.
// One persistent CTA per SM takes tiles blockIdx.x, blockIdx.x + grid, ...
// over the whole H (no split, no cluster), with three roles:
//   * warp 0 (one lane): TMA loads of the W_head slice and the hidden slice
//     of each stage into an 8-stage ring;
//   * warp 1 (one lane): tcgen05.mma (M = 128, N = 64, K = 16, bf16 -> fp32)
//     into one of two tensor-memory accumulators, so a tile's epilogue runs
//     while the next tile accumulates;
//   * warps 4-7: the epilogue, tcgen05.ld of the accumulator (thread j holds
//     W_head row row0 + j, i.e. logits column row0 + j, for the 64 hidden
//     rows) and coalesced logits stores.
// Every wait is bounded (NS_FLAG_TIMEOUT).
#include <cuda.h>

#include "ns_umma_tile.cuh"

namespace ns {
namespace {

constexpr int kDStages = 8;
constexpr int kDThreads = 256;
constexpr int kDRing = kDStages * kStage;
constexpr uint32_t kDTmemCols = 2 * kUN;  // two accumulators of 64 fp32 columns
constexpr int kDSmem = kDRing + 256 + 1024;  // ring, barriers and slot, alignment slack

__global__ void __launch_bounds__(kDThreads, 1)
    dense_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH, float *logits,
                 int ld, int rows, int n, int H, uint32_t *err) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte-swizzled stages need 1024-byte alignment
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t bar_full = base + kDRing, bar_empty = bar_full + 8 * kDStages;
  const uint32_t bar_accf = bar_empty + 8 * kDStages, bar_acce = bar_accf + 16;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kDRing + 8 * (2 * kDStages + 4));

  if (tid == 0) {
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);   // the TMA issuer's arrival with the bytes
      mbar_init(bar_empty + 8 * s, 1);  // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_accf + 8 * b, 1);  // the last MMA commit of a tile
      mbar_init(bar_acce + 8 * b, 4);  // the four epilogue warps
    }
    mbar_fence_init();
    tma_prefetch(&tmW);
    tma_prefetch(&tmH);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kDTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int T = (rows + kUM - 1) / kUM, KC = H / kUK;
  if (warp == 0 && lane == 0) {  // producer
    int g = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
      for (int kt = 0; kt < KC; ++kt, ++g) {
        const int s = g % kDStages;
        if (g >= kDStages && !(ok = mbar_wait(bar_empty + 8 * s, ((g / kDStages) - 1) & 1, err))) break;
        const uint32_t A = base + s * kStage;
        mbar_expect_tx(bar_full + 8 * s, kStage);
        tma_load_2d(A, &tmW, kt * kUK, t * kUM, bar_full + 8 * s);
        tma_load_2d(A + kStageA, &tmH, kt * kUK, 0, bar_full + 8 * s);
      }
    }
    // nothing may still be landing in shared memory when the CTA leaves
    const int first = g > kDStages ? g - kDStages : 0;
    for (int q = first; q < g; ++q) mbar_wait(bar_full + 8 * (q % kDStages), (q / kDStages) & 1, err);
  } else if (warp == 1 && lane == 0) {  // MMA issuer
    int g = 0, i = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < T && ok; t += gridDim.x, ++i) {
      const int b = i & 1;
      if (i >= 2 && !(ok = mbar_wait(bar_acce + 8 * b, ((i >> 1) - 1) & 1, err))) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(b * kUN);
      for (int kt = 0; kt < KC; ++kt, ++g) {
        const int s = g % kDStages;
        if (!(ok = mbar_wait(bar_full + 8 * s, (g / kDStages) & 1, err))) break;
        tc_fence_after();
        const uint32_t A = base + s * kStage;
#pragma unroll
        for (int kk = 0; kk < kUK / 16; ++kk)
          umma_bf16(acc, sw128_desc(A + kk * 32), sw128_desc(A + kStageA + kk * 32), (kt | kk) != 0);
        umma_commit(bar_empty + 8 * s);
      }
      if (ok) umma_commit(bar_accf + 8 * b);
    }
  } else if (warp >= 4) {  // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
    const int wq = warp - 4;
    int i = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, ++i) {
      const int b = i & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bar_accf + 8 * b, (i >> 1) & 1, err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      mbar_try_wait(bar_accf + 8 * b, (i >> 1) & 1);  // every lane takes the completed phase
      tc_fence_after();
      const int col = t * kUM + wq * 32 + lane;
      const uint32_t taddr = tmem + (uint32_t)(b * kUN) + ((uint32_t)(wq * 32) << 16);
#pragma unroll
      for (int c = 0; c < kUN; c += 16) {
        float v[16];
        tmem_ld16(taddr + c, v);
        tmem_ld_wait();
        if (col < rows) {
#pragma unroll
          for (int q = 0; q < 16; ++q)
            if (c + q < n) logits[(size_t)(c + q) * ld + col] = v[q];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acce + 8 * b);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kDTmemCols);
}

int g_dense_sms = 0;

}  // namespace

cudaError_t prepare_dense_kernel() {
  cudaError_t e = cudaFuncSetAttribute(dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmem);
  if (e != cudaSuccess) return e;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(&g_dense_sms, cudaDevAttrMultiProcessorCount, dev);
}

cudaError_t launch_dense(const uint16_t *W, int rows, const uint16_t *hid, int n, int H, float *logits, int ld,
                         uint32_t *err, cudaStream_t st) {
  CUtensorMap tmW, tmH;
  if (!encode_bf16_2d(&tmW, W, H, rows, kUK, kUM) || !encode_bf16_2d(&tmH, hid, H, n, kUK, kUN))
    return cudaErrorInvalidValue;
  const int T = (rows + kUM - 1) / kUM;
  const int grid = T < g_dense_sms ? T : g_dense_sms;
  dense_kernel<<<grid > 0 ? grid : 1, kDThreads, kDSmem, st>>>(tmW, tmH, logits, ld, rows, n, H, err);
  return cudaGetLastError();
}

}  // namespace ns
