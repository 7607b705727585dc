// Per-row top-k of a dense head's logits (the draft head's top-k of
// MicroSpec §3.3, here over every row of a full-vocabulary or static head):
// the k largest logits of each hidden row, ties to the smaller column, NaN
// never ranked, ids = column numbers (or idmap[column]).  Values are ranked
// by their order keys (a larger key is a larger value; NaN has the key of an
// empty entry).  Two launches:
//   * slice_topk_kernel: CTA (s, r) ranks columns [s * kTopkSliceCols, ...)
//     of row r in two passes of eight consecutive columns per thread (all
//     sixteen loads in flight at once): each lane sorts its eight keys, each
//     warp takes its k best in k rounds of a warp-wide best-of-heads, and
//     warp 0 merges the sixteen warp lists into the slice's k best;
//   * merge_topk_kernel: CTA r merges the slices' lists of row r (up to 32
//     lists per warp, then warp 0 merges the warps' results).
#include "ns_internal.cuh"

namespace ns {
namespace {

constexpr int kSliceThreads = kTopkSliceCols / 16;  // sixteen columns per thread
constexpr int kSliceWarps = kSliceThreads / kWarp;
constexpr int kMergeWarps = 4;                        // up to 128 slices per row
static_assert(kSliceWarps * 2 <= kWarp, "warp 0 merges every warp's two lists");

__global__ void __launch_bounds__(kSliceThreads) slice_topk_kernel(const float *logits, int ld, int m, int k, int S,
                                                                   bool vec, uint32_t *ck, uint32_t *ci) {
  __shared__ uint32_t wl_k[2 * kSliceWarps * NS_MAX_TOPK], wl_i[2 * kSliceWarps * NS_MAX_TOPK];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, r = blockIdx.y;
  const int c0 = s * kTopkSliceCols;
  const float *row = logits + (size_t)r * ld;
  float v[2][8];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int j0 = c0 + p * (kTopkSliceCols / 2) + 8 * tid;
    if (vec && j0 + 8 <= m) {
      const float4 a = __ldcs(reinterpret_cast<const float4 *>(row + j0));
      const float4 b = __ldcs(reinterpret_cast<const float4 *>(row + j0 + 4));
      v[p][0] = a.x, v[p][1] = a.y, v[p][2] = a.z, v[p][3] = a.w;
      v[p][4] = b.x, v[p][5] = b.y, v[p][6] = b.z, v[p][7] = b.w;
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) v[p][q] = j0 + q < m ? __ldcs(row + j0 + q) : __int_as_float(0x7fffffff);
    }
  }
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int j0 = c0 + p * (kTopkSliceCols / 2) + 8 * tid;
    uint32_t hk[8], hi[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      hk[q] = order_key(v[p][q]);  // padding is NaN: key 0, never ranks
      hi[q] = hk[q] != 0u ? (uint32_t)(j0 + q) : (uint32_t)kEmptyId;
    }
    uint32_t wk, wi;
    warp_topk8_lanes(hk, hi, k, &wk, &wi);
    if (lane < k) {
      wl_k[(p * kSliceWarps + warp) * k + lane] = wk;
      wl_i[(p * kSliceWarps + warp) * k + lane] = wi;
    }
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t lk, li;
    const size_t o = ((size_t)r * S + s) * k;
    warp_merge_lists(wl_k, wl_i, 2 * kSliceWarps, k, ck + o, ci + o, lk, li);
  }
}

__global__ void __launch_bounds__(kMergeWarps * kWarp) merge_topk_kernel(const uint32_t *ck, const uint32_t *ci, int S,
                                                                         int k, const int32_t *idmap, int32_t *ids,
                                                                         float *vals) {
  __shared__ uint32_t wl_k[kMergeWarps * NS_MAX_TOPK], wl_i[kMergeWarps * NS_MAX_TOPK];
  __shared__ uint32_t rk[NS_MAX_TOPK], ri[NS_MAX_TOPK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x;
  const int nw = (S + kWarp - 1) / kWarp;
  if (warp < nw) {
    const int l0 = warp * kWarp, nl = S - l0 < kWarp ? S - l0 : kWarp;
    const size_t o = ((size_t)r * S + l0) * k;
    uint32_t lk, li;
    warp_merge_lists(ck + o, ci + o, nl, k, wl_k + warp * k, wl_i + warp * k, lk, li);
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t lk, li;
    warp_merge_lists(wl_k, wl_i, nw, k, rk, ri, lk, li);
    if (lane < k) {
      const uint32_t key = rk[lane];
      const int j = (int)ri[lane];
      ids[(size_t)r * k + lane] = key != 0u ? (idmap ? idmap[j] : j) : -1;
      vals[(size_t)r * k + lane] = key != 0u ? key_value(key) : -__int_as_float(0x7f800000);
    }
  }
}

}  // namespace

cudaError_t launch_topk(const float *logits, int ld, int rows, const int32_t *idmap, int n, int k, int32_t *ids,
                        float *vals, uint32_t *cand_k, uint32_t *cand_i, cudaStream_t st) {
  const int S = topk_slices(rows);
  if (S > kMergeWarps * kWarp) return cudaErrorInvalidValue;
  const bool vec = (ld % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
  slice_topk_kernel<<<dim3((unsigned)S, (unsigned)n), kSliceThreads, 0, st>>>(logits, ld, rows, k, S, vec, cand_k,
                                                                              cand_i);
  merge_topk_kernel<<<n, kMergeWarps * kWarp, 0, st>>>(cand_k, cand_i, S, k, idmap, ids, vals);
  return cudaGetLastError();
}

}  // namespace ns
