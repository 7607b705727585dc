// Internal declarations of the dynamic-vocabulary draft LM head library.
//
// Device state of one sequence, small device helpers shared by the kernels,
// and the launch wrappers the C ABI (ns_api.cu) calls.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nanospec.h"

namespace ns {

constexpr int kWarp = 32;
constexpr int kProjBM = 64;      // W_head rows per projection tile
constexpr int kProjBN = 64;      // hidden rows per tile (NS_MAX_ROWS)
constexpr int kProjBK = 64;      // k per pipeline stage (128 bytes of a bf16 row)
constexpr int kProjStages = 4;   // cp.async pipeline depth
constexpr int kProjThreads = 128;
constexpr int kProjMaxSplit = 16;  // most K-splits of one row tile
constexpr int kStateThreads = 1024;
constexpr int kTopkThreads = 256;
constexpr int kInitTopkThreads = 256;

// Device pointers of one sequence's state.  Everything lives in one
// allocation owned by the handle.
struct SeqDev {
  int32_t *ring;      // [W_max] stream entry at position p lives at ring[p % W_max]
  uint32_t *counts;   // [V] occurrences of each id among the last W_max entries
  uint32_t *bitmap;   // [nwords_pad] bit i%32 of word i/32 <=> id i in window
  int32_t *active;    // [W_max] I_t ascending
  int32_t *count;     // [1] |I_t|
  long long *length;  // [1] |S|
  uint16_t *packed;   // [W_max x H] bf16 rows W_head[I_t[j], :]
  float *logits;      // [kProjBN x ld_scratch] fp32 logits when the caller passes none
  float *ppart;       // [proj_grid x kProjBN x kProjBM] split-K partial tiles
  int32_t *pticket;   // [proj_grid] per-tile arrival counters
  int32_t *first;     // [V] first flat index of an id in the prefill union (init only)
  int32_t *cand;      // [max_prompt x K_pre] prefill Top-K ids (init only)
  int32_t *sinit;     // [max_prompt x (1 + K_pre)] S_init entries (init only)
  float *cand_v;      // [umma tiles x 64 x max_k] per-tile top-k candidates
  int32_t *cand_i;
  int32_t *slice_ticket;  // [umma cluster] arrival counters of the row slices
};

struct Dims {
  int32_t V, H, W_max, K_pre, K_ver, nwords, nwords_pad, ld_scratch;
  int32_t state_cluster;  // CTAs of the state-update cluster (16 where the device allows, else 8)
};

// ---------------------------------------------------------------------------
// Ordering used by every Top-K: larger value first, then the smaller id.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

constexpr int kEmptyId = 0x7fffffff;

// Per-thread sorted (best first) candidate list of compile-time length KMAX.
template <int KMAX>
struct TopList {
  float v[KMAX];
  int id[KMAX];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int q = 0; q < KMAX; ++q) {
      v[q] = -__int_as_float(0x7f800000);
      id[q] = kEmptyId;
    }
  }
  __device__ __forceinline__ void insert(float x, int i) {
    if (!better(x, i, v[KMAX - 1], id[KMAX - 1])) return;
    bool placed = false;
#pragma unroll
    for (int q = KMAX - 1; q > 0; --q) {
      if (!placed) {
        if (better(x, i, v[q - 1], id[q - 1])) {
          v[q] = v[q - 1];
          id[q] = id[q - 1];
        } else {
          v[q] = x;
          id[q] = i;
          placed = true;
        }
      }
    }
    if (!placed) {
      v[0] = x;
      id[0] = i;
    }
  }
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int q = 0; q < KMAX - 1; ++q) {
      v[q] = v[q + 1];
      id[q] = id[q + 1];
    }
    v[KMAX - 1] = -__int_as_float(0x7f800000);
    id[KMAX - 1] = kEmptyId;
  }
};

// K rounds of warp-wide argmax over the lanes' list heads.  Every lane ends
// with the same winners; lane 0 stores them to out_v/out_i (K entries).
template <int KMAX>
__device__ __forceinline__ void warp_select(TopList<KMAX> &L, int K, float *out_v, int *out_i) {
  const int lane = threadIdx.x & (kWarp - 1);
  for (int q = 0; q < K; ++q) {
    float bv = L.v[0];
    int bi = L.id[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      out_v[q] = bv;
      out_i[q] = bi;
    }
    if (L.id[0] == bi && L.v[0] == bv) L.pop();
  }
}

// Block-wide Top-K of the threads' lists.  Needs shared scratch of
// (blockDim/32) * K floats and ints; the K winners end in res_v/res_i
// (shared, K entries).  Ids must be unique across threads (empty entries
// excepted).  Contains __syncthreads(); call from every thread.
template <int KMAX>
__device__ void block_select(TopList<KMAX> &L, int K, float *sc_v, int *sc_i, float *res_v, int *res_i) {
  const int warp = threadIdx.x / kWarp;
  const int nwarps = blockDim.x / kWarp;
  warp_select<KMAX>(L, K, sc_v + warp * K, sc_i + warp * K);
  __syncthreads();
  if (warp == 0) {
    TopList<KMAX> M;
    M.clear();
    const int lane = threadIdx.x & (kWarp - 1);
    for (int q = lane; q < nwarps * K; q += kWarp) M.insert(sc_v[q], sc_i[q]);
    warp_select<KMAX>(M, K, res_v, res_i);
  }
  __syncthreads();
}

// Warp-wide streaming Top-K (K <= 32).  Lane q < K holds the q-th best value
// pushed so far (larger value first, then smaller id); (tv, ti) is the K-th
// best, uniform across the warp.  Each push hands one value per lane; a value
// costs a compare and a vote unless it beats the K-th best, which is rare, and
// only then is it merged into the lane-distributed list.
struct WarpStreamTopK {
  float lv, tv;
  int li, ti, K;
  __device__ __forceinline__ void init(int k) {
    K = k;
    lv = tv = -__int_as_float(0x7f800000);
    li = ti = kEmptyId;
  }
  __device__ __forceinline__ void push(float x, int i) {
    const int lane = threadIdx.x & (kWarp - 1);
    unsigned m = __ballot_sync(0xffffffffu, better(x, i, tv, ti));
    while (m) {
      const int src = __ffs(m) - 1;
      m &= m - 1;
      const float cx = __shfl_sync(0xffffffffu, x, src);
      const int ci = __shfl_sync(0xffffffffu, i, src);
      if (!better(cx, ci, tv, ti)) continue;  // the threshold rose since the vote
      const int pos = __popc(__ballot_sync(0xffffffffu, lane < K && better(lv, li, cx, ci)));
      const float uv = __shfl_up_sync(0xffffffffu, lv, 1);
      const int ui = __shfl_up_sync(0xffffffffu, li, 1);
      if (lane < K && lane > pos) {
        lv = uv;
        li = ui;
      } else if (lane == pos) {
        lv = cx;
        li = ci;
      }
      tv = __shfl_sync(0xffffffffu, lv, K - 1);
      ti = __shfl_sync(0xffffffffu, li, K - 1);
    }
  }
};

// Sorts one (value, id) per lane across the warp, best first (bitonic network).
__device__ __forceinline__ void warp_sort_desc(float &v, int &i) {
  const int lane = threadIdx.x & (kWarp - 1);
#pragma unroll
  for (int k = 2; k <= kWarp; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, j);
      const int oi = __shfl_xor_sync(0xffffffffu, i, j);
      const bool take_better = ((lane & j) == 0) == ((lane & k) == 0);
      if (take_better ? better(ov, oi, v, i) : better(v, i, ov, oi)) {
        v = ov;
        i = oi;
      }
    }
  }
}

__device__ __forceinline__ void set_flag(uint32_t *err, uint32_t f) { atomicOr(err, f); }

// ---------------------------------------------------------------------------
// Launch wrappers (return cudaError_t of the launch).
// ---------------------------------------------------------------------------
cudaError_t launch_init(const SeqDev &s, const Dims &d, const int32_t *prompt, int L, const float *prefill,
                        uint32_t *err, cudaStream_t st);
cudaError_t launch_append(const SeqDev &s, const Dims &d, const int32_t *tree, int n_tree,
                          const float *verify_row_ptr, bool build, uint32_t *err, cudaStream_t st);
// Sets the state kernels' shared-memory limits and picks d->state_cluster.
cudaError_t prepare_state_kernels(Dims *d);
cudaError_t launch_build(const SeqDev &s, const Dims &d, uint32_t *err, cudaStream_t st);
cudaError_t launch_gather(const SeqDev &s, const Dims &d, const uint16_t *W, int grid, cudaStream_t st);

// Projection source modes.
enum ProjMode { kFromPacked = 0, kGatherRows = 1, kDenseRows = 2 };

struct ProjArgs {
  const uint16_t *rows;      // packed buffer (kFromPacked) or W_head
  const int32_t *idx;        // I_t (kGatherRows)
  const int32_t *count_ptr;  // device row count (kFromPacked / kGatherRows)
  int32_t rows_host;         // row count (kDenseRows)
  uint16_t *packed_out;      // packed buffer to fill (kGatherRows)
  const uint16_t *hid;       // [n x H]
  int32_t n, H;
  float *logits;             // [n x ld]
  int32_t ld;
  float *part;               // split-K partial tiles
  int32_t *tickets;          // per-tile arrival counters
};

cudaError_t launch_project(ProjMode mode, const ProjArgs &a, int grid, cudaStream_t st);
cudaError_t launch_topk(const float *logits, int ld, const int32_t *count_ptr, int rows_host,
                        const int32_t *idmap, int n, int k, int32_t *ids, float *vals, cudaStream_t st);

size_t project_smem_bytes();
cudaError_t prepare_project_kernels();

// Fused gather + projection + top-k on tcgen05 tensor cores (ns_umma.cu).
struct UmmaLaunch {
  const uint16_t *W;         // W_head [V x H]
  int32_t V, H;
  const uint16_t *hid;       // [n x H]
  int32_t n;
  uint16_t *packed;          // [W_max x H]
  int32_t W_max;
  const int32_t *idx;        // I_t
  const int32_t *count_ptr;  // |I_t|
  int32_t k;
  float *logits;             // [n x ld]
  int32_t ld;
  float *cand_v;             // [umma_tiles(W_max) x 64 x k]
  int32_t *cand_i;
  int32_t *slice_ticket;     // [umma_cluster()]
  int32_t *out_ids;          // [n x k]
  float *out_vals;
  uint32_t *err;
  bool programmatic;         // may start while the preceding kernel finishes
};
int umma_tiles(int W_max);
int umma_cluster();
cudaError_t prepare_umma_kernels();
cudaError_t launch_umma_step(const UmmaLaunch &L, cudaStream_t st);

}  // namespace ns
