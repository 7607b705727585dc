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
constexpr int kProjBN = 64;      // hidden rows of a projection (NS_MAX_ROWS): rows of the logits scratch
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
  long long *active_len;  // [1] |S| when active and count were last built (another |S|: they are stale)
  long long *length;  // [2] |S|, then |S| mod W_max (the ring slot of the next entry)
  uint16_t *packed;   // [W_max x H] bf16 rows W_head[I_t[j], :]
  float *logits;      // [kProjBN x ld_scratch] fp32 logits when the caller passes none
  int32_t *first;     // [V] first flat index of an id in the prefill union (init only)
  int32_t *cand;      // [max_prompt x K_pre] prefill Top-K ids (init only)
  int32_t *sinit;     // [max_prompt x (1 + K_pre)] S_init entries (init only)
  uint32_t *cand_k;   // [umma tiles x 64 x max_k] per-tile top-k candidates (order keys)
  uint32_t *cand_i;
  int32_t *slice_ticket;  // [umma cluster] arrival counters of the row slices
  // slot-stable buffer (incremental gather of the rows of newly active ids)
  int32_t *slot_id;     // [W_max] id whose row slot s holds, -1 = free
  uint32_t *held;       // [nwords_pad] bit id <=> id holds a slot (the window bitmap at the last slot update)
  int32_t *slot_meta;   // [2] high-water mark (one past the highest occupied slot), rows the last update gathered
  int32_t *new_slot;    // [W_max] (slot, id) of each row the last update gathered, in assignment order
  int32_t *new_id;      // [W_max]
  uint16_t *slot_rows;  // [W_max x H] bf16 slot buffer
  int32_t *slot_of;     // [V] slot of each id that holds one (entries of other ids are stale)
  uint32_t *slot_free;  // [slot_words(W_max)] bit s of word s/32: slot s < W_max is free (other bits 0)
  long long *slot_len;  // [1] |S| at the last slot update (-1 after a reset: the table is empty)
  // one-launch step (ns_step.cu)
  unsigned long long *gbar;  // [1] grid barrier counter (grows by the grid size per step)
  uint32_t *vcand_k;         // [kMaxStepCtas x K_ver] each CTA's verify Top-K: order keys
  uint32_t *vcand_i;         //   and ids
};

// Words of a sequence's free-slot bitmap (a multiple of 4, for 16-byte copies).
__host__ __device__ inline int slot_words(int W_max) { return (((W_max + 31) / 32) + 3) & ~3; }

struct Dims {
  int32_t V, H, W_max, K_pre, K_ver, nwords, nwords_pad, ld_scratch;
  int32_t state_cluster;  // CTAs of the state-update cluster (16 where the device allows, else 8)
  int32_t state_max16, state_max8;  // state-update clusters of 16 and of 8 CTAs resident at once
};

// The handle lays every sequence's state out identically, one sequence after
// the other, so sequence b's buffers are sequence 0's moved by b * stride
// bytes.  Null pointers (buffers a configuration does not have) stay null.
template <typename T>
__host__ __device__ inline void move_ptr(T *&p, long long off) {
  if (p) p = reinterpret_cast<T *>(reinterpret_cast<char *>(p) + off);
}
__host__ __device__ inline SeqDev seq_at(SeqDev s, long long off) {
  move_ptr(s.ring, off), move_ptr(s.counts, off), move_ptr(s.bitmap, off), move_ptr(s.active, off);
  move_ptr(s.count, off), move_ptr(s.length, off), move_ptr(s.packed, off), move_ptr(s.logits, off);
  move_ptr(s.first, off), move_ptr(s.cand, off), move_ptr(s.sinit, off), move_ptr(s.cand_k, off);
  move_ptr(s.cand_i, off), move_ptr(s.slice_ticket, off), move_ptr(s.slot_id, off), move_ptr(s.held, off);
  move_ptr(s.slot_meta, off), move_ptr(s.new_slot, off), move_ptr(s.new_id, off), move_ptr(s.slot_rows, off);
  move_ptr(s.gbar, off), move_ptr(s.vcand_k, off), move_ptr(s.vcand_i, off), move_ptr(s.active_len, off);
  move_ptr(s.slot_of, off), move_ptr(s.slot_free, off), move_ptr(s.slot_len, off);
  return s;
}

// One batched launch covers up to kMaxBatchLaunch consecutive sequences.
constexpr int kMaxBatchLaunch = 32;

// Where sequence b (0-based within the launch) finds its step inputs: state
// at seq_at(s, b * seq_bytes), tree ids at tree + b * tree_stride, verify row
// at verify + b * z_stride + vrow[b] * V.
struct StepBatch {
  long long seq_bytes;
  long long z_stride;
  int32_t tree_stride;
  int32_t vrow[kMaxBatchLaunch];
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

// Ranking order of a float as an unsigned key: a larger key is a larger
// value, so (key descending, id ascending) is the Top-K order of `better`.
// NaN maps to 0, the key of an empty entry, and never ranks; -0.0 takes the
// key of +0.0 so that the two tie.
__device__ __forceinline__ uint32_t order_key(float x) {
  if (x != x) return 0u;
  const uint32_t u = x == 0.f ? 0u : __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The value of a nonzero key (+0.0 for a key that came from -0.0).
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The best (key, id) held by the warp's lanes: the largest key, then the
// smallest id.  An empty entry is (0, kEmptyId).
__device__ __forceinline__ void warp_best(uint32_t k, uint32_t i, uint32_t &bk, uint32_t &bi) {
  bk = __reduce_max_sync(0xffffffffu, k);
  bi = __reduce_min_sync(0xffffffffu, k == bk ? i : 0xffffffffu);
}

// One warp: the K best entries of `nl` (<= 32) lists that are sorted best
// first, K entries each (list l at lk/li[l * K]).  Lane l follows list l; each
// round the best head wins and its list advances.  Winners go to ok/oi[r]
// when ok is not null (outputs must not overlap the lists); every lane
// returns the K-th winner in lastk/lasti.
__device__ __forceinline__ void warp_merge_lists(const uint32_t *lk, const uint32_t *li, int nl, int K,
                                                 uint32_t *ok, uint32_t *oi, uint32_t &lastk, uint32_t &lasti) {
  const int lane = threadIdx.x & (kWarp - 1);
  int p = 0;
  lastk = 0u;
  lasti = (uint32_t)kEmptyId;
#pragma unroll 1  // code size: these loops run once per call
  for (int r = 0; r < K; ++r) {
    uint32_t hk = 0u, hi = (uint32_t)kEmptyId;
    if (lane < nl && p < K) {
      hk = lk[lane * K + p];
      hi = li[lane * K + p];
    }
    uint32_t bk, bi;
    warp_best(hk, hi, bk, bi);
    if (ok != nullptr && lane == 0) {
      ok[r] = bk;
      oi[r] = bi;
    }
    if (bk != 0u && hk == bk && hi == bi) ++p;
    lastk = bk;
    lasti = bi;
  }
  __syncwarp();
}

// Sorts four (key, id) pairs best first (key descending, then id ascending).
__device__ __forceinline__ void sort4_desc(uint32_t *k, uint32_t *i) {
  auto cs = [&](int x, int y) {
    if (k[y] > k[x] || (k[y] == k[x] && i[y] < i[x])) {
      const uint32_t tk = k[x], ti = i[x];
      k[x] = k[y];
      i[x] = i[y];
      k[y] = tk;
      i[y] = ti;
    }
  };
  cs(0, 1);
  cs(2, 3);
  cs(0, 2);
  cs(1, 3);
  cs(1, 2);
}

// One warp: the K best of four (key, id) pairs per lane, held in registers:
// each lane sorts its four, then K rounds of a warp-wide best-of-heads, the
// winner's lane moving to its next entry.  Lane 0 writes winner r to ok/oi[r]
// (global or shared).
__device__ __forceinline__ void warp_topk4(uint32_t *hk, uint32_t *hi, int K, uint32_t *ok, uint32_t *oi) {
  const int lane = threadIdx.x & (kWarp - 1);
  sort4_desc(hk, hi);
#pragma unroll 1  // code size: these loops run once per call
  for (int r = 0; r < K; ++r) {
    uint32_t bk, bi;
    warp_best(hk[0], hi[0], bk, bi);
    if (lane == 0) {
      ok[r] = bk;
      oi[r] = bi;
    }
    if (bk != 0u && hk[0] == bk && hi[0] == bi) {
      hk[0] = hk[1];
      hi[0] = hi[1];
      hk[1] = hk[2];
      hi[1] = hi[2];
      hk[2] = hk[3];
      hi[2] = hi[3];
      hk[3] = 0u;
      hi[3] = (uint32_t)kEmptyId;
    }
  }
  __syncwarp();
}

// warp_topk4 on two independent sets of four pairs per lane at once (their
// rounds overlap), with the winners kept in registers: lane r ends with
// winner r (r < K) of each set, so each set's K entries leave in one
// coalesced store.
__device__ __forceinline__ void warp_topk4_pair(uint32_t *ka, uint32_t *ia, uint32_t *kb, uint32_t *ib, int K,
                                                uint32_t *wak, uint32_t *wai, uint32_t *wbk, uint32_t *wbi) {
  const int lane = threadIdx.x & (kWarp - 1);
  sort4_desc(ka, ia);
  sort4_desc(kb, ib);
  *wak = 0u, *wai = (uint32_t)kEmptyId, *wbk = 0u, *wbi = (uint32_t)kEmptyId;
  auto pop = [](uint32_t *k, uint32_t *i) {
    k[0] = k[1], i[0] = i[1], k[1] = k[2], i[1] = i[2], k[2] = k[3], i[2] = i[3];
    k[3] = 0u, i[3] = (uint32_t)kEmptyId;
  };
#pragma unroll 1  // code size: these loops run once per call
  for (int r = 0; r < K; ++r) {
    uint32_t ak, ai, bk, bi;
    warp_best(ka[0], ia[0], ak, ai);
    warp_best(kb[0], ib[0], bk, bi);
    if (lane == r) {
      *wak = ak, *wai = ai, *wbk = bk, *wbi = bi;
    }
    if (ak != 0u && ka[0] == ak && ia[0] == ai) pop(ka, ia);
    if (bk != 0u && kb[0] == bk && ib[0] == bi) pop(kb, ib);
  }
}

// Sorts eight (key, id) pairs best first (key descending, then id
// ascending): Batcher's odd-even merge network, 19 compare-exchanges.
__device__ __forceinline__ void sort8_desc(uint32_t *k, uint32_t *i) {
  auto cs = [&](int x, int y) {
    if (k[y] > k[x] || (k[y] == k[x] && i[y] < i[x])) {
      const uint32_t tk = k[x], ti = i[x];
      k[x] = k[y];
      i[x] = i[y];
      k[y] = tk;
      i[y] = ti;
    }
  };
  cs(0, 1), cs(2, 3), cs(4, 5), cs(6, 7);
  cs(0, 2), cs(1, 3), cs(4, 6), cs(5, 7);
  cs(1, 2), cs(5, 6);
  cs(0, 4), cs(1, 5), cs(2, 6), cs(3, 7);
  cs(2, 4), cs(3, 5);
  cs(1, 2), cs(3, 4), cs(5, 6);
}

// One warp: the K best of eight (key, id) pairs per lane; lane r ends with
// winner r (r < K) in *wk/*wi.
__device__ __forceinline__ void warp_topk8_lanes(uint32_t *hk, uint32_t *hi, int K, uint32_t *wk, uint32_t *wi) {
  const int lane = threadIdx.x & (kWarp - 1);
  sort8_desc(hk, hi);
  *wk = 0u;
  *wi = (uint32_t)kEmptyId;
#pragma unroll 1
  for (int r = 0; r < K; ++r) {
    uint32_t bk, bi;
    warp_best(hk[0], hi[0], bk, bi);
    if (lane == r) {
      *wk = bk;
      *wi = bi;
    }
    if (bk != 0u && hk[0] == bk && hi[0] == bi) {
#pragma unroll
      for (int q = 0; q < 7; ++q) {
        hk[q] = hk[q + 1];
        hi[q] = hi[q + 1];
      }
      hk[7] = 0u;
      hi[7] = (uint32_t)kEmptyId;
    }
  }
}

// One warp: the K best of n unsorted entries at ck/ci (K rounds; each
// round's winner is struck out in place).  Winners go to ok/oi[r].
__device__ __forceinline__ void warp_select_keys(uint32_t *ck, uint32_t *ci, int n, int K, uint32_t *ok,
                                                 uint32_t *oi) {
  const int lane = threadIdx.x & (kWarp - 1);
#pragma unroll 1  // code size: these loops run once per call
  for (int r = 0; r < K; ++r) {
    uint32_t lk = 0u, li = (uint32_t)kEmptyId;
    int lq = -1;
    for (int q = lane; q < n; q += kWarp) {
      const uint32_t k = ck[q], i = ci[q];
      if (k > lk || (k == lk && k != 0u && i < li)) {
        lk = k;
        li = i;
        lq = q;
      }
    }
    uint32_t bk, bi;
    warp_best(lk, li, bk, bi);
    if (lane == 0) {
      ok[r] = bk;
      oi[r] = bi;
    }
    if (bk != 0u && lq >= 0 && lk == bk && li == bi) {
      ck[lq] = 0u;
      ci[lq] = (uint32_t)kEmptyId;
    }
    __syncwarp();
  }
}

__device__ __forceinline__ void set_flag(uint32_t *err, uint32_t f) { atomicOr(err, f); }

__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & (kWarp - 1);
#pragma unroll
  for (int off = 1; off < kWarp; off <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Exclusive prefix sum of one int per thread over the block.  `sh` needs
// blockDim/32 ints.  Returns the exclusive prefix; *total gets the block sum.
__device__ inline int block_exclusive_scan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & (kWarp - 1);
  const int warp = threadIdx.x / kWarp;
  const int nwarps = blockDim.x / kWarp;
  int incl = warp_inclusive_scan(v);
  if (lane == kWarp - 1) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = lane < nwarps ? sh[lane] : 0;
    t = warp_inclusive_scan(t);
    if (lane < nwarps) sh[lane] = t;
  }
  __syncthreads();
  const int warp_off = warp > 0 ? sh[warp - 1] : 0;
  *total = sh[nwarps - 1];
  __syncthreads();
  return warp_off + incl - v;
}

// ---------------------------------------------------------------------------
// Launch wrappers (return cudaError_t of the launch).
// ---------------------------------------------------------------------------
cudaError_t launch_init(const SeqDev &s, const Dims &d, const int32_t *prompt, int L, const float *prefill,
                        uint32_t *err, cudaStream_t st);
cudaError_t launch_append(const SeqDev &s, const Dims &d, const int32_t *tree, int n_tree,
                          const float *verify_row_ptr, bool build, uint32_t *err, cudaStream_t st);
// The state update (append + active vocabulary) of nseq <= kMaxBatchLaunch
// sequences in one launch, one cluster per sequence; s is the first one's.
cudaError_t launch_append_batch(const SeqDev &s, const Dims &d, int nseq, const int32_t *tree, int n_tree,
                                const float *verify, const StepBatch &bt, uint32_t *err, cudaStream_t st);
// Sets the state kernels' shared-memory limits and picks d->state_cluster.
cudaError_t prepare_state_kernels(Dims *d);
cudaError_t launch_build(const SeqDev &s, const Dims &d, uint32_t *err, cudaStream_t st);
// A restored checkpoint: resets the sequence (as ns_stream_init), copies the
// ring image h_ring [W_max] (host memory; the window's entries at their ring
// slots), counts the window into the counts and bitmap, sets |S| = len and
// builds I_t.
cudaError_t launch_restore(const SeqDev &s, const Dims &d, const int32_t *h_ring, long long len, uint32_t *err,
                           cudaStream_t st);
// out[w] = OR over sequences b < nseq of sequence b's bitmap word w (sequence
// b's state is b * seq_bytes past s's).
cudaError_t launch_union_bitmap(const SeqDev &s, const Dims &d, int nseq, long long seq_bytes, uint32_t *out,
                                cudaStream_t st);
cudaError_t launch_gather(const SeqDev &s, const Dims &d, const uint16_t *W, int grid, cudaStream_t st);

// Slot-stable buffer (ns_slots.cu): update the slot table to I_t, then copy
// the rows of the newly placed ids from W_head.
cudaError_t prepare_slot_kernels(const Dims &d);
cudaError_t launch_slot_update(const SeqDev &s, const Dims &d, const uint16_t *W, int copy_grid, uint32_t *err,
                               cudaStream_t st);

// Per-row top-k of a dense head's logits (ns_topk.cu): two launches, the
// slices' lists (order keys and columns) in cand_k/cand_i, n x
// topk_slices(rows) x k entries each; at most 128 slices.
constexpr int kTopkSliceCols = 4096;
__host__ __device__ inline int topk_slices(int rows) { return (rows + kTopkSliceCols - 1) / kTopkSliceCols; }
cudaError_t launch_topk(const float *logits, int ld, int rows, const int32_t *idmap, int n, int k, int32_t *ids,
                        float *vals, uint32_t *cand_k, uint32_t *cand_i, cudaStream_t st);

// Dense head on tcgen05 (ns_dense.cu): logits[r, j] = hid[r, :] . W[j, :] for
// r < n, j < rows, written to logits[r * ld + j]; W 16-byte aligned, H a
// multiple of 64.  The top-k is a separate launch_topk.
cudaError_t prepare_dense_kernel();
cudaError_t launch_dense(const uint16_t *W, int rows, const uint16_t *hid, int n, int H, float *logits, int ld,
                         uint32_t *err, cudaStream_t st);

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
  uint32_t *cand_k;          // [umma_tiles(W_max) x 64 x k]
  uint32_t *cand_i;
  int32_t *slice_ticket;     // [umma_cluster()]
  int32_t *out_ids;          // [n x k]
  float *out_vals;
  uint32_t *err;
  bool programmatic;         // may start while the preceding kernel finishes
  bool in_place;             // rows already in a contiguous buffer W (row j = id idx[j], -1 = skip), not stored
  // nseq > 1: consecutive sequences in one launch (gather mode only); hid is
  // [nseq x n x H], the per-sequence buffers above are sequence 0's and move
  // by seq_bytes per sequence, logits by logits_bytes, outputs by n * k
  int32_t nseq;
  long long seq_bytes, logits_bytes;
  bool rows_by_id;           // in_place over W_head itself: row j = W row idx[j]
  // union mode (in_place with nseq sequences): idx/count are one list shared
  // by all; mask is sequence 0's window bitmap (moved by seq_bytes); the
  // candidate lists and tickets move by cand_stride (0: seq_bytes)
  const uint32_t *mask;
  long long cand_stride;
};
int umma_tiles(int W_max);
int umma_cluster();
cudaError_t prepare_umma_kernels();
cudaError_t launch_umma_step(const UmmaLaunch &L, cudaStream_t st);

// One-launch decode step (ns_step.cu): the state update and the fused
// gather + projection + top-k of one sequence in one cooperative launch.
constexpr int kMaxStepCtas = 256;  // most CTAs of a step launch (the verify-candidate buffer's rows)
struct StepLaunch {
  SeqDev s;
  Dims d;
  const uint16_t *W;         // W_head [V x H]
  const uint16_t *hid;       // [n x H]
  int32_t n, k;
  float *logits;             // [n x ld]
  int32_t ld;
  int32_t *out_ids;          // [n x k]
  float *out_vals;
  uint32_t *err;
  const int32_t *tree;       // [n_tree]
  int32_t n_tree;
  const float *zrow;         // the verify row (null when K_ver = 0)
  int32_t clusters, tiles_per_cluster, cluster_size;  // from step_plan
  bool probe;                // launch check: every CTA returns at once
  bool slots;                // the slot-stable variant (the slot table must match the window)
};
// Sets the kernel's shared-memory limit and counts its resident clusters.
cudaError_t prepare_step_kernel();
// Clusters of a step launch for these dimensions (0: the configuration needs
// the two-launch path); *tiles_per_cluster gets the tiles each cluster runs,
// *cluster_size its CTAs.
int step_plan(const Dims &d, bool slots, int *tiles_per_cluster, int *cluster_size);
cudaError_t launch_step(const StepLaunch &L, cudaStream_t st);

}  // namespace ns
