// One-launch decode step: the whole hot path of one sequence (verify Top-K,
// draft-tree dedup, stream append and eviction, window bitmap, ascending
// compaction into I_t, gather of W_head[I_t, :] into the packed buffer,
// projection and top-k) in a single cooperative launch.
//
// Sources: MicroSpec §3.2 (stream-update and sliding-window equations; Draft
// and Verify Candidates), §3.3 (GPU-resident state, the contiguous sub-head
// buffer) and §3.1 Eq. 1 restricted to I_t.
//
// Why one launch.  The state update moves almost no bytes but is a chain of
// dependent steps (read the verify row, rank it, merge, append, update the
// bitmap, compact), and the product can only start once I_t is known.  Here
// every CTA of the product's grid takes part in the state update, so the
// chain runs on the whole GPU, and the row reads of the product start at the
// first cycle: I_t differs from I_{t-1} by the few ids that enter or leave,
// so each CTA prefetches into L2 the rows it read in the previous step while
// the state update runs.
//
// Phase A (every CTA, from the first cycle):
//   * bulk copies of the window bitmap, the ring and |S| into shared memory;
//   * its slice of the verify row: the slice's Top-K_ver, sorted, to global;
//   * C_draft from the tree ids (warp 1);
//   * L2 prefetch of the rows of its tiles in the previous I_t, and of the
//     tree ids' rows;
//   * the ids of the ring entries that may leave the window, and for each the
//     last position at which it occurs in the window (from the ring copy).
// Grid barrier: one arrival per CTA on a 64-bit counter (bounded wait).
// Phase B (every CTA computes the same thing):
//   * merge of every CTA's Top-K list into C_ver;
//   * what enters (appended) and what leaves (evicted with no later
//     occurrence and not appended again): the updated bitmap in shared memory;
//   * block scan of the bitmap into I_t positions and the ids of its own tiles;
//   * the last CTA writes the ring, |S|, the window counts and the changed
//     bitmap words; each CTA writes its share of I_t.
// Then the tcgen05 tile (ns_umma_tile.cuh) on the CTA's tiles.
//
// Reads of the old state all happen before a CTA arrives at the grid barrier,
// writes of the new state all after it, so no CTA sees a half-updated state.
#include <cuda.h>

#include "ns_umma_tile.cuh"

namespace ns {
namespace {

constexpr int kStepWarps = kUThreads / kWarp;
constexpr int kMaxAppendStep = NS_MAX_ROWS + NS_MAX_SELECT_K;
constexpr int kStepHash = 256;  // > the distinct ids one step appends or evicts (2 x 80)
constexpr int kMaxTilesPerCluster = 4;
constexpr int kFilterWords = 128;  // 4096-bit filter of the evictable ids (hashed), ahead of the table
static_assert(kMaxStepCtas <= kStepWarps * kWarp, "the Top-K merge takes one list per lane of 8 warps");
static_assert(kMaxTilesPerCluster * ((kUM + 3) / 4) <= 4 * kWarp, "the gather warps hold the prefetched row ids");
constexpr long long kBarrierNs = 1000000000LL;    // grid barrier gives up after ~1 s

struct StepArgs {
  UmmaArgs u;                 // the tiles' part (W_head, hiddens, logits, candidates, outputs, error word)
  int32_t *ring;
  uint32_t *counts;
  uint32_t *bitmap;
  int32_t *active;
  int32_t *count;
  long long *length;
  unsigned long long *gbar;   // grid barrier counter
  uint32_t *vk, *vi;          // [CTAs x K_ver] each CTA's verify Top-K (order keys, ids)
  const int32_t *tree;
  int32_t n_tree;
  const float *zrow;          // the verify row (null when K_ver = 0)
  int32_t K, nwords_pad, ring_words, tiles_per_cluster, vec;
  int32_t probe;              // launch check only: every CTA returns at once
};

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Streaming loads of the verify row, issued where they stand (volatile) so
// that they leave before the other loads of the prologue.
__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
  float4 v;
  asm volatile("ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_stream_f32(const float *p) {
  float v;
  asm volatile("ld.global.cs.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Every CTA of the (co-resident) grid arrives once; returns false on every
// thread when the wait ran out (NS_FLAG_TIMEOUT is set).  The counter only
// grows by the grid size per barrier, so generation g ends at (g + 1) * P.
__device__ bool grid_barrier(unsigned long long *ctr, unsigned long long P, uint32_t *err, int *s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    const unsigned long long old = atomicAdd(ctr, 1ull);
    const unsigned long long target = (old / P + 1) * P;
    int ok = 1;
    if (ld_acquire_u64(ctr) < target) {
      const unsigned long long t0 = globaltimer_ns();
      while (ld_acquire_u64(ctr) < target) {
        if (globaltimer_ns() - t0 > (unsigned long long)kBarrierNs) {
          atomicOr(err, NS_FLAG_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// The r-th (0-based) set bit of w, which has more than r set bits.
__device__ __forceinline__ int select_bit(uint32_t w, int r) {
  int b = 0, c = __popc(w & 0xffffu);
  if (r >= c) { r -= c; b += 16; w >>= 16; }
  c = __popc(w & 0xffu);
  if (r >= c) { r -= c; b += 8; w >>= 8; }
  c = __popc(w & 0xfu);
  if (r >= c) { r -= c; b += 4; w >>= 4; }
  c = __popc(w & 0x3u);
  if (r >= c) { r -= c; b += 2; w >>= 2; }
  if (r >= (int)(w & 1u)) b += 1;
  return b;
}

// Slot of `id` in the open-addressing table (inserted when absent); -1 when
// the table is full (cannot happen: fewer distinct ids than slots).
__device__ __forceinline__ int hash_insert(int *keys, int id) {
  unsigned slot = ((unsigned)id * 2654435761u) >> 24;
#pragma unroll 1
  for (int probe = 0; probe < kStepHash; ++probe, slot = (slot + 1) & (kStepHash - 1)) {
    const int prev = atomicCAS(&keys[slot], -1, id);
    if (prev == -1 || prev == id) return (int)slot;
  }
  return -1;
}
__device__ __forceinline__ int hash_find(const int *keys, int id) {
  unsigned slot = ((unsigned)id * 2654435761u) >> 24;
#pragma unroll 1
  for (int probe = 0; probe < kStepHash; ++probe, slot = (slot + 1) & (kStepHash - 1)) {
    const int k = keys[slot];
    if (k == id) return (int)slot;
    if (k == -1) return -1;
  }
  return -1;
}

// Word offsets of the phase A/B arrays inside the stage ring (the bulk-copy
// destinations and the bitmap's uint4 reads need 16-byte alignment).
struct StepSmem {
  int bits, ring, len, goff, vk, vi, hash, filt, wl, small, total;
};
__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }
__host__ __device__ inline StepSmem step_smem(int nwords_pad, int ring_words, int P, int K) {
  StepSmem L;
  L.bits = 0;
  L.ring = L.bits + nwords_pad;                 // nwords_pad and ring_words are multiples of 4
  L.len = L.ring + ring_words;                  // two int64
  L.goff = L.len + 4;
  L.vk = L.goff + round4(nwords_pad / 4);
  L.vi = L.vk + round4(P * K);
  L.hash = L.vi + round4(P * K);
  L.filt = L.hash + 4 * kStepHash;
  L.wl = L.filt + kFilterWords;
  L.small = L.wl + 2 * (kStepWarps + 1) * NS_MAX_SELECT_K + 2 * NS_MAX_SELECT_K;
  L.total = L.small + round4(NS_MAX_ROWS + 2 * kMaxAppendStep + 4 + kStepWarps);
  return L;
}

template <int kCL>
__global__ void __cluster_dims__(kCL, 1, 1) __launch_bounds__(kUThreads, 1)
    step_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmP, StepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) unsigned long long s_sbar;
  __shared__ int s_tiles[kMaxTilesPerCluster * kUM];  // the row ids of this CTA's tiles
  if (a.probe) return;

  const UmmaSmem S = umma_smem(smem_raw);
  const UmmaArgs &u = a.u;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_rank();
  const int P = (int)gridDim.x, cta = (int)blockIdx.x;
  const int cid = cta / kCL, ncid = P / kCL;
  const int V = u.V, W = u.W_max, K = a.K, n_tree = a.n_tree;
  const bool writer = cta == P - 1;
  // Phase A/B working set, inside the stage ring (free until the tiles run).
  const StepSmem L = step_smem(a.nwords_pad, a.ring_words, P, K);
  int32_t *wbase = reinterpret_cast<int32_t *>(S.gbase);
  uint32_t *s_bits = reinterpret_cast<uint32_t *>(wbase + L.bits);
  int32_t *s_ring = wbase + L.ring;
  long long *s_len = reinterpret_cast<long long *>(wbase + L.len);
  int32_t *s_goff = wbase + L.goff;
  int *h_key = wbase + L.hash, *h_last = h_key + kStepHash, *h_ev = h_last + kStepHash, *h_ap = h_ev + kStepHash;
  uint32_t *s_filt = reinterpret_cast<uint32_t *>(wbase + L.filt);
  uint32_t *wl_k = reinterpret_cast<uint32_t *>(wbase + L.wl), *wl_i = wl_k + (kStepWarps + 1) * NS_MAX_SELECT_K;
  uint32_t *res_k = wl_i + (kStepWarps + 1) * NS_MAX_SELECT_K, *res_i = res_k + NS_MAX_SELECT_K;
  int *s_tree = wbase + L.small, *s_app = s_tree + NS_MAX_ROWS, *s_evid = s_app + kMaxAppendStep;
  int *s_misc = s_evid + kMaxAppendStep, *sh_scan = s_misc + 4;
  uint32_t *s_vk = reinterpret_cast<uint32_t *>(wbase + L.vk);
  uint32_t *s_vi = reinterpret_cast<uint32_t *>(wbase + L.vi);
  const uint32_t sbar = smem_u32(&s_sbar);

  // ---- phase A: the loads of the old state and of the verify slice ---------
  if (tid == 0) {
    mbar_init(sbar, 1);
    umma_init_barriers(S, false);  // ends with the barrier-init fence
    mbar_expect_tx(sbar, (uint32_t)(a.nwords_pad + a.ring_words) * 4u + 16u);
    bulk_load(smem_u32(s_bits), a.bitmap, (uint32_t)a.nwords_pad * 4u, sbar);
    bulk_load(smem_u32(s_ring), a.ring, (uint32_t)a.ring_words * 4u, sbar);
    bulk_load(smem_u32(s_len), a.length, 16u, sbar);
    tma_prefetch(&tmH);
    tma_prefetch(&tmP);
  }
  // this CTA's slice of the verify row: values [lo, lo + nsl)
  int lo = 0, nsl = 0;
  if (K > 0) {
    const int per = (((V + 3) / 4 + P - 1) / P) * 4;
    lo = cta * per;
    nsl = V - lo < per ? V - lo : per;
    if (nsl < 0) nsl = 0;
  }
  // the first two passes (4 values per thread each) load at once
  float x[4], x2[4];
  auto load_pass = [&](int c0, float *v) {
    const int n = nsl - c0;
    if (a.vec) {
      float4 f = make_float4(__int_as_float(0x7fffffff), __int_as_float(0x7fffffff), __int_as_float(0x7fffffff),
                             __int_as_float(0x7fffffff));
      if (4 * tid < n) f = ld_stream_f4(a.zrow + lo + c0 + 4 * tid);
      v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = q * kUThreads + tid;
        v[q] = e < n ? ld_stream_f32(a.zrow + lo + c0 + e) : __int_as_float(0x7fffffff);
      }
    }
  };
  if (nsl > 0) load_pass(0, x);
  if (nsl > 4 * kUThreads) load_pass(4 * kUThreads, x2);
  const int tree_id = tid < n_tree ? a.tree[tid] : 0;
  // the previous I_t's rows of this CTA's share of its tiles (rows
  // [128c/C, 128(c+1)/C) of each), loaded by the gather warps, which also
  // issue the prefetches
  const int tpc = a.tiles_per_cluster;
  const int sh0 = (kUM * (int)crank) / kCL, shn = (kUM * ((int)crank + 1)) / kCL - sh0;
  const int pt = tid - 4 * kWarp;
  int pf_pos = -1, pf_id = -1, old_m = 0;
  if (pt >= 0 && pt < shn * tpc) {
    pf_pos = (cid + (pt / shn) * ncid) * kUM + sh0 + pt % shn;
    if (pf_pos < W) {
      old_m = *a.count;
      pf_id = a.active[pf_pos];
    }
  }
  for (int q = tid; q < kStepHash; q += kUThreads) {
    h_key[q] = -1;
    h_last[q] = -1;
    h_ev[q] = 0;
    h_ap[q] = 0;
  }
  for (int q = tid; q < kFilterWords; q += kUThreads) s_filt[q] = 0u;
  if (warp == 1) tmem_alloc(smem_u32(S.tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *S.tmem_slot;

  const size_t row_bytes = (size_t)u.H * 2;
  // The rows of the previous I_t of this CTA's tiles start streaming into L2
  // (they were loaded before the barrier above; the critical loads left first).
  // The gather warps issue them, so the thread that arrives at the grid
  // barrier has none outstanding.
  if (pf_pos >= 0 && pf_pos < old_m && (unsigned)pf_id < (unsigned)V)
    prefetch_l2(u.W + (size_t)pf_id * u.H, (uint32_t)row_bytes);
  if (tid < n_tree) s_tree[tid] = tree_id;

  // the old window: |S|, its ring slot, the entries that may leave
  bool have = __syncthreads_and(mbar_wait(sbar, 0, u.err));
  if (!have) mbar_wait(sbar, 0, u.err);  // a second bounded wait for the copies in flight
  if (tid == kUThreads - 1 && cta < n_tree && (unsigned)s_tree[cta] < (unsigned)V)  // tree id c by CTA c
    prefetch_l2(u.W + (size_t)s_tree[cta] * u.H, (uint32_t)row_bytes);
  const long long len0 = s_len[0];
  const int head = (int)s_len[1];
  const long long old_start = len0 > W ? len0 - W : 0;
  const int n_old = (int)(len0 - old_start);
  int max_ev = n_tree + K;
  if (max_ev > n_old) max_ev = n_old;
  if (tid < max_ev) {  // position old_start + tid
    const int slot = len0 > W ? (head + tid >= W ? head + tid - W : head + tid) : tid;
    int id = s_ring[slot];
    if ((unsigned)id >= (unsigned)V) {  // the ring only ever holds valid ids
      if (writer) set_flag(u.err, NS_FLAG_INTERNAL | (2u << 8));
      id = -1;
    }
    s_evid[tid] = id;
    if (id >= 0) {
      hash_insert(h_key, id);
      const uint32_t f = ((uint32_t)id * 2654435761u) >> 20;
      atomicOr(&s_filt[f >> 5], 1u << (f & 31));
    }
  }
  __syncthreads();

  // C_draft: distinct valid tree ids in first-occurrence node order (warp 1)
  if (warp == 1) {
    const int ta = lane < n_tree ? s_tree[lane] : 0;
    const int tb = lane + 32 < n_tree ? s_tree[lane + 32] : 0;
    const bool va = lane < n_tree && (unsigned)ta < (unsigned)V;
    const bool vb = lane + 32 < n_tree && (unsigned)tb < (unsigned)V;
    if (writer && ((lane < n_tree && !va) || (lane + 32 < n_tree && !vb))) set_flag(u.err, NS_FLAG_BAD_ID);
    const int ka = va ? ta : -1 - lane, kb = vb ? tb : -33 - lane;
    const unsigned ma = __match_any_sync(0xffffffffu, ka);
    const unsigned mb = __match_any_sync(0xffffffffu, kb);
    bool in_a = false;
#pragma unroll 4
    for (int j = 0; j < kWarp; ++j) in_a |= __shfl_sync(0xffffffffu, ka, j) == kb;
    const bool keep_a = va && __ffs(ma) - 1 == lane;
    const bool keep_b = vb && __ffs(mb) - 1 == lane && !in_a;
    const unsigned ba = __ballot_sync(0xffffffffu, keep_a), bb = __ballot_sync(0xffffffffu, keep_b);
    const unsigned lt = (1u << lane) - 1u;
    if (keep_a) s_app[__popc(ba & lt)] = ta;
    if (keep_b) s_app[__popc(ba) + __popc(bb & lt)] = tb;
    if (lane == 0) s_misc[0] = __popc(ba) + __popc(bb);
  }

  // last position (relative to old_start) of each evictable id in the
  // window: a filter bit first (one shared load for almost every entry), the
  // table only for the few entries that pass it
  for (int b0 = 0; b0 < n_old; b0 += 4 * kUThreads) {
    int ids[4];
    bool hit[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int sl = b0 + q * kUThreads + tid;
      ids[q] = sl < n_old ? s_ring[sl] : -1;
      const uint32_t f = ((uint32_t)ids[q] * 2654435761u) >> 20;
      hit[q] = ids[q] >= 0 && ((s_filt[f >> 5] >> (f & 31)) & 1u);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (hit[q]) {
        const int sl = b0 + q * kUThreads + tid;
        const int h = hash_find(h_key, ids[q]);
        if (h >= 0) atomicMax(&h_last[h], len0 > W ? (sl >= head ? sl - head : sl - head + W) : sl);
      }
    }
  }

  // the slice's Top-K: per pass, each warp's K best of its lanes' four
  // values, then warp 0 merges the warps' lists with the running result
  if (tid < K) {
    wl_k[kStepWarps * K + tid] = 0u;  // the running Top-K starts empty
    wl_i[kStepWarps * K + tid] = (uint32_t)kEmptyId;
  }
  for (int c0 = 0; c0 < nsl; c0 += 4 * kUThreads) {
    if (c0 == 4 * kUThreads) {
#pragma unroll
      for (int q = 0; q < 4; ++q) x[q] = x2[q];
    } else if (c0 > 0) {
      load_pass(c0, x);
    }
    uint32_t hk[4], hi[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      hk[q] = order_key(x[q]);  // padding is NaN: key 0, never ranks
      hi[q] = hk[q] != 0u ? (uint32_t)(a.vec ? lo + c0 + 4 * tid + q : lo + c0 + q * kUThreads + tid)
                          : (uint32_t)kEmptyId;
    }
    warp_topk4(hk, hi, K, wl_k + warp * K, wl_i + warp * K);
    __syncthreads();
    if (warp == 0) {
      uint32_t lk, li;
      warp_merge_lists(wl_k, wl_i, kStepWarps + 1, K, res_k, res_i, lk, li);
      if (lane < K) {
        wl_k[kStepWarps * K + lane] = res_k[lane];
        wl_i[kStepWarps * K + lane] = res_i[lane];
      }
    }
    __syncthreads();
  }
  if (tid < K) {
    a.vk[cta * K + tid] = wl_k[kStepWarps * K + tid];
    a.vi[cta * K + tid] = wl_i[kStepWarps * K + tid];
  }

  // ---- grid barrier: every CTA's Top-K is out, every old-state read done ---
  bool ok = have && grid_barrier(a.gbar, (unsigned long long)P, u.err, &s_misc[3]);

  // ---- phase B: C_ver, the window update, I_t ------------------------------
  int m_act = 0;
  if (ok) {
    for (int q = tid; q < P * K; q += kUThreads) {
      s_vk[q] = __ldcg(a.vk + q);
      s_vi[q] = __ldcg(a.vi + q);
    }
    __syncthreads();
    if (K > 0) {  // two rounds of list merging: 8 groups of at most 32 lists, then the 8 results
      const int per_warp = (P + kStepWarps - 1) / kStepWarps;
      const int l0 = warp * per_warp;
      const int nl = P - l0 < per_warp ? (P - l0 > 0 ? P - l0 : 0) : per_warp;
      uint32_t lk, li;
      warp_merge_lists(s_vk + l0 * K, s_vi + l0 * K, nl, K, wl_k + warp * K, wl_i + warp * K, lk, li);
      __syncthreads();
      if (warp == 0) {
        warp_merge_lists(wl_k, wl_i, kStepWarps, K, res_k, res_i, lk, li);
        const int n_draft = s_misc[0];
        const bool got = lane < K && res_k[lane] != 0u;
        const int n_ver = __popc(__ballot_sync(0xffffffffu, got));
        if (got) {
          int y = (int)res_i[lane];
          if ((unsigned)y >= (unsigned)V) {  // cannot happen for a well-formed merge
            if (writer) set_flag(u.err, NS_FLAG_INTERNAL | (1u << 8));
            y = 0;
          }
          s_app[n_draft + lane] = y;
        }
        if (lane == 0) {
          if (writer && n_ver < K) set_flag(u.err, NS_FLAG_BAD_ID);
          s_misc[1] = n_draft + n_ver;
        }
      }
    } else if (tid == 0) {
      s_misc[1] = s_misc[0];
    }
    __syncthreads();
    const int m = s_misc[1];
    if (cta == 0 && tid >= kWarp * 2 && tid < kWarp * 2 + m - s_misc[0]) {  // the entering verify ids' rows
      const int y = s_app[s_misc[0] + tid - kWarp * 2];
      prefetch_l2(u.W + (size_t)y * u.H, (uint32_t)row_bytes);
    }
    // positions: evicted [old_start, old_start + n_ev), appended [ap_begin, len1)
    const long long len1 = len0 + m;
    const long long new_start = len1 > W ? len1 - W : 0;
    const long long ev_end = len0 < new_start ? len0 : new_start;
    const int n_ev = ev_end > old_start ? (int)(ev_end - old_start) : 0;
    const long long ap_begin = len0 > new_start ? len0 : new_start;
    const int n_ap = (int)(len1 - ap_begin);
    const int ap_off = (int)(ap_begin - len0);
    if (tid < n_ap) {
      const int h = hash_insert(h_key, s_app[ap_off + tid]);
      if (h >= 0) atomicAdd(&h_ap[h], 1);
    } else if (tid >= kMaxAppendStep && tid < kMaxAppendStep + n_ev) {
      const int id = s_evid[tid - kMaxAppendStep];
      const int h = id >= 0 ? hash_find(h_key, id) : -1;
      if (h >= 0) atomicAdd(&h_ev[h], 1);
    }
    __syncthreads();
    // One thread per distinct id: an appended id is in the window; an evicted
    // one stays only if it occurs again at a position that is not evicted.
    int wchg = -1;
    if (tid < kStepHash) {
      const int id = h_key[tid];
      if (id >= 0) {
        const int ap = h_ap[tid], ev = h_ev[tid];
        const uint32_t bit = 1u << (id & 31);
        if (ap > 0) {
          if (!(s_bits[id >> 5] & bit)) {
            atomicOr(&s_bits[id >> 5], bit);
            wchg = id >> 5;
          }
        } else if (ev > 0 && h_last[tid] < n_ev) {
          atomicAnd(&s_bits[id >> 5], ~bit);
          wchg = id >> 5;
        }
        if (writer && ap != ev) atomicAdd(&a.counts[id], (unsigned)(ap - ev));
      }
    }
    if (writer) {
      if (tid < n_ap) a.ring[(head + ap_off + tid) % W] = s_app[ap_off + tid];
      if (tid == 0) {
        a.length[0] = len1;
        a.length[1] = (head + m) % W;
      }
    }
    __syncthreads();
    if (writer && wchg >= 0) a.bitmap[wchg] = s_bits[wchg];

    // compaction: per 4-word group, the number of ids before it (block scan)
    const int ng = a.nwords_pad / 4;
    const int G = (ng + kUThreads - 1) / kUThreads;
    const uint4 *b4 = reinterpret_cast<const uint4 *>(s_bits);
    int cnt = 0;
    for (int g = tid * G; g < tid * G + G && g < ng; ++g) {
      const uint4 w4 = b4[g];
      cnt += __popc(w4.x) + __popc(w4.y) + __popc(w4.z) + __popc(w4.w);
    }
    int total;
    int off = block_exclusive_scan(cnt, sh_scan, &total);
    for (int g = tid * G; g < tid * G + G && g < ng; ++g) {
      s_goff[g] = off;
      const uint4 w4 = b4[g];
      off += __popc(w4.x) + __popc(w4.y) + __popc(w4.z) + __popc(w4.w);
    }
    m_act = total < W ? total : W;
    if (writer && tid == 0) {
      if (total > W) set_flag(u.err, NS_FLAG_OVERFLOW);
      *a.count = m_act;
    }
    __syncthreads();
    // this CTA's tiles: position p -> the group holding it (the last group
    // whose offset is <= p), then the word and the bit
    for (int j = 0; j < tpc; ++j) {
      const int p = (cid + j * ncid) * kUM + tid;
      if (tid < kUM && p < m_act) {
        int lo_g = 0, hi_g = ng - 1;
        while (lo_g < hi_g) {
          const int mid = (lo_g + hi_g + 1) >> 1;
          if (s_goff[mid] <= p) lo_g = mid;
          else hi_g = mid - 1;
        }
        int r = p - s_goff[lo_g], wi = 4 * lo_g;
        uint32_t w = s_bits[wi];
        while (r >= __popc(w)) {
          r -= __popc(w);
          w = s_bits[++wi];
        }
        const int id = wi * 32 + select_bit(w, r);
        s_tiles[j * kUM + tid] = id;
        if (tid >= sh0 && tid < sh0 + shn) a.active[p] = id;  // this CTA's share of the tile
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the ring area goes back to the tiles
    __syncthreads();
  }

  // ---- the tiles --------------------------------------------------------------
  const int T = (m_act + kUM - 1) / kUM;
  const int KC = u.H / kUK;
  const int nk = KC > (int)crank ? (KC - (int)crank + kCL - 1) / kCL : 0;
  int iter = 0;
  for (int j = 0; j < tpc; ++j) {
    const int tile = cid + j * ncid;
    if (!ok || tile >= T) break;  // uniform across the cluster
    const int row0 = tile * kUM;
    if (tid < kUM) S.s_rows[tid] = s_tiles[j * kUM + (row0 + tid < m_act ? tid : m_act - 1 - row0)];
    __syncthreads();
    umma_tile<kCL, false, false, false>(S, tmem, tmH, tmP, u, iter, nk, tile, 0, m_act, T);
    ++iter;
  }

  // ---- top-k: every CTA ranks whole rows of the logits the tiles wrote ----
  // (rows cta, cta + P, ...; 8 columns per thread per pass, ties to the
  // smaller column, which is the smaller id as I_t ascends)
  if (ok) ok = grid_barrier(a.gbar, (unsigned long long)P, u.err, &s_misc[3]);
  if (ok) {
    uint32_t *rk = reinterpret_cast<uint32_t *>(S.gbase);  // [(warps + 1) x K] lists, then the result
    uint32_t *ri = rk + (kStepWarps + 1) * NS_MAX_TOPK;
    uint32_t *ok_k = ri + (kStepWarps + 1) * NS_MAX_TOPK, *ok_i = ok_k + NS_MAX_TOPK;
    const int k = u.k;
    const bool vec_l = (u.ld % 4 == 0) && (reinterpret_cast<uintptr_t>(u.logits) % 16 == 0);
    for (int r = cta; r < u.n; r += P) {
      const float *row = u.logits + (size_t)r * u.ld;
      if (tid < k) {
        rk[kStepWarps * k + tid] = 0u;
        ri[kStepWarps * k + tid] = (uint32_t)kEmptyId;
      }
      for (int c0 = 0; c0 < m_act; c0 += 8 * kUThreads) {
        uint32_t hk[8], hi[8];
        const int j0 = c0 + 8 * tid;
        if (vec_l && j0 + 8 <= m_act) {
          const float4 f0 = __ldcg(reinterpret_cast<const float4 *>(row + j0));
          const float4 f1 = __ldcg(reinterpret_cast<const float4 *>(row + j0 + 4));
          const float v[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
          for (int q = 0; q < 8; ++q) hk[q] = order_key(v[q]);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) hk[q] = j0 + q < m_act ? order_key(__ldcg(row + j0 + q)) : 0u;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) hi[q] = hk[q] != 0u ? (uint32_t)(j0 + q) : (uint32_t)kEmptyId;
        uint32_t wk, wi;
        warp_topk8_lanes(hk, hi, k, &wk, &wi);
        if (lane < k) {
          rk[warp * k + lane] = wk;
          ri[warp * k + lane] = wi;
        }
        __syncthreads();
        if (warp == 0) {
          uint32_t lk, li;
          warp_merge_lists(rk, ri, kStepWarps + 1, k, ok_k, ok_i, lk, li);
          if (lane < k) {
            rk[kStepWarps * k + lane] = ok_k[lane];
            ri[kStepWarps * k + lane] = ok_i[lane];
          }
        }
        __syncthreads();
      }
      if (tid < k) {  // column -> id through I_t
        const uint32_t key = rk[kStepWarps * k + tid];
        const int j = (int)ri[kStepWarps * k + tid];
        u.out_ids[r * k + tid] = key != 0u ? __ldcg(a.active + j) : -1;
        u.out_vals[r * k + tid] = key != 0u ? key_value(key) : -__int_as_float(0x7f800000);
      }
      __syncthreads();
    }
  }
  if (warp == 2 && lane == 0) bulk_wait_all();  // the packed-buffer stores are complete before the CTA leaves
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

constexpr int kStepSizes[] = {8, 6, 5, 4};  // cluster sizes the one-launch step can take
constexpr int kNumStepSizes = 4;
int g_step_clusters[kNumStepSizes] = {0, 0, 0, 0};  // resident clusters of each size (prepare_step_kernel)

template <int CL>
int prepare_one() {
  cudaError_t e = cudaFuncSetAttribute(step_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, kUSmem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, 1, 1);
  cfg.blockDim = dim3(kUThreads, 1, 1);
  cfg.dynamicSmemBytes = kUSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, step_kernel<CL>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    clusters = 0;
  }
  return clusters;
}

}  // namespace

cudaError_t prepare_step_kernel() {
  g_step_clusters[0] = prepare_one<8>();
  g_step_clusters[1] = prepare_one<6>();
  g_step_clusters[2] = prepare_one<5>();
  g_step_clusters[3] = prepare_one<4>();
  return cudaSuccess;
}

// The grid must be resident at once (its CTAs wait for each other), so it
// has at most the resident clusters, which then run several tiles each.
// Take the cluster size with the fewest tiles per cluster, then the largest
// (a smaller share of H per CTA).
int step_plan(const Dims &d, int *tiles_per_cluster, int *cluster_size) {
  const int tiles = (d.W_max + kUM - 1) / kUM;
  int best_ncl = 0, best_tpc = 0, best_size = 0;
  for (int i = 0; i < kNumStepSizes; ++i) {
    const int size = kStepSizes[i];
    int ncl = g_step_clusters[i] < kMaxStepCtas / size ? g_step_clusters[i] : kMaxStepCtas / size;
    if (ncl > tiles) ncl = tiles;
    if (ncl < 1) continue;
    const int tpc = (tiles + ncl - 1) / ncl;
    if (tpc > kMaxTilesPerCluster) continue;
    const StepSmem L = step_smem(d.nwords_pad, (d.W_max + 3) & ~3, ncl * size, d.K_ver);
    if ((size_t)L.total * 4 > (size_t)kRingBytes) continue;
    if (best_ncl == 0 || tpc < best_tpc) {
      best_ncl = ncl;
      best_tpc = tpc;
      best_size = size;
    }
  }
  *tiles_per_cluster = best_tpc;
  *cluster_size = best_size;
  return best_ncl;
}

cudaError_t launch_step(const StepLaunch &L, cudaStream_t st) {
  CUtensorMap tmH, tmP;
  if (!L.probe && (!encode_bf16_2d(&tmH, L.hid, L.d.H, L.n, kUK, kUN) ||
                   !encode_bf16_2d(&tmP, L.s.packed, L.d.H, L.d.W_max, kUK, kUM)))
    return cudaErrorInvalidValue;
  if (L.probe) memset(&tmH, 0, sizeof(tmH)), memset(&tmP, 0, sizeof(tmP));
  StepArgs a{};
  UmmaArgs &u = a.u;
  u.W = L.W;
  u.idx = L.s.active;
  u.count_ptr = L.s.count;
  u.V = L.d.V;
  u.H = L.d.H;
  u.n = L.n;
  u.k = L.k;
  u.W_max = L.d.W_max;
  u.logits = L.logits;
  u.ld = L.ld;
  u.cand_k = L.s.cand_k;
  u.cand_i = L.s.cand_i;
  u.slice_ticket = L.s.slice_ticket;
  u.out_ids = L.out_ids;
  u.out_vals = L.out_vals;
  u.err = L.err;
  u.nseq = 1;
  u.tiles_per_seq = (L.d.W_max + kUM - 1) / kUM;
  a.ring = L.s.ring;
  a.counts = L.s.counts;
  a.bitmap = L.s.bitmap;
  a.active = L.s.active;
  a.count = L.s.count;
  a.length = L.s.length;
  a.gbar = L.s.gbar;
  a.vk = L.s.vcand_k;
  a.vi = L.s.vcand_i;
  a.tree = L.tree;
  a.n_tree = L.n_tree;
  a.zrow = L.zrow;
  a.K = L.d.K_ver;
  a.nwords_pad = L.d.nwords_pad;
  a.ring_words = (L.d.W_max + 3) & ~3;
  a.tiles_per_cluster = L.tiles_per_cluster;
  a.vec = L.d.K_ver > 0 && (L.d.V % 4 == 0) && (reinterpret_cast<uintptr_t>(L.zrow) % 16 == 0);
  a.probe = L.probe ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(L.clusters * L.cluster_size));
  cfg.blockDim = dim3(kUThreads);
  cfg.dynamicSmemBytes = kUSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA waits for every other at the grid barrier
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (L.cluster_size) {
    case 8: return cudaLaunchKernelEx(&cfg, step_kernel<8>, tmH, tmP, a);
    case 6: return cudaLaunchKernelEx(&cfg, step_kernel<6>, tmH, tmP, a);
    case 5: return cudaLaunchKernelEx(&cfg, step_kernel<5>, tmH, tmP, a);
    case 4: return cudaLaunchKernelEx(&cfg, step_kernel<4>, tmH, tmP, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ns
