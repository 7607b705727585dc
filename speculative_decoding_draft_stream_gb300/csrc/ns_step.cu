// One-launch decode step: the whole hot path of one sequence (verify Top-K,
// draft-tree dedup, stream append and eviction, window bitmap, ascending
// compaction into I_t, gather of W_head[I_t, :] into the packed buffer,
// projection and top-k) in a single cooperative launch.
//
// Sources: MicroSpec §3.2 (stream-update and sliding-window equations; Draft
// and Verify Candidates), §3.3 (GPU-resident state, the contiguous sub-head
// buffer) and §3.1 Eq. 1 restricted to I_t.
//
// Why the projection does not wait for I_t.  The state update moves almost
// no bytes but is a chain of dependent steps (read the verify row, rank it,
// merge across the grid, append, evict, compact), while the product moves
// the bytes.  Each logit is one dot product, so where a column sits in I_t
// does not change its value, and I_t differs from I_{t-1} only by the ids
// that enter (this step's draft and verify candidates) and leave.  So the
// product starts at the first cycle on what is already known:
//   * one work item per 128 ids of I_{t-1} (read before anything changes);
//   * one item for the draft-tree ids (inputs of the step);
//   * the few verify Top-K ids (K_ver of them) by CUDA-core dot products,
//     once the grid has ranked the verify row.
// When the state update has produced I_t, every column is written at the
// position of its id in I_t: an id of I_{t-1} that stays by its old item,
// an id that enters by the draft item or the verify products (the first
// candidate that holds it), an id that leaves by nobody, so each column of
// I_t is written exactly once.  The packed buffer (W_head[I_t, :] in I_t
// order) is filled by bulk row copies that run beside the top-k.
//
// A CTA runs three groups of warps side by side:
//   * tile group, warps 0-1 and 4-11: its cluster's items (tcgen05 tiles
//     split over H across the cluster: TMA hidden loads, cp.async row
//     gathers into the 128-byte-swizzled layout, MMA into tensor memory,
//     split-K partials summed through distributed shared memory in rank
//     order), then the logits writes;
//   * verify group, warps 2-3: the verify ids' logits;
//   * state group, warps 12-15: the state update, computed identically by
//     every CTA (its slice of the verify row, a grid barrier, the merge of
//     all slices into C_ver, the window update and the compaction), then its
//     share of I_t and of the packed buffer.
// The groups meet through mbarriers (old-state reads done; C_ver known; I_t
// known; the stage ring free), so none waits at another's block barriers.  Warps 0-11 then take the second grid
// barrier together and rank whole rows.
//
// Reads of the old state (I_{t-1}, |I_{t-1}|, the bitmap, the ring, |S|)
// all happen before a CTA arrives at the first grid barrier, writes of the
// new state all after it.  Every wait is bounded (about a second); a wait
// that runs out sets NS_FLAG_TIMEOUT and the kernel still follows the same
// barrier sequence.
//
// The slot-stable variant (kSlots) is the same step on the slot buffer of
// NanoSpec's incremental gather (only the rows of newly active ids are
// copied; an id keeps its row slot while it stays active).  It needs the
// slot table to match the window at launch (the host takes the multi-launch
// path otherwise).  Then a column's slot is known before the state update:
//   * the old items are the tiles of slots [0, high-water mark), their rows
//     read from the slot buffer itself; a slot whose id stays is written in
//     place, a slot left free gets NaN (never ranked);
//   * the state group frees the slots of the ids that leave and gives the
//     entering ids the lowest free slots in ascending id order, so the draft
//     item and the verify products write them at their new slots;
//   * the row top-k maps a column to its id through the slot table, and the
//     rows of the entering ids are copied into their slots once every CTA is
//     past the second grid barrier (no tile reads a slot row any more).
// No compaction is on the logits' path and there is no packed copy.
#include <cuda.h>

#include "ns_umma_tile.cuh"

namespace ns {
namespace {

constexpr int kSThreads = 512;                        // the whole CTA
constexpr int kKThreads = 384;                        // warps 0-11: the second grid barrier and the row top-k
constexpr int kTGroup = 320;                          // tile group: warps 0-1 and 4-11
constexpr int kVGroup = 64;                           // verify group: warps 2-3
constexpr int kSgThreads = kSThreads - kKThreads;     // state group: warps 12-15
constexpr int kSgWarps = kSgThreads / kWarp;
constexpr int kKWarps = kKThreads / kWarp;
constexpr int kBarT = 1, kBarS = 2, kBarK = 3;        // named barriers of the groups
constexpr int kVerPairs = 16;                         // most (verify id, hidden row) products of one CTA
constexpr int kCopyOff = 8192;                        // packed-copy staging in the ring, past the top-k lists
constexpr int kMinStepCtas = 120;                     // grid the state update wants (slices of the verify row)
constexpr int kSStages = 6;                           // stage ring of the tiles
constexpr int kSRing = kSStages * kStage;
constexpr int kMaxItemsPerCluster = 2;
constexpr int kFRows = (kUN + 3) / 4;                 // most hidden rows one CTA sums (clusters of >= 4)
constexpr int kFBytes = kFRows * kUM * 4;
constexpr int kStepMiscBytes = 1536;                  // barriers, TMEM slot, flags, the items' row ids
constexpr int kMaxAppendStep = NS_MAX_ROWS + NS_MAX_SELECT_K;
constexpr int kVerRow0 = NS_MAX_ROWS;                 // writer-row code of verify id v: kVerRow0 + v
constexpr int kStepHash = 256;                        // > the distinct ids one step appends or evicts (2 x 80)
constexpr int kHashArrays = 7;                        // key, count, ev, ap, writer row, enters, changed word
constexpr int kMaxSmem = 232448;                      // dynamic shared memory one CTA can take
constexpr long long kBarrierNs = 1000000000LL;        // grid barrier gives up after ~1 s
static_assert(kMaxStepCtas <= kSgWarps * 2 * kWarp, "the C_ver merge takes two lists per lane of the state warps");
static_assert(kPartBytes <= kSRing, "partial tile fits in the stage ring");
static_assert((kKWarps + 1) * 2 * NS_MAX_TOPK * 4 + 2 * NS_MAX_TOPK * 4 <= kCopyOff, "top-k lists before the staging");
static_assert(kMaxItemsPerCluster * kUM * 4 + 512 <= kStepMiscBytes, "row ids fit the misc area");
static_assert(kUM == 128 && kTGroup >= 2 * kUM, "logits writes: one column per thread, two row groups");

struct StepArgs {
  UmmaArgs u;                 // W_head, hiddens, logits, outputs, error word
  int32_t *ring;
  uint32_t *counts;
  uint32_t *bitmap;
  int32_t *active;
  int32_t *count;
  long long *length;
  long long *active_len;      // |S| when active/count were built
  uint16_t *packed;
  const uint16_t *hid;        // hidden rows [n x H] (the verify products read them directly)
  unsigned long long *gbar;   // grid barrier counter
  uint32_t *vk, *vi;          // [CTAs x K_ver] each CTA's verify Top-K (order keys, ids)
  const int32_t *tree;
  int32_t n_tree;
  const float *zrow;          // the verify row (null when K_ver = 0)
  int32_t K, nwords_pad, ring_words, items_per_cluster, t_max, vec;
  int32_t probe;              // launch check only: every CTA returns at once
  // slot-stable variant only
  int32_t *slot_id;           // [W_max] id a slot holds, -1 = free
  int32_t *slot_of;           // [V] slot of each id that holds one
  uint32_t *slot_free;        // [fs_words] bit s of word s/32: slot s < W_max is free
  uint32_t *held;             // [nwords_pad] ids holding a slot (the window bitmap at the last slot update)
  int32_t *slot_meta;         // [2] high-water mark, rows the last update copied
  int32_t *new_slot, *new_id;  // [W_max] (slot, id) of those rows, in assignment order
  uint16_t *slot_rows;        // [W_max x H]
  long long *slot_len;        // [1] |S| at the last slot update
  int32_t fs_words;           // words of slot_free (a multiple of 4)
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
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// Arrival on a barrier of a CTA of this cluster (its shared::cluster address),
// releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a phase completed by arrivals from the cluster's CTAs.
static __device__ __noinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint32_t *err) {
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(err, NS_FLAG_TIMEOUT);
      return false;
    }
  }
  return true;
}

// One arrival per CTA (by `leader`, after a barrier of its group) on a 64-bit
// counter that only grows by the grid size per barrier, so generation g ends
// at (g + 1) * P.  Returns false on every thread of the group when the wait
// ran out (NS_FLAG_TIMEOUT is set).
__device__ bool grid_barrier(unsigned long long *ctr, unsigned long long P, uint32_t *err, int *s_ok, int bar_id,
                             int threads, bool leader) {
  named_sync(bar_id, threads);
  if (leader) {
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
  named_sync(bar_id, threads);
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

// Id at position p (< |I_t|) of I_t: the last 4-word group whose count of
// earlier ids is <= p, then the word and the bit.
__device__ __forceinline__ int nth_id(const uint32_t *bits, const int32_t *goff, int ng, int p) {
  int lo_g = 0, hi_g = ng - 1;
  while (lo_g < hi_g) {
    const int mid = (lo_g + hi_g + 1) >> 1;
    if (goff[mid] <= p) lo_g = mid;
    else hi_g = mid - 1;
  }
  int r = p - goff[lo_g], wi = 4 * lo_g;
  uint32_t w = bits[wi];
  while (r >= __popc(w)) {
    r -= __popc(w);
    w = bits[++wi];
  }
  return wi * 32 + select_bit(w, r);
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

// One warp: the K best entries of `nl` (<= 64) lists sorted best first, K
// entries each (list l at lk/li[l * K]); lane l follows lists l and l + 32.
// Winners go to ok/oi[r] (lane 0 writes).
__device__ __forceinline__ void warp_merge_lists64(const uint32_t *lk, const uint32_t *li, int nl, int K,
                                                   uint32_t *ok, uint32_t *oi) {
  const int lane = threadIdx.x & (kWarp - 1);
  int pa = 0, pb = 0;
  const int la = lane, lb = lane + kWarp;
#pragma unroll 1
  for (int r = 0; r < K; ++r) {
    uint32_t ak = 0u, ai = (uint32_t)kEmptyId, bk = 0u, bi = (uint32_t)kEmptyId;
    if (la < nl && pa < K) {
      ak = lk[la * K + pa];
      ai = li[la * K + pa];
    }
    if (lb < nl && pb < K) {
      bk = lk[lb * K + pb];
      bi = li[lb * K + pb];
    }
    const bool take_b = bk > ak || (bk == ak && bi < ai);
    const uint32_t hk = take_b ? bk : ak, hi = take_b ? bi : ai;
    uint32_t wk, wi;
    warp_best(hk, hi, wk, wi);
    if (lane == 0) {
      ok[r] = wk;
      oi[r] = wi;
    }
    if (wk != 0u && hk == wk && hi == wi) {
      if (take_b) ++pb;
      else ++pa;
    }
  }
  __syncwarp();
}

// Exclusive prefix sum of one int per thread over the state group.  `sh`
// needs kSgWarps ints.
__device__ __forceinline__ int sg_exclusive_scan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & (kWarp - 1), w = ((int)threadIdx.x - kKThreads) >> 5;
  const int incl = warp_inclusive_scan(v);
  if (lane == kWarp - 1) sh[w] = incl;
  named_sync(kBarS, kSgThreads);
  int off = 0, tot = 0;
#pragma unroll
  for (int q = 0; q < kSgWarps; ++q) {
    if (q < w) off += sh[q];
    tot += sh[q];
  }
  *total = tot;
  return off + incl - v;
}

// Word offsets of the state group's arrays (the bulk-copy destinations need
// 16-byte alignment).
struct StepSmem {
  int bits, ring, len, goff, vk, vi, hash, wl, small, share, slot, total;
};
// The slot-stable variant's arrays (at L.slot): the free-slot words, their
// exclusive prefix counts, two hash arrays (an evictable id's old slot, an
// entering id's new slot) and five lists of the entering ids.
constexpr int kSlotHashArrays = 2;
constexpr int kSlotLists = 5;
__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }
__host__ __device__ inline int share_of(int W, int P) { return (W + P - 1) / P; }
__host__ __device__ inline StepSmem step_smem(int nwords_pad, int ring_words, int W, int P, int K, bool slots) {
  StepSmem L;
  L.bits = 0;
  L.ring = L.bits + nwords_pad;                 // nwords_pad and ring_words are multiples of 4
  L.len = L.ring + ring_words;                  // two int64
  L.goff = L.len + 4;
  L.vk = L.goff + round4(nwords_pad / 4);
  L.vi = L.vk + round4(P * K);
  L.hash = L.vi + round4(P * K);
  L.wl = L.hash + kHashArrays * kStepHash;
  L.small = L.wl + 2 * (kSgWarps + 1) * NS_MAX_SELECT_K + 2 * NS_MAX_SELECT_K;
  L.share = L.small + round4(NS_MAX_ROWS + 3 * kMaxAppendStep + 8 + kSgWarps + 3 * kVerPairs);
  L.slot = L.share + round4(share_of(W, P));
  L.total = L.slot + (slots ? 2 * slot_words(W) + kSlotHashArrays * kStepHash + kSlotLists * kMaxAppendStep : 0);
  return L;
}
__host__ __device__ inline int step_smem_bytes(const StepSmem &L) {
  return 1024 + kSRing + kMaxItemsPerCluster * kFBytes + kStepMiscBytes + 4 * L.total;
}

template <int kCL, bool kSlots>
__global__ void __cluster_dims__(kCL, 1, 1) __launch_bounds__(kSThreads, 1)
    step_kernel(const __grid_constant__ CUtensorMap tmH, StepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  if (a.probe) return;

  const UmmaArgs &u = a.u;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool tgrp = warp < 2 || (warp >= 4 && warp < kKWarps);  // tile group
  const bool vgrp = warp == 2 || warp == 3;                      // verify group
  const bool sgrp = warp >= kKWarps;                             // state group
  const int ttid = warp < 2 ? tid : tid - kVGroup;               // index in the tile group
  const int stid = tid - kKThreads;                              // index in the state group
  const uint32_t crank = cluster_rank();
  const int P = (int)gridDim.x, cta = (int)blockIdx.x;
  const int cid = cta / kCL, ncid = P / kCL;
  const int V = u.V, W = u.W_max, K = a.K, n_tree = a.n_tree, H = u.H;
  const bool writer = cta == P - 1;

  // ---- shared memory ----------------------------------------------------------
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte-swizzled stages need 1024-byte alignment
  uint8_t *gbase = smem_raw + (base - raw);
  float *Fbuf = reinterpret_cast<float *>(gbase + kSRing);  // [items][kFRows][kUM] summed tiles
  uint8_t *misc = gbase + kSRing + kMaxItemsPerCluster * kFBytes;
  const uint32_t bar_full = smem_u32(misc), bar_empty = bar_full + 8 * kSStages;
  const uint32_t bar_acc = bar_empty + 8 * kSStages, bar_pready = bar_acc + 8, bar_pdone = bar_pready + 8;
  const uint32_t bar_old = bar_pdone + 8, bar_cver = bar_old + 8, bar_state = bar_cver + 8;
  const uint32_t bar_ring = bar_state + 8, bar_copy = bar_ring + 8, sbar = bar_copy + 8;
  const uint32_t bar_tbl = sbar + 8, bar_k2 = bar_tbl + 8;  // slot-stable variant: table copy landed; past barrier 2
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + 256);
  int *s_flag = reinterpret_cast<int *>(misc + 272);   // [1] state failed, [2], [3] barrier words, [5] past barrier 2
  int *s_tiles = reinterpret_cast<int *>(misc + 512);  // [items][kUM] ids of the items' rows (-1: none)
  int32_t *wbase = reinterpret_cast<int32_t *>(misc + kStepMiscBytes);
  const StepSmem L = step_smem(a.nwords_pad, a.ring_words, W, P, K, kSlots);
  uint32_t *s_bits = reinterpret_cast<uint32_t *>(wbase + L.bits);
  int32_t *s_ring = wbase + L.ring;
  long long *s_len = reinterpret_cast<long long *>(wbase + L.len);
  int32_t *s_goff = wbase + L.goff;
  int *h_key = wbase + L.hash, *h_cnt = h_key + kStepHash, *h_ev = h_cnt + kStepHash, *h_ap = h_ev + kStepHash;
  int *h_wrow = h_ap + kStepHash, *h_ent = h_wrow + kStepHash, *h_chg = h_ent + kStepHash;
  uint32_t *wl_k = reinterpret_cast<uint32_t *>(wbase + L.wl), *wl_i = wl_k + (kSgWarps + 1) * NS_MAX_SELECT_K;
  uint32_t *res_k = wl_i + (kSgWarps + 1) * NS_MAX_SELECT_K, *res_i = res_k + NS_MAX_SELECT_K;
  int *s_tree = wbase + L.small, *s_app = s_tree + NS_MAX_ROWS, *s_arow = s_app + kMaxAppendStep;
  int *s_evid = s_arow + kMaxAppendStep, *s_misc = s_evid + kMaxAppendStep, *sh_scan = s_misc + 8;
  float *s_vdot = reinterpret_cast<float *>(sh_scan + kSgWarps);  // [kVerPairs] verify products
  int *s_vpair = reinterpret_cast<int *>(s_vdot + kVerPairs);     // [kVerPairs] their pair index
  int32_t *s_share = wbase + L.share;
  uint32_t *s_vk = reinterpret_cast<uint32_t *>(wbase + L.vk);
  uint32_t *s_vi = reinterpret_cast<uint32_t *>(wbase + L.vi);
  // slot-stable variant: free slots (updated in place by the state group),
  // their prefix counts, the hash arrays of old and new slots, the entering
  // ids (as found, then ranked) and their new slots; the table of slot ids
  // for the row top-k lives in the stage ring past the top-k lists
  const int fsw = kSlots ? a.fs_words : 0;
  uint32_t *s_fs = reinterpret_cast<uint32_t *>(wbase + L.slot);
  int *s_fsp = reinterpret_cast<int *>(s_fs + fsw);
  int *h_sold = s_fsp + fsw, *h_nslot = h_sold + kStepHash;
  int *e_id = h_nslot + kStepHash, *e_h = e_id + kMaxAppendStep;
  int *p_id = e_h + kMaxAppendStep, *p_slot = p_id + kMaxAppendStep, *p_h = p_slot + kMaxAppendStep;
  int32_t *s_tbl = reinterpret_cast<int32_t *>(gbase + kCopyOff);

  const int nitems = a.items_per_cluster;
  const int t_max = a.t_max;
  const int KC = H / kUK;
  const int nk = KC > (int)crank ? (KC - (int)crank + kCL - 1) / kCL : 0;  // this CTA's k slices
  const int r0 = (kUN * (int)crank) / kCL, nr = (kUN * ((int)crank + 1)) / kCL - r0;  // hidden rows it sums

  // ---- setup: barriers, the state group's copies, loads issued early --------
  if (tid == 0) {
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(bar_full + 8 * s, 1 + kGatherThreads);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    mbar_init(bar_pready, kCL);
    mbar_init(bar_pdone, kCL);
    mbar_init(bar_old, 1);
    mbar_init(bar_cver, 1);
    mbar_init(bar_state, 1);
    mbar_init(bar_ring, 1);
    mbar_init(bar_copy, 1);
    if (kSlots) {
      mbar_init(bar_tbl, 1);
      mbar_init(bar_k2, 1);
    }
    s_flag[1] = 0;
    s_flag[4] = 0;
    mbar_fence_init();
  }
  if (tid == kKThreads) {  // the state group's copies leave first
    mbar_init(sbar, 1);
    mbar_fence_init();
    mbar_expect_tx(sbar, (uint32_t)(a.nwords_pad + a.ring_words + fsw) * 4u + 16u);
    bulk_load(smem_u32(s_bits), a.bitmap, (uint32_t)a.nwords_pad * 4u, sbar);
    bulk_load(smem_u32(s_ring), a.ring, (uint32_t)a.ring_words * 4u, sbar);
    bulk_load(smem_u32(s_len), a.length, 16u, sbar);
    if (kSlots) bulk_load(smem_u32(s_fs), a.slot_free, (uint32_t)fsw * 4u, sbar);
  }
  if (tid == 32) tma_prefetch(&tmH);
  // tile group: the ids of its items' rows (old items: I_{t-1}; the draft
  // item: the tree ids) into registers now, published after the setup barrier
  int t_id[kMaxItemsPerCluster];
  int m_old = 0;
  long long built_len = 0, cur_len = 0;
  if (tgrp || vgrp) {  // compared after the setup barrier (the loads are in flight meanwhile)
    m_old = kSlots ? a.slot_meta[0] : *a.count;  // slot-stable: the old items cover [0, high-water mark)
    built_len = *a.active_len;
    cur_len = a.length[0];
  }
  if (tgrp) {
#pragma unroll
    for (int j = 0; j < kMaxItemsPerCluster; ++j) {
      t_id[j] = -1;
      const int it = cid + j * ncid;
      if (ttid < kUM && j < nitems) {
        if (it < t_max) {
          if (it * kUM + ttid < W) t_id[j] = kSlots ? a.slot_id[it * kUM + ttid] : a.active[it * kUM + ttid];
        } else if (it == t_max && ttid < n_tree) {
          t_id[j] = a.tree[ttid];
        }
      }
    }
  }
  // state group: its slice of the verify row (values [lo, lo + nsl)), one
  // pass of eight values per thread in flight
  int lo = 0, nsl = 0;
  if (K > 0) {
    const int per = (((V + 3) / 4 + P - 1) / P) * 4;
    lo = cta * per;
    nsl = V - lo < per ? V - lo : per;
    if (nsl < 0) nsl = 0;
  }
  constexpr int kPass = 8 * kSgThreads;
  constexpr int kFold = 4;  // extra values a thread can fold into the one pass
  // With K_ver <= 8 a thread's values beyond its 8 best never reach the
  // Top-K, so a slice up to kFold values per thread longer than a pass is
  // ranked in one pass: the extra values (loaded with the pass) replace a
  // thread's worst.
  const bool fold = K <= 8 && nsl > kPass && nsl <= kPass + kFold * kSgThreads;
  float x[8], xe[kFold];
  auto load_pass = [&](int c0) {
    const int n = nsl - c0;
    if (a.vec) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float4 f = make_float4(__int_as_float(0x7fffffff), __int_as_float(0x7fffffff), __int_as_float(0x7fffffff),
                               __int_as_float(0x7fffffff));
        const int e = 4 * (h2 * kSgThreads + stid);
        if (e < n) f = ld_stream_f4(a.zrow + lo + c0 + e);
        x[4 * h2] = f.x, x[4 * h2 + 1] = f.y, x[4 * h2 + 2] = f.z, x[4 * h2 + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = q * kSgThreads + stid;
        x[q] = e < n ? ld_stream_f32(a.zrow + lo + c0 + e) : __int_as_float(0x7fffffff);
      }
    }
  };
  auto load_extra = [&]() {
#pragma unroll
    for (int q = 0; q < kFold; ++q) xe[q] = __int_as_float(0x7fffffff);
    if (a.vec) {
      const int e = kPass + 4 * stid;
      if (e < nsl) {
        const float4 f = ld_stream_f4(a.zrow + lo + e);
        xe[0] = f.x, xe[1] = f.y, xe[2] = f.z, xe[3] = f.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < kFold; ++q) {
        const int e = kPass + q * kSgThreads + stid;
        if (e < nsl) xe[q] = ld_stream_f32(a.zrow + lo + e);
      }
    }
  };
  int tree_id = 0;
  if (sgrp) {
    if (nsl > 0) load_pass(0);
    if (fold) load_extra();
    tree_id = stid < n_tree ? a.tree[stid] : 0;
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // every CTA of the cluster has initialized its barriers before the first
  // remote arrival (the tile group waits on this before its first one)
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  // I_{t-1} was not built from the current window (then the tiles wait for
  // I_t); the slot-stable variant's columns do not depend on I_{t-1}
  const bool stale = !kSlots && built_len != cur_len;

  if (tgrp) {
    // ======================== tile group ======================================
    if (ttid < kUM) {
#pragma unroll
      for (int j = 0; j < kMaxItemsPerCluster; ++j) {
        const int it = cid + j * ncid;
        int id = t_id[j];
        if (it < t_max && it * kUM + ttid >= m_old) id = -1;  // past |I_{t-1}|
        if ((unsigned)id >= (unsigned)V) id = -1;              // invalid tree ids are flagged by the state group
        s_tiles[j * kUM + ttid] = id;
      }
    }
    named_sync(kBarT, kTGroup);
    if (ttid == 0) mbar_arrive(bar_old);  // this group's reads of the old state are done
    int t_old = (m_old + kUM - 1) / kUM;
    if (stale) {  // tiles of I_t itself, at their positions, once it is known
      const bool okw = mbar_wait(bar_state, 0, u.err);
      const int m_new = okw ? s_misc[3] : 0;
      t_old = (m_new + kUM - 1) / kUM;
      if (ttid < kUM) {
        for (int j = 0; j < nitems; ++j) {
          const int it = cid + j * ncid, p = it * kUM + ttid;
          s_tiles[j * kUM + ttid] = it < t_max && p < m_new ? nth_id(s_bits, s_goff, a.nwords_pad / 4, p) : -1;
        }
      }
      named_sync(kBarT, kTGroup);
    }
    bool cluster_ready = false;
    int iter = 0;
    for (int j = 0; j < nitems; ++j) {
      const int it = cid + j * ncid;
      const bool active = it < t_max ? it < t_old : (it == t_max && !stale && n_tree > 0);
      if (!active) continue;  // uniform across the cluster
      const int *rows = s_tiles + j * kUM;
      // ---- main loop ----------------------------------------------------------
      if (warp == 0 && lane == 0) {  // hidden slices by TMA
        int issued = 0;
        for (int kt = 0; kt < nk; ++kt) {
          const int g = iter * nk + kt, s = g % kSStages;
          if (g >= kSStages && !mbar_wait(bar_empty + 8 * s, ((g / kSStages) - 1) & 1, u.err)) break;
          issued = kt + 1;
          mbar_expect_tx(bar_full + 8 * s, kStageB);
          tma_load_2d(base + s * kStage + kStageA, &tmH, ((int)crank + kt * kCL) * kUK, 0, bar_full + 8 * s);
        }
        // nothing may still be landing in shared memory when the ring is reused
        const int first = issued > kSStages ? issued - kSStages : 0;
        for (int kt = first; kt < issued; ++kt) {
          const int g = iter * nk + kt;
          mbar_wait(bar_full + 8 * (g % kSStages), (g / kSStages) & 1, u.err);
        }
      } else if (warp >= 4) {  // W_head rows by cp.async (rows without an id stay unread)
        const int p = tid - 128, wl = p >> 5, c = lane & 7;
        // the slot-stable variant's old items read the slot buffer's own rows
        const bool from_slots = kSlots && it < t_max;
        const uint16_t *src0 = from_slots ? a.slot_rows + (size_t)it * kUM * H : u.W;
        for (int kt = 0; kt < nk; ++kt) {
          const int g = iter * nk + kt, s = g % kSStages;
          if (g >= kSStages) mbar_wait(bar_empty + 8 * s, ((g / kSStages) - 1) & 1, u.err);
          const uint32_t A = base + s * kStage;
          const int col = ((int)crank + kt * kCL) * kUK + c * 8;
#pragma unroll
          for (int rg = 0; rg < kUM / (4 * kGatherWarps); ++rg) {
            const int row = (rg * kGatherWarps + wl) * 4 + (lane >> 3);
            const int id = rows[row];
            if (id >= 0)
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(A + row * 128 + ((c ^ (row & 7)) << 4)),
                           "l"(src0 + (size_t)(from_slots ? row : id) * H + col)
                           : "memory");
          }
          asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar_full + 8 * s) : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");  // nothing of this thread is still landing
      } else if (warp == 1 && lane == 0) {
        bool ok = true;
        for (int kt = 0; kt < nk && ok; ++kt) {
          const int g = iter * nk + kt, s = g % kSStages;
          ok = mbar_wait(bar_full + 8 * s, (g / kSStages) & 1, u.err);
          if (!ok) break;
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the gathered rows, for the tensor core
          tc_fence_after();
          const uint32_t A = base + s * kStage;
#pragma unroll
          for (int kk = 0; kk < kUK / 16; ++kk)
            umma_bf16(tmem, sw128_desc(A + kk * 32), sw128_desc(A + kStageA + kk * 32), (kt | kk) != 0);
          umma_commit(bar_empty + 8 * s);
        }
        if (nk > 0 && ok) umma_commit(bar_acc);
        else mbar_arrive(bar_acc);
      }
      __syncwarp();
      // ---- accumulator -> this CTA's partial tile, then the cluster's sum ----
      float *Pt = reinterpret_cast<float *>(gbase);  // [64][128], reuses the ring
      if (warp >= 4 && warp < 8) {  // warp w reads tensor-memory lanes 32 (w % 4) .. + 31
        const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_acc, iter & 1, u.err));
        tc_fence_after();
        const int jj = (warp - 4) * 32 + lane;
        const uint32_t t0 = tmem + ((uint32_t)((warp - 4) * 32) << 16);
#pragma unroll
        for (int c = 0; c < kUN; c += 16) {
          float v[16];
          if (nk > 0 && ok) {
            tmem_ld16(t0 + c, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = 0.f;
          }
#pragma unroll
          for (int q = 0; q < 16; ++q) Pt[(c + q) * kUM + jj] = v[q];
        }
      }
      tc_fence_before();
      named_sync(kBarT, kTGroup);
      if (!cluster_ready) {  // every peer's barriers are initialized
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        cluster_ready = true;
      }
      if (ttid == 0) {
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        for (uint32_t p = 0; p < (uint32_t)kCL; ++p) mbar_arrive_cluster(map_peer(bar_pready, p));
      }
      mbar_wait_cluster(bar_pready, iter & 1, u.err);
      // hidden rows [r0, r0 + nr) summed over the C partials in rank order
      float *F = Fbuf + j * kFRows * kUM;
      for (int t = ttid; t < nr * (kUM / 4); t += kTGroup) {
        const int rr = t / (kUM / 4), c4 = (t % (kUM / 4)) * 4;
        const uint32_t off = base + (uint32_t)(((r0 + rr) * kUM + c4) * 4);
        float4 s4 = ld_peer_f4(map_peer(off, 0));
#pragma unroll
        for (uint32_t p = 1; p < (uint32_t)kCL; ++p) {
          const float4 q = ld_peer_f4(map_peer(off, p));
          s4.x += q.x;
          s4.y += q.y;
          s4.z += q.z;
          s4.w += q.w;
        }
        *reinterpret_cast<float4 *>(F + rr * kUM + c4) = s4;
      }
      named_sync(kBarT, kTGroup);
      if (ttid == 0) {
        for (uint32_t p = 0; p < (uint32_t)kCL; ++p) mbar_arrive_cluster(map_peer(bar_pdone, p));
      }
      mbar_wait_cluster(bar_pdone, iter & 1, u.err);  // no peer still reads this CTA's partial
      ++iter;
    }
    if (!cluster_ready) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (ttid == 0) mbar_arrive(bar_ring);  // the ring is free past the top-k lists
    if (kSlots && ttid == 0) {  // the old slot table, for the row top-k (its changed entries are patched below)
      const int nt = round4(m_old < 0 ? 0 : (m_old > W ? W : m_old));
      if (nt > 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(bar_tbl, (uint32_t)nt * 4u);
        bulk_load(smem_u32(s_tbl), a.slot_id, (uint32_t)nt * 4u, bar_tbl);
      } else {
        mbar_arrive(bar_tbl);
      }
    }

    // ---- the columns at their positions in I_t ------------------------------
    const bool okst = mbar_wait(bar_state, 0, u.err);
    const int m_act = s_misc[3];
    if (kSlots && ttid < 2 * kUM && okst && m_act >= 0) {
      // slot-stable: a slot whose id stays is written in place, a slot left
      // free below the new high-water mark gets NaN, a slot an entering id
      // took is left to the draft item or the verify products
      const int col = ttid & (kUM - 1), rg = ttid / kUM;
      for (int j = 0; j < nitems; ++j) {
        const int it = cid + j * ncid;
        const bool active = it < t_max ? it < t_old : (it == t_max && n_tree > 0);
        if (!active) continue;
        const int id = s_tiles[j * kUM + col];
        int pos = -1;
        bool hole = false;
        if (it < t_max) {
          const int sl = it * kUM + col;
          if (id >= 0 && ((s_bits[id >> 5] >> (id & 31)) & 1u)) {
            pos = sl;
          } else if (sl < m_act && ((s_fs[sl >> 5] >> (sl & 31)) & 1u)) {
            pos = sl;
            hole = true;
          }
        } else if (id >= 0) {
          const int h = hash_find(h_key, id);
          if (h >= 0 && h_ent[h] != 0 && h_wrow[h] == col) pos = h_nslot[h];
        }
        if (pos >= 0 && pos < W) {
          const float *F = Fbuf + j * kFRows * kUM;
          for (int rr = rg; rr < nr; rr += 2)
            if (r0 + rr < u.n)
              u.logits[(size_t)(r0 + rr) * u.ld + pos] = hole ? __int_as_float(0x7fffffff) : F[rr * kUM + col];
        }
      }
    }
    if (kSlots) {  // the new slots of the entering ids into the table copy
      if (ttid == 0 && !mbar_wait(bar_tbl, 0, u.err)) s_flag[4] = 1;
      named_sync(kBarT, kTGroup);
      const int n_new = okst && m_act >= 0 ? s_misc[4] : 0;
      if (ttid < n_new && ttid < kMaxAppendStep && (unsigned)p_slot[ttid] < (unsigned)W) s_tbl[p_slot[ttid]] = p_id[ttid];
    }
    if (!kSlots && ttid < 2 * kUM && okst) {
      const int col = ttid & (kUM - 1), rg = ttid / kUM;  // one column per thread, two row groups
      for (int j = 0; j < nitems; ++j) {
        const int it = cid + j * ncid;
        const bool active = it < t_max ? it < t_old : (it == t_max && !stale && n_tree > 0);
        if (!active) continue;
        const int id = s_tiles[j * kUM + col];
        int pos = -1;
        if (stale) {
          if (id >= 0 && it * kUM + col < m_act) pos = it * kUM + col;
        } else if (id >= 0) {
          const uint32_t w = s_bits[id >> 5], bit = 1u << (id & 31);
          bool put;
          if (it < t_max) {
            put = (w & bit) != 0u;  // stays in the window
          } else {
            const int h = hash_find(h_key, id);
            put = h >= 0 && h_ent[h] != 0 && h_wrow[h] == col;
          }
          if (put) {
            const int g4 = id >> 7;
            pos = s_goff[g4];
            for (int q = 4 * g4; q < (id >> 5); ++q) pos += __popc(s_bits[q]);
            pos += __popc(w & (bit - 1u));
            if (pos >= m_act) pos = -1;
          }
        }
        if (pos >= 0) {
          const float *F = Fbuf + j * kFRows * kUM;
          for (int rr = rg; rr < nr; rr += 2)
            if (r0 + rr < u.n) u.logits[(size_t)(r0 + rr) * u.ld + pos] = F[rr * kUM + col];
        }
      }
    }
  } else if (vgrp) {
    // ======================== verify group ====================================
    // The verify ids that enter the window and are not tree ids: their
    // logits by CUDA-core dot products, one warp per (id, hidden row) pair;
    // this CTA takes pairs cta, cta + P, ...
    const int vw = warp - 2;
    int npair = 0;
    const bool okc = mbar_wait(bar_cver, 0, u.err);
    const int n_draft = s_misc[0], n_ver = okc && !stale ? s_misc[2] : 0;
    const int n = u.n;
    for (int i = vw;; i += 2) {
      const int q = cta + i * P;
      if (q >= n_ver * n || i >= kVerPairs) break;
      const int v = q / n, r = q - v * n;
      const int id = s_app[n_draft + v];
      const uint4 *wr = reinterpret_cast<const uint4 *>(u.W + (size_t)id * H);
      const uint4 *hr = reinterpret_cast<const uint4 *>(a.hid + (size_t)r * H);
      float acc = 0.f;
      for (int c = lane; c < (H >> 3); c += kWarp) {
        const uint4 w4 = __ldg(wr + c), h4 = __ldg(hr + c);
        const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w}, hv[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = fmaf(__uint_as_float(wv[e] << 16), __uint_as_float(hv[e] << 16), acc);
          acc = fmaf(__uint_as_float(wv[e] & 0xffff0000u), __uint_as_float(hv[e] & 0xffff0000u), acc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) {
        s_vdot[i] = acc;
        s_vpair[i] = q;
      }
      ++npair;
    }
    __syncwarp();
    const bool okst = mbar_wait(bar_state, 0, u.err);
    const int m_act = s_misc[3];
    if (okst && lane < npair) {  // lane l writes the warp's pair l
      const int i = vw + 2 * lane, q = s_vpair[i];
      const int v = q / n, r = q - v * n, id = s_app[n_draft + v];
      const int h = hash_find(h_key, id);
      if (h >= 0 && h_ent[h] != 0 && h_wrow[h] == kVerRow0 + v) {
        int pos;
        if (kSlots) {
          pos = h_nslot[h];  // the slot it took
          if (pos >= W) pos = -1;
        } else {
          const uint32_t w = s_bits[id >> 5], bit = 1u << (id & 31);
          const int g4 = id >> 7;
          pos = s_goff[g4];
          for (int qq = 4 * g4; qq < (id >> 5); ++qq) pos += __popc(s_bits[qq]);
          pos += __popc(w & (bit - 1u));
        }
        if (pos >= 0 && pos < m_act) u.logits[(size_t)r * u.ld + pos] = s_vdot[i];
      }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }

  if (!sgrp) {
    // ---- every CTA's columns are out: rank whole rows ------------------------
    // (the bitmap and group counts of I_t in this CTA's shared memory map a
    // column back to its id)
    bool ok = grid_barrier(a.gbar, (unsigned long long)P, u.err, &s_flag[2], kBarK, kKThreads, tid == 0) &&
              s_misc[3] >= 0;
    if (kSlots) {
      if (tid == 0) mbar_arrive(bar_k2);  // the state group may now write slot rows and the slot table
      ok = ok && s_flag[4] == 0;          // the table copy landed
    }
    const int m_act = s_misc[3];
    if (ok) {
      uint32_t *rk = reinterpret_cast<uint32_t *>(gbase);  // [(warps + 1) x k] lists, then the result
      uint32_t *ri = rk + (kKWarps + 1) * NS_MAX_TOPK;
      uint32_t *ok_k = ri + (kKWarps + 1) * NS_MAX_TOPK, *ok_i = ok_k + NS_MAX_TOPK;
      const int k = u.k;
      const bool vec_l = (u.ld % 4 == 0) && (reinterpret_cast<uintptr_t>(u.logits) % 16 == 0);
      for (int r = cta; r < u.n; r += P) {
        const float *row = u.logits + (size_t)r * u.ld;
        if (tid < k) {
          rk[kKWarps * k + tid] = 0u;
          ri[kKWarps * k + tid] = (uint32_t)kEmptyId;
        }
        for (int c0 = 0; c0 < m_act; c0 += 8 * kKThreads) {
          uint32_t hk[8], hi[8];
          const int j0 = c0 + 8 * tid;
          // every lane takes the same path (a lane that straddles m_act
          // would otherwise wait for a second round of loads): 16-byte
          // groups that start below m_act (inside the row: m_act <= W_max <=
          // ld, both groups and ld multiples of four), then a mask
          float v[8];
          if (vec_l) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
              if (j0 + 4 * h2 < m_act) f = __ldcg(reinterpret_cast<const float4 *>(row + j0 + 4 * h2));
              v[4 * h2] = f.x;
              v[4 * h2 + 1] = f.y;
              v[4 * h2 + 2] = f.z;
              v[4 * h2 + 3] = f.w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = j0 + q < m_act ? __ldcg(row + j0 + q) : 0.f;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) hk[q] = j0 + q < m_act ? order_key(v[q]) : 0u;
          if (kSlots) {  // slot-stable: rank by (value, id), the id from the slot table
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int idq = hk[q] != 0u ? s_tbl[j0 + q] : -1;
              hi[q] = idq >= 0 ? (uint32_t)idq : (uint32_t)kEmptyId;
              if (idq < 0) hk[q] = 0u;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) hi[q] = hk[q] != 0u ? (uint32_t)(j0 + q) : (uint32_t)kEmptyId;
          }
          uint32_t wk, wi;
          warp_topk8_lanes(hk, hi, k, &wk, &wi);
          if (lane < k) {
            rk[warp * k + lane] = wk;
            ri[warp * k + lane] = wi;
          }
          named_sync(kBarK, kKThreads);
          if (warp == 0) {
            uint32_t lk, li;
            warp_merge_lists(rk, ri, kKWarps + 1, k, ok_k, ok_i, lk, li);
            if (lane < k) {
              rk[kKWarps * k + lane] = ok_k[lane];
              ri[kKWarps * k + lane] = ok_i[lane];
            }
          }
          named_sync(kBarK, kKThreads);
        }
        if (tid < k) {  // column -> id through I_t
          const uint32_t key = rk[kKWarps * k + tid];
          const int jc = (int)ri[kKWarps * k + tid];
          u.out_ids[r * k + tid] = key == 0u ? -1 : (kSlots ? jc : nth_id(s_bits, s_goff, a.nwords_pad / 4, jc));
          u.out_vals[r * k + tid] = key != 0u ? key_value(key) : -__int_as_float(0x7f800000);
        }
        named_sync(kBarK, kKThreads);
      }
    }
  } else {
    // ======================== state group =====================================
    const int swarp = stid >> 5;
    for (int q = stid; q < kStepHash; q += kSgThreads) {
      h_key[q] = -1;
      h_cnt[q] = 0;
      h_ev[q] = 0;
      h_ap[q] = 0;
      h_wrow[q] = 0x7fffffff;
      h_ent[q] = 0;
      h_chg[q] = -1;
      if (kSlots) {
        h_sold[q] = -1;
        h_nslot[q] = -1;
      }
    }
    if (kSlots && stid == 0) {
      s_misc[5] = 0;  // entering ids found
      s_misc[6] = 0;  // new high-water mark
    }
    if (stid < n_tree) s_tree[stid] = tree_id;
    // the old window: |S|, its ring slot, the entries that may leave and
    // their counts in the window
    if (!mbar_wait(sbar, 0, u.err)) s_flag[1] = 1;
    named_sync(kBarS, kSgThreads);
    const bool have = s_flag[1] == 0;
    const long long len0 = s_len[0];
    const int head = (int)s_len[1];
    // the slot table must match the window the step starts from (the host
    // takes the multi-launch path otherwise)
    if (kSlots && writer && stid == 0 && have && __ldcg(a.slot_len) != len0) set_flag(u.err, NS_FLAG_INTERNAL | (7u << 8));
    const long long old_start = len0 > W ? len0 - W : 0;
    const int n_old = (int)(len0 - old_start);
    int max_ev = n_tree + K;
    if (max_ev > n_old) max_ev = n_old;
    int ev_id = -1, ev_slot = -1;
    uint32_t ev_cnt = 0u;
    if (stid < max_ev) {  // position old_start + stid
      const int slot = len0 > W ? (head + stid >= W ? head + stid - W : head + stid) : stid;
      ev_id = s_ring[slot];
      if ((unsigned)ev_id >= (unsigned)V) {  // the ring only ever holds valid ids
        if (writer) set_flag(u.err, NS_FLAG_INTERNAL | (2u << 8));
        ev_id = -1;
      }
      if (ev_id >= 0) {  // read before the grid barrier, used after it
        ev_cnt = __ldcg(a.counts + ev_id);
        if (kSlots) ev_slot = __ldcg(a.slot_of + ev_id);  // an id in the window holds a slot
      }
      s_evid[stid] = ev_id;
    }

    // C_draft: distinct valid tree ids in first-occurrence node order, with
    // the tree row of each (state warp 0)
    if (swarp == 0) {
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
      for (int q = 0; q < kWarp; ++q) in_a |= __shfl_sync(0xffffffffu, ka, q) == kb;
      const bool keep_a = va && __ffs(ma) - 1 == lane;
      const bool keep_b = vb && __ffs(mb) - 1 == lane && !in_a;
      const unsigned ba = __ballot_sync(0xffffffffu, keep_a), bb = __ballot_sync(0xffffffffu, keep_b);
      const unsigned lt = (1u << lane) - 1u;
      if (keep_a) {
        s_app[__popc(ba & lt)] = ta;
        s_arow[__popc(ba & lt)] = lane;
      }
      if (keep_b) {
        s_app[__popc(ba) + __popc(bb & lt)] = tb;
        s_arow[__popc(ba) + __popc(bb & lt)] = lane + 32;
      }
      if (lane == 0) s_misc[0] = __popc(ba) + __popc(bb);
    }

    // the slice's Top-K: per pass of eight values per thread, each warp's K
    // best, then state warp 0 merges the warps' lists with the running one
    if (stid < K) {
      wl_k[kSgWarps * K + stid] = 0u;  // the running Top-K starts empty
      wl_i[kSgWarps * K + stid] = (uint32_t)kEmptyId;
    }
    for (int c0 = 0; c0 < (fold ? kPass : nsl); c0 += kPass) {
      if (c0 > 0) load_pass(c0);
      uint32_t hk[8], hi[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = a.vec ? 4 * ((q >> 2) * kSgThreads + stid) + (q & 3) : q * kSgThreads + stid;
        hk[q] = order_key(x[q]);  // padding is NaN: key 0, never ranks
        hi[q] = hk[q] != 0u ? (uint32_t)(lo + c0 + e) : (uint32_t)kEmptyId;
      }
      if (fold) {  // each extra value replaces this thread's worst entry when better
#pragma unroll
        for (int f = 0; f < kFold; ++f) {
          const int e = a.vec ? kPass + 4 * stid + f : kPass + f * kSgThreads + stid;
          const uint32_t ek = order_key(xe[f]);
          const uint32_t ei = ek != 0u ? (uint32_t)(lo + e) : (uint32_t)kEmptyId;
          int w = 0;  // the worst entry: smallest key, then largest id
          uint32_t wk = hk[0], wi = hi[0];
#pragma unroll
          for (int q = 1; q < 8; ++q)
            if (hk[q] < wk || (hk[q] == wk && hi[q] > wi)) w = q, wk = hk[q], wi = hi[q];
          if (ek > wk || (ek == wk && ei < wi)) {
#pragma unroll
            for (int z = 0; z < 8; ++z)
              if (z == w) hk[z] = ek, hi[z] = ei;
          }
        }
      }
      uint32_t wk, wi;
      warp_topk8_lanes(hk, hi, K, &wk, &wi);
      if (lane < K) {
        wl_k[swarp * K + lane] = wk;
        wl_i[swarp * K + lane] = wi;
      }
      named_sync(kBarS, kSgThreads);
      if (swarp == 0) {
        uint32_t lk, li;
        warp_merge_lists(wl_k, wl_i, kSgWarps + 1, K, res_k, res_i, lk, li);
        if (lane < K) {
          wl_k[kSgWarps * K + lane] = res_k[lane];
          wl_i[kSgWarps * K + lane] = res_i[lane];
        }
      }
      named_sync(kBarS, kSgThreads);
    }
    if (stid < K) {
      a.vk[cta * K + stid] = wl_k[kSgWarps * K + stid];
      a.vi[cta * K + stid] = wl_i[kSgWarps * K + stid];
    }
    if (ev_id >= 0) {  // the evictable ids and their window counts
      const int h = hash_insert(h_key, ev_id);
      if (h >= 0) {
        h_cnt[h] = (int)ev_cnt;  // every occurrence of an id read the same count
        if (kSlots) h_sold[h] = ev_slot;
      }
    }

    // ---- grid barrier: every CTA's Top-K is out, every old-state read done --
    if (stid == 0 && !mbar_wait(bar_old, 0, u.err)) s_flag[1] = 1;
    const bool ok = grid_barrier(a.gbar, (unsigned long long)P, u.err, &s_flag[3], kBarS, kSgThreads, stid == 0) &&
                    have && s_flag[1] == 0;

    // ---- C_ver, the window update, I_t --------------------------------------
    int m_act = 0;
    long long len_new = 0;  // |S| after the append
    if (ok) {
      for (int q = stid; q < P * K; q += kSgThreads) {
        s_vk[q] = __ldcg(a.vk + q);
        s_vi[q] = __ldcg(a.vi + q);
      }
      named_sync(kBarS, kSgThreads);
      if (K > 0) {  // two rounds of list merging: 4 groups of at most 64 lists, then the 4 results
        const int per_warp = (P + kSgWarps - 1) / kSgWarps;
        const int l0 = swarp * per_warp;
        const int nl = P - l0 < per_warp ? (P - l0 > 0 ? P - l0 : 0) : per_warp;
        warp_merge_lists64(s_vk + l0 * K, s_vi + l0 * K, nl, K, wl_k + swarp * K, wl_i + swarp * K);
        named_sync(kBarS, kSgThreads);
        if (swarp == 0) {
          uint32_t lk, li;
          warp_merge_lists(wl_k, wl_i, kSgWarps, K, res_k, res_i, lk, li);
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
            s_arow[n_draft + lane] = kVerRow0 + lane;
          }
          if (lane == 0) {
            if (writer && n_ver < K) set_flag(u.err, NS_FLAG_BAD_ID);
            s_misc[1] = n_draft + n_ver;
            s_misc[2] = n_ver;
          }
        }
      } else if (stid == 0) {
        s_misc[1] = s_misc[0];
        s_misc[2] = 0;
      }
      named_sync(kBarS, kSgThreads);
      if (stid == 0) mbar_arrive(bar_cver);  // the verify group may take its products
      const int m = s_misc[1];
      // positions: evicted [old_start, old_start + n_ev), appended [ap_begin, len1)
      const long long len1 = len0 + m;
      const long long new_start = len1 > W ? len1 - W : 0;
      const long long ev_end = len0 < new_start ? len0 : new_start;
      const int n_ev = ev_end > old_start ? (int)(ev_end - old_start) : 0;
      const long long ap_begin = len0 > new_start ? len0 : new_start;
      const int n_ap = (int)(len1 - ap_begin);
      const int ap_off = (int)(ap_begin - len0);
      if (stid < n_ap) {
        const int h = hash_insert(h_key, s_app[ap_off + stid]);
        if (h >= 0) {
          atomicAdd(&h_ap[h], 1);
          atomicMin(&h_wrow[h], s_arow[ap_off + stid]);
        }
      }
      for (int q = stid; q < n_ev; q += kSgThreads) {
        const int id = s_evid[q];
        const int h = id >= 0 ? hash_find(h_key, id) : -1;
        if (h >= 0) atomicAdd(&h_ev[h], 1);
      }
      named_sync(kBarS, kSgThreads);
      // One thread per distinct id: an appended id is in the window (it
      // enters if its bit was clear); an evicted one leaves when its count
      // in the window drops to zero.
      for (int q = stid; q < kStepHash; q += kSgThreads) {
        const int id = h_key[q];
        if (id >= 0) {
          const int ap = h_ap[q], ev = h_ev[q];
          const uint32_t bit = 1u << (id & 31);
          if (ap > 0) {
            if (!(s_bits[id >> 5] & bit)) {
              atomicOr(&s_bits[id >> 5], bit);
              h_ent[q] = 1;
              h_chg[q] = id >> 5;
              if (kSlots) {
                const int e = atomicAdd(&s_misc[5], 1);  // fewer than kMaxAppendStep: one per appended id
                e_id[e] = id;
                e_h[e] = q;
              }
            }
          } else if (ev > 0) {
            const int now = h_cnt[q] - ev;
            if (now < 0 && writer) set_flag(u.err, NS_FLAG_OVERFLOW);
            if (now <= 0) {
              atomicAnd(&s_bits[id >> 5], ~bit);
              h_chg[q] = id >> 5;
              if (kSlots) {  // its slot is free again
                const int sl = h_sold[q];
                if ((unsigned)sl < (unsigned)W) atomicOr(&s_fs[sl >> 5], 1u << (sl & 31));
                else if (writer) set_flag(u.err, NS_FLAG_INTERNAL | (8u << 8));
              }
            }
          }
          if (writer && ap != ev) atomicAdd(&a.counts[id], (unsigned)(ap - ev));
        }
      }
      if (writer) {
        if (stid < n_ap) a.ring[(head + ap_off + stid) % W] = s_app[ap_off + stid];
        if (stid == 0) {
          a.length[0] = len1;
          a.length[1] = (head + m) % W;
          *a.active_len = len1;
        }
      }
      named_sync(kBarS, kSgThreads);
      if (writer) {
        for (int q = stid; q < kStepHash; q += kSgThreads)
          if (h_chg[q] >= 0) a.bitmap[h_chg[q]] = s_bits[h_chg[q]];
      }
      len_new = len1;

      if (kSlots) {
        // ---- the slot update: the entering ids, ascending, take the lowest
        // free slots (the slots of the ids that left are free again)
        const int n_new = s_misc[5];
        if (stid < n_new) {
          const int id = e_id[stid];
          int rk = 0;
          for (int q = 0; q < n_new; ++q) rk += e_id[q] < id ? 1 : 0;
          p_id[rk] = id;
          p_h[rk] = e_h[stid];
        }
        const int G2 = (fsw + kSgThreads - 1) / kSgThreads;
        int nfree_mine = 0;
        for (int w = stid * G2; w < stid * G2 + G2 && w < fsw; ++w) nfree_mine += __popc(s_fs[w]);
        int nfree;
        int fo = sg_exclusive_scan(nfree_mine, sh_scan, &nfree);
        for (int w = stid * G2; w < stid * G2 + G2 && w < fsw; ++w) {
          s_fsp[w] = fo;
          fo += __popc(s_fs[w]);
        }
        named_sync(kBarS, kSgThreads);
        if (stid < n_new) {
          int sl = -1;
          if (stid < nfree) {  // the last word with fewer free slots before it than this rank
            int lo_w = 0, hi_w = fsw - 1;
            while (lo_w < hi_w) {
              const int mid = (lo_w + hi_w + 1) >> 1;
              if (s_fsp[mid] <= stid) lo_w = mid;
              else hi_w = mid - 1;
            }
            sl = 32 * lo_w + select_bit(s_fs[lo_w], stid - s_fsp[lo_w]);
          }
          if ((unsigned)sl >= (unsigned)W) {  // more active ids than slots: cannot happen while |I_t| <= W_max
            if (writer) set_flag(u.err, NS_FLAG_OVERFLOW);
            sl = -1;
          }
          p_slot[stid] = sl;
          h_nslot[p_h[stid]] = sl;
        }
        named_sync(kBarS, kSgThreads);
        if (stid < n_new && p_slot[stid] >= 0) atomicAnd(&s_fs[p_slot[stid] >> 5], ~(1u << (p_slot[stid] & 31)));
        named_sync(kBarS, kSgThreads);
        int top = 0;  // one past the highest occupied slot
        for (int w = stid; w < fsw; w += kSgThreads) {
          const int b0 = 32 * w;
          uint32_t occ = b0 < W ? ~s_fs[w] : 0u;
          if (b0 < W && W - b0 < 32) occ &= (1u << (W - b0)) - 1u;
          if (occ != 0u) top = b0 + 32 - __clz(occ);
        }
        if (top > 0) atomicMax(&s_misc[6], top);
        named_sync(kBarS, kSgThreads);
        if (stid == 0) {
          s_misc[3] = s_misc[6];  // the columns the tile and verify groups write and the top-k ranks
          s_misc[4] = n_new;
        }
        named_sync(kBarS, kSgThreads);
        if (stid == 0) mbar_arrive(bar_state);  // the tile and verify groups may place their columns
      }

      // compaction: per 4-word group, the number of ids before it.  State
      // warp w scans the groups [w * C, (w + 1) * C), 32 consecutive groups
      // per round (one per lane: conflict-free 16-byte reads, a shuffle scan
      // per round), then adds the warps before it.
      const int ng = a.nwords_pad / 4;
      const int C = (((ng + kSgWarps - 1) / kSgWarps) + kWarp - 1) & ~(kWarp - 1);
      const int g0 = swarp * C;
      const uint4 *b4 = reinterpret_cast<const uint4 *>(s_bits);
      int wtot = 0;
#pragma unroll 4
      for (int c0 = 0; c0 < C; c0 += kWarp) {
        const int g = g0 + c0 + lane;
        int cnt = 0;
        if (g < ng) {
          const uint4 w4 = b4[g];
          cnt = __popc(w4.x) + __popc(w4.y) + __popc(w4.z) + __popc(w4.w);
        }
        const int incl = warp_inclusive_scan(cnt);
        if (g < ng) s_goff[g] = wtot + incl - cnt;
        wtot += __shfl_sync(0xffffffffu, incl, kWarp - 1);
      }
      if (lane == 0) sh_scan[swarp] = wtot;
      named_sync(kBarS, kSgThreads);
      int woff = 0, total = 0;
#pragma unroll
      for (int q = 0; q < kSgWarps; ++q) {
        if (q < swarp) woff += sh_scan[q];
        total += sh_scan[q];
      }
      if (woff != 0) {
        for (int c0 = 0; c0 < C; c0 += kWarp) {
          const int g = g0 + c0 + lane;
          if (g < ng) s_goff[g] += woff;
        }
      }
      m_act = total < W ? total : W;
      if (!kSlots && stid == 0) s_misc[3] = m_act;
      if (writer && stid == 0) {
        if (total > W) set_flag(u.err, NS_FLAG_OVERFLOW);
        *a.count = m_act;
      }
      named_sync(kBarS, kSgThreads);
      if (!kSlots && stid == 0) mbar_arrive(bar_state);  // the tile and verify groups may place their columns
      // this CTA's share of I_t: positions [p0, p0 + share)
      const int share = share_of(W, P), p0 = cta * share;
      for (int i = stid; i < share; i += kSgThreads) {
        const int p = p0 + i;
        int id = -1;
        if (p < m_act) {
          id = nth_id(s_bits, s_goff, ng, p);
          a.active[p] = id;
        }
        s_share[i] = id;
      }
    } else if (stid == 0) {
      s_misc[3] = -1;  // no columns, no ranking
      s_misc[4] = 0;   // no new slots
      mbar_arrive(bar_cver);
      mbar_arrive(bar_state);
    }
    named_sync(kBarS, kSgThreads);
    // ---- the packed buffer: the rows of this CTA's share by bulk copies
    // through the stage ring (once the tile group is done with it), beside
    // the top-k
    if (!kSlots && ok && stid == 0) {
      const int share = share_of(W, P), p0 = cta * share;
      int nsh = m_act - p0;
      if (nsh > share) nsh = share;
      const uint32_t rb = (uint32_t)H * 2u;  // row bytes (a multiple of 16)
      const int nbuf = (int)((kSRing - kCopyOff) / rb);
      if (nsh > 0 && nbuf > 0 && mbar_wait(bar_ring, 0, u.err)) {
        const uint32_t stage = base + kCopyOff;
        int phase = 0;
        for (int i0 = 0; i0 < nsh; i0 += nbuf, ++phase) {
          const int nb = nsh - i0 < nbuf ? nsh - i0 : nbuf;
          mbar_expect_tx(bar_copy, (uint32_t)nb * rb);
          for (int b = 0; b < nb; ++b) bulk_load(stage + b * rb, u.W + (size_t)s_share[i0 + b] * H, rb, bar_copy);
          if (!mbar_wait(bar_copy, phase & 1, u.err)) break;
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          for (int b = 0; b < nb; ++b)
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             a.packed + (size_t)(p0 + i0 + b) * H),
                         "r"(stage + b * rb), "r"(rb)
                         : "memory");
          bulk_commit();
          bulk_wait_read_all();  // the staging may be refilled
        }
        bulk_wait_all();
      }
    }
    if (kSlots && ok) {
      // ---- slot-stable: once every CTA is past the second grid barrier (no
      // tile reads a slot row or the old table any more), the entering ids'
      // rows into their slots, and (the last CTA) the new slot state
      if (stid == 0) s_flag[5] = mbar_wait(bar_k2, 0, u.err) ? 1 : 0;
      named_sync(kBarS, kSgThreads);
      if (s_flag[5]) {
        const int n_new = s_misc[4];
        const int upr = H >> 3;  // 16-byte units per row
        for (int r = cta; r < n_new; r += P) {
          const int id = p_id[r], sl = p_slot[r];
          if ((unsigned)id < (unsigned)V && (unsigned)sl < (unsigned)W) {
            const uint4 *src = reinterpret_cast<const uint4 *>(u.W + (size_t)id * H);
            uint4 *dst = reinterpret_cast<uint4 *>(a.slot_rows + (size_t)sl * H);
#pragma unroll 4
            for (int c = stid; c < upr; c += kSgThreads) dst[c] = __ldg(src + c);
          }
        }
        if (writer) {
          for (int q = stid; q < kStepHash; q += kSgThreads) {
            if (h_key[q] >= 0 && h_chg[q] >= 0) {
              a.held[h_chg[q]] = s_bits[h_chg[q]];  // the ids holding a slot: the window's
              const int sl = h_sold[q];             // a slot left free by an id that left
              if (h_ent[q] == 0 && (unsigned)sl < (unsigned)W && ((s_fs[sl >> 5] >> (sl & 31)) & 1u))
                a.slot_id[sl] = -1;
            }
          }
          for (int r = stid; r < n_new; r += kSgThreads) {
            const int sl = p_slot[r], id = p_id[r];
            a.new_slot[r] = sl;
            a.new_id[r] = id;
            if (sl >= 0) {
              a.slot_id[sl] = id;
              a.slot_of[id] = sl;
            }
          }
          for (int w = stid; w < fsw; w += kSgThreads) a.slot_free[w] = s_fs[w];
          if (stid == 0) {
            a.slot_meta[0] = s_misc[3];
            a.slot_meta[1] = n_new;
            *a.slot_len = len_new;
          }
        }
      }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

constexpr int kStepSizes[] = {8, 6, 5, 4};  // cluster sizes the one-launch step can take
constexpr int kNumStepSizes = 4;
// resident clusters of each size (prepare_step_kernel), of the canonical and
// of the slot-stable variant
int g_step_clusters[2][kNumStepSizes] = {{0, 0, 0, 0}, {0, 0, 0, 0}};

template <int CL, bool SLOTS>
int prepare_one() {
  cudaError_t e =
      cudaFuncSetAttribute(step_kernel<CL, SLOTS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, 1, 1);
  cfg.blockDim = dim3(kSThreads, 1, 1);
  cfg.dynamicSmemBytes = kMaxSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, step_kernel<CL, SLOTS>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    clusters = 0;
  }
  return clusters;
}

}  // namespace

cudaError_t prepare_step_kernel() {
  g_step_clusters[0][0] = prepare_one<8, false>();
  g_step_clusters[0][1] = prepare_one<6, false>();
  g_step_clusters[0][2] = prepare_one<5, false>();
  g_step_clusters[0][3] = prepare_one<4, false>();
  g_step_clusters[1][0] = prepare_one<8, true>();
  g_step_clusters[1][1] = prepare_one<6, true>();
  g_step_clusters[1][2] = prepare_one<5, true>();
  g_step_clusters[1][3] = prepare_one<4, true>();
  return cudaSuccess;
}

// The grid must be resident at once (its CTAs wait for each other).  Its work
// items are the tiles of W_max rows plus the draft item; take
// the cluster size that runs them with the fewest items per cluster, then the
// largest (a smaller share of H per CTA), and just enough clusters.
int step_plan(const Dims &d, bool slots, int *tiles_per_cluster, int *cluster_size) {
  const int items = (d.W_max + kUM - 1) / kUM + 1;
  int best_ncl = 0, best_tpc = 0, best_size = 0;
  // the slot-stable variant keeps a copy of the slot table in the stage ring
  if (slots && kCopyOff + 4 * round4(d.W_max) > kSRing) {
    *tiles_per_cluster = 0;
    *cluster_size = 0;
    return 0;
  }
  for (int i = 0; i < kNumStepSizes; ++i) {
    const int size = kStepSizes[i];
    const int res = g_step_clusters[slots ? 1 : 0][i];
    const int most = res < kMaxStepCtas / size ? res : kMaxStepCtas / size;
    if (most < 1) continue;
    const int tpc = (items + most - 1) / most;
    if (tpc > kMaxItemsPerCluster) continue;
    int ncl = (items + tpc - 1) / tpc;
    // enough CTAs for the verify products (kVerPairs per CTA)
    const int pairs = d.K_ver * NS_MAX_ROWS, ctas = (pairs + kVerPairs - 1) / kVerPairs;
    if (ncl * size < ctas) ncl = (ctas + size - 1) / size;
    if (ncl > most) continue;
    // the state update runs on every CTA (the verify row in slices): take
    // about as many CTAs as a full window would, where they are resident
    const int want = (kMinStepCtas + size - 1) / size;
    if (ncl < want) ncl = want < most ? want : most;
    const StepSmem L = step_smem(d.nwords_pad, (d.W_max + 3) & ~3, d.W_max, ncl * size, d.K_ver, slots);
    if (step_smem_bytes(L) > kMaxSmem) continue;
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
  CUtensorMap tmH;
  if (!L.probe && !encode_bf16_2d(&tmH, L.hid, L.d.H, L.n, kUK, kUN)) return cudaErrorInvalidValue;
  if (L.probe) memset(&tmH, 0, sizeof(tmH));
  StepArgs a{};
  UmmaArgs &u = a.u;
  u.W = L.W;
  u.V = L.d.V;
  u.H = L.d.H;
  u.n = L.n;
  u.k = L.k;
  u.W_max = L.d.W_max;
  u.logits = L.logits;
  u.ld = L.ld;
  u.out_ids = L.out_ids;
  u.out_vals = L.out_vals;
  u.err = L.err;
  a.ring = L.s.ring;
  a.counts = L.s.counts;
  a.bitmap = L.s.bitmap;
  a.active = L.s.active;
  a.count = L.s.count;
  a.length = L.s.length;
  a.active_len = L.s.active_len;
  a.packed = L.s.packed;
  a.hid = L.hid;
  a.gbar = L.s.gbar;
  a.vk = L.s.vcand_k;
  a.vi = L.s.vcand_i;
  a.tree = L.tree;
  a.n_tree = L.n_tree;
  a.zrow = L.zrow;
  a.K = L.d.K_ver;
  a.nwords_pad = L.d.nwords_pad;
  a.ring_words = (L.d.W_max + 3) & ~3;
  a.items_per_cluster = L.tiles_per_cluster;
  a.t_max = (L.d.W_max + kUM - 1) / kUM;
  a.vec = L.d.K_ver > 0 && (L.d.V % 4 == 0) && (reinterpret_cast<uintptr_t>(L.zrow) % 16 == 0);
  a.probe = L.probe ? 1 : 0;
  if (L.slots) {
    a.slot_id = L.s.slot_id;
    a.slot_of = L.s.slot_of;
    a.slot_free = L.s.slot_free;
    a.held = L.s.held;
    a.slot_meta = L.s.slot_meta;
    a.new_slot = L.s.new_slot;
    a.new_id = L.s.new_id;
    a.slot_rows = L.s.slot_rows;
    a.slot_len = L.s.slot_len;
    a.fs_words = slot_words(L.d.W_max);
  }
  const int P = L.clusters * L.cluster_size;
  const StepSmem S = step_smem(L.d.nwords_pad, a.ring_words, L.d.W_max, P, L.d.K_ver, L.slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = (size_t)step_smem_bytes(S);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA waits for every other at the grid barriers
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.slots) {
    switch (L.cluster_size) {
      case 8: return cudaLaunchKernelEx(&cfg, step_kernel<8, true>, tmH, a);
      case 6: return cudaLaunchKernelEx(&cfg, step_kernel<6, true>, tmH, a);
      case 5: return cudaLaunchKernelEx(&cfg, step_kernel<5, true>, tmH, a);
      case 4: return cudaLaunchKernelEx(&cfg, step_kernel<4, true>, tmH, a);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (L.cluster_size) {
    case 8: return cudaLaunchKernelEx(&cfg, step_kernel<8, false>, tmH, a);
    case 6: return cudaLaunchKernelEx(&cfg, step_kernel<6, false>, tmH, a);
    case 5: return cudaLaunchKernelEx(&cfg, step_kernel<5, false>, tmH, a);
    case 4: return cudaLaunchKernelEx(&cfg, step_kernel<4, false>, tmH, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ns
