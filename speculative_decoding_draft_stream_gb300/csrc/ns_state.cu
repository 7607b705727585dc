// GPU-resident candidate-stream state: prefill initialisation, the decode-step
// append with the verify Top-K, the window counts and bitmap, and the
// ascending compaction of the bitmap into I_t.
//
// Sources: MicroSpec §3.2 (stream-initialisation, stream-update and
// sliding-window equations; Draft/Verify Candidates) and MicroSpec §3.3
// "Eliminating Overhead via GPU-Resident State Management" (window kept in
// VRAM bitmaps, updated by lock-free kernels without host round-trips).
//
// Representation.  Only the last W_max stream entries are kept, in a ring:
// stream position p lives at ring[p % W_max].  counts[id] is the number of
// occurrences of id among those entries, and bitmap bit id is counts[id] > 0,
// i.e. id in Unique(Suffix(S, W_max)).  Appending entry p overwrites the slot
// of entry p - W_max, which is exactly the entry that leaves the window.
#include "ns_internal.cuh"
#include "ns_ptx.cuh"

namespace ns {
namespace {

constexpr int kMaxAppend = NS_MAX_ROWS + NS_MAX_SELECT_K;

// I_t = set bits of the bitmap (in shared memory) in ascending order, by one
// CTA of kStateThreads threads, in two phases.
//  Scan: thread t takes G consecutive groups of four words (a contiguous run
//  of 128 * G ids); one block scan of the per-thread counts of set bits and
//  of nonzero words lists every nonzero word, in order, with the output
//  offset of its first id (nz_w / nz_o, shared, nwords_pad ints each).
//  Emit: the listed words are dealt so that neighbouring entries go to
//  different warps (the dense run of frequent low ids is spread over all
//  warps) and the lanes of a warp read different banks.  A thread writes the
//  ids of a sparse word itself; the lanes of a warp write a dense word's ids
//  together, one bit each.
// Most words are zero when |I_t| << V; only the listed ones cost work after
// the scan.
constexpr int kCompactMaxG = 4;   // groups of four words per thread (V <= 4 * 4 * 1024 * 32)
constexpr int kDenseBits = 8;     // a word with more set bits is emitted by its whole warp
static_assert(kStateThreads == kWarp * kWarp, "the block scan takes one warp of warp totals");

__device__ void compact_bitmap(const uint32_t *bits, int nwords, int nwords_pad, int32_t *nz_w, int32_t *nz_o,
                               int32_t *active, int32_t *count, int W_max, uint32_t *err,
                               int *sh /* 2 * kWarp ints */) {
  const int T = kStateThreads, tid = threadIdx.x;
  const int lane = tid & (kWarp - 1), warp = tid / kWarp;
  const int ng = nwords_pad / 4;
  const int G = (ng + T - 1) / T;
  const uint4 *bits4 = reinterpret_cast<const uint4 *>(bits);
  uint4 w4[kCompactMaxG];
  int cb = 0, cn = 0;  // set bits, nonzero words
#pragma unroll
  for (int g = 0; g < kCompactMaxG; ++g) {
    w4[g] = make_uint4(0u, 0u, 0u, 0u);
    const int gi = tid * G + g;
    if (g < G && gi < ng) {
      w4[g] = bits4[gi];
      cb += __popc(w4[g].x) + __popc(w4[g].y) + __popc(w4[g].z) + __popc(w4[g].w);
      cn += (w4[g].x != 0u) + (w4[g].y != 0u) + (w4[g].z != 0u) + (w4[g].w != 0u);
    }
  }
  int ib = cb, in = cn;  // inclusive warp scans of both counts
#pragma unroll
  for (int d = 1; d < kWarp; d <<= 1) {
    const int xb = __shfl_up_sync(0xffffffffu, ib, d), xn = __shfl_up_sync(0xffffffffu, in, d);
    if (lane >= d) {
      ib += xb;
      in += xn;
    }
  }
  if (lane == kWarp - 1) {
    sh[warp] = ib;
    sh[kWarp + warp] = in;
  }
  __syncthreads();
  if (warp == 0) {
    int vb = sh[lane], vn = sh[kWarp + lane];
#pragma unroll
    for (int d = 1; d < kWarp; d <<= 1) {
      const int xb = __shfl_up_sync(0xffffffffu, vb, d), xn = __shfl_up_sync(0xffffffffu, vn, d);
      if (lane >= d) {
        vb += xb;
        vn += xn;
      }
    }
    sh[lane] = vb;
    sh[kWarp + lane] = vn;
  }
  __syncthreads();
  const int total = sh[kWarp - 1], n_nz = sh[2 * kWarp - 1];
  int ob = (warp > 0 ? sh[warp - 1] : 0) + ib - cb;
  int on = (warp > 0 ? sh[kWarp + warp - 1] : 0) + in - cn;
#pragma unroll
  for (int g = 0; g < kCompactMaxG; ++g) {
    if (g < G && (w4[g].x | w4[g].y | w4[g].z | w4[g].w) != 0u) {
      const uint32_t ws[4] = {w4[g].x, w4[g].y, w4[g].z, w4[g].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (ws[e] != 0u) {
          nz_w[on] = 4 * (tid * G + g) + e;
          nz_o[on] = ob;
          ++on;
          ob += __popc(ws[e]);
        }
      }
    }
  }
  __syncthreads();
  int32_t *out = active;
  const uint32_t lt = (1u << lane) - 1u;
  for (int r = 0; r * T < n_nz; ++r) {
    const int k = r * T + kWarp * lane + ((warp + lane) & (kWarp - 1));
    const int w = k < n_nz ? nz_w[k] : 0;
    const int o = k < n_nz ? nz_o[k] : 0;
    const uint32_t word = k < n_nz ? bits[w] : 0u;
    const bool dense = __popc(word) > kDenseBits;
    unsigned m = __ballot_sync(0xffffffffu, dense);
    while (m) {
      const int src = __ffs(m) - 1;
      m &= m - 1;
      const uint32_t wd = __shfl_sync(0xffffffffu, word, src);
      const int od = __shfl_sync(0xffffffffu, o, src);
      const int wi = __shfl_sync(0xffffffffu, w, src);
      if ((wd >> lane) & 1u) {
        const int p = od + __popc(wd & lt);
        if (p < W_max) out[p] = wi * 32 + lane;
      }
    }
    if (!dense) {
      uint32_t b = word;
      int p = o;
      while (b) {
        const int i = __ffs(b) - 1;
        b &= b - 1;
        if (p < W_max) out[p] = w * 32 + i;
        ++p;
      }
    }
  }
  const int n = total < W_max ? total : W_max;
  if (tid == 0) {
    if (total > W_max) set_flag(err, NS_FLAG_OVERFLOW);
    *count = n;
  }
}

// Dynamic shared memory of the state kernels, in words: the bitmap, the list
// of nonzero words and their offsets.
__host__ __device__ inline int state_smem_words(int nwords_pad) { return 3 * nwords_pad; }

// ---------------------------------------------------------------------------
// Prefill initialisation (per request)
// ---------------------------------------------------------------------------
// Entries the reset touches: the counts, the bitmaps and the slot table.
__host__ __device__ inline int reset_extent(const Dims &d) {
  int n = d.V > d.nwords_pad ? d.V : d.nwords_pad;
  n = n > d.W_max ? n : d.W_max;
  return n > slot_words(d.W_max) ? n : slot_words(d.W_max);
}

// An empty stream: no entries, an empty window, and an empty slot table.
__global__ void init_reset_kernel(SeqDev s, Dims d) {
  const int n = reset_extent(d);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (i < d.V) {
      s.counts[i] = 0u;
      if (d.K_pre > 0) s.first[i] = 0x7fffffff;
    }
    if (i < d.nwords_pad) {
      s.bitmap[i] = 0u;
      s.held[i] = 0u;
    }
    if (i < d.W_max) s.slot_id[i] = -1;
    if (i < slot_words(d.W_max)) {  // every slot free
      const int b0 = 32 * i;
      s.slot_free[i] = b0 >= d.W_max ? 0u : (d.W_max - b0 >= 32 ? 0xffffffffu : (1u << (d.W_max - b0)) - 1u);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    s.length[0] = 0;
    s.length[1] = 0;
    *s.count = 0;
    *s.active_len = 0;  // the empty I_t matches the empty stream
    s.slot_meta[0] = 0;
    s.slot_meta[1] = 0;
    *s.slot_len = -1;  // the empty table matches no window
    *s.gbar = 0ull;
  }
}

// T_Kpre of prefill row blockIdx.x -> cand[row * K_pre + rank].
template <int KMAX, bool VEC>
__global__ void __launch_bounds__(kInitTopkThreads) prefill_topk_kernel(SeqDev s, Dims d, const float *Z) {
  __shared__ float sc_v[(kInitTopkThreads / kWarp) * NS_MAX_SELECT_K];
  __shared__ int sc_i[(kInitTopkThreads / kWarp) * NS_MAX_SELECT_K];
  __shared__ float res_v[NS_MAX_SELECT_K];
  __shared__ int res_i[NS_MAX_SELECT_K];
  const int K = d.K_pre;
  const float *z = Z + (size_t)blockIdx.x * d.V;
  TopList<KMAX> L;
  L.clear();
  if (VEC) {
    const int n4 = d.V >> 2;
    for (int q = threadIdx.x; q < n4; q += blockDim.x) {
      const float4 f = __ldcs(reinterpret_cast<const float4 *>(z) + q);
      L.insert(f.x, 4 * q);
      L.insert(f.y, 4 * q + 1);
      L.insert(f.z, 4 * q + 2);
      L.insert(f.w, 4 * q + 3);
    }
  } else {
    for (int q = threadIdx.x; q < d.V; q += blockDim.x) L.insert(__ldcs(z + q), q);
  }
  block_select<KMAX>(L, K, sc_v, sc_i, res_v, res_i);
  if (threadIdx.x < K) s.cand[(size_t)blockIdx.x * K + threadIdx.x] = res_i[threadIdx.x];
}

// first[id] = smallest flat index f = row * K_pre + rank at which id occurs.
__global__ void init_first_kernel(SeqDev s, Dims d, int L) {
  const int n = L * d.K_pre;
  for (int f = blockIdx.x * blockDim.x + threadIdx.x; f < n; f += gridDim.x * blockDim.x) {
    const int x = s.cand[f];
    if ((unsigned)x < (unsigned)d.V) atomicMin(&s.first[x], f);  // an all-NaN row leaves empty slots
  }
}

// One CTA: S_init = prompt (+) first occurrences of the union, then the last
// W_max entries into the ring, counts and bitmap.
__global__ void __launch_bounds__(kStateThreads) init_compose_kernel(SeqDev s, Dims d, const int32_t *prompt, int L,
                                                                     uint32_t *err) {
  __shared__ int sh[kStateThreads / kWarp];
  const int nent = L + L * d.K_pre;
  int off = 0;
  for (int base = 0; base < nent; base += blockDim.x) {
    const int e = base + threadIdx.x;
    int keep = 0, x = 0;
    if (e < L) {
      x = prompt[e];
      keep = (unsigned)x < (unsigned)d.V;
      if (!keep) set_flag(err, NS_FLAG_BAD_ID);
    } else if (e < nent) {
      const int f = e - L;
      x = s.cand[f];
      keep = (unsigned)x < (unsigned)d.V && s.first[x] == f;
    }
    int total;
    const int p = block_exclusive_scan(keep, sh, &total);
    if (keep) s.sinit[off + p] = x;
    off += total;
  }
  __syncthreads();
  const long long Ltot = off;
  const long long start = Ltot > d.W_max ? Ltot - d.W_max : 0;
  for (long long p = start + threadIdx.x; p < Ltot; p += blockDim.x) {
    const int x = s.sinit[p];
    s.ring[p % d.W_max] = x;
    atomicAdd(&s.counts[x], 1u);
    atomicOr(&s.bitmap[x >> 5], 1u << (x & 31));
  }
  if (threadIdx.x == 0) {
    s.length[0] = Ltot;
    s.length[1] = Ltot % d.W_max;
  }
}

// The window counts and bitmap of a ring written by the host (a restored
// checkpoint): positions [|S| - min(|S|, W_max), |S|) hold the window, which
// this counts as init_compose_kernel does; then |S| and its ring slot.
__global__ void restore_window_kernel(SeqDev s, Dims d, long long len, uint32_t *err) {
  const long long start = len > d.W_max ? len - d.W_max : 0;
  for (long long p = start + blockIdx.x * (long long)blockDim.x + threadIdx.x; p < len;
       p += (long long)gridDim.x * blockDim.x) {
    const int x = s.ring[p % d.W_max];
    if ((unsigned)x >= (unsigned)d.V) {  // the host checked every entry
      set_flag(err, NS_FLAG_BAD_ID);
      continue;
    }
    atomicAdd(&s.counts[x], 1u);
    atomicOr(&s.bitmap[x >> 5], 1u << (x & 31));
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    s.length[0] = len;
    s.length[1] = len % d.W_max;
  }
}

// ---------------------------------------------------------------------------
// Decode-step append (+ optional compaction): one cluster of 16 CTAs (8 where
// the device cannot hold 16)
// ---------------------------------------------------------------------------
constexpr int kMaxStateCluster = 16;

__device__ __forceinline__ uint32_t state_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ int state_cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ void state_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t leader_addr(const void *p) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)));
  return r;
}

// The cluster's CTAs other than the leader rank one slice each of the verify
// row and hand their Top-K to the leader through distributed shared memory.  A CTA ranks its slice in
// passes of 16 values per thread, held in registers: each thread takes the
// best of its 16; the K-th best of those 1024 maxima is a threshold T that
// every value of the pass's Top-K reaches, and only values at or above T (at
// most K * 16: they all belong to the K threads whose maximum reaches T) are
// collected and ranked exactly by one warp, together with the earlier passes'
// Top-K.  Meanwhile the leader has pulled the tree ids, |S|, the ring slots
// that can be evicted, their ids' window counts and (by a bulk copy) the
// whole bitmap into shared memory, so after the cluster barrier it makes no
// global round trip: the net change of every touched id's window count
// (summed in a shared hash table) and the bitmap say which bits flip, and the
// count and bitmap updates are fire-and-forget atomics.  It then rewrites the
// ring and (BUILD) compacts the updated shared-memory bitmap into I_t.
constexpr int kRankPer = 16;                           // verify values per thread per pass
constexpr int kRankPass = kRankPer * kStateThreads;    // values per CTA per pass
constexpr int kMaxCand = NS_MAX_SELECT_K * kRankPer;   // a pass's threshold candidates, at most
constexpr int kStateWarps = kStateThreads / kWarp;
constexpr int kHashSlots = 256;                        // >= the most distinct ids one step touches

// BATCH: one cluster per sequence; cluster b steps sequence b of the launch
// (its state, tree ids and verify row located through `bt`).
template <bool VEC, bool BUILD, bool BATCH>
__global__ void __launch_bounds__(kStateThreads, 1) append_kernel(SeqDev s, Dims d, const int32_t *tree, int n_tree,
                                                                  const float *zrow, uint32_t *err, StepBatch bt) {
  extern __shared__ uint4 s_dyn4[];  // leader: the bitmap and the nonzero-word list (nwords_pad words each)
  __shared__ uint32_t wl_k[kStateWarps * NS_MAX_SELECT_K], wl_i[kStateWarps * NS_MAX_SELECT_K];
  __shared__ uint32_t cand_k[NS_MAX_SELECT_K + kMaxCand], cand_i[NS_MAX_SELECT_K + kMaxCand];
  __shared__ uint32_t res_k[NS_MAX_SELECT_K], res_i[NS_MAX_SELECT_K];
  __shared__ uint32_t cl_k[kMaxStateCluster * NS_MAX_SELECT_K], cl_i[kMaxStateCluster * NS_MAX_SELECT_K];
  __shared__ uint32_t s_thr[2];
  __shared__ int s_ncand;
  __shared__ int s_tree[NS_MAX_ROWS];
  __shared__ int s_app[kMaxAppend];
  __shared__ int s_evict[kMaxAppend];
  __shared__ uint32_t s_evc[kMaxAppend];
  __shared__ int h_key[kHashSlots];
  __shared__ int h_dl[kHashSlots];
  __shared__ uint32_t h_old[kHashSlots];
  __shared__ int s_misc[4];
  __shared__ long long s_len;
  __shared__ int s_head;  // |S| mod W_max
  __shared__ __align__(8) unsigned long long s_bar;  // the bitmap copy
  __shared__ int sh_scan[2 * kWarp];

  const int tid = threadIdx.x;
  const int warp = tid / kWarp, lane = tid & (kWarp - 1);
  const int K = d.K_ver;
  const uint32_t rank = state_cluster_rank();
  const int nct = state_cluster_size();
  const bool leader = rank == 0;
  if (BATCH) {
    const int b = (int)(blockIdx.x / nct);
    s = seq_at(s, b * bt.seq_bytes);
    tree += (long long)b * bt.tree_stride;
    if (zrow) zrow += b * bt.z_stride + (long long)bt.vrow[b] * d.V;
  }
  uint32_t *s_bits = reinterpret_cast<uint32_t *>(s_dyn4);
  int32_t *s_nzw = reinterpret_cast<int32_t *>(s_bits + d.nwords_pad);
  int32_t *s_nzo = s_nzw + d.nwords_pad;

  // ---- leader: the bitmap starts streaming into shared memory -------------
  if (leader && tid == 0) {
    mbar_init(smem_u32(&s_bar), 1);
    mbar_fence_init();
    mbar_expect_tx(smem_u32(&s_bar), (uint32_t)d.nwords_pad * 4);
    bulk_load(smem_u32(s_bits), s.bitmap, (uint32_t)d.nwords_pad * 4, smem_u32(&s_bar));
  }
  // Distributed shared memory may only be written once every CTA of the
  // cluster is running: arrive now, wait just before the first remote store.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // ---- this CTA's slice of the verify row; the first pass's loads ----------
  // The leader ranks nothing when the cluster has other CTAs: its own loads
  // (|S|, the tree, the ring slots and counts it will update) overlap their
  // ranking instead of delaying its share of it.
  int lo = 0, nslice = 0;
  const int nrank = nct > 1 ? nct - 1 : 1, slice = nct > 1 ? (int)rank - 1 : 0;
  if (K > 0 && slice >= 0) {
    const int S = (((d.V + 3) / 4 + nrank - 1) / nrank) * 4;  // values per ranking CTA, a multiple of 4
    lo = slice * S;
    nslice = d.V - lo < S ? d.V - lo : S;
    if (nslice < 0) nslice = 0;
  }
  float x[kRankPer];
  auto load_pass = [&](int c0) {
    const int n = nslice - c0 < kRankPass ? nslice - c0 : kRankPass;
    if (VEC) {  // zrow is 16-byte aligned and lo, c0, n are multiples of 4
      const float4 *z4 = reinterpret_cast<const float4 *>(zrow + lo + c0);
#pragma unroll
      for (int q = 0; q < kRankPer / 4; ++q) {
        const int u = q * kStateThreads + tid;
        float4 f = make_float4(__int_as_float(0x7fffffff), __int_as_float(0x7fffffff), __int_as_float(0x7fffffff),
                               __int_as_float(0x7fffffff));
        if (4 * u < n) f = __ldcs(z4 + u);
        x[4 * q] = f.x;
        x[4 * q + 1] = f.y;
        x[4 * q + 2] = f.z;
        x[4 * q + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < kRankPer; ++q) {
        const int u = q * kStateThreads + tid;
        x[q] = u < n ? __ldcs(zrow + lo + c0 + u) : __int_as_float(0x7fffffff);
      }
    }
  };
  // id of x[q] in the pass starting at c0 (ascending in q for each thread)
  auto id_of = [&](int c0, int q) -> uint32_t {
    return VEC ? (uint32_t)(lo + c0 + 4 * ((q >> 2) * kStateThreads + tid) + (q & 3))
               : (uint32_t)(lo + c0 + q * kStateThreads + tid);
  };
  // whether group g (x[4g .. 4g+3]) holds any value of the pass starting at c0
  // (the rest of the thread's slots are padding; uniform across most warps)
  auto group_live = [&](int c0, int g) -> bool {
    const int n = nslice - c0 < kRankPass ? nslice - c0 : kRankPass;
    return VEC ? 4 * (g * kStateThreads + tid) < n : 4 * g * kStateThreads + tid < n;
  };
  if (nslice > 0) load_pass(0);

  // ---- leader prologue: |S|, the tree ids -----------------------------------
  if (leader) {
    if (tid == 0) {  // |S| and the ring slot of the next entry, one 16-byte load
      const longlong2 lv = *reinterpret_cast<const longlong2 *>(s.length);
      s_len = lv.x;
      s_head = (int)lv.y;
    }
    if (tid < n_tree) s_tree[tid] = tree[tid];
    for (int q = tid; q < kHashSlots; q += blockDim.x) {
      h_key[q] = -1;
      h_dl[q] = 0;
    }
  }
  if (tid < K) {  // the running Top-K starts empty
    res_k[tid] = 0u;
    res_i[tid] = (uint32_t)kEmptyId;
  }
  __syncthreads();  // the leader's s_len and s_tree; its barrier is initialised

  const int W = d.W_max;
  const long long len0 = s_len;
  const long long old_start = len0 > W ? len0 - W : 0;
  const int max_ev = (n_tree + K) < W ? (n_tree + K) : W;  // no step evicts more
  int ev_id = -1;
  if (leader && tid < max_ev) {  // position old_start + tid (old_start = len0 - W past a full window)
    const int r0 = len0 > W ? s_head : 0;
    ev_id = s.ring[r0 + tid >= W ? r0 + tid - W : r0 + tid];  // used after the ranking
  }

  // ---- rank the slice -------------------------------------------------------
  for (int c0 = 0; c0 < nslice; c0 += kRankPass) {
    if (c0 > 0) load_pass(c0);
    // this thread's best, compared as floats (NaN never wins; -0.0 ties
    // +0.0); ids ascend with q, so the first of equal values stays
    float mv = -__int_as_float(0x7f800000);
    int mq = -1;
#pragma unroll
    for (int g = 0; g < kRankPer / 4; ++g) {
      if (group_live(c0, g)) {
#pragma unroll
        for (int q = 4 * g; q < 4 * g + 4; ++q) {
          if (x[q] > mv) {
            mv = x[q];
            mq = q;
          }
        }
      }
    }
    if (mq < 0) {  // nothing above -inf: the first -inf, if any
      for (int q = 0; q < kRankPer; ++q) {
        if (x[q] == mv) {
          mq = q;
          break;
        }
      }
    }
    uint32_t mk = 0u, mi = (uint32_t)kEmptyId;
    if (mq >= 0) {
      mk = order_key(mv);
      mi = id_of(c0, mq);
    }
    for (int r = 0; r < K; ++r) {  // this warp's K best maxima, best first
      uint32_t bk, bi;
      warp_best(mk, mi, bk, bi);
      if (lane == 0) {
        wl_k[warp * K + r] = bk;
        wl_i[warp * K + r] = bi;
      }
      if (mk == bk && mi == bi) {
        mk = 0u;
        mi = (uint32_t)kEmptyId;
      }
    }
    if (tid == 0) s_ncand = K;  // entries [0, K) hold the earlier passes' Top-K
    if (tid < K) {
      cand_k[tid] = res_k[tid];
      cand_i[tid] = res_i[tid];
    }
    __syncthreads();
    if (warp == 0) {  // T = the K-th best of the CTA's maxima
      uint32_t tk, ti;
      warp_merge_lists(wl_k, wl_i, kStateWarps, K, nullptr, nullptr, tk, ti);
      if (lane == 0) {
        s_thr[0] = tk;
        s_thr[1] = ti;
      }
    }
    __syncthreads();
    const uint32_t tk = s_thr[0], ti = s_thr[1];
    const float tv = tk != 0u ? key_value(tk) : -__int_as_float(0x7f800000);
#pragma unroll
    for (int g = 0; g < kRankPer / 4; ++g) {
      // one compare per group of four (fmaxf skips NaN; padding is NaN), then per value
      if (fmaxf(fmaxf(x[4 * g], x[4 * g + 1]), fmaxf(x[4 * g + 2], x[4 * g + 3])) >= tv) {
#pragma unroll
        for (int q = 4 * g; q < 4 * g + 4; ++q) {
          if (x[q] >= tv) {  // rare: the exact test in key order
            const uint32_t k = order_key(x[q]), i = id_of(c0, q);
            if (k != 0u && (k > tk || (k == tk && i <= ti))) {
              const int slot = atomicAdd(&s_ncand, 1);
              if (slot < NS_MAX_SELECT_K + kMaxCand) {
                cand_k[slot] = k;
                cand_i[slot] = i;
              } else {  // cannot happen: at most K * kRankPer values reach T
                set_flag(err, NS_FLAG_INTERNAL | (4u << 8));
              }
            }
          }
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      const int n = s_ncand < NS_MAX_SELECT_K + kMaxCand ? s_ncand : NS_MAX_SELECT_K + kMaxCand;
      if (n <= 4 * kWarp) {  // the usual case: a few candidates, ranked from registers
        uint32_t hk[4], hi[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = lane + q * kWarp;
          hk[q] = e < n ? cand_k[e] : 0u;
          hi[q] = e < n ? cand_i[e] : (uint32_t)kEmptyId;
        }
        warp_topk4(hk, hi, K, res_k, res_i);
      } else {
        warp_select_keys(cand_k, cand_i, n, K, res_k, res_i);
      }
    }
    __syncthreads();  // res is complete; x, wl and cand may be reused
  }

  // ---- leader: C_draft (warp 1), evicted ids' counts -------------------------
  if (leader && warp == 1) {
    // C_draft: distinct valid tree ids in first-occurrence order.  Lane l
    // holds nodes l and l + 32; invalid ids get keys that match nothing.
    const int a = lane < n_tree ? s_tree[lane] : 0;
    const int b = lane + 32 < n_tree ? s_tree[lane + 32] : 0;
    const bool va = lane < n_tree && (unsigned)a < (unsigned)d.V;
    const bool vb = lane + 32 < n_tree && (unsigned)b < (unsigned)d.V;
    if ((lane < n_tree && !va) || (lane + 32 < n_tree && !vb)) set_flag(err, NS_FLAG_BAD_ID);
    const int ka = va ? a : -1 - lane, kb = vb ? b : -33 - lane;
    const unsigned ma = __match_any_sync(0xffffffffu, ka);
    const unsigned mb = __match_any_sync(0xffffffffu, kb);
    bool in_a = false;
#pragma unroll
    for (int j = 0; j < kWarp; ++j) in_a |= __shfl_sync(0xffffffffu, ka, j) == kb;
    const bool keep_a = va && __ffs(ma) - 1 == lane;
    const bool keep_b = vb && __ffs(mb) - 1 == lane && !in_a;
    const unsigned ba = __ballot_sync(0xffffffffu, keep_a), bb = __ballot_sync(0xffffffffu, keep_b);
    const unsigned lt = (1u << lane) - 1u;
    if (keep_a) s_app[__popc(ba & lt)] = a;
    if (keep_b) s_app[__popc(ba) + __popc(bb & lt)] = b;
    if (lane == 0) s_misc[2] = __popc(ba) + __popc(bb);
    asm volatile("bar.arrive 1, 64;" ::: "memory");  // C_draft and its length, for warp 0
  }
  uint32_t ev_cnt = 0u;
  if (ev_id >= 0) {
    if ((unsigned)ev_id >= (unsigned)d.V) {  // the ring only ever holds valid ids
      set_flag(err, NS_FLAG_INTERNAL | (2u << 8));
      ev_id = -1;
    } else {
      ev_cnt = s.counts[ev_id];  // used after the merge
    }
  }

  // ---- the CTAs' Top-K to the leader ---------------------------------------
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (K > 0 && warp == 0 && lane < K) {
    const uint32_t ak = leader_addr(cl_k + rank * K + lane), ai = leader_addr(cl_i + rank * K + lane);
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ak), "r"(res_k[lane]) : "memory");
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ai), "r"(res_i[lane]) : "memory");
  }
  if (leader) {  // the leader publishes nothing here, so its arrival need not wait for its own loads
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  } else {
    state_cluster_sync();
    return;
  }

  // Warp 0 merges the CTAs' Top-K and appends C_ver after C_draft: the
  // ranked ids are best first; a row without enough orderable (non-NaN)
  // values leaves empty slots at the end, which are not appended.
  if (warp == 0) {
    asm volatile("bar.sync 1, 64;" ::: "memory");  // warp 1 has written C_draft
    const int n_draft = s_misc[2];
    int n_ver = 0;
    if (K > 0) {
      uint32_t lk, li;
      warp_merge_lists(cl_k, cl_i, nct, K, res_k, res_i, lk, li);
      const bool ok = lane < K && res_k[lane] != 0u;
      n_ver = __popc(__ballot_sync(0xffffffffu, ok));
      if (ok) {
        int y = (int)res_i[lane];
        if ((unsigned)y >= (unsigned)d.V) {  // cannot happen for a well-formed merge
          set_flag(err, NS_FLAG_INTERNAL | (1u << 8));
          y = 0;
        }
        s_app[n_draft + lane] = y;
      }
    }
    if (lane == 0) {
      if (n_ver < K) set_flag(err, NS_FLAG_BAD_ID);
      s_misc[3] = n_draft + n_ver;
    }
  }
  if (tid < max_ev) {
    s_evict[tid] = ev_id;
    s_evc[tid] = ev_cnt;
  }
  __syncthreads();  // the appended entries, their count and the evictable ids
  // Let a programmatically launched successor start its prologue; it waits
  // for this grid's results before reading them.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int m = s_misc[3];

  // ---- window: what enters (+1), what leaves (-1), net per distinct id -----
  const long long len1 = len0 + m;
  const long long new_start = len1 > W ? len1 - W : 0;
  const long long ev_end = len0 < new_start ? len0 : new_start;
  const int n_ev = ev_end > old_start ? (int)(ev_end - old_start) : 0;
  const long long ap_begin = len0 > new_start ? len0 : new_start;
  const int n_ap = (int)(len1 - ap_begin);
  if (tid < n_ap + n_ev) {
    int id, dl;
    uint32_t old = 0u;
    if (tid < n_ap) {
      id = s_app[ap_begin + tid - len0];
      dl = 1;
    } else {
      id = s_evict[tid - n_ap];
      old = s_evc[tid - n_ap];
      dl = -1;
    }
    if (id >= 0) {
      unsigned slot = ((unsigned)id * 2654435761u) >> 24;  // 8-bit hash
      for (int probe = 0; probe < kHashSlots; ++probe, slot = (slot + 1) & (kHashSlots - 1)) {
        const int prev = atomicCAS(&h_key[slot], -1, id);
        if (prev == -1 || prev == id) {
          atomicAdd(&h_dl[slot], dl);
          if (dl < 0) h_old[slot] = old;  // every eviction of an id read the same count
          break;
        }
      }
    }
  }
  if (tid < n_ap) {  // position p = ap_begin + tid goes to ring[p % W]
    const int off = (int)(ap_begin - len0) + tid;
    s.ring[(s_head + off) % W] = s_app[off];
  }
  if (tid == 0) {
    s.length[0] = len1;
    s.length[1] = (s_head + m) % W;
  }
  // The bitmap copy must have landed before its bits are read.  If the wait
  // gave up (NS_FLAG_TIMEOUT), the bitmap and I_t are left as they were.
  const bool have_bits = __syncthreads_and(mbar_wait(smem_u32(&s_bar), 0, err));
  // One thread per distinct id.  A net gain sets the bit of an id that was
  // outside the window (bit clear: count 0); a net loss happens only to an
  // evicted id, whose count was read above, and clears the bit when the
  // count reaches 0.
  if (tid < kHashSlots) {
    const int id = h_key[tid], net = h_dl[tid];
    if (id >= 0 && net != 0) {
      atomicAdd(&s.counts[id], (unsigned)net);
      const unsigned bit = 1u << (id & 31);
      if (net > 0) {
        if (have_bits && !(s_bits[id >> 5] & bit)) {
          atomicOr(&s_bits[id >> 5], bit);
          atomicOr(&s.bitmap[id >> 5], bit);
        }
      } else {
        const long long now = (long long)h_old[tid] + net;
        if (now < 0) set_flag(err, NS_FLAG_OVERFLOW);
        if (now == 0 && have_bits) {
          atomicAnd(&s_bits[id >> 5], ~bit);
          atomicAnd(&s.bitmap[id >> 5], ~bit);
        }
      }
    }
  }
  __syncthreads();

  if (BUILD && have_bits) {
    compact_bitmap(s_bits, d.nwords, d.nwords_pad, s_nzw, s_nzo, s.active, s.count, d.W_max, err, sh_scan);
    if (tid == 0 && s.active_len) *s.active_len = len1;
  }
}

__global__ void __launch_bounds__(kStateThreads) build_kernel(SeqDev s, Dims d, uint32_t *err) {
  extern __shared__ uint4 s_dyn4[];  // the bitmap and the nonzero-word list (nwords_pad words each)
  __shared__ int sh_scan[2 * kWarp];
  uint32_t *s_bits = reinterpret_cast<uint32_t *>(s_dyn4);
  int32_t *s_nzw = reinterpret_cast<int32_t *>(s_bits + d.nwords_pad);
  int32_t *s_nzo = s_nzw + d.nwords_pad;
  const uint4 *g4 = reinterpret_cast<const uint4 *>(s.bitmap);
  for (int q = threadIdx.x; q < d.nwords_pad / 4; q += blockDim.x) s_dyn4[q] = g4[q];
  __syncthreads();
  compact_bitmap(s_bits, d.nwords, d.nwords_pad, s_nzw, s_nzo, s.active, s.count, d.W_max, err, sh_scan);
  if (threadIdx.x == 0 && s.active_len && s.length) *s.active_len = s.length[0];
}

// The union of several sequences' windows: word w of every bitmap ORed.
__global__ void union_bitmap_kernel(const uint32_t *bitmap0, int nwords_pad, int nseq, long long seq_bytes,
                                    uint32_t *out) {
  for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < nwords_pad; w += gridDim.x * blockDim.x) {
    uint32_t v = 0u;
    for (int b = 0; b < nseq; ++b)
      v |= __ldg(reinterpret_cast<const uint32_t *>(reinterpret_cast<const char *>(bitmap0) + b * seq_bytes) + w);
    out[w] = v;
  }
}

// packed[j, :] = W[I_t[j], :]; each CTA copies 4 rows per iteration with all
// 16-byte loads of those rows issued before the stores.
constexpr int kGatherThreads = 256;
constexpr int kGatherRows = 4;
constexpr int kGatherMaxUnits = 16;  // per thread per iteration (H <= 8192)

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(SeqDev s, Dims d, const uint16_t *W) {
  const int m = *s.count;
  const int upr = d.H >> 3;  // 16-byte units per row
  const int units = kGatherRows * upr;
  for (int r0 = blockIdx.x * kGatherRows; r0 < m; r0 += gridDim.x * kGatherRows) {
    uint4 buf[kGatherMaxUnits];
#pragma unroll
    for (int q = 0; q < kGatherMaxUnits; ++q) {
      const int u = threadIdx.x + q * kGatherThreads;
      if (u < units) {
        const int r = r0 + u / upr;
        if (r < m) {
          const int c = u - (u / upr) * upr;
          const int id = s.active[r];
          buf[q] = __ldcs(reinterpret_cast<const uint4 *>(W + (size_t)id * d.H) + c);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kGatherMaxUnits; ++q) {
      const int u = threadIdx.x + q * kGatherThreads;
      if (u < units) {
        const int r = r0 + u / upr;
        if (r < m) {
          const int c = u - (u / upr) * upr;
          reinterpret_cast<uint4 *>(s.packed + (size_t)r * d.H)[c] = buf[q];
        }
      }
    }
  }
}

template <int KMAX, bool VEC>
cudaError_t launch_prefill_topk(const SeqDev &s, const Dims &d, const float *Z, int L, cudaStream_t st) {
  prefill_topk_kernel<KMAX, VEC><<<L, kInitTopkThreads, 0, st>>>(s, d, Z);
  return cudaGetLastError();
}

template <bool VEC, bool BUILD, bool BATCH = false>
cudaError_t launch_append_k(const SeqDev &s, const Dims &d, const int32_t *tree, int n_tree, const float *zrow,
                            uint32_t *err, cudaStream_t st, const StepBatch &bt = StepBatch{}, int nseq = 1,
                            int cluster = 0) {
  if (cluster == 0) cluster = d.state_cluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster * nseq, 1, 1);
  cfg.blockDim = dim3(kStateThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)state_smem_words(d.nwords_pad) * 4;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel<VEC, BUILD, BATCH>, s, d, tree, n_tree, zrow, err, bt);
}

template <bool VEC, bool BUILD, bool BATCH = false>
cudaError_t allow_append(int bytes) {
  cudaError_t e =
      cudaFuncSetAttribute(append_kernel<VEC, BUILD, BATCH>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(append_kernel<VEC, BUILD, BATCH>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

// How many clusters of `n` append CTAs with `bytes` of dynamic shared memory
// can be resident at once on this device.
int resident_clusters(int n, int bytes) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n, 1, 1);
  cfg.blockDim = dim3(kStateThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = n;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  const cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, append_kernel<true, true, false>, &cfg);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

bool cluster_fits(int n, int bytes) { return resident_clusters(n, bytes) >= 1; }

}  // namespace

cudaError_t launch_init(const SeqDev &s, const Dims &d, const int32_t *prompt, int L, const float *prefill,
                        uint32_t *err, cudaStream_t st) {
  const int n = reset_extent(d);
  init_reset_kernel<<<(n + 255) / 256, 256, 0, st>>>(s, d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || L == 0) return e;  // an empty prompt leaves the stream empty
  if (d.K_pre > 0) {
    const bool vec = (d.V % 4 == 0) && (reinterpret_cast<uintptr_t>(prefill) % 16 == 0);
    const int K = d.K_pre;
    if (vec) {
      e = K <= 4 ? launch_prefill_topk<4, true>(s, d, prefill, L, st)
          : K <= 8 ? launch_prefill_topk<8, true>(s, d, prefill, L, st)
                   : launch_prefill_topk<16, true>(s, d, prefill, L, st);
    } else {
      e = K <= 4 ? launch_prefill_topk<4, false>(s, d, prefill, L, st)
          : K <= 8 ? launch_prefill_topk<8, false>(s, d, prefill, L, st)
                   : launch_prefill_topk<16, false>(s, d, prefill, L, st);
    }
    if (e != cudaSuccess) return e;
    const int nf = L * d.K_pre;
    init_first_kernel<<<(nf + 255) / 256, 256, 0, st>>>(s, d, L);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  init_compose_kernel<<<1, kStateThreads, 0, st>>>(s, d, prompt, L, err);
  return cudaGetLastError();
}

cudaError_t prepare_state_kernels(Dims *d) {
  const int bytes = state_smem_words(d->nwords_pad) * 4;
  cudaError_t e = cudaSuccess;
  const cudaError_t r[] = {allow_append<true, true>(bytes), allow_append<true, false>(bytes),
                           allow_append<false, true>(bytes), allow_append<false, false>(bytes),
                           allow_append<true, true, true>(bytes), allow_append<false, true, true>(bytes),
                           cudaFuncSetAttribute(build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)};
  for (cudaError_t x : r)
    if (x != cudaSuccess) e = x;
  if (e != cudaSuccess) return e;
  d->state_max16 = resident_clusters(kMaxStateCluster, bytes);
  d->state_max8 = resident_clusters(8, bytes);
  d->state_cluster = d->state_max16 >= 1 ? kMaxStateCluster : 8;
  return cluster_fits(d->state_cluster, bytes) ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t launch_append(const SeqDev &s, const Dims &d, const int32_t *tree, int n_tree, const float *zrow,
                          bool build, uint32_t *err, cudaStream_t st) {
  const bool vec = d.K_ver > 0 && (d.V % 4 == 0) && (reinterpret_cast<uintptr_t>(zrow) % 16 == 0);
  if (vec) {
    return build ? launch_append_k<true, true>(s, d, tree, n_tree, zrow, err, st)
                 : launch_append_k<true, false>(s, d, tree, n_tree, zrow, err, st);
  }
  return build ? launch_append_k<false, true>(s, d, tree, n_tree, zrow, err, st)
               : launch_append_k<false, false>(s, d, tree, n_tree, zrow, err, st);
}

cudaError_t launch_append_batch(const SeqDev &s, const Dims &d, int nseq, const int32_t *tree, int n_tree,
                                const float *verify, const StepBatch &bt, uint32_t *err, cudaStream_t st) {
  if (nseq < 1 || nseq > kMaxBatchLaunch) return cudaErrorInvalidValue;
  // 16-CTA clusters rank faster, but take whichever size needs fewer waves
  const int w16 = d.state_max16 > 0 ? (nseq + d.state_max16 - 1) / d.state_max16 : 1 << 30;
  const int w8 = d.state_max8 > 0 ? (nseq + d.state_max8 - 1) / d.state_max8 : 1 << 30;
  const int cluster = w16 <= w8 ? kMaxStateCluster : 8;
  const bool vec = d.K_ver > 0 && (d.V % 4 == 0) && (reinterpret_cast<uintptr_t>(verify) % 16 == 0);
  return vec ? launch_append_k<true, true, true>(s, d, tree, n_tree, verify, err, st, bt, nseq, cluster)
             : launch_append_k<false, true, true>(s, d, tree, n_tree, verify, err, st, bt, nseq, cluster);
}

cudaError_t launch_restore(const SeqDev &s, const Dims &d, const int32_t *h_ring, long long len, uint32_t *err,
                           cudaStream_t st) {
  const int n = reset_extent(d);
  init_reset_kernel<<<(n + 255) / 256, 256, 0, st>>>(s, d);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(s.ring, h_ring, (size_t)d.W_max * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  const long long win = len < d.W_max ? len : d.W_max;
  const int blocks = win > 0 ? (int)((win + 255) / 256) : 1;
  restore_window_kernel<<<blocks, 256, 0, st>>>(s, d, len, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_build(s, d, err, st);
}

cudaError_t launch_build(const SeqDev &s, const Dims &d, uint32_t *err, cudaStream_t st) {
  build_kernel<<<1, kStateThreads, (size_t)state_smem_words(d.nwords_pad) * 4, st>>>(s, d, err);
  return cudaGetLastError();
}

cudaError_t launch_union_bitmap(const SeqDev &s, const Dims &d, int nseq, long long seq_bytes, uint32_t *out,
                                cudaStream_t st) {
  const int blocks = (d.nwords_pad + 255) / 256;
  union_bitmap_kernel<<<blocks, 256, 0, st>>>(s.bitmap, d.nwords_pad, nseq, seq_bytes, out);
  return cudaGetLastError();
}

cudaError_t launch_gather(const SeqDev &s, const Dims &d, const uint16_t *W, int grid, cudaStream_t st) {
  gather_kernel<<<grid, kGatherThreads, 0, st>>>(s, d, W);
  return cudaGetLastError();
}

}  // namespace ns
