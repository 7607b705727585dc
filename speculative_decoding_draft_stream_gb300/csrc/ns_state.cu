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

namespace ns {
namespace {

constexpr int kMaxAppend = NS_MAX_ROWS + NS_MAX_SELECT_K;
constexpr int kCompactPerThread = 4;  // uint4 bitmap chunks per thread in one CTA

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
__device__ int block_exclusive_scan(int v, int *sh, int *total) {
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

// I_t = set bits of the bitmap in ascending order, by one CTA: each thread
// pop-counts a contiguous run of words, a block scan gives every thread its
// output offset, and each thread emits its ids in order.
__device__ void compact_bitmap(const uint32_t *bitmap, int nwords_pad, int32_t *active, int32_t *count,
                               int W_max, uint32_t *err, int *sh_scan) {
  const int nw4 = nwords_pad / 4;
  const int per = (nw4 + blockDim.x - 1) / blockDim.x;  // <= kCompactPerThread (host checks V)
  const int v0 = threadIdx.x * per;
  uint4 w[kCompactPerThread];
  int c = 0;
#pragma unroll
  for (int q = 0; q < kCompactPerThread; ++q) {
    w[q] = make_uint4(0u, 0u, 0u, 0u);
    if (q < per && v0 + q < nw4) w[q] = __ldcg(reinterpret_cast<const uint4 *>(bitmap) + v0 + q);
    c += __popc(w[q].x) + __popc(w[q].y) + __popc(w[q].z) + __popc(w[q].w);
  }
  int total;
  int pos = block_exclusive_scan(c, sh_scan, &total);
#pragma unroll
  for (int q = 0; q < kCompactPerThread; ++q) {
    const uint32_t ws[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t bits = ws[e];
      const int base = ((v0 + q) * 4 + e) * 32;
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        if (pos < W_max) active[pos] = base + b;
        ++pos;
      }
    }
  }
  if (threadIdx.x == 0) {
    if (total > W_max) set_flag(err, NS_FLAG_OVERFLOW);
    *count = total < W_max ? total : W_max;
  }
}

// ---------------------------------------------------------------------------
// Prefill initialisation (per request)
// ---------------------------------------------------------------------------
__global__ void init_reset_kernel(SeqDev s, Dims d) {
  const int n = d.V > d.nwords_pad ? d.V : d.nwords_pad;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (i < d.V) {
      s.counts[i] = 0u;
      if (d.K_pre > 0) s.first[i] = 0x7fffffff;
    }
    if (i < d.nwords_pad) s.bitmap[i] = 0u;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *s.length = 0;
    *s.count = 0;
    *s.vticket = 0;
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
  if (threadIdx.x == 0) *s.length = Ltot;
}

// ---------------------------------------------------------------------------
// Decode-step append (+ optional compaction)
// ---------------------------------------------------------------------------
// All CTAs rank a slice of the verify row; the last CTA to finish merges the
// slices into C_ver, builds C_draft, appends C_draft (+) C_ver to the ring,
// updates counts and bitmap, and (BUILD) compacts the bitmap into I_t.
template <int KMAX, bool VEC, bool BUILD>
__global__ void __launch_bounds__(kStateThreads) append_kernel(SeqDev s, Dims d, const int32_t *tree, int n_tree,
                                                               const float *zrow, uint32_t *err) {
  __shared__ float sc_v[(kStateThreads / kWarp) * NS_MAX_SELECT_K];
  __shared__ int sc_i[(kStateThreads / kWarp) * NS_MAX_SELECT_K];
  __shared__ float res_v[NS_MAX_SELECT_K];
  __shared__ int res_i[NS_MAX_SELECT_K];
  __shared__ int s_tree[NS_MAX_ROWS];
  __shared__ int s_app[kMaxAppend];
  __shared__ int s_ev[kMaxAppend];
  __shared__ int s_misc[4];
  __shared__ int sh_scan[kStateThreads / kWarp];

  const int tid = threadIdx.x;
  const int K = d.K_ver;

  // ---- C_ver = T_Kver(z_verify) -------------------------------------------
  if (K > 0) {
    TopList<KMAX> L;
    L.clear();
    const int gstride = gridDim.x * blockDim.x;
    if (VEC) {
      const int n4 = d.V >> 2;
      for (int q = blockIdx.x * blockDim.x + tid; q < n4; q += gstride) {
        const float4 f = __ldcs(reinterpret_cast<const float4 *>(zrow) + q);
        L.insert(f.x, 4 * q);
        L.insert(f.y, 4 * q + 1);
        L.insert(f.z, 4 * q + 2);
        L.insert(f.w, 4 * q + 3);
      }
    } else {
      for (int q = blockIdx.x * blockDim.x + tid; q < d.V; q += gstride) L.insert(__ldcs(zrow + q), q);
    }
    block_select<KMAX>(L, K, sc_v, sc_i, res_v, res_i);
    if (gridDim.x > 1) {
      if (tid < K) {
        s.vpart_v[blockIdx.x * K + tid] = res_v[tid];
        s.vpart_i[blockIdx.x * K + tid] = res_i[tid];
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) s_misc[0] = (atomicAdd(s.vticket, 1) == (int)gridDim.x - 1);
      __syncthreads();
      if (!s_misc[0]) return;
      __threadfence();
      if (tid == 0) *s.vticket = 0;
      L.clear();
      for (int q = tid; q < (int)gridDim.x * K; q += blockDim.x) L.insert(__ldcg(s.vpart_v + q), __ldcg(s.vpart_i + q));
      block_select<KMAX>(L, K, sc_v, sc_i, res_v, res_i);
    }
  }

  // Only this CTA is left: let a programmatically launched successor start
  // its prologue; it waits for this grid's results before reading them.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- C_draft: distinct valid tree ids in first-occurrence order ----------
  if (tid < n_tree) s_tree[tid] = tree[tid];
  __syncthreads();
  const int warp = tid / kWarp, lane = tid & (kWarp - 1);
  int keep = 0, x = 0;
  if (tid < n_tree) {
    x = s_tree[tid];
    keep = (unsigned)x < (unsigned)d.V;
    if (!keep) set_flag(err, NS_FLAG_BAD_ID);
    for (int j = 0; j < tid && keep; ++j)
      if (s_tree[j] == x) keep = 0;
  }
  unsigned ball = 0;
  if (warp < 2) ball = __ballot_sync(0xffffffffu, keep);
  if (warp == 0 && lane == 0) s_misc[1] = __popc(ball);
  __syncthreads();
  if (warp < 2) {
    const int pos = __popc(ball & ((1u << lane) - 1u)) + (warp == 1 ? s_misc[1] : 0);
    if (keep) s_app[pos] = x;
    if (warp == 1 && lane == 0) s_misc[2] = s_misc[1] + __popc(ball);
  }
  __syncthreads();
  const int n_draft = s_misc[2];
  // C_ver: the ranked ids are best first; a row without enough orderable
  // (non-NaN) values leaves empty slots at the end, which are not appended.
  int n_ver = 0;
  for (int q = 0; q < K; ++q) n_ver += res_i[q] != kEmptyId;
  if (tid < n_ver) s_app[n_draft + tid] = res_i[tid];
  if (tid == 0 && n_ver < K) set_flag(err, NS_FLAG_BAD_ID);
  const int m = n_draft + n_ver;

  // ---- append to the ring, evict, update counts and bitmap ----------------
  const long long W = d.W_max;
  const long long len0 = *s.length;
  const long long len1 = len0 + m;
  const long long new_start = len1 > W ? len1 - W : 0;
  const long long old_start = len0 > W ? len0 - W : 0;
  const long long ev_end = len0 < new_start ? len0 : new_start;
  const int n_ev = ev_end > old_start ? (int)(ev_end - old_start) : 0;
  const long long ap_begin = len0 > new_start ? len0 : new_start;
  const int n_ap = (int)(len1 - ap_begin);
  if (tid < n_ev) s_ev[tid] = s.ring[(old_start + tid) % W];
  __syncthreads();
  if (tid < n_ap) {
    const long long p = ap_begin + tid;
    const int y = s_app[p - len0];
    s.ring[p % W] = y;
    atomicAdd(&s.counts[y], 1u);
  }
  if (tid >= 128 && tid - 128 < n_ev) {
    const unsigned old = atomicSub(&s.counts[s_ev[tid - 128]], 1u);
    if (old == 0u) set_flag(err, NS_FLAG_OVERFLOW);
  }
  __threadfence();
  __syncthreads();
  int fix = -1;
  if (tid < n_ap) fix = s_app[ap_begin + tid - len0];
  else if (tid >= 128 && tid - 128 < n_ev) fix = s_ev[tid - 128];
  if (fix >= 0) {
    const unsigned c = atomicAdd(&s.counts[fix], 0u);
    const unsigned bit = 1u << (fix & 31);
    if (c) atomicOr(&s.bitmap[fix >> 5], bit);
    else atomicAnd(&s.bitmap[fix >> 5], ~bit);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *s.length = len1;

  if (BUILD) compact_bitmap(s.bitmap, d.nwords_pad, s.active, s.count, d.W_max, err, sh_scan);
}

__global__ void __launch_bounds__(kStateThreads) build_kernel(SeqDev s, Dims d, uint32_t *err) {
  __shared__ int sh_scan[kStateThreads / kWarp];
  compact_bitmap(s.bitmap, d.nwords_pad, s.active, s.count, d.W_max, err, sh_scan);
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

template <bool VEC, bool BUILD>
cudaError_t launch_append_k(const SeqDev &s, const Dims &d, int vgrid, const int32_t *tree, int n_tree,
                            const float *zrow, uint32_t *err, cudaStream_t st) {
  const int K = d.K_ver;
  if (K <= 4) append_kernel<4, VEC, BUILD><<<vgrid, kStateThreads, 0, st>>>(s, d, tree, n_tree, zrow, err);
  else if (K <= 8) append_kernel<8, VEC, BUILD><<<vgrid, kStateThreads, 0, st>>>(s, d, tree, n_tree, zrow, err);
  else append_kernel<16, VEC, BUILD><<<vgrid, kStateThreads, 0, st>>>(s, d, tree, n_tree, zrow, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_init(const SeqDev &s, const Dims &d, const int32_t *prompt, int L, const float *prefill,
                        uint32_t *err, cudaStream_t st) {
  const int n = d.V > d.nwords_pad ? d.V : d.nwords_pad;
  init_reset_kernel<<<(n + 255) / 256, 256, 0, st>>>(s, d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
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

cudaError_t launch_append(const SeqDev &s, const Dims &d, int vgrid, const int32_t *tree, int n_tree,
                          const float *zrow, bool build, uint32_t *err, cudaStream_t st) {
  const bool vec = d.K_ver > 0 && (d.V % 4 == 0) && (reinterpret_cast<uintptr_t>(zrow) % 16 == 0);
  const int grid = d.K_ver > 0 ? vgrid : 1;
  if (vec) {
    return build ? launch_append_k<true, true>(s, d, grid, tree, n_tree, zrow, err, st)
                 : launch_append_k<true, false>(s, d, grid, tree, n_tree, zrow, err, st);
  }
  return build ? launch_append_k<false, true>(s, d, grid, tree, n_tree, zrow, err, st)
               : launch_append_k<false, false>(s, d, grid, tree, n_tree, zrow, err, st);
}

cudaError_t launch_build(const SeqDev &s, const Dims &d, uint32_t *err, cudaStream_t st) {
  build_kernel<<<1, kStateThreads, 0, st>>>(s, d, err);
  return cudaGetLastError();
}

cudaError_t launch_gather(const SeqDev &s, const Dims &d, const uint16_t *W, int grid, cudaStream_t st) {
  gather_kernel<<<grid, kGatherThreads, 0, st>>>(s, d, W);
  return cudaGetLastError();
}

}  // namespace ns
