// Fused sub-head step on the 5th-generation tensor cores: gather of
// W_head[I_t, :] into the packed buffer, projection of the draft hidden
// states through it, and per-row top-k remapped to global ids
// (MicroSpec §3.3 gathering into a contiguous buffer + dense product; §3.1
// Eq. 1 restricted to the active rows).
//
// Tile: 128 W_head rows (UMMA M) x 64 hidden rows (UMMA N, n <= 64).
// Each tile belongs to one cluster of C CTAs (16 where the device holds such
// clusters, else 8) that split H C ways; the 64-wide k slices are dealt
// round-robin (CTA c takes slices c, c+C, ...), so at any moment a cluster
// reads C * 128-byte runs of each row.
// Per CTA and per k slice (a 4-stage ring overlaps the roles):
//   * warps 4-7 gather the tile's 128 rows with 16-byte cp.async (four rows
//     of 128 contiguous bytes per warp instruction) into the 128-byte-
//     swizzled operand layout, then fence the async proxy and arrive on the
//     stage's "full" barrier;
//   * warp 0 (one lane) loads the hidden slice with a tiled TMA load onto the
//     same barrier;
//   * warp 1 (one lane) issues four tcgen05.mma (K = 16 each) into a
//     128 x 64 fp32 accumulator in tensor memory and commits to the stage's
//     "empty" barrier;
//   * warp 2 (one lane) stores the gathered stage to the packed buffer with a
//     TMA tile store, so each W_head row crosses HBM once per step.
// Epilogue: warps 4-7 read the accumulator (tcgen05.ld, one row per thread),
// every CTA publishes its partial tile in shared memory, and after a cluster
// barrier CTA c adds the C partials for hidden rows [64c/C, 64(c+1)/C)
// through distributed shared memory in a fixed order (deterministic), ranks each
// row's 128 columns (one warp per row) and writes those logits.  The
// per-tile candidates (sorted) of a row slice are merged by the last CTA of
// that slice to finish (release/acquire ticket) into the final top-k.
//
// Every wait is bounded (about a second); a wait that runs out sets
// NS_FLAG_TIMEOUT and the kernel still follows the same barrier sequence and
// frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ns_internal.cuh"
#include "ns_ptx.cuh"

namespace ns {
namespace {

constexpr int kUM = 128;                     // W rows per tile
constexpr int kUN = 64;                      // hidden rows per tile
constexpr int kUK = 64;                      // k per stage: one 128-byte swizzled row
constexpr int kUStages = 4;
constexpr int kUThreads = 256;
constexpr int kGatherThreads = 128;          // warps 4-7
constexpr int kInFlight = 3;                 // cp.async stages a gather thread keeps in flight
constexpr int kStoresInFlight = 1;           // packed-buffer stores still reading a stage
// A stage is published kInFlight-1 iterations after it is issued and released
// by the store issuer kStoresInFlight stores later; the gather threads wait for
// the release of the stage they reuse kUStages iterations on.  Reuse can only
// make progress when the two lags fit in the ring.
static_assert((kInFlight - 1) + kStoresInFlight <= kUStages - 1, "stage ring too short for the pipeline lags");
constexpr int kStageA = kUM * kUK * 2;       // 16 KB
constexpr int kStageB = kUN * kUK * 2;       // 8 KB
constexpr int kStage = kStageA + kStageB;    // 24 KB (1024-byte multiple)
constexpr int kRingBytes = kUStages * kStage;
constexpr int kPartBytes = kUN * kUM * 4;    // one CTA's partial tile, [r][j] fp32
constexpr int kMiscBytes = 1280;             // barriers, TMEM slot, ticket flag, row ids, slot ids
constexpr int kUSmem = kRingBytes + kMiscBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 64;

constexpr int kMergeLists = 24;  // tiles' lists merged per round of the final merge (+ the running list)
constexpr int kMergeWarpWords = (kMergeLists + 1) * NS_MAX_TOPK;
constexpr int kMergeBatch = 8;   // candidate loads a lane keeps in flight while staging
// hidden rows reduced by one CTA: kUN / cluster size, at most 8
static_assert(kPartBytes + 8 * kUM * 4 + 8 * (2 * kMergeWarpWords + 2 * NS_MAX_TOPK) * 4 <= kRingBytes,
              "epilogue buffers reuse the stage ring");

// D = fp32, A = B = bf16, both K-major, N = 64, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kUN >> 3) << 17) |
                            ((uint32_t)(kUM >> 4) << 24);

// ---- TMA ------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- tcgen05 ----------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (sm_100 descriptor version 1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused with a 128-byte swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // SWIZZLE_128B
  return d;
}
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- cluster ----------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_peer_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

struct UmmaArgs {
  const uint16_t *W;         // W_head [V x H]
  const int32_t *idx;        // I_t ascending
  const int32_t *count_ptr;  // |I_t|
  int32_t V, H, n, k, W_max;
  float *logits;             // [n x ld]
  int32_t ld;
  uint32_t *cand_k;          // [tiles x 64 x k] per-tile candidates: order keys, best first
  uint32_t *cand_i;          // and their ids
  int32_t *slice_ticket;     // [cluster size]
  int32_t *out_ids;          // [n x k]
  float *out_vals;
  uint32_t *err;
  // kBatch: nseq sequences of tiles_per_seq tiles (of W_max) each; sequence
  // b's state (idx, count, candidates, tickets) is b * seq_bytes past
  // sequence 0's, its logits b * logits_bytes past, its outputs b * n * k
  // entries past
  long long seq_bytes, logits_bytes;
  int32_t nseq, tiles_per_seq;
  int32_t rows_by_id;  // kInPlace: row j is W row idx[j] (an indexed product, nothing packed)
};

// kInPlace: the rows come from a buffer that already holds them (the packed
// buffer after a separate gather, or the slot buffer): row j of a tile is
// buffer row row0 + j, read in place and not stored back, and the top-k maps
// row j to the id idx[j], skipping rows whose id is -1 (free slots; count_ptr
// is then the slot table's high-water mark).  With rows_by_id the buffer is
// W_head itself and row j is W_head row idx[j]: the indexed product without a
// packed copy.
//
// kBatch: one launch for several sequences (the hidden and packed tensor maps
// get a third, per-sequence dimension); the clusters loop over the work items
// (a tile of a sequence), see below.
template <int kUCluster, bool kInPlace, bool kBatch = false>
__global__ void __cluster_dims__(kUCluster, 1, 1) __launch_bounds__(kUThreads, 2)
    umma_step_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmP,
                     UmmaArgs a) {
  constexpr int kSlice = kUN / kUCluster;  // hidden rows [kSlice * c, kSlice * (c + 1)) are reduced by CTA c
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte-swizzled tiles need 1024-byte alignment
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t bar_full = base + kRingBytes;
  const uint32_t bar_empty = bar_full + 8 * kUStages;
  const uint32_t bar_acc = bar_empty + 8 * kUStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kRingBytes + 16 * kUStages + 8);
  int *s_flag = reinterpret_cast<int *>(gbase + kRingBytes + 16 * kUStages + 16);
  int *s_rows = reinterpret_cast<int *>(gbase + kRingBytes + 256);  // 128 source rows (ids, or slots)
  int *s_ids = s_rows + kUM;                                         // 128 ids of the rows (kInPlace)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_rank();
  // One sequence: clusters take tiles cid, cid + ncid, ... (one each when the
  // grid holds them all).  kBatch: clusters take work items cid, cid + ncid,
  // ... of nseq * tiles_per_seq; item i is tile i / nseq of sequence i % nseq
  // (tile-major, so the tiles that exist come first), and the items past a
  // sequence's |I_t| are skipped.
  const int cid = blockIdx.x / kUCluster, ncid = gridDim.x / kUCluster;
  __shared__ int s_cnt[kMaxBatchLaunch];  // kBatch: |I_t| of every sequence

  // ---- prologue (overlaps the state update when launched programmatically) --
  if (tid == 0) {
    tma_prefetch(&tmH);
    tma_prefetch(&tmP);
    for (int s = 0; s < kUStages; ++s) {
      mbar_init(bar_full + 8 * s, 1 + kGatherThreads);  // the TMA issuer and every gather thread
      mbar_init(bar_empty + 8 * s, kInPlace ? 1 : 2);     // the MMA commit (and the packed-store issuer)
    }
    mbar_init(bar_acc, 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependency_wait();  // I_t and |I_t| come from the state update
  // The first tile's row ids load together with |I_t| (one round trip); the
  // entries past |I_t| are not used.
  int id_first = 0, m0 = 0, T0 = 0;
  if (kBatch) {
    const int t0 = cid / a.nseq, b0 = cid % a.nseq;
    const int32_t *idx0 = reinterpret_cast<const int32_t *>(reinterpret_cast<const char *>(a.idx) + b0 * a.seq_bytes);
    if (tid < kUM && t0 * kUM + tid < a.W_max) id_first = idx0[t0 * kUM + tid];
    if (tid < a.nseq)
      s_cnt[tid] = *reinterpret_cast<const int32_t *>(reinterpret_cast<const char *>(a.count_ptr) + tid * a.seq_bytes);
    __syncthreads();
  } else {
    if (tid < kUM && cid * kUM + tid < a.W_max) id_first = a.idx[cid * kUM + tid];
    m0 = *a.count_ptr;
    T0 = (m0 + kUM - 1) / kUM;
    if (cid >= T0) {  // uniform across the cluster
      if (T0 == 0 && cid == 0) {
        const int r = (int)crank * kSlice + warp;
        if (warp < kSlice && r < a.n && lane < a.k) {
          a.out_ids[r * a.k + lane] = -1;
          a.out_vals[r * a.k + lane] = -__int_as_float(0x7f800000);
        }
      }
      __syncwarp();
      if (warp == 1) tmem_dealloc(tmem, kTmemCols);
      return;
    }
  }

  const int KC = a.H / kUK;
  // k slices of this CTA: crank, crank + C, ... (nk of them, the same for every tile)
  const int nk = KC > (int)crank ? (KC - (int)crank + kUCluster - 1) / kUCluster : 0;
  // Stage use g = iter * nk + kt runs on across tiles: ring slot g % kUStages,
  // mbarrier phase g / kUStages.
  int iter = 0;  // work items processed so far
  for (int item = cid;; item += ncid) {
  int tile, bseq = 0, m, T;
  if (kBatch) {
    if (item >= a.nseq * a.tiles_per_seq) break;
    tile = item / a.nseq;
    bseq = item % a.nseq;
    m = s_cnt[bseq];
    T = (m + kUM - 1) / kUM;
  } else {
    tile = item;
    m = m0;
    T = T0;
    if (tile >= T) break;
  }
  // this sequence's state and outputs
  const long long so = bseq * a.seq_bytes;
  const int32_t *idx = reinterpret_cast<const int32_t *>(reinterpret_cast<const char *>(a.idx) + so);
  uint32_t *cand_k = reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(a.cand_k) + so);
  uint32_t *cand_i = reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(a.cand_i) + so);
  int32_t *ticket = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(a.slice_ticket) + so);
  float *logits = reinterpret_cast<float *>(reinterpret_cast<char *>(a.logits) + bseq * a.logits_bytes);
  int32_t *out_ids = a.out_ids + (long long)bseq * a.n * a.k;
  float *out_vals = a.out_vals + (long long)bseq * a.n * a.k;
  if (kBatch && tile >= T) {  // uniform across the cluster
    if (T == 0 && tile == 0) {  // an empty I_t: padding only
      const int r = (int)crank * kSlice + warp;
      if (warp < kSlice && r < a.n && lane < a.k) {
        out_ids[r * a.k + lane] = -1;
        out_vals[r * a.k + lane] = -__int_as_float(0x7f800000);
      }
    }
    continue;
  }
  const int row0 = tile * kUM;
  if (tid < kUM) {
    const int j = row0 + tid;
    if (j < m) {
      int id = item == cid ? id_first : idx[j];
      if (kInPlace) {
        if (id < -1 || id >= a.V) {  // a row holds a valid id or is a free slot (-1)
          atomicOr(a.err, NS_FLAG_INTERNAL | (3u << 8));
          id = -1;
        }
        s_ids[tid] = id;
        s_rows[tid] = a.rows_by_id ? (id < 0 ? 0 : id) : j;  // rows_by_id: W_head rows, no packed copy
      } else {
        if ((unsigned)id >= (unsigned)a.V) {  // I_t only holds valid ids
          atomicOr(a.err, NS_FLAG_INTERNAL | (3u << 8));
          id = 0;
        }
        s_rows[tid] = id;
      }
    }
  }
  __syncthreads();
  if (tid < kUM && row0 + tid >= m) s_rows[tid] = s_rows[m - 1 - row0];  // rows past |I_t| repeat the last
  __syncthreads();

  // ---- main loop -------------------------------------------------------------
  if (warp == 0 && lane == 0) {  // hidden slices by TMA
    int issued = 0;
    for (int kt = 0; kt < nk; ++kt) {
      const int g = iter * nk + kt, s = g % kUStages;
      if (g >= kUStages && !mbar_wait(bar_empty + 8 * s, ((g / kUStages) - 1) & 1, a.err)) break;
      issued = kt + 1;
      mbar_expect_tx(bar_full + 8 * s, kStageB);
      if (kBatch)
        tma_load_3d(base + s * kStage + kStageA, &tmH, ((int)crank + kt * kUCluster) * kUK, 0, bseq,
                    bar_full + 8 * s);
      else
        tma_load_2d(base + s * kStage + kStageA, &tmH, ((int)crank + kt * kUCluster) * kUK, 0, bar_full + 8 * s);
    }
    // nothing may still be landing in shared memory when the CTA leaves
    const int first = issued > kUStages ? issued - kUStages : 0;
    for (int kt = first; kt < issued; ++kt) {
      const int g = iter * nk + kt;
      mbar_wait(bar_full + 8 * (g % kUStages), (g / kUStages) & 1, a.err);
    }
  } else if (warp >= 4) {  // W_head rows by cp.async
    const int p = tid - 128, wl = p >> 5, c = lane & 7;
    int arrived = 0;
    for (int kt = 0; kt < nk; ++kt) {
      const int g = iter * nk + kt, s = g % kUStages;
      if (g >= kUStages) mbar_wait(bar_empty + 8 * s, ((g / kUStages) - 1) & 1, a.err);
      const uint32_t A = base + s * kStage;
      const int col = ((int)crank + kt * kUCluster) * kUK + c * 8;
#pragma unroll
      for (int rg = 0; rg < kUM / 16; ++rg) {
        const int row = rg * 16 + wl * 4 + (lane >> 3);
        const uint16_t *src = a.W + (size_t)s_rows[row] * a.H + col;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(A + row * 128 + ((c ^ (row & 7)) << 4)),
                     "l"(src)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      if (kt + 1 - arrived >= kInFlight) {  // the oldest pending stage has landed: publish it
        asm volatile("cp.async.wait_group %0;" ::"n"(kInFlight - 1) : "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(bar_full + 8 * ((iter * nk + arrived) % kUStages));
        ++arrived;
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (; arrived < nk; ++arrived) mbar_arrive(bar_full + 8 * ((iter * nk + arrived) % kUStages));
  } else if (warp == 1 && lane == 0) {
    bool ok = true;
    for (int kt = 0; kt < nk && ok; ++kt) {
      const int g = iter * nk + kt, s = g % kUStages;
      ok = mbar_wait(bar_full + 8 * s, (g / kUStages) & 1, a.err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t A = base + s * kStage;
#pragma unroll
      for (int kk = 0; kk < kUK / 16; ++kk)
        umma_bf16(tmem, sw128_desc(A + kk * 32), sw128_desc(A + kStageA + kk * 32), (kt | kk) != 0);
      umma_commit(bar_empty + 8 * s);
    }
    if (nk > 0 && ok) umma_commit(bar_acc);
    else mbar_arrive(bar_acc);
  } else if (!kInPlace && warp == 2 && lane == 0) {
    int released = 0;
    for (int kt = 0; kt < nk; ++kt) {
      const int g = iter * nk + kt, s = g % kUStages;
      if (!mbar_wait(bar_full + 8 * s, (g / kUStages) & 1, a.err)) break;
      if (kBatch)
        tma_store_3d(&tmP, base + s * kStage, ((int)crank + kt * kUCluster) * kUK, row0, bseq);
      else
        tma_store_2d(&tmP, base + s * kStage, ((int)crank + kt * kUCluster) * kUK, row0);
      bulk_commit();
      if (kt + 1 - released > kStoresInFlight) {  // the oldest store has read its stage
        asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kStoresInFlight) : "memory");
        mbar_arrive(bar_empty + 8 * ((iter * nk + released) % kUStages));
        ++released;
      }
    }
    bulk_wait_read_all();  // the ring may be reused; the global writes finish in the background
    for (; released < nk; ++released) mbar_arrive(bar_empty + 8 * ((iter * nk + released) % kUStages));
  }

  // ---- epilogue: accumulator -> partial tile in shared memory ---------------
  tc_fence_before();
  __syncthreads();  // every role is done with the ring (MMAs issued, packed stores have read it)
  float *P = reinterpret_cast<float *>(gbase);  // [64][128] partial of this CTA
  if (warp >= 4) {
    // tcgen05.ld is warp-collective: the whole warp takes the same branch
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_acc, iter & 1, a.err));
    tc_fence_after();
    const int j = (warp - 4) * 32 + lane;
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
      for (int q = 0; q < 16; ++q) P[(c + q) * kUM + j] = v[q];
    }
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();

  // ---- reduce hidden rows [8c, 8c+8) over the eight partials ---------------
  float *F = reinterpret_cast<float *>(gbase + kPartBytes);  // [8][128]
  if (tid < kSlice * (kUM / 4)) {
    const int rr = tid / (kUM / 4), j = (tid % (kUM / 4)) * 4;  // a float4 of the kSlice x 128 block each
    const uint32_t off = base + (uint32_t)(((crank * kSlice + rr) * kUM + j) * 4);
    float4 s4 = ld_peer_f4(map_peer(off, 0));
#pragma unroll
    for (uint32_t p = 1; p < kUCluster; ++p) {
      const float4 q = ld_peer_f4(map_peer(off, p));
      s4.x += q.x;
      s4.y += q.y;
      s4.z += q.z;
      s4.w += q.w;
    }
    *reinterpret_cast<float4 *>(F + rr * kUM + j) = s4;
  }
  __syncthreads();

  // ---- per-tile top-k of each row (one warp per hidden row) -----------------
  // Each lane sorts its four columns (value descending, then id ascending; I_t
  // is ascending, so ids ascend with the column), and k rounds of a warp-wide
  // best-of-heads write the tile's k best, best first, with global ids.
  const int r = (int)crank * kSlice + warp;
  const bool row_warp = warp < kSlice && r < a.n;
  if (row_warp) {
    uint32_t hk[4], hi[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane + 32 * q;
      const bool live = row0 + j < m && (!kInPlace || s_ids[j] >= 0);
      hk[q] = live ? order_key(F[warp * kUM + j]) : 0u;
      hi[q] = hk[q] != 0u ? (uint32_t)(kInPlace ? s_ids[j] : s_rows[j]) : (uint32_t)kEmptyId;
    }
    const size_t o = ((size_t)tile * kUN + r) * a.k;
    warp_topk4(hk, hi, a.k, cand_k + o, cand_i + o);
  }
  __syncthreads();  // every warp's candidates are written before the ticket is taken
  if (tid == 0) {   // release this CTA's candidates; the last CTA acquires everyone's
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(ticket + crank) : "memory");
    *s_flag = old == T - 1;
  }
  for (int i = tid; i < kSlice * kUM; i += kUThreads) {
    const int rr = i / kUM, j = i % kUM;
    const int rw = (int)crank * kSlice + rr, jg = row0 + j;
    if (rw < a.n && jg < m) logits[(size_t)rw * a.ld + jg] = F[i];
  }
  __syncthreads();
  if (*s_flag) {  // last tile of this row slice: merge every tile's sorted candidates
    if (tid == 0) ticket[crank] = 0;
    if (row_warp) {
      const int K = a.k;
      uint32_t *ep = reinterpret_cast<uint32_t *>(gbase + kPartBytes + kSlice * kUM * 4);
      uint32_t *Lk = ep + warp * 2 * kMergeWarpWords, *Li = Lk + kMergeWarpWords;
      uint32_t *Rk = ep + kSlice * 2 * kMergeWarpWords + warp * 2 * NS_MAX_TOPK, *Ri = Rk + NS_MAX_TOPK;
      for (int q = lane; q < K; q += kWarp) {
        Rk[q] = 0u;
        Ri[q] = (uint32_t)kEmptyId;
      }
      // up to kMergeLists tiles at a time, together with the running result
      for (int t0 = 0; t0 < T; t0 += kMergeLists) {
        const int nl = T - t0 < kMergeLists ? T - t0 : kMergeLists;
        // entry e = l * K + q (list l, rank q) goes to Lk/Li[e]; each lane
        // takes e = lane, lane + 32, ..., loading a batch before storing it
        const int ne = nl * K, dl = kWarp / K, dq = kWarp - dl * K;
        int l = lane / K, q = lane - (lane / K) * K;
        for (int e0 = 0; e0 < ne; e0 += kMergeBatch * kWarp) {
          uint32_t bk[kMergeBatch], bi[kMergeBatch];
#pragma unroll
          for (int b = 0; b < kMergeBatch; ++b) {
            if (e0 + b * kWarp + lane < ne) {
              const size_t src = ((size_t)(t0 + l) * kUN + r) * K + q;
              bk[b] = __ldcg(cand_k + src);
              bi[b] = __ldcg(cand_i + src);
            }
            q += dq;
            l += dl;
            if (q >= K) {
              q -= K;
              ++l;
            }
          }
#pragma unroll
          for (int b = 0; b < kMergeBatch; ++b) {
            const int e = e0 + b * kWarp + lane;
            if (e < ne) {
              Lk[e] = bk[b];
              Li[e] = bi[b];
            }
          }
        }
        for (int q = lane; q < K; q += kWarp) {
          Lk[nl * K + q] = Rk[q];
          Li[nl * K + q] = Ri[q];
        }
        __syncwarp();
        uint32_t lk, li;
        warp_merge_lists(Lk, Li, nl + 1, K, Rk, Ri, lk, li);
      }
      if (lane < K) {
        const uint32_t k = Rk[lane];
        out_ids[r * K + lane] = k != 0u ? (int)Ri[lane] : -1;
        out_vals[r * K + lane] = k != 0u ? key_value(k) : -__int_as_float(0x7f800000);
      }
    }
  }
  __syncwarp();
  cluster_sync();  // peers may still be reading this CTA's partial tile
  ++iter;
  }  // work items
  if (!kInPlace && warp == 2 && lane == 0) bulk_wait_all();  // the packed-buffer stores are complete before the CTA leaves
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---- host side ---------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2-D bf16 tensor [outer x inner] with rows of `inner` elements, 128-byte swizzle.
bool encode_bf16_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                    uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor [outer x mid x inner]: rows of `inner` elements, `mid` rows
// per block, blocks `outer_stride` bytes apart; 128-byte swizzle.
bool encode_bf16_3d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t mid, uint64_t outer,
                    uint64_t outer_stride, uint32_t box_inner, uint32_t box_mid) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * 2, outer_stride};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int umma_tiles(int W_max) { return (W_max + kUM - 1) / kUM; }
// Clusters of 16 CTAs halve each CTA's share of H (a shorter gather chain),
// but far fewer of them are resident at once than clusters of 8, and a tile
// that waits for a second wave costs more than the halved chain saves.  So a
// launch uses 16 only when every tile of W_max gets a resident cluster (by
// the occupancy query), else 8.  The grid has one cluster per tile of W_max;
// the kernel's tile loop also covers a grid of fewer clusters.
int g_max16 = 0, g_max8 = 0;  // resident clusters of each size, from prepare_umma_kernels

int umma_cluster() { return 16; }  // the most row slices a launch can use

// How many clusters of `CL` fused-kernel CTAs can be resident at once.
template <int CL>
int max_clusters() {
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
  if (cudaOccupancyMaxActiveClusters(&clusters, umma_step_kernel<CL, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

template <int CL, bool IN_PLACE, bool BATCH = false>
cudaError_t allow_umma() {
  cudaError_t e = cudaFuncSetAttribute(umma_step_kernel<CL, IN_PLACE, BATCH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kUSmem);
  if (e == cudaSuccess && CL > 8)
    e = cudaFuncSetAttribute(umma_step_kernel<CL, IN_PLACE, BATCH>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t prepare_umma_kernels() {
  cudaError_t e = allow_umma<8, false>();
  if (e == cudaSuccess) e = allow_umma<16, false>();
  if (e == cudaSuccess) e = allow_umma<8, true>();
  if (e == cudaSuccess) e = allow_umma<16, true>();
  if (e == cudaSuccess) e = allow_umma<8, false, true>();
  if (e == cudaSuccess) e = allow_umma<16, false, true>();
  if (e != cudaSuccess) return e;
  if (!encoder()) return cudaErrorNotSupported;
  g_max16 = max_clusters<16>();
  g_max8 = max_clusters<8>();
  return g_max16 > 0 || g_max8 > 0 ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t launch_umma_step(const UmmaLaunch &L, cudaStream_t st) {
  const bool batch = L.nseq > 1;
  if (L.in_place && batch) return cudaErrorInvalidValue;
  CUtensorMap tmH, tmP;
  const bool maps =
      batch ? encode_bf16_3d(&tmH, L.hid, L.H, L.n, L.nseq, (uint64_t)L.n * L.H * 2, kUK, kUN) &&
                  encode_bf16_3d(&tmP, L.packed, L.H, L.W_max, L.nseq, (uint64_t)L.seq_bytes, kUK, kUM)
            : encode_bf16_2d(&tmH, L.hid, L.H, L.n, kUK, kUN) && encode_bf16_2d(&tmP, L.packed, L.H, L.W_max, kUK, kUM);
  if (!maps) return cudaErrorInvalidValue;
  UmmaArgs a{};
  a.W = L.W;
  a.idx = L.idx;
  a.count_ptr = L.count_ptr;
  a.V = L.V;
  a.W_max = L.W_max;
  a.H = L.H;
  a.n = L.n;
  a.k = L.k;
  a.logits = L.logits;
  a.ld = L.ld;
  a.cand_k = L.cand_k;
  a.cand_i = L.cand_i;
  a.slice_ticket = L.slice_ticket;
  a.out_ids = L.out_ids;
  a.out_vals = L.out_vals;
  a.err = L.err;
  const int nseq = batch ? L.nseq : 1;
  a.seq_bytes = L.seq_bytes;
  a.logits_bytes = L.logits_bytes;
  a.nseq = nseq;
  a.tiles_per_seq = umma_tiles(L.W_max);
  a.rows_by_id = L.rows_by_id ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  // one cluster per tile of W_max; a batch gets as many 8-CTA clusters as are
  // resident at once, which loop over the work items (tiles of every sequence)
  int clusters = umma_tiles(L.W_max) * nseq;
  const int CL = clusters <= g_max16 || g_max8 == 0 ? 16 : 8;
  if (batch && CL == 8 && clusters > g_max8) clusters = g_max8;
  cfg.gridDim = dim3((unsigned)(clusters * CL));
  cfg.blockDim = dim3(kUThreads);
  cfg.dynamicSmemBytes = kUSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = L.programmatic ? 1 : 0;
  if (batch) {
    if (CL == 16) return cudaLaunchKernelEx(&cfg, umma_step_kernel<16, false, true>, tmH, tmP, a);
    return cudaLaunchKernelEx(&cfg, umma_step_kernel<8, false, true>, tmH, tmP, a);
  }
  if (L.in_place) {
    if (CL == 16) return cudaLaunchKernelEx(&cfg, umma_step_kernel<16, true>, tmH, tmP, a);
    return cudaLaunchKernelEx(&cfg, umma_step_kernel<8, true>, tmH, tmP, a);
  }
  if (CL == 16) return cudaLaunchKernelEx(&cfg, umma_step_kernel<16, false>, tmH, tmP, a);
  return cudaLaunchKernelEx(&cfg, umma_step_kernel<8, false>, tmH, tmP, a);
}

}  // namespace ns
