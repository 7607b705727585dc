// The tcgen05 tile of the sub-head product, shared by the kernels that run it
// (the fused gather + projection + top-k of ns_umma.cu and the one-launch
// decode step of ns_step.cu).
//
// Tile: 128 W_head rows (UMMA M) x 64 hidden rows (UMMA N, n <= 64), owned by
// one cluster of C CTAs that split H C ways; the 64-wide k slices are dealt
// round-robin (CTA c takes slices c, c+C, ...).  Per CTA and per k slice a
// 4-stage ring overlaps the roles:
//   * warps 4-7 gather the tile's 128 rows with 16-byte cp.async (four rows
//     of 128 contiguous bytes per warp instruction) into the 128-byte-
//     swizzled operand layout, fence the async proxy and arrive on the
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
// through distributed shared memory in a fixed order (deterministic), ranks
// each row's 128 columns (one warp per row) and writes those logits.  The
// per-tile candidates (sorted) of a row slice are merged by the last CTA of
// that slice to finish (release/acquire ticket) into the final top-k.
//
// Every wait is bounded (about a second); a wait that runs out sets
// NS_FLAG_TIMEOUT and the kernel still follows the same barrier sequence.
#pragma once

#include <cuda.h>

#include "ns_internal.cuh"
#include "ns_ptx.cuh"

namespace ns {
namespace {

constexpr int kUM = 128;                     // W rows per tile
constexpr int kUN = 64;                      // hidden rows per tile
constexpr int kUK = 64;                      // k per stage: one 128-byte swizzled row
constexpr int kUStages = 8;
constexpr int kUThreads = 384;
constexpr int kGatherThreads = 256;          // warps 4-11
constexpr int kGatherWarps = kGatherThreads / 32;
static_assert(kUM % (4 * kGatherWarps) == 0, "each gather warp instruction copies four 128-byte rows");
constexpr int kStoresInFlight = 1;           // packed-buffer stores still reading a stage
// A stage is released by the store issuer kStoresInFlight stores later; the
// gather threads wait for the release of the stage they reuse kUStages
// iterations on.
static_assert(kStoresInFlight <= kUStages - 1, "stage ring too short for the store lag");
constexpr int kStageA = kUM * kUK * 2;       // 16 KB
constexpr int kStageB = kUN * kUK * 2;       // 8 KB
constexpr int kStage = kStageA + kStageB;    // 24 KB (1024-byte multiple)
constexpr int kRingBytes = kUStages * kStage;
constexpr int kPartBytes = kUN * kUM * 4;    // one CTA's partial tile, [r][j] fp32
constexpr int kMiscBytes = 1280;             // barriers, TMEM slot, ticket flag, row ids, slot ids
constexpr int kUSmem = kRingBytes + kMiscBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 64;

constexpr int kMergeLists = 24;  // tiles' lists merged per round of the final merge (+ the running list)
constexpr int kMergeBatch = 8;   // candidate loads a lane keeps in flight while staging
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
  // batch strides in bytes: the row ids and their count (0 when the
  // sequences share one list) and the candidate lists and tickets; mask
  // (nullable): sequence 0's window bitmap, moved by mask_stride -- a row
  // whose id is outside a sequence's window is computed but not ranked for it
  long long idx_stride, cand_stride, mask_stride;
  const uint32_t *mask;
  int32_t rows_by_id;  // kInPlace: row j is W row idx[j] (an indexed product, nothing packed)
};

// Shared-memory carve-up of a CTA that runs tiles: the 1024-byte-aligned
// stage ring, its barriers, the tensor-memory slot, the last-tile flag and
// the tile's row ids.
struct UmmaSmem {
  uint32_t base;      // shared address of the stage ring (1024-byte aligned)
  uint8_t *gbase;     // the same, generic
  uint32_t bar_full, bar_empty, bar_acc;
  uint32_t *tmem_slot;
  int *s_flag;
  int *s_rows;        // [kUM] source rows of the tile (ids, or buffer rows)
  int *s_ids;         // [kUM] ids of the rows (in-place modes)
};

__device__ __forceinline__ UmmaSmem umma_smem(uint8_t *smem_raw) {
  UmmaSmem S;
  const uint32_t raw = smem_u32(smem_raw);
  S.base = (raw + 1023u) & ~1023u;  // 128-byte-swizzled tiles need 1024-byte alignment
  S.gbase = smem_raw + (S.base - raw);
  S.bar_full = S.base + kRingBytes;
  S.bar_empty = S.bar_full + 8 * kUStages;
  S.bar_acc = S.bar_empty + 8 * kUStages;
  S.tmem_slot = reinterpret_cast<uint32_t *>(S.gbase + kRingBytes + 16 * kUStages + 8);
  S.s_flag = reinterpret_cast<int *>(S.gbase + kRingBytes + 16 * kUStages + 16);
  S.s_rows = reinterpret_cast<int *>(S.gbase + kRingBytes + 256);
  S.s_ids = S.s_rows + kUM;
  return S;
}

// Top-k padding of an empty I_t, written by the CTAs of one cluster (each
// its own hidden rows): ids -1, values -inf.
template <int kUCluster>
__device__ __forceinline__ void umma_pad_topk(int32_t *out_ids, float *out_vals, int n, int k) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = (int)cluster_rank();
  const int r0 = (kUN * crank) / kUCluster, r1 = (kUN * (crank + 1)) / kUCluster;
  for (int r = r0 + warp; r < r1 && r < n; r += kUThreads / kWarp) {
    if (lane < k) {
      out_ids[r * k + lane] = -1;
      out_vals[r * k + lane] = -__int_as_float(0x7f800000);
    }
  }
}

// One thread: the ring's barriers (the TMA issuer and every gather thread
// fill a stage; the MMA commit, and in gather mode the packed-store issuer,
// release it).
__device__ __forceinline__ void umma_init_barriers(const UmmaSmem &S, bool in_place) {
  for (int s = 0; s < kUStages; ++s) {
    mbar_init(S.bar_full + 8 * s, 1 + kGatherThreads);
    mbar_init(S.bar_empty + 8 * s, in_place ? 1 : 2);
  }
  mbar_init(S.bar_acc, 1);
  mbar_fence_init();
}

// One tile (work item) of a cluster: main loop and epilogue.  s_rows (and
// s_ids in the in-place modes) hold the tile's rows, published by a
// __syncthreads.  `iter` counts the items this CTA ran before (the stage
// ring's slots and phases run on across items); nk = this CTA's k slices;
// row0 = tile * kUM; m = rows of the sequence (|I_t|), T = its tiles.  The
// sequence's candidate lists, ticket, logits and outputs are a's, moved by
// bseq sequences (kBatch).  Ends with a cluster barrier.
// kTopk: rank each row's tile columns and merge the tiles' lists into the
// top-k (the last tile of a row slice to finish merges).  Without it the
// tile only writes its logits, and the caller ranks the rows afterwards.
template <int kUCluster, bool kInPlace, bool kBatch, bool kTopk = true>
__device__ __forceinline__ void umma_tile(const UmmaSmem &S, uint32_t tmem, const CUtensorMap &tmH,
                                          const CUtensorMap &tmP, const UmmaArgs &a, int iter, int nk, int tile,
                                          int bseq, int m, int T) {
  constexpr int kRows = (kUN + kUCluster - 1) / kUCluster;  // most hidden rows one CTA reduces
  static_assert(kPartBytes + kRows * kUM * 4 + (kUThreads / kWarp) * 4 * (kMergeLists + 1) * NS_MAX_TOPK * 4 <=
                    kRingBytes,
                "epilogue buffers reuse the stage ring");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_rank();
  const uint32_t base = S.base, bar_full = S.bar_full, bar_empty = S.bar_empty, bar_acc = S.bar_acc;
  uint8_t *gbase = S.gbase;
  int *s_rows = S.s_rows, *s_ids = S.s_ids, *s_flag = S.s_flag;
  const long long so = bseq * a.cand_stride;
  uint32_t *cand_k = reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(a.cand_k) + so);
  uint32_t *cand_i = reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(a.cand_i) + so);
  int32_t *ticket = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(a.slice_ticket) + so);
  float *logits = reinterpret_cast<float *>(reinterpret_cast<char *>(a.logits) + bseq * a.logits_bytes);
  int32_t *out_ids = a.out_ids + (long long)bseq * a.n * a.k;
  float *out_vals = a.out_vals + (long long)bseq * a.n * a.k;
  const int row0 = tile * kUM;
  (void)s_ids;

  // ---- main loop -------------------------------------------------------------
  // In place, row j of the tile is row row0 + j of the buffer tmP maps, so the
  // rows of a stage are one tiled TMA load (the rows past |I_t| are loaded
  // too and never ranked); otherwise the gather warps copy them by id.
  const bool tma_rows = kInPlace && !a.rows_by_id;
  if (warp == 0 && lane == 0) {  // hidden slices (and, in place, the row tiles) by TMA
    int issued = 0;
    for (int kt = 0; kt < nk; ++kt) {
      const int g = iter * nk + kt, s = g % kUStages;
      if (g >= kUStages && !mbar_wait(bar_empty + 8 * s, ((g / kUStages) - 1) & 1, a.err)) break;
      issued = kt + 1;
      mbar_expect_tx(bar_full + 8 * s, tma_rows ? kStage : kStageB);
      if (tma_rows) tma_load_2d(base + s * kStage, &tmP, ((int)crank + kt * kUCluster) * kUK, row0, bar_full + 8 * s);
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
    // Each thread's copies of a stage arrive on the stage's "full" barrier by
    // themselves when they land (cp.async.mbarrier.arrive), so issuing runs
    // ahead as far as the ring allows; the consumers fence the async proxy.
    const int p = tid - 128, wl = p >> 5, c = lane & 7;  // warp wl of the gather warps
    for (int kt = 0; kt < nk; ++kt) {
      const int g = iter * nk + kt, s = g % kUStages;
      if (g >= kUStages) mbar_wait(bar_empty + 8 * s, ((g / kUStages) - 1) & 1, a.err);
      const uint32_t A = base + s * kStage;
      const int col = ((int)crank + kt * kUCluster) * kUK + c * 8;
      if (!tma_rows) {
#pragma unroll
        for (int rg = 0; rg < kUM / (4 * kGatherWarps); ++rg) {
          const int row = (rg * kGatherWarps + wl) * 4 + (lane >> 3);
          const uint16_t *src = a.W + (size_t)s_rows[row] * a.H + col;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(A + row * 128 + ((c ^ (row & 7)) << 4)),
                       "l"(src)
                       : "memory");
        }
      }
      // (with no copy of this thread in flight the arrival is immediate)
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar_full + 8 * s) : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // nothing of this thread is still landing
  } else if (warp == 1 && lane == 0) {
    bool ok = true;
    for (int kt = 0; kt < nk && ok; ++kt) {
      const int g = iter * nk + kt, s = g % kUStages;
      ok = mbar_wait(bar_full + 8 * s, (g / kUStages) & 1, a.err);
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
  } else if (!kInPlace && warp == 2 && lane == 0) {
    int released = 0;
    for (int kt = 0; kt < nk; ++kt) {
      const int g = iter * nk + kt, s = g % kUStages;
      if (!mbar_wait(bar_full + 8 * s, (g / kUStages) & 1, a.err)) break;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the gathered rows, for the TMA store
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
  if (warp >= 4 && warp < 8) {  // warp w reads TMEM lanes 32 (w % 4) .. +32
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

  // ---- reduce hidden rows [r0, r1) over the C partials ---------------------
  // CTA c of the cluster owns hidden rows [64c/C, 64(c+1)/C) (C need not
  // divide 64: the shares differ by at most one row).
  const int r0 = (kUN * (int)crank) / kUCluster, nr = (kUN * ((int)crank + 1)) / kUCluster - r0;
  float *F = reinterpret_cast<float *>(gbase + kPartBytes);  // [kRows][128]
  for (int t = tid; t < nr * (kUM / 4); t += kUThreads) {
    const int rr = t / (kUM / 4), j = (t % (kUM / 4)) * 4;  // a float4 of the nr x 128 block each
    const uint32_t off = base + (uint32_t)(((r0 + rr) * kUM + j) * 4);
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

  if (!kTopk) {  // logits only
    for (int i = tid; i < nr * kUM; i += kUThreads) {
      const int rr = i / kUM, j = i % kUM;
      const int rw = r0 + rr, jg = row0 + j;
      if (rw < a.n && jg < m) logits[(size_t)rw * a.ld + jg] = F[i];
    }
    __syncwarp();
    cluster_sync();  // peers may still be reading this CTA's partial tile
    return;
  }

  // ---- per-tile top-k of each row (a warp takes rows w and w + 8) ----------
  // Each lane sorts its four columns (value descending, then id ascending; I_t
  // is ascending, so ids ascend with the column), and k rounds of a warp-wide
  // best-of-heads give the tile's k best, best first, with global ids; a
  // warp's two rows run in lockstep so their rounds overlap.
  static_assert(kRows <= 2 * (kUThreads / kWarp), "a warp takes at most two hidden rows");
  const int rA = warp, rB = warp + kUThreads / kWarp;
  const bool hasA = rA < nr && r0 + rA < a.n, hasB = rB < nr && r0 + rB < a.n;
  if (hasA) {
    uint32_t ka[4], ia[4], kb[4], ib[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane + 32 * q;
      const bool live = row0 + j < m && (!kInPlace || s_ids[j] >= 0);
      const uint32_t id = (uint32_t)(kInPlace ? s_ids[j] : s_rows[j]);
      ka[q] = live ? order_key(F[rA * kUM + j]) : 0u;
      ia[q] = ka[q] != 0u ? id : (uint32_t)kEmptyId;
      kb[q] = live && hasB ? order_key(F[rB * kUM + j]) : 0u;
      ib[q] = kb[q] != 0u ? id : (uint32_t)kEmptyId;
    }
    uint32_t wa_k, wa_i, wb_k, wb_i;
    warp_topk4_pair(ka, ia, kb, ib, a.k, &wa_k, &wa_i, &wb_k, &wb_i);
    if (lane < a.k) {
      const size_t oa = ((size_t)tile * kUN + r0 + rA) * a.k + lane;
      cand_k[oa] = wa_k;
      cand_i[oa] = wa_i;
      if (hasB) {
        const size_t ob = ((size_t)tile * kUN + r0 + rB) * a.k + lane;
        cand_k[ob] = wb_k;
        cand_i[ob] = wb_i;
      }
    }
  }
  __syncthreads();  // every warp's candidates are written before the ticket is taken
  if (tid == 0) {   // release this CTA's candidates; the last CTA acquires everyone's
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(ticket + crank) : "memory");
    *s_flag = old == T - 1;
  }
  for (int i = tid; i < nr * kUM; i += kUThreads) {
    const int rr = i / kUM, j = i % kUM;
    const int rw = r0 + rr, jg = row0 + j;
    if (rw < a.n && jg < m) logits[(size_t)rw * a.ld + jg] = F[i];
  }
  __syncthreads();
  if (*s_flag) {  // last tile of this row slice: merge every tile's sorted candidates
    if (tid == 0) ticket[crank] = 0;
    if (hasA) {
      // Each warp merges its rows' lists, up to kMergeLists tiles at a time
      // together with the running result: it stages the lists in its own
      // shared-memory area (every load of a round issued before any store),
      // then k rounds of best-of-heads per row, the two rows in lockstep.
      const int K = a.k;
      constexpr int kL = kMergeLists + 1;
      uint32_t *wk0 = reinterpret_cast<uint32_t *>(gbase + kPartBytes + kRows * kUM * 4) + warp * 4 * kL * NS_MAX_TOPK;
      uint32_t *wi0 = wk0 + kL * NS_MAX_TOPK, *wk1 = wi0 + kL * NS_MAX_TOPK, *wi1 = wk1 + kL * NS_MAX_TOPK;
      uint32_t rka = 0u, ria = (uint32_t)kEmptyId, rkb = 0u, rib = (uint32_t)kEmptyId;  // lane q: entry q
      const int dl = kWarp / K, dq = kWarp - dl * K;
      for (int t0 = 0; t0 < T; t0 += kMergeLists) {
        const int nl = T - t0 < kMergeLists ? T - t0 : kMergeLists;
        const int ne = nl * K;
        int l = lane / K, q = lane - (lane / K) * K;  // entry e = l * K + q
        for (int e0 = 0; e0 < ne; e0 += kMergeBatch * kWarp) {
          uint32_t bka[kMergeBatch], bia[kMergeBatch], bkb[kMergeBatch], bib[kMergeBatch];
#pragma unroll
          for (int b2 = 0; b2 < kMergeBatch; ++b2) {
            if (e0 + b2 * kWarp + lane < ne) {
              const size_t src = ((size_t)(t0 + l) * kUN + r0 + rA) * K + q;
              bka[b2] = __ldcg(cand_k + src);
              bia[b2] = __ldcg(cand_i + src);
              if (hasB) {
                const size_t srb = src + (size_t)(rB - rA) * K;
                bkb[b2] = __ldcg(cand_k + srb);
                bib[b2] = __ldcg(cand_i + srb);
              }
            }
            q += dq;
            l += dl;
            if (q >= K) {
              q -= K;
              ++l;
            }
          }
#pragma unroll
          for (int b2 = 0; b2 < kMergeBatch; ++b2) {
            const int e = e0 + b2 * kWarp + lane;
            if (e < ne) {
              wk0[e] = bka[b2];
              wi0[e] = bia[b2];
              if (hasB) {
                wk1[e] = bkb[b2];
                wi1[e] = bib[b2];
              }
            }
          }
        }
        if (lane < K) {  // the running result is list nl
          wk0[ne + lane] = rka;
          wi0[ne + lane] = ria;
          wk1[ne + lane] = rkb;
          wi1[ne + lane] = rib;
        }
        __syncwarp();
        int pa = 0, pb = 0;
#pragma unroll 1
        for (int r = 0; r < K; ++r) {
          uint32_t hka = 0u, hia = (uint32_t)kEmptyId, hkb = 0u, hib = (uint32_t)kEmptyId;
          if (lane <= nl) {
            if (pa < K) {
              hka = wk0[lane * K + pa];
              hia = wi0[lane * K + pa];
            }
            if (hasB && pb < K) {
              hkb = wk1[lane * K + pb];
              hib = wi1[lane * K + pb];
            }
          }
          uint32_t ta, tia, tb, tib;
          warp_best(hka, hia, ta, tia);
          warp_best(hkb, hib, tb, tib);
          if (lane == r) {
            rka = ta;
            ria = tia;
            rkb = tb;
            rib = tib;
          }
          if (ta != 0u && hka == ta && hia == tia) ++pa;
          if (tb != 0u && hkb == tb && hib == tib) ++pb;
        }
        __syncwarp();
      }
      if (lane < K) {
        const int ra = r0 + rA;
        out_ids[ra * K + lane] = rka != 0u ? (int)ria : -1;
        out_vals[ra * K + lane] = rka != 0u ? key_value(rka) : -__int_as_float(0x7f800000);
        if (hasB) {
          const int rb = r0 + rB;
          out_ids[rb * K + lane] = rkb != 0u ? (int)rib : -1;
          out_vals[rb * K + lane] = rkb != 0u ? key_value(rkb) : -__int_as_float(0x7f800000);
        }
      }
    }
  }
  __syncwarp();
  cluster_sync();  // peers may still be reading this CTA's partial tile
}

}  // namespace

// 2-D bf16 tensor map [outer x inner] (rows of `inner` elements), box
// box_inner x box_outer, 128-byte swizzle (ns_umma.cu).
bool encode_bf16_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                    uint32_t box_outer);

}  // namespace ns
