// Fused sub-head step on the 5th-generation tensor cores: gather of
// W_head[I_t, :] into the packed buffer, projection of the draft hidden
// states through it, and per-row top-k remapped to global ids
// (MicroSpec §3.3 gathering into a contiguous buffer + dense product; §3.1
// Eq. 1 restricted to the active rows).  The tile itself (roles, stage ring,
// cluster reduce, top-k) is in ns_umma_tile.cuh; this file holds the kernel
// that walks a sequence's (or a batch's) tiles after the state update, and
// its host side.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ns_umma_tile.cuh"

namespace ns {
namespace {

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
// (a tile of a sequence), see below.  kBatch with kInPlace: every sequence
// projects the same buffer (the union of the sequences' active rows), and
// ranks only the rows its own window holds (a.mask).
template <int kUCluster, bool kInPlace, bool kBatch = false>
__global__ void __cluster_dims__(kUCluster, 1, 1) __launch_bounds__(kUThreads, 1)
    umma_step_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmP,
                     UmmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const UmmaSmem S = umma_smem(smem_raw);
  int *s_rows = S.s_rows, *s_ids = S.s_ids;

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
    umma_init_barriers(S, kInPlace);
  }
  if (warp == 1) tmem_alloc(smem_u32(S.tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *S.tmem_slot;

  grid_dependency_wait();  // I_t and |I_t| come from the state update
  // The first tile's row ids load together with |I_t| (one round trip); the
  // entries past |I_t| are not used.
  int id_first = 0, m0 = 0, T0 = 0;
  if (kBatch) {
    const int t0 = cid / a.nseq, b0 = cid % a.nseq;
    const int32_t *idx0 = reinterpret_cast<const int32_t *>(reinterpret_cast<const char *>(a.idx) + b0 * a.idx_stride);
    if (tid < kUM && t0 * kUM + tid < a.W_max) id_first = idx0[t0 * kUM + tid];
    if (tid < a.nseq)
      s_cnt[tid] = *reinterpret_cast<const int32_t *>(reinterpret_cast<const char *>(a.count_ptr) + tid * a.idx_stride);
    __syncthreads();
  } else {
    if (tid < kUM && cid * kUM + tid < a.W_max) id_first = a.idx[cid * kUM + tid];
    m0 = *a.count_ptr;
    T0 = (m0 + kUM - 1) / kUM;
    if (cid >= T0) {  // uniform across the cluster
      if (T0 == 0 && cid == 0) umma_pad_topk<kUCluster>(a.out_ids, a.out_vals, a.n, a.k);
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
  const int32_t *idx = reinterpret_cast<const int32_t *>(reinterpret_cast<const char *>(a.idx) + bseq * a.idx_stride);
  const uint32_t *mask =
      a.mask ? reinterpret_cast<const uint32_t *>(reinterpret_cast<const char *>(a.mask) + bseq * a.mask_stride)
             : nullptr;
  int32_t *out_ids = a.out_ids + (long long)bseq * a.n * a.k;
  float *out_vals = a.out_vals + (long long)bseq * a.n * a.k;
  if (kBatch && tile >= T) {  // uniform across the cluster
    if (T == 0 && tile == 0) umma_pad_topk<kUCluster>(out_ids, out_vals, a.n, a.k);  // an empty I_t: padding only
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
        if (mask && id >= 0 && !((mask[id >> 5] >> (id & 31)) & 1u)) id = -1;  // not this sequence's
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

  umma_tile<kUCluster, kInPlace, kBatch>(S, tmem, tmH, tmP, a, iter, nk, tile, bseq, m, T);
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

int umma_tiles(int W_max) { return (W_max + kUM - 1) / kUM; }

// A kernel that allocates tensor memory runs one CTA per SM, so how many
// clusters are resident at once depends on the cluster size and on how the
// GPCs' SMs divide by it.  A launch takes the size that runs its work items
// (tiles) in the fewest waves, then the largest (a smaller share of H per
// CTA); the grid holds at most the resident clusters, which loop over the
// items.
constexpr int kClusterSizes[] = {16, 8, 6, 5, 4};
constexpr int kNumClusterSizes = 5;
int g_maxcl[kNumClusterSizes] = {0, 0, 0, 0, 0};  // resident clusters of each size (prepare_umma_kernels)

int umma_cluster() { return 16; }  // the most row slices a launch can use

template <int CL, bool IN_PLACE, bool BATCH>
cudaError_t allow_umma() {
  static_assert(CL <= 16, "cluster size");
  cudaError_t e = cudaFuncSetAttribute(umma_step_kernel<CL, IN_PLACE, BATCH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kUSmem);
  if (e == cudaSuccess && CL > 8)
    e = cudaFuncSetAttribute(umma_step_kernel<CL, IN_PLACE, BATCH>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

// How many clusters of `CL` fused-kernel CTAs can be resident at once.
template <int CL>
int max_clusters() {
  if (allow_umma<CL, false, false>() != cudaSuccess || allow_umma<CL, true, false>() != cudaSuccess ||
      allow_umma<CL, false, true>() != cudaSuccess || allow_umma<CL, true, true>() != cudaSuccess) {
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
  if (cudaOccupancyMaxActiveClusters(&clusters, umma_step_kernel<CL, false, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

template <int CL>
cudaError_t launch_cl(cudaLaunchConfig_t &cfg, bool in_place, bool batch, const CUtensorMap &tmH,
                      const CUtensorMap &tmP, const UmmaArgs &a) {
  cfg.gridDim = dim3(cfg.gridDim.x * CL);
  if (batch && in_place) return cudaLaunchKernelEx(&cfg, umma_step_kernel<CL, true, true>, tmH, tmP, a);
  if (batch) return cudaLaunchKernelEx(&cfg, umma_step_kernel<CL, false, true>, tmH, tmP, a);
  if (in_place) return cudaLaunchKernelEx(&cfg, umma_step_kernel<CL, true, false>, tmH, tmP, a);
  return cudaLaunchKernelEx(&cfg, umma_step_kernel<CL, false, false>, tmH, tmP, a);
}

cudaError_t prepare_umma_kernels() {
  if (!encoder()) return cudaErrorNotSupported;
  g_maxcl[0] = max_clusters<16>();
  g_maxcl[1] = max_clusters<8>();
  g_maxcl[2] = max_clusters<6>();
  g_maxcl[3] = max_clusters<5>();
  g_maxcl[4] = max_clusters<4>();
  for (int i = 0; i < kNumClusterSizes; ++i)
    if (g_maxcl[i] > 0) return cudaSuccess;
  return cudaErrorNotSupported;
}

int pick_cluster_size(int items, int *clusters) {
  int best = -1, best_waves = 0;
  for (int i = 0; i < kNumClusterSizes; ++i) {
    if (g_maxcl[i] <= 0) continue;
    const int waves = (items + g_maxcl[i] - 1) / g_maxcl[i];
    if (best < 0 || waves < best_waves) {
      best = i;
      best_waves = waves;
    }
  }
  if (best < 0) return 0;
  *clusters = items < g_maxcl[best] ? items : g_maxcl[best];
  return kClusterSizes[best];
}

cudaError_t launch_umma_step(const UmmaLaunch &L, cudaStream_t st) {
  const bool batch = L.nseq > 1 || L.mask != nullptr;
  if (L.in_place && batch && L.mask == nullptr) return cudaErrorInvalidValue;  // only the union mode
  CUtensorMap tmH, tmP;
  // in place, nothing is stored: the packed map only needs to be valid
  const bool maps =
      batch ? encode_bf16_3d(&tmH, L.hid, L.H, L.n, L.nseq, (uint64_t)L.n * L.H * 2, kUK, kUN) &&
                  (L.in_place ? encode_bf16_2d(&tmP, L.packed, L.H, L.W_max, kUK, kUM)
                              : encode_bf16_3d(&tmP, L.packed, L.H, L.W_max, L.nseq, (uint64_t)L.seq_bytes, kUK, kUM))
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
  a.idx_stride = L.mask ? 0 : L.seq_bytes;  // the union mode: one row-id list for every sequence
  a.cand_stride = L.cand_stride ? L.cand_stride : L.seq_bytes;
  a.mask = L.mask;
  a.mask_stride = L.seq_bytes;
  a.logits_bytes = L.logits_bytes;
  a.nseq = nseq;
  a.tiles_per_seq = umma_tiles(L.W_max);
  a.rows_by_id = L.rows_by_id ? 1 : 0;
  int clusters = 0;
  const int CL = pick_cluster_size(umma_tiles(L.W_max) * nseq, &clusters);
  if (CL == 0) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)clusters);  // times CL in launch_cl
  cfg.blockDim = dim3(kUThreads);
  cfg.dynamicSmemBytes = kUSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = L.programmatic ? 1 : 0;
  switch (CL) {
    case 16: return launch_cl<16>(cfg, L.in_place, batch, tmH, tmP, a);
    case 8: return launch_cl<8>(cfg, L.in_place, batch, tmH, tmP, a);
    case 6: return launch_cl<6>(cfg, L.in_place, batch, tmH, tmP, a);
    case 5: return launch_cl<5>(cfg, L.in_place, batch, tmH, tmP, a);
    default: return launch_cl<4>(cfg, L.in_place, batch, tmH, tmP, a);
  }
}

}  // namespace ns
