// Slot-stable packed buffer: the incremental reading of NanoSpec's
// "Avoiding Sparse Computation via Asynchronous Gathering" paragraph, where
// only the weights of newly active tokens are gathered into the pre-allocated
// contiguous buffer.
//
// The pages give no slot rule; the one used here: a slot whose id left I_t is
// freed, then the ids of I_t that hold no slot take the free slots in
// ascending id order, lowest slot first.  An id keeps its slot (and its row
// stays in place) for as long as it stays active, so a decode step copies
// only |I_t \ I_{t-1}| rows (at most the ids one append brings in), instead
// of the |I_t| rows of a full repack.  The first update after the stream is
// initialised lays I_1 out ascending, the layout of the full repack.
//
// State per sequence: slot_id[W_max] (the id a slot holds, -1 = free), the
// bitmap `held` of ids holding a slot, slot_meta = {high-water mark, rows
// gathered by the last update} and the (slot, id) list of those rows.  After
// an update exactly the active ids hold slots, so `held` is the window
// bitmap as of the last update: an id of I_t is new iff its `held` bit is
// clear, and a slot is freed iff the window bitmap lost its id.
#include "ns_internal.cuh"

namespace ns {
namespace {

constexpr int kSlotThreads = 1024;
constexpr int kCopyThreads = 256;
constexpr int kCopyUnits = 4;  // 16-byte loads a lane keeps in flight

__device__ __forceinline__ bool has_bit(const uint32_t *w, int id) { return (w[id >> 5] >> (id & 31)) & 1u; }

// One CTA.  Reads I_t, |I_t| and the window bitmap; updates slot_id, held,
// slot_meta and the list of rows to gather (new_slot / new_id), and the
// state the one-launch slot step keeps besides: the slot of each placed id
// (slot_of), the free-slot bitmap and the |S| the table now matches.
__global__ void __launch_bounds__(kSlotThreads) slot_update_kernel(SeqDev s, Dims d, uint32_t *err) {
  extern __shared__ uint4 s_dyn4[];  // the window bitmap, then `held` (nwords_pad words each)
  __shared__ int sh[kSlotThreads / kWarp];
  __shared__ int s_hw;
  uint32_t *s_win = reinterpret_cast<uint32_t *>(s_dyn4);
  uint32_t *s_held = s_win + d.nwords_pad;
  const int tid = threadIdx.x, nq = d.nwords_pad / 4;
  const uint4 *w4 = reinterpret_cast<const uint4 *>(s.bitmap);
  const uint4 *h4 = reinterpret_cast<const uint4 *>(s.held);
  for (int q = tid; q < nq; q += blockDim.x) {
    s_dyn4[q] = w4[q];
    s_dyn4[nq + q] = h4[q];
  }
  if (tid == 0) s_hw = 0;
  int m = *s.count;
  if (m < 0 || m > d.W_max) {  // I_t never holds more than W_max ids
    if (tid == 0) set_flag(err, NS_FLAG_OVERFLOW);
    m = m < 0 ? 0 : d.W_max;
  }
  __syncthreads();

  // 1. how many ids of I_t hold no slot
  int n_new = 0;
  for (int j0 = 0; j0 < m; j0 += blockDim.x) {
    const int j = j0 + tid;
    bool fresh = false;
    if (j < m) {
      const int id = s.active[j];
      fresh = (unsigned)id < (unsigned)d.V && !has_bit(s_held, id);
    }
    n_new += __syncthreads_count(fresh);
  }

  // 2. free the slots whose id left the window; list the lowest n_new free
  //    slots, ascending, in new_slot
  int hw = 0, nfree = 0;
  for (int s0 = 0; s0 < d.W_max; s0 += blockDim.x) {
    const int sl = s0 + tid;
    bool is_free = false;
    if (sl < d.W_max) {
      const int id = s.slot_id[sl];
      if (id >= 0 && (id >= d.V || !has_bit(s_win, id))) {
        if (id >= d.V) set_flag(err, NS_FLAG_INTERNAL | (5u << 8));
        s.slot_id[sl] = -1;
        is_free = true;
      } else {
        is_free = id < 0;
      }
      if (!is_free) hw = sl + 1;
    }
    int total;
    const int rank = nfree + block_exclusive_scan(is_free ? 1 : 0, sh, &total);
    if (is_free && rank < n_new) s.new_slot[rank] = sl;
    nfree += total;
  }
  if (n_new > nfree) {  // more active ids than slots: cannot happen while |I_t| <= W_max
    if (tid == 0) set_flag(err, NS_FLAG_OVERFLOW);
    n_new = nfree;
  }
  atomicMax(&s_hw, hw);
  __syncthreads();  // new_slot[] (global, this block) is visible to every thread

  // 3. the ids without a slot, in I_t's ascending order, take new_slot[0..n_new)
  int placed = 0;
  for (int j0 = 0; j0 < m; j0 += blockDim.x) {
    const int j = j0 + tid;
    int id = -1;
    bool fresh = false;
    if (j < m) {
      id = s.active[j];
      fresh = (unsigned)id < (unsigned)d.V && !has_bit(s_held, id);
    }
    int total;
    const int rank = placed + block_exclusive_scan(fresh ? 1 : 0, sh, &total);
    if (fresh && rank < n_new) {
      const int sl = s.new_slot[rank];
      s.slot_id[sl] = id;
      s.slot_of[id] = sl;
      s.new_id[rank] = id;
    }
    placed += total;
  }
  __syncthreads();  // the table is final (global, this block)

  // the free-slot bitmap of the final table: warp w of a round covers 32
  // consecutive slots, one word
  const int nfw = slot_words(d.W_max);
  for (int s0 = 0; s0 < 32 * nfw; s0 += blockDim.x) {
    const int sl = s0 + tid;
    const bool is_free = sl < d.W_max && s.slot_id[sl] < 0;
    const unsigned word = __ballot_sync(0xffffffffu, is_free);
    if ((tid & (kWarp - 1)) == 0 && sl < 32 * nfw) s.slot_free[sl >> 5] = word;
  }

  // 4. held := the window bitmap; the high-water mark and the row count
  uint4 *ho = reinterpret_cast<uint4 *>(s.held);
  for (int q = tid; q < nq; q += blockDim.x) ho[q] = s_dyn4[q];
  if (tid == 0) {
    int top = s_hw;
    if (n_new > 0 && s.new_slot[n_new - 1] + 1 > top) top = s.new_slot[n_new - 1] + 1;
    s.slot_meta[0] = top;
    s.slot_meta[1] = n_new;
    *s.slot_len = s.length[0];
  }
}

// slot_rows[new_slot[i], :] = W[new_id[i], :] for i < slot_meta[1].  The rows
// are cut into 16-byte chunks numbered row-major; each warp copies 128
// consecutive chunks per round, four loads per lane in flight.
__global__ void __launch_bounds__(kCopyThreads) slot_copy_kernel(SeqDev s, Dims d, const uint16_t *W, uint32_t *err) {
  // a programmatically launched projection may start its prologue; it waits
  // for this grid to finish before it reads the slot buffer
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int n = s.slot_meta[1];
  const int upr = d.H >> 3;  // 16-byte chunks per row
  const long long total = (long long)n * upr;
  const int lane = threadIdx.x & (kWarp - 1);
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  constexpr int kChunk = kWarp * kCopyUnits;
  for (long long c0 = gw * kChunk; c0 < total; c0 += nw * kChunk) {
    uint4 v[kCopyUnits];
    int dst[kCopyUnits], col[kCopyUnits];
#pragma unroll
    for (int q = 0; q < kCopyUnits; ++q) {
      const long long c = c0 + lane + kWarp * q;
      dst[q] = -1;
      if (c < total) {
        const int r = (int)(c / upr);
        col[q] = (int)(c - (long long)r * upr);
        const int id = s.new_id[r], sl = s.new_slot[r];
        if ((unsigned)id < (unsigned)d.V && (unsigned)sl < (unsigned)d.W_max) {
          dst[q] = sl;
          v[q] = __ldcs(reinterpret_cast<const uint4 *>(W + (size_t)id * d.H) + col[q]);
        } else if (col[q] == 0) {
          set_flag(err, NS_FLAG_INTERNAL | (6u << 8));
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kCopyUnits; ++q)
      if (dst[q] >= 0) reinterpret_cast<uint4 *>(s.slot_rows + (size_t)dst[q] * d.H)[col[q]] = v[q];
  }
}

}  // namespace

cudaError_t prepare_slot_kernels(const Dims &d) {
  return cudaFuncSetAttribute(slot_update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              2 * d.nwords_pad * 4);
}

cudaError_t launch_slot_update(const SeqDev &s, const Dims &d, const uint16_t *W, int copy_grid, uint32_t *err,
                               cudaStream_t st) {
  slot_update_kernel<<<1, kSlotThreads, (size_t)2 * d.nwords_pad * 4, st>>>(s, d, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  slot_copy_kernel<<<copy_grid, kCopyThreads, 0, st>>>(s, d, W, err);
  return cudaGetLastError();
}

}  // namespace ns
