// C ABI of the dynamic-vocabulary draft LM head (declared in include/nanospec.h).
//
// The handle owns one device allocation holding every sequence's state
// (MicroSpec §3.3: all window state resident in VRAM, a pre-allocated
// contiguous buffer for the packed sub-head) plus scratch.  Calls validate
// their arguments on the host, then only enqueue kernels on the caller's
// stream: no host synchronisation and no allocation after ns_create.
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "ns_internal.cuh"

struct ns_handle {
  ns_config cfg;
  ns::Dims dims;
  int device = 0;
  int num_sms = 0;
  int ggrid = 1;  // CTAs of the gather
  int sgrid = 1;  // CTAs of the slot-row copy
  char *base = nullptr;
  size_t bytes = 0;
  uint32_t *err = nullptr;
  std::vector<ns::SeqDev> seqs;
  std::vector<char> inited;
  float *dense_logits = nullptr;  // [kProjBN x dense_ld]
  uint32_t *dense_cand_k = nullptr;  // [NS_MAX_ROWS x topk slices of V x NS_MAX_TOPK] slices' top-k lists
  uint32_t *dense_cand_i = nullptr;
  int dense_ld = 0;
  int step_clusters = 0;  // clusters of the one-launch step (0: two launches)
  int step_tpc = 0;       // tiles per cluster of the one-launch step
  int step_cl = 0;        // CTAs per cluster of the one-launch step
  int slot_clusters = 0;  // the same for the one-launch slot-stable step (0: the multi-launch chain)
  int slot_tpc = 0;
  int slot_cl = 0;
  // per sequence: the slot table matches the window (the calls enqueued so
  // far end with a slot update; any later change of the window clears it)
  std::vector<char> slots_synced;
  // union of the sequences' active vocabularies (batch > 1): its bitmap, ids
  // and count, the packed rows W_head[U, :], logits scratch and, per
  // sequence, candidate lists and tickets of the union projection
  long long u_cap = 0;  // most union rows: min(batch * W_max, V)
  int u_ld = 0;
  uint32_t *u_bitmap = nullptr;
  int32_t *u_ids = nullptr, *u_count = nullptr;
  uint16_t *u_packed = nullptr;
  float *u_logits = nullptr;
  uint32_t *u_cand = nullptr;
  long long u_cand_words = 0;   // one candidate array of one sequence
  long long u_block_words = 0;  // one sequence's block: keys, ids, tickets
  cudaEvent_t trace[4] = {nullptr, nullptr, nullptr, nullptr};
  bool tracing = false;
  // device staging of ns_step_host: tree ids, verify row, hidden rows, top-k
  int32_t *st_tree = nullptr;
  float *st_verify = nullptr;
  uint16_t *st_hidden = nullptr;
  int32_t *st_ids = nullptr;
  float *st_vals = nullptr;
  long long seq_bytes = 0;  // distance between consecutive sequences' state
};

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxV = 524288;  // one CTA compacts the bitmap (4 uint4 words per thread)
constexpr int kMaxH = 8192;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Two passes over the same layout: the first (base == nullptr) only sums sizes.
struct Carver {
  char *base;
  size_t off = 0;
  explicit Carver(char *b) : base(b) {}
  template <typename T>
  T *take(size_t count) {
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += align_up(count * sizeof(T) + (count == 0 ? 1 : 0));
    return p;
  }
};

void layout(ns_handle *h, Carver &cv) {
  const ns_config &c = h->cfg;
  const ns::Dims &d = h->dims;
  h->err = cv.take<uint32_t>(1);
  h->seqs.assign(c.batch, ns::SeqDev{});
  for (int b = 0; b < c.batch; ++b) {
    ns::SeqDev &s = h->seqs[b];
    s.ring = cv.take<int32_t>(c.W_max);
    s.counts = cv.take<uint32_t>(c.V);
    s.bitmap = cv.take<uint32_t>(d.nwords_pad);
    s.active = cv.take<int32_t>(c.W_max);
    s.count = cv.take<int32_t>(1);
    s.length = cv.take<long long>(2);
    s.active_len = cv.take<long long>(1);
    s.packed = cv.take<uint16_t>((size_t)c.W_max * c.H);
    s.logits = cv.take<float>((size_t)ns::kProjBN * d.ld_scratch);
    s.first = c.K_pre > 0 ? cv.take<int32_t>(c.V) : nullptr;
    s.cand = c.K_pre > 0 ? cv.take<int32_t>((size_t)c.max_prompt * c.K_pre) : nullptr;
    s.sinit = cv.take<int32_t>((size_t)c.max_prompt * (1 + c.K_pre));
    const size_t ncand = (size_t)ns::umma_tiles(c.W_max) * ns::kProjBN * c.max_k;
    s.cand_k = cv.take<uint32_t>(ncand);
    s.cand_i = cv.take<uint32_t>(ncand);
    s.slice_ticket = cv.take<int32_t>(ns::umma_cluster());
    s.slot_id = cv.take<int32_t>(c.W_max);
    s.held = cv.take<uint32_t>(d.nwords_pad);
    s.slot_meta = cv.take<int32_t>(2);
    s.new_slot = cv.take<int32_t>(c.W_max);
    s.new_id = cv.take<int32_t>(c.W_max);
    s.slot_rows = cv.take<uint16_t>((size_t)c.W_max * c.H);
    s.slot_of = cv.take<int32_t>(c.V);
    s.slot_free = cv.take<uint32_t>(ns::slot_words(c.W_max));
    s.slot_len = cv.take<long long>(1);
    s.gbar = cv.take<unsigned long long>(1);
    s.vcand_k = cv.take<uint32_t>((size_t)ns::kMaxStepCtas * (c.K_ver > 0 ? c.K_ver : 1));
    s.vcand_i = cv.take<uint32_t>((size_t)ns::kMaxStepCtas * (c.K_ver > 0 ? c.K_ver : 1));
  }
  if (c.batch > 1) {
    const long long cap = (long long)c.batch * c.W_max;
    h->u_cap = cap < c.V ? cap : c.V;
    h->u_ld = (int)((h->u_cap + 3) & ~3LL);
    h->u_bitmap = cv.take<uint32_t>(d.nwords_pad);
    h->u_ids = cv.take<int32_t>((size_t)h->u_cap);
    h->u_count = cv.take<int32_t>(1);
    h->u_packed = cv.take<uint16_t>((size_t)h->u_cap * c.H);
    h->u_logits = cv.take<float>((size_t)c.batch * ns::kProjBN * h->u_ld);
    h->u_cand_words = (long long)ns::umma_tiles((int)h->u_cap) * ns::kProjBN * c.max_k;
    h->u_block_words = ((2 * h->u_cand_words + ns::umma_cluster()) + 63) & ~63LL;
    h->u_cand = cv.take<uint32_t>((size_t)c.batch * h->u_block_words);
  }
  h->dense_ld = (c.V + 3) & ~3;
  h->dense_logits = cv.take<float>((size_t)ns::kProjBN * h->dense_ld);
  h->st_tree = cv.take<int32_t>(c.max_tree > 0 ? c.max_tree : 1);
  h->st_verify = cv.take<float>(c.K_ver > 0 ? c.V : 1);
  h->st_hidden = cv.take<uint16_t>((size_t)NS_MAX_ROWS * c.H);
  h->st_ids = cv.take<int32_t>((size_t)NS_MAX_ROWS * c.max_k);
  h->st_vals = cv.take<float>((size_t)NS_MAX_ROWS * c.max_k);
  const size_t ncand = (size_t)NS_MAX_ROWS * ns::topk_slices(c.V) * NS_MAX_TOPK;
  h->dense_cand_k = cv.take<uint32_t>(ncand);
  h->dense_cand_i = cv.take<uint32_t>(ncand);
}

bool valid_seq(const ns_handle *h, int32_t seq) { return h && seq >= 0 && seq < h->cfg.batch; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
ns_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NS_OK : NS_ERR_CUDA; }

}  // namespace

extern "C" {

const char *ns_status_string(ns_status s) {
  switch (s) {
    case NS_OK: return "ok";
    case NS_ERR_ARG: return "invalid argument";
    case NS_ERR_CUDA: return "CUDA error";
    case NS_ERR_OOM: return "out of device memory";
    case NS_ERR_TIMEOUT: return "device wait timed out";
    case NS_ERR_STATE: return "call out of order";
    default: return "unknown status";
  }
}

ns_status ns_create(const ns_config *cfg, ns_handle **out) {
  if (!cfg || !out) return NS_ERR_ARG;
  *out = nullptr;
  const ns_config c = *cfg;
  if (c.V < 1 || c.V > kMaxV || c.H < 64 || c.H > kMaxH || c.H % 64 != 0 || c.W_max < 1 ||
      c.W_max > (1 << 20) || c.K_pre < 0 || c.K_pre > NS_MAX_SELECT_K || c.K_pre > c.V || c.K_ver < 0 ||
      c.K_ver > NS_MAX_SELECT_K || c.K_ver > c.V || c.max_tree < 0 || c.max_tree > NS_MAX_ROWS || c.max_k < 1 ||
      c.max_k > NS_MAX_TOPK || c.batch < 1 || c.batch > 4096 || c.max_prompt < 1 || c.max_prompt > (1 << 20))
    return NS_ERR_ARG;
  ns_handle *h = new (std::nothrow) ns_handle();
  if (!h) return NS_ERR_OOM;
  h->cfg = c;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
      ns::prepare_umma_kernels() != cudaSuccess ||
      ns::prepare_step_kernel() != cudaSuccess || ns::prepare_dense_kernel() != cudaSuccess) {
    delete h;
    return NS_ERR_CUDA;
  }
  ns::Dims &d = h->dims;
  d.V = c.V;
  d.H = c.H;
  d.W_max = c.W_max;
  d.K_pre = c.K_pre;
  d.K_ver = c.K_ver;
  d.nwords = (c.V + 31) / 32;
  d.nwords_pad = (d.nwords + 3) & ~3;
  d.ld_scratch = (c.W_max + 3) & ~3;
  if (ns::prepare_state_kernels(&d) != cudaSuccess || ns::prepare_slot_kernels(d) != cudaSuccess) {
    delete h;
    return NS_ERR_CUDA;
  }
  h->ggrid = 4 * h->num_sms;
  h->sgrid = 2 * h->num_sms;

  Carver sizing(nullptr);
  layout(h, sizing);
  h->bytes = sizing.off;
  if (cudaMalloc(reinterpret_cast<void **>(&h->base), h->bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return NS_ERR_OOM;
  }
  Carver carve(h->base);
  layout(h, carve);
  if (c.batch > 1)
    h->seq_bytes = reinterpret_cast<char *>(h->seqs[1].ring) - reinterpret_cast<char *>(h->seqs[0].ring);
  if (cudaMemset(h->base, 0, h->bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(h->base);
    delete h;
    return NS_ERR_CUDA;
  }
  h->inited.assign(c.batch, 0);
  h->slots_synced.assign(c.batch, 0);
  // The one-launch steps need every CTA of their grid resident at once (a
  // cooperative launch); check once that the device takes such a launch.
  for (int v = 0; v < 2; ++v) {
    const bool slots = v == 1;
    int &ncl = slots ? h->slot_clusters : h->step_clusters;
    int &tpc = slots ? h->slot_tpc : h->step_tpc;
    int &cl = slots ? h->slot_cl : h->step_cl;
    ncl = ns::step_plan(d, slots, &tpc, &cl);
    if (ncl > 0) {
      ns::StepLaunch L{};
      L.s = h->seqs[0];
      L.d = d;
      L.clusters = ncl;
      L.tiles_per_cluster = tpc;
      L.cluster_size = cl;
      L.probe = true;
      L.slots = slots;
      if (ns::launch_step(L, nullptr) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        ncl = 0;
      }
    }
  }
  *out = h;
  return NS_OK;
}

ns_status ns_destroy(ns_handle *h) {
  if (!h) return NS_ERR_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (h->base) cudaFree(h->base);
  delete h;
  return cuda_status(e);
}

int64_t ns_device_bytes(const ns_handle *h) { return h ? (int64_t)h->bytes : 0; }

int32_t ns_step_launches(const ns_handle *h) { return h ? (h->step_clusters > 0 ? 1 : 2) : 0; }

int32_t ns_step_slots_fused(const ns_handle *h, int32_t seq) {
  if (!valid_seq(h, seq)) return 0;
  return h->slot_clusters > 0 && h->slots_synced[seq] ? 1 : 0;
}

ns_status ns_stream_init(ns_handle *h, int32_t seq, const int32_t *d_prompt, int32_t L,
                         const float *d_prefill_logits, ns_stream stream) {
  if (!valid_seq(h, seq) || L < 0 || L > h->cfg.max_prompt || (L > 0 && !d_prompt)) return NS_ERR_ARG;
  if (h->cfg.K_pre > 0 && L > 0 && !d_prefill_logits) return NS_ERR_ARG;
  ns_status st = cuda_status(ns::launch_init(h->seqs[seq], h->dims, d_prompt, L, d_prefill_logits, h->err,
                                             static_cast<cudaStream_t>(stream)));
  if (st == NS_OK) h->inited[seq] = 1;
  h->slots_synced[seq] = 0;  // the table is empty, the window is not
  return st;
}

static ns_status check_append_args(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                                   const float *d_verify_logits, int32_t n_verify, int32_t verify_row) {
  if (!valid_seq(h, seq) || n_tree < 0 || n_tree > h->cfg.max_tree || (n_tree > 0 && !d_tree_ids))
    return NS_ERR_ARG;
  if (h->cfg.K_ver > 0 && (!d_verify_logits || n_verify < 1 || verify_row < 0 || verify_row >= n_verify))
    return NS_ERR_ARG;
  if (!h->inited[seq]) return NS_ERR_STATE;
  return NS_OK;
}

ns_status ns_stream_append(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                           const float *d_verify_logits, int32_t n_verify, int32_t verify_row, ns_stream stream) {
  ns_status st = check_append_args(h, seq, d_tree_ids, n_tree, d_verify_logits, n_verify, verify_row);
  if (st != NS_OK) return st;
  const float *zrow = h->cfg.K_ver > 0 ? d_verify_logits + (size_t)verify_row * h->cfg.V : nullptr;
  h->slots_synced[seq] = 0;
  return cuda_status(ns::launch_append(h->seqs[seq], h->dims, d_tree_ids, n_tree, zrow, false, h->err,
                                       static_cast<cudaStream_t>(stream)));
}

ns_status ns_build_active_vocab(ns_handle *h, int32_t seq, ns_stream stream) {
  if (!valid_seq(h, seq)) return NS_ERR_ARG;
  if (!h->inited[seq]) return NS_ERR_STATE;
  return cuda_status(ns::launch_build(h->seqs[seq], h->dims, h->err, static_cast<cudaStream_t>(stream)));
}

ns_status ns_gather_head_rows(ns_handle *h, int32_t seq, const uint16_t *d_W_head, ns_stream copy_stream,
                              ns_event done) {
  if (!valid_seq(h, seq) || !d_W_head || !aligned16(d_W_head)) return NS_ERR_ARG;
  if (!h->inited[seq]) return NS_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(copy_stream);
  cudaError_t e = ns::launch_gather(h->seqs[seq], h->dims, d_W_head, h->ggrid, st);
  if (e == cudaSuccess && done) e = cudaEventRecord(static_cast<cudaEvent_t>(done), st);
  return cuda_status(e);
}

static ns_status check_proj_args(ns_handle *h, const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                                 int32_t ld_logits, int32_t min_ld, int32_t *d_ids, float *d_vals) {
  if (!d_hidden || !aligned16(d_hidden) || n < 1 || n > NS_MAX_ROWS || k < 1 || k > h->cfg.max_k || !d_ids ||
      !d_vals)
    return NS_ERR_ARG;
  if (d_logits && ld_logits < min_ld) return NS_ERR_ARG;
  return NS_OK;
}

// Trace events are recorded as external event nodes when the stream is being
// captured into a CUDA graph (so a captured step still times its kernels) and
// as plain records otherwise (the external flag is only valid in capture).
static cudaError_t trace_record(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return e;
  if (cap == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}

// Where the fused tcgen05 kernel reads the rows of the sub-head from.
enum class Rows {
  kGather,  // W_head through I_t, storing them to the packed buffer on the way
  kPacked,  // the packed buffer, row j = I_t[j] (after a separate gather)
  kSlots,   // the slot buffer, row s = slot_id[s] (-1: free, not ranked)
  kIndexed, // W_head rows through I_t, nothing packed (the indexed product)
};

// Projection + top-k (one tcgen05 kernel).  `mid` (nullable) is recorded
// after it.  With `programmatic` the kernel may begin while the preceding
// kernel finishes.
static cudaError_t enqueue_gather_project(ns_handle *h, int32_t seq, const uint16_t *d_W_head,
                                          const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                                          int32_t ld_logits, int32_t *d_ids, float *d_vals, cudaStream_t cs,
                                          cudaEvent_t mid, bool programmatic, Rows rows = Rows::kGather) {
  const ns::SeqDev &s = h->seqs[seq];
  ns::UmmaLaunch L{};
  L.W = rows == Rows::kGather || rows == Rows::kIndexed ? d_W_head : rows == Rows::kPacked ? s.packed : s.slot_rows;
  L.V = h->cfg.V;
  L.H = h->cfg.H;
  L.hid = d_hidden;
  L.n = n;
  L.packed = rows == Rows::kSlots ? s.slot_rows : s.packed;
  L.W_max = h->cfg.W_max;
  L.idx = rows == Rows::kSlots ? s.slot_id : s.active;
  L.count_ptr = rows == Rows::kSlots ? s.slot_meta : s.count;
  L.in_place = rows != Rows::kGather;
  L.rows_by_id = rows == Rows::kIndexed;
  L.k = k;
  L.logits = d_logits ? d_logits : s.logits;
  L.ld = d_logits ? ld_logits : h->dims.ld_scratch;
  L.cand_k = s.cand_k;
  L.cand_i = s.cand_i;
  L.slice_ticket = s.slice_ticket;
  L.out_ids = d_ids;
  L.out_vals = d_vals;
  L.err = h->err;
  L.programmatic = programmatic;
  cudaError_t e = ns::launch_umma_step(L, cs);
  if (e == cudaSuccess && mid) e = trace_record(mid, cs);
  return e;
}

ns_status ns_sub_lm_head_logits_topk(ns_handle *h, int32_t seq, const uint16_t *d_hidden, int32_t n, int32_t k,
                                     float *d_logits, int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                                     ns_stream stream) {
  if (!valid_seq(h, seq)) return NS_ERR_ARG;
  ns_status st = check_proj_args(h, d_hidden, n, k, d_logits, ld_logits, h->cfg.W_max, d_topk_ids, d_topk_vals);
  if (st != NS_OK) return st;
  if (!h->inited[seq]) return NS_ERR_STATE;
  return cuda_status(enqueue_gather_project(h, seq, nullptr, d_hidden, n, k, d_logits, ld_logits, d_topk_ids,
                                            d_topk_vals, static_cast<cudaStream_t>(stream), nullptr, false,
                                            Rows::kPacked));
}

ns_status ns_state_update(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                          const float *d_verify_logits, int32_t n_verify, int32_t verify_row, ns_stream stream) {
  ns_status st = check_append_args(h, seq, d_tree_ids, n_tree, d_verify_logits, n_verify, verify_row);
  if (st != NS_OK) return st;
  const float *zrow = h->cfg.K_ver > 0 ? d_verify_logits + (size_t)verify_row * h->cfg.V : nullptr;
  h->slots_synced[seq] = 0;
  return cuda_status(ns::launch_append(h->seqs[seq], h->dims, d_tree_ids, n_tree, zrow, true, h->err,
                                       static_cast<cudaStream_t>(stream)));
}

static ns_status check_gather_project_args(ns_handle *h, int32_t seq, const uint16_t *d_W_head,
                                           const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                                           int32_t ld_logits, int32_t *d_ids, float *d_vals) {
  if (!valid_seq(h, seq) || !d_W_head || !aligned16(d_W_head)) return NS_ERR_ARG;
  ns_status st = check_proj_args(h, d_hidden, n, k, d_logits, ld_logits, h->cfg.W_max, d_ids, d_vals);
  if (st != NS_OK) return st;
  if (!h->inited[seq]) return NS_ERR_STATE;
  return NS_OK;
}

ns_status ns_gather_sub_lm_head_topk(ns_handle *h, int32_t seq, const uint16_t *d_W_head, const uint16_t *d_hidden,
                                     int32_t n, int32_t k, float *d_logits, int32_t ld_logits, int32_t *d_topk_ids,
                                     float *d_topk_vals, ns_stream stream) {
  ns_status st = check_gather_project_args(h, seq, d_W_head, d_hidden, n, k, d_logits, ld_logits, d_topk_ids,
                                           d_topk_vals);
  if (st != NS_OK) return st;
  return cuda_status(enqueue_gather_project(h, seq, d_W_head, d_hidden, n, k, d_logits, ld_logits, d_topk_ids,
                                            d_topk_vals, static_cast<cudaStream_t>(stream), nullptr, false));
}

ns_status ns_sub_lm_head_indexed_topk(ns_handle *h, int32_t seq, const uint16_t *d_W_head, const uint16_t *d_hidden,
                                      int32_t n, int32_t k, float *d_logits, int32_t ld_logits, int32_t *d_topk_ids,
                                      float *d_topk_vals, ns_stream stream) {
  ns_status st = check_gather_project_args(h, seq, d_W_head, d_hidden, n, k, d_logits, ld_logits, d_topk_ids,
                                           d_topk_vals);
  if (st != NS_OK) return st;
  return cuda_status(enqueue_gather_project(h, seq, d_W_head, d_hidden, n, k, d_logits, ld_logits, d_topk_ids,
                                            d_topk_vals, static_cast<cudaStream_t>(stream), nullptr, false,
                                            Rows::kIndexed));
}

static cudaError_t enqueue_step(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                                const float *d_verify_logits, int32_t verify_row, const uint16_t *d_W_head,
                                const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits, int32_t ld_logits,
                                int32_t *d_topk_ids, float *d_topk_vals, cudaStream_t cs, bool tr);

ns_status ns_step(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                  const float *d_verify_logits, int32_t n_verify, int32_t verify_row, const uint16_t *d_W_head,
                  const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits, int32_t ld_logits,
                  int32_t *d_topk_ids, float *d_topk_vals, ns_stream stream) {
  ns_status st = check_append_args(h, seq, d_tree_ids, n_tree, d_verify_logits, n_verify, verify_row);
  if (st != NS_OK) return st;
  st = check_gather_project_args(h, seq, d_W_head, d_hidden, n, k, d_logits, ld_logits, d_topk_ids, d_topk_vals);
  if (st != NS_OK) return st;
  return cuda_status(enqueue_step(h, seq, d_tree_ids, n_tree, d_verify_logits, verify_row, d_W_head, d_hidden, n, k,
                                  d_logits, ld_logits, d_topk_ids, d_topk_vals, static_cast<cudaStream_t>(stream),
                                  h->tracing));
}

// The step's launches on cs (arguments checked by the caller); with `tr`
// the four trace events bracket them.
static cudaError_t enqueue_step(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                                const float *d_verify_logits, int32_t verify_row, const uint16_t *d_W_head,
                                const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits, int32_t ld_logits,
                                int32_t *d_topk_ids, float *d_topk_vals, cudaStream_t cs, bool tr) {
  h->slots_synced[seq] = 0;
  cudaError_t e = tr ? trace_record(h->trace[0], cs) : cudaSuccess;
  const float *zrow = h->cfg.K_ver > 0 ? d_verify_logits + (size_t)verify_row * h->cfg.V : nullptr;
  if (h->step_clusters > 0) {  // one launch: state update, gather, projection, top-k
    if (e == cudaSuccess && tr) e = trace_record(h->trace[1], cs);
    ns::StepLaunch L{};
    L.s = h->seqs[seq];
    L.d = h->dims;
    L.W = d_W_head;
    L.hid = d_hidden;
    L.n = n;
    L.k = k;
    L.logits = d_logits ? d_logits : h->seqs[seq].logits;
    L.ld = d_logits ? ld_logits : h->dims.ld_scratch;
    L.out_ids = d_topk_ids;
    L.out_vals = d_topk_vals;
    L.err = h->err;
    L.tree = d_tree_ids;
    L.n_tree = n_tree;
    L.zrow = zrow;
    L.clusters = h->step_clusters;
    L.tiles_per_cluster = h->step_tpc;
    L.cluster_size = h->step_cl;
    if (e == cudaSuccess) e = ns::launch_step(L, cs);
    if (e == cudaSuccess && tr) e = trace_record(h->trace[2], cs);
    if (e == cudaSuccess && tr) e = trace_record(h->trace[3], cs);
    return e;
  }
  if (e == cudaSuccess) e = ns::launch_append(h->seqs[seq], h->dims, d_tree_ids, n_tree, zrow, true, h->err, cs);
  if (e == cudaSuccess && tr) e = trace_record(h->trace[1], cs);
  if (e == cudaSuccess)
    e = enqueue_gather_project(h, seq, d_W_head, d_hidden, n, k, d_logits, ld_logits, d_topk_ids, d_topk_vals, cs,
                               tr ? h->trace[2] : nullptr, !tr);
  if (e == cudaSuccess && tr) e = trace_record(h->trace[3], cs);
  return e;
}

// The device address of a page-locked host buffer the device can reach, or
// null (pageable memory, or a null pointer).
static void *device_view(const void *p) {
  if (!p) return nullptr;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

ns_status ns_step_host(ns_handle *h, int32_t seq, const int32_t *h_tree_ids, int32_t n_tree,
                       const float *h_verify_row, const uint16_t *d_W_head, const uint16_t *h_hidden, int32_t n,
                       int32_t k, int32_t *h_topk_ids, float *h_topk_vals, ns_stream stream) {
  ns_status st = check_append_args(h, seq, h->st_tree, n_tree, h->st_verify, 1, 0);
  if (st != NS_OK) return st;
  if ((n_tree > 0 && !h_tree_ids) || (h->cfg.K_ver > 0 && !h_verify_row) || !h_hidden || !h_topk_ids ||
      !h_topk_vals)
    return NS_ERR_ARG;
  st = check_gather_project_args(h, seq, d_W_head, h->st_hidden, n, k, nullptr, 0, h->st_ids, h->st_vals);
  if (st != NS_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool tr = h->tracing;
  // Page-locked host buffers that the device can address are read (tree ids,
  // verify row) and written (top-k) by the step kernel in place, over the
  // host link; other host buffers go through the device staging.  The
  // hidden rows are always staged: the kernel reads them by TMA.
  const int32_t *tree_d = reinterpret_cast<const int32_t *>(device_view(h_tree_ids));
  const float *verify_d = reinterpret_cast<const float *>(device_view(h_verify_row));
  int32_t *ids_d = reinterpret_cast<int32_t *>(device_view(h_topk_ids));
  float *vals_d = reinterpret_cast<float *>(device_view(h_topk_vals));
  const bool out_direct = ids_d != nullptr && vals_d != nullptr;
  cudaError_t e = tr ? trace_record(h->trace[0], cs) : cudaSuccess;
  if (e == cudaSuccess && n_tree > 0 && !tree_d) {
    e = cudaMemcpyAsync(h->st_tree, h_tree_ids, (size_t)n_tree * 4, cudaMemcpyHostToDevice, cs);
    tree_d = h->st_tree;
  }
  if (e == cudaSuccess && h->cfg.K_ver > 0 && !verify_d) {
    e = cudaMemcpyAsync(h->st_verify, h_verify_row, (size_t)h->cfg.V * 4, cudaMemcpyHostToDevice, cs);
    verify_d = h->st_verify;
  }
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h->st_hidden, h_hidden, (size_t)n * h->cfg.H * 2, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess && tr) e = trace_record(h->trace[1], cs);
  if (e == cudaSuccess)
    e = enqueue_step(h, seq, n_tree > 0 ? tree_d : h->st_tree, n_tree, verify_d ? verify_d : h->st_verify, 0,
                     d_W_head, h->st_hidden, n, k, nullptr, 0, out_direct ? ids_d : h->st_ids,
                     out_direct ? vals_d : h->st_vals, cs, false);
  if (e == cudaSuccess && tr) e = trace_record(h->trace[2], cs);
  if (e == cudaSuccess && !out_direct)
    e = cudaMemcpyAsync(h_topk_ids, h->st_ids, (size_t)n * k * 4, cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess && !out_direct)
    e = cudaMemcpyAsync(h_topk_vals, h->st_vals, (size_t)n * k * 4, cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess && tr) e = trace_record(h->trace[3], cs);
  return cuda_status(e);
}

ns_status ns_set_copy_ctas(ns_handle *h, int32_t ctas) {
  if (!h || ctas < 0) return NS_ERR_ARG;
  h->ggrid = ctas > 0 ? ctas : 4 * h->num_sms;
  h->sgrid = ctas > 0 ? ctas : 2 * h->num_sms;
  return NS_OK;
}

ns_status ns_gather_new_head_rows(ns_handle *h, int32_t seq, const uint16_t *d_W_head, ns_stream copy_stream,
                                  ns_event done) {
  if (!valid_seq(h, seq) || !d_W_head || !aligned16(d_W_head)) return NS_ERR_ARG;
  if (!h->inited[seq]) return NS_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(copy_stream);
  cudaError_t e = ns::launch_slot_update(h->seqs[seq], h->dims, d_W_head, h->sgrid, h->err, st);
  h->slots_synced[seq] = e == cudaSuccess ? 1 : 0;
  if (e == cudaSuccess && done) e = cudaEventRecord(static_cast<cudaEvent_t>(done), st);
  return cuda_status(e);
}

ns_status ns_slot_lm_head_logits_topk(ns_handle *h, int32_t seq, const uint16_t *d_hidden, int32_t n, int32_t k,
                                      float *d_logits, int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                                      ns_stream stream) {
  if (!valid_seq(h, seq)) return NS_ERR_ARG;
  ns_status st = check_proj_args(h, d_hidden, n, k, d_logits, ld_logits, h->cfg.W_max, d_topk_ids, d_topk_vals);
  if (st != NS_OK) return st;
  if (!h->inited[seq]) return NS_ERR_STATE;
  return cuda_status(enqueue_gather_project(h, seq, nullptr, d_hidden, n, k, d_logits, ld_logits, d_topk_ids,
                                            d_topk_vals, static_cast<cudaStream_t>(stream), nullptr, false,
                                            Rows::kSlots));
}

ns_status ns_step_slots(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                        const float *d_verify_logits, int32_t n_verify, int32_t verify_row, const uint16_t *d_W_head,
                        const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits, int32_t ld_logits,
                        int32_t *d_topk_ids, float *d_topk_vals, ns_stream stream) {
  ns_status st = check_append_args(h, seq, d_tree_ids, n_tree, d_verify_logits, n_verify, verify_row);
  if (st != NS_OK) return st;
  st = check_gather_project_args(h, seq, d_W_head, d_hidden, n, k, d_logits, ld_logits, d_topk_ids, d_topk_vals);
  if (st != NS_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const float *zrow = h->cfg.K_ver > 0 ? d_verify_logits + (size_t)verify_row * h->cfg.V : nullptr;
  cudaError_t e = cudaSuccess;
  if (h->slot_clusters > 0 && h->slots_synced[seq]) {
    // one launch: the state and slot updates, the new rows' copy, the
    // projection of the slot buffer and the top-k
    ns::StepLaunch L{};
    L.s = h->seqs[seq];
    L.d = h->dims;
    L.W = d_W_head;
    L.hid = d_hidden;
    L.n = n;
    L.k = k;
    L.logits = d_logits ? d_logits : h->seqs[seq].logits;
    L.ld = d_logits ? ld_logits : h->dims.ld_scratch;
    L.out_ids = d_topk_ids;
    L.out_vals = d_topk_vals;
    L.err = h->err;
    L.tree = d_tree_ids;
    L.n_tree = n_tree;
    L.zrow = zrow;
    L.clusters = h->slot_clusters;
    L.tiles_per_cluster = h->slot_tpc;
    L.cluster_size = h->slot_cl;
    L.slots = true;
    e = ns::launch_step(L, cs);
  } else {
    e = ns::launch_append(h->seqs[seq], h->dims, d_tree_ids, n_tree, zrow, true, h->err, cs);
    if (e == cudaSuccess) e = ns::launch_slot_update(h->seqs[seq], h->dims, d_W_head, h->sgrid, h->err, cs);
    if (e == cudaSuccess)
      e = enqueue_gather_project(h, seq, nullptr, d_hidden, n, k, d_logits, ld_logits, d_topk_ids, d_topk_vals, cs,
                                 nullptr, true, Rows::kSlots);
  }
  h->slots_synced[seq] = e == cudaSuccess ? 1 : 0;
  return cuda_status(e);
}

ns_status ns_step_batch(ns_handle *h, int32_t n_seq, const int32_t *d_tree_ids, int32_t n_tree,
                        const float *d_verify_logits, int32_t n_verify, const int32_t *verify_rows,
                        const uint16_t *d_W_head, const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                        int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals, ns_stream stream) {
  if (!h || n_seq < 1 || n_seq > h->cfg.batch) return NS_ERR_ARG;
  if (n_tree < 0 || n_tree > h->cfg.max_tree || (n_tree > 0 && !d_tree_ids)) return NS_ERR_ARG;
  const int V = h->cfg.V, H = h->cfg.H;
  if (h->cfg.K_ver > 0) {
    if (!d_verify_logits || n_verify < 1 || !verify_rows) return NS_ERR_ARG;
    for (int b = 0; b < n_seq; ++b)
      if (verify_rows[b] < 0 || verify_rows[b] >= n_verify) return NS_ERR_ARG;
  }
  if (!d_W_head || !aligned16(d_W_head)) return NS_ERR_ARG;
  ns_status st = check_proj_args(h, d_hidden, n, k, d_logits, ld_logits, h->cfg.W_max, d_topk_ids, d_topk_vals);
  if (st != NS_OK) return st;
  for (int b = 0; b < n_seq; ++b)
    if (!h->inited[b]) return NS_ERR_STATE;
  for (int b = 0; b < n_seq; ++b) h->slots_synced[b] = 0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  for (int c0 = 0; c0 < n_seq && e == cudaSuccess; c0 += ns::kMaxBatchLaunch) {
    const int nb = n_seq - c0 < ns::kMaxBatchLaunch ? n_seq - c0 : ns::kMaxBatchLaunch;
    const ns::SeqDev &s0 = h->seqs[c0];
    ns::StepBatch bt{};
    bt.seq_bytes = h->seq_bytes;
    bt.tree_stride = n_tree;
    bt.z_stride = (long long)n_verify * V;
    const float *verify = nullptr;
    if (h->cfg.K_ver > 0) {
      verify = d_verify_logits + (size_t)c0 * n_verify * V;
      for (int b = 0; b < nb; ++b) bt.vrow[b] = verify_rows[c0 + b];
    }
    e = ns::launch_append_batch(s0, h->dims, nb, n_tree > 0 ? d_tree_ids + (size_t)c0 * n_tree : d_tree_ids,
                                n_tree, verify, bt, h->err, cs);
    if (e != cudaSuccess) break;
    ns::UmmaLaunch L{};
    L.W = d_W_head;
    L.V = V;
    L.H = H;
    L.hid = d_hidden + (size_t)c0 * n * H;
    L.n = n;
    L.packed = s0.packed;
    L.W_max = h->cfg.W_max;
    L.idx = s0.active;
    L.count_ptr = s0.count;
    L.k = k;
    L.logits = d_logits ? d_logits + (size_t)c0 * n * ld_logits : s0.logits;
    L.ld = d_logits ? ld_logits : h->dims.ld_scratch;
    L.cand_k = s0.cand_k;
    L.cand_i = s0.cand_i;
    L.slice_ticket = s0.slice_ticket;
    L.out_ids = d_topk_ids + (size_t)c0 * n * k;
    L.out_vals = d_topk_vals + (size_t)c0 * n * k;
    L.err = h->err;
    L.programmatic = true;
    L.nseq = nb;
    L.seq_bytes = h->seq_bytes;
    L.logits_bytes = d_logits ? (long long)n * ld_logits * 4 : h->seq_bytes;
    e = ns::launch_umma_step(L, cs);
  }
  return cuda_status(e);
}

ns_status ns_step_batch_union(ns_handle *h, int32_t n_seq, const int32_t *d_tree_ids, int32_t n_tree,
                              const float *d_verify_logits, int32_t n_verify, const int32_t *verify_rows,
                              const uint16_t *d_W_head, const uint16_t *d_hidden, int32_t n, int32_t k,
                              float *d_logits, int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                              ns_stream stream) {
  if (!h || n_seq < 1 || n_seq > h->cfg.batch) return NS_ERR_ARG;
  if (h->u_cap == 0) return NS_ERR_STATE;  // a handle of one sequence has no union buffers
  if (n_tree < 0 || n_tree > h->cfg.max_tree || (n_tree > 0 && !d_tree_ids)) return NS_ERR_ARG;
  const int V = h->cfg.V, H = h->cfg.H;
  if (h->cfg.K_ver > 0) {
    if (!d_verify_logits || n_verify < 1 || !verify_rows) return NS_ERR_ARG;
    for (int b = 0; b < n_seq; ++b)
      if (verify_rows[b] < 0 || verify_rows[b] >= n_verify) return NS_ERR_ARG;
  }
  if (!d_W_head || !aligned16(d_W_head)) return NS_ERR_ARG;
  ns_status st = check_proj_args(h, d_hidden, n, k, d_logits, ld_logits, (int32_t)h->u_cap, d_topk_ids, d_topk_vals);
  if (st != NS_OK) return st;
  for (int b = 0; b < n_seq; ++b)
    if (!h->inited[b]) return NS_ERR_STATE;
  for (int b = 0; b < n_seq; ++b) h->slots_synced[b] = 0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  // 1. every sequence's state update and its own I_t
  for (int c0 = 0; c0 < n_seq && e == cudaSuccess; c0 += ns::kMaxBatchLaunch) {
    const int nb = n_seq - c0 < ns::kMaxBatchLaunch ? n_seq - c0 : ns::kMaxBatchLaunch;
    ns::StepBatch bt{};
    bt.seq_bytes = h->seq_bytes;
    bt.tree_stride = n_tree;
    bt.z_stride = (long long)n_verify * V;
    const float *verify = nullptr;
    if (h->cfg.K_ver > 0) {
      verify = d_verify_logits + (size_t)c0 * n_verify * V;
      for (int b = 0; b < nb; ++b) bt.vrow[b] = verify_rows[c0 + b];
    }
    e = ns::launch_append_batch(h->seqs[c0], h->dims, nb, n_tree > 0 ? d_tree_ids + (size_t)c0 * n_tree : d_tree_ids,
                                n_tree, verify, bt, h->err, cs);
  }
  // 2. U = the union of their windows, ascending; 3. one gather of W_head[U, :]
  ns::SeqDev u{};
  u.bitmap = h->u_bitmap;
  u.active = h->u_ids;
  u.count = h->u_count;
  u.packed = h->u_packed;
  ns::Dims du = h->dims;
  du.W_max = (int32_t)h->u_cap;
  if (e == cudaSuccess) e = ns::launch_union_bitmap(h->seqs[0], h->dims, n_seq, h->seq_bytes, h->u_bitmap, cs);
  if (e == cudaSuccess) e = ns::launch_build(u, du, h->err, cs);
  if (e == cudaSuccess) e = ns::launch_gather(u, du, d_W_head, h->ggrid, cs);
  // 4. every sequence's hidden rows through the union rows, each ranking its own
  for (int c0 = 0; c0 < n_seq && e == cudaSuccess; c0 += ns::kMaxBatchLaunch) {
    const int nb = n_seq - c0 < ns::kMaxBatchLaunch ? n_seq - c0 : ns::kMaxBatchLaunch;
    ns::UmmaLaunch L{};
    L.W = h->u_packed;
    L.V = V;
    L.H = H;
    L.hid = d_hidden + (size_t)c0 * n * H;
    L.n = n;
    L.packed = h->u_packed;
    L.W_max = (int32_t)h->u_cap;
    L.idx = h->u_ids;
    L.count_ptr = h->u_count;
    L.k = k;
    L.logits = d_logits ? d_logits + (size_t)c0 * n * ld_logits : h->u_logits + (size_t)c0 * ns::kProjBN * h->u_ld;
    L.ld = d_logits ? ld_logits : h->u_ld;
    uint32_t *blk = h->u_cand + (size_t)c0 * h->u_block_words;
    L.cand_k = blk;
    L.cand_i = blk + h->u_cand_words;
    L.slice_ticket = reinterpret_cast<int32_t *>(blk + 2 * h->u_cand_words);
    L.cand_stride = h->u_block_words * 4;
    L.out_ids = d_topk_ids + (size_t)c0 * n * k;
    L.out_vals = d_topk_vals + (size_t)c0 * n * k;
    L.err = h->err;
    L.in_place = true;
    L.nseq = nb;
    L.seq_bytes = h->seq_bytes;
    L.logits_bytes = d_logits ? (long long)n * ld_logits * 4 : (long long)ns::kProjBN * h->u_ld * 4;
    L.mask = h->seqs[c0].bitmap;
    e = ns::launch_umma_step(L, cs);
  }
  return cuda_status(e);
}

ns_status ns_get_union(ns_handle *h, const int32_t **ids, const int32_t **count, const uint32_t **bitmap,
                       const uint16_t **packed, int64_t *capacity) {
  if (!h) return NS_ERR_ARG;
  if (h->u_cap == 0) return NS_ERR_STATE;
  if (ids) *ids = h->u_ids;
  if (count) *count = h->u_count;
  if (bitmap) *bitmap = h->u_bitmap;
  if (packed) *packed = h->u_packed;
  if (capacity) *capacity = h->u_cap;
  return NS_OK;
}

ns_status ns_trace_events(ns_handle *h, ns_event *events, int32_t n_events) {
  if (!h) return NS_ERR_ARG;
  if (n_events == 0 && !events) {
    h->tracing = false;
    return NS_OK;
  }
  if (!events || n_events != 4) return NS_ERR_ARG;
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return NS_ERR_ARG;
    h->trace[i] = static_cast<cudaEvent_t>(events[i]);
  }
  h->tracing = true;
  return NS_OK;
}

ns_status ns_dense_lm_head_topk(ns_handle *h, const uint16_t *d_W_head, int32_t rows, const uint16_t *d_hidden,
                                int32_t n, int32_t k, float *d_logits, int32_t ld_logits, int32_t *d_topk_ids,
                                float *d_topk_vals, ns_stream stream) {
  if (!h || !d_W_head || !aligned16(d_W_head) || rows < 1 || rows > h->cfg.V) return NS_ERR_ARG;
  ns_status st = check_proj_args(h, d_hidden, n, k, d_logits, ld_logits, rows, d_topk_ids, d_topk_vals);
  if (st != NS_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  float *logits = d_logits ? d_logits : h->dense_logits;
  const int ld = d_logits ? ld_logits : h->dense_ld;
  cudaError_t e = ns::launch_dense(d_W_head, rows, d_hidden, n, h->cfg.H, logits, ld, h->err, cs);
  if (e == cudaSuccess)
    e = ns::launch_topk(logits, ld, rows, nullptr, n, k, d_topk_ids, d_topk_vals, h->dense_cand_k, h->dense_cand_i, cs);
  return cuda_status(e);
}

ns_status ns_get_active(ns_handle *h, int32_t seq, const int32_t **ids, const int32_t **count,
                        const uint32_t **bitmap, const uint16_t **packed) {
  if (!valid_seq(h, seq)) return NS_ERR_ARG;
  const ns::SeqDev &s = h->seqs[seq];
  if (ids) *ids = s.active;
  if (count) *count = s.count;
  if (bitmap) *bitmap = s.bitmap;
  if (packed) *packed = s.packed;
  return NS_OK;
}

ns_status ns_get_state(ns_handle *h, int32_t seq, const int32_t **ring, const int64_t **length,
                       const uint32_t **counts) {
  if (!valid_seq(h, seq)) return NS_ERR_ARG;
  const ns::SeqDev &s = h->seqs[seq];
  if (ring) *ring = s.ring;
  if (length) *length = reinterpret_cast<const int64_t *>(s.length);
  if (counts) *counts = s.counts;
  return NS_OK;
}

// Checkpoint of one sequence (little-endian): a 32-byte header, then the
// window's stream entries oldest first.
namespace {
constexpr char kCkptMagic[4] = {'N', 'S', 'S', 'T'};
constexpr uint32_t kCkptVersion = 1;
struct CkptHeader {
  char magic[4];
  uint32_t version;
  int32_t V, W_max;
  int64_t length;  // |S|
  int32_t n;       // entries that follow: min(|S|, W_max)
  int32_t reserved;
};
static_assert(sizeof(CkptHeader) == 32, "checkpoint header layout");
}  // namespace

int64_t ns_state_export_bytes(const ns_handle *h) {
  return h ? (int64_t)sizeof(CkptHeader) + 4 * (int64_t)h->cfg.W_max : 0;
}

ns_status ns_state_export(ns_handle *h, int32_t seq, void *host_buf, int64_t buf_bytes, int64_t *written,
                          ns_stream stream) {
  if (!valid_seq(h, seq) || !written) return NS_ERR_ARG;
  if (!h->inited[seq]) return NS_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const ns::SeqDev &s = h->seqs[seq];
  const int W = h->cfg.W_max;
  long long len[2] = {0, 0};
  std::vector<int32_t> ring((size_t)W);
  cudaError_t e = cudaMemcpyAsync(len, s.length, sizeof(len), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ring.data(), s.ring, (size_t)W * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  const long long n = len[0] < W ? len[0] : W;
  const int64_t need = (int64_t)sizeof(CkptHeader) + 4 * n;
  *written = need;
  if (!host_buf) return NS_OK;  // the size only
  if (buf_bytes < need) return NS_ERR_ARG;
  CkptHeader hd{};
  std::memcpy(hd.magic, kCkptMagic, 4);
  hd.version = kCkptVersion;
  hd.V = h->cfg.V;
  hd.W_max = W;
  hd.length = len[0];
  hd.n = (int32_t)n;
  char *out = static_cast<char *>(host_buf);
  std::memcpy(out, &hd, sizeof(hd));
  int32_t *ent = reinterpret_cast<int32_t *>(out + sizeof(hd));
  for (long long i = 0; i < n; ++i) {
    const int32_t x = ring[(size_t)((len[0] - n + i) % W)];
    std::memcpy(ent + i, &x, 4);
  }
  return NS_OK;
}

ns_status ns_state_import(ns_handle *h, int32_t seq, const void *host_buf, int64_t bytes, ns_stream stream) {
  if (!valid_seq(h, seq) || !host_buf || bytes < (int64_t)sizeof(CkptHeader)) return NS_ERR_ARG;
  CkptHeader hd;
  std::memcpy(&hd, host_buf, sizeof(hd));
  const int W = h->cfg.W_max;
  if (std::memcmp(hd.magic, kCkptMagic, 4) != 0 || hd.version != kCkptVersion || hd.V != h->cfg.V ||
      hd.W_max != W || hd.length < 0 || hd.n < 0 || hd.n != (hd.length < W ? hd.length : W) ||
      bytes < (int64_t)sizeof(CkptHeader) + 4 * (int64_t)hd.n)
    return NS_ERR_ARG;
  const char *in = static_cast<const char *>(host_buf) + sizeof(hd);
  std::vector<int32_t> ring((size_t)W, 0);
  for (int i = 0; i < hd.n; ++i) {
    int32_t x;
    std::memcpy(&x, in + 4 * (size_t)i, 4);
    if (x < 0 || x >= h->cfg.V) return NS_ERR_ARG;
    ring[(size_t)((hd.length - hd.n + i) % W)] = x;
  }
  // the copy from this pageable vector is staged before cudaMemcpyAsync returns
  const cudaError_t e =
      ns::launch_restore(h->seqs[seq], h->dims, ring.data(), hd.length, h->err, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) h->inited[seq] = 1;
  h->slots_synced[seq] = 0;  // the slot table restarts empty
  return cuda_status(e);
}

ns_status ns_get_slots(ns_handle *h, int32_t seq, const int32_t **slot_id, const int32_t **meta,
                       const int32_t **new_slots, const int32_t **new_ids, const uint16_t **rows) {
  if (!valid_seq(h, seq)) return NS_ERR_ARG;
  const ns::SeqDev &s = h->seqs[seq];
  if (slot_id) *slot_id = s.slot_id;
  if (meta) *meta = s.slot_meta;
  if (new_slots) *new_slots = s.new_slot;
  if (new_ids) *new_ids = s.new_id;
  if (rows) *rows = s.slot_rows;
  return NS_OK;
}

ns_status ns_get_error(ns_handle *h, uint32_t *flags, int32_t clear) {
  if (!h || !flags) return NS_ERR_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(flags, h->err, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(h->err, 0, sizeof(uint32_t));
  if (e == cudaSuccess && clear) e = cudaDeviceSynchronize();
  return cuda_status(e);
}

}  // extern "C"
