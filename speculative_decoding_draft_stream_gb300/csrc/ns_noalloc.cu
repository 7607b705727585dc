// A dense LM head with top-k that needs no allocation at all.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory pool or a fixed device-memory budget, a plugin that is
// only handed pointers, or a process whose allocator is locked down while it
// serves.  ns_create allocates, so those callers cannot hold a handle.  This
// entry point computes the same dense head as ns_dense_lm_head_topk using
// only the caller's inputs and outputs plus a fixed scratch array that is part
// of the library image itself (a file-scope __device__ array, so it is
// reserved on every GPU that loads the library and held until the process
// exits).
#include <mutex>

#include "ns_internal.cuh"

namespace {

// Scratch layout (floats, 256-byte aligned pieces; 6,817,792 bytes in all):
//   [0, kTicketWords)                 per-tile arrival counters (int32)
//   [kPartOff, kPartOff + kPartFloats) split-K partial tiles
//   [kLogitsOff, + NS_NOALLOC_MAX_LOGITS) logits when the caller passes none
constexpr int kSlots = 160;  // most CTAs of one call; also the most split-K partial tiles
constexpr size_t kTileFloats = (size_t)ns::kProjBN * ns::kProjBM;
constexpr size_t kTicketWords = 256;
constexpr size_t kPartOff = kTicketWords;
constexpr size_t kPartFloats = (size_t)kSlots * kTileFloats;
constexpr size_t kLogitsOff = kPartOff + kPartFloats;
constexpr size_t kScratchFloats = kLogitsOff + (size_t)NS_NOALLOC_MAX_LOGITS;

static_assert(kTicketWords >= kSlots, "one arrival counter per tile");

// The scratch itself.  Host code must not use this name as an address: on
// the host it is only a stand-in, so the device address is looked up once per
// device with cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool ready = false;
  float *scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int grid = 0;
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: find the scratch's device
// address, size the grid and allow the projection's shared-memory footprint.
cudaError_t setup_current_device(DeviceSetup **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup &s = g_setup[dev];
  if (!s.ready) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = ns::prepare_project_kernels();
    if (e != cudaSuccess) return e;
    s.scratch = static_cast<float *>(ptr);
    // one CTA per SM (at most kSlots): the handle's dense head runs two per
    // SM, so this one is slower on large heads and splits K differently
    // (the same logits up to fp32 summation order)
    s.grid = sms < kSlots ? sms : kSlots;
    s.ready = true;
  }
  *out = &s;
  return cudaSuccess;
}

}  // namespace

extern "C" ns_status ns_dense_lm_head_topk_noalloc(const uint16_t *d_W_head, int32_t rows, int32_t H,
                                                   const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                                                   int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                                                   ns_stream stream) {
  if (!d_W_head || (reinterpret_cast<uintptr_t>(d_W_head) & 15u) || rows < 1 || H < 64 || H > 8192 || H % 64 ||
      !d_hidden || (reinterpret_cast<uintptr_t>(d_hidden) & 15u) || n < 1 || n > NS_MAX_ROWS || k < 1 ||
      k > NS_MAX_TOPK || !d_topk_ids || !d_topk_vals)
    return NS_ERR_ARG;
  if (d_logits && ld_logits < rows) return NS_ERR_ARG;
  // Without a caller logits buffer the logits live in the scratch, which
  // holds at most NS_NOALLOC_MAX_LOGITS values.
  if (!d_logits && (int64_t)n * rows > (int64_t)NS_NOALLOC_MAX_LOGITS) return NS_ERR_ARG;

  DeviceSetup *s = nullptr;
  if (setup_current_device(&s) != cudaSuccess) return NS_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // The scratch address is the current device's copy: a stream of another
  // device would run the kernels against the wrong GPU's array.
  int cur = 0, sdev = 0;
  if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(cs, &sdev) != cudaSuccess) return NS_ERR_CUDA;
  if (sdev != cur) return NS_ERR_ARG;
  float *base = s->scratch;
  int32_t *tickets = reinterpret_cast<int32_t *>(base);
  // The arrival counters must start at zero; everything else is written
  // before it is read.
  if (cudaMemsetAsync(tickets, 0, kTicketWords * sizeof(int32_t), cs) != cudaSuccess) return NS_ERR_CUDA;

  ns::ProjArgs a{};
  a.rows = d_W_head;
  a.rows_host = rows;
  a.hid = d_hidden;
  a.n = n;
  a.H = H;
  a.logits = d_logits ? d_logits : base + kLogitsOff;
  a.ld = d_logits ? ld_logits : rows;
  a.part = base + kPartOff;
  a.tickets = tickets;
  cudaError_t e = ns::launch_project(a, s->grid, cs);
  if (e == cudaSuccess) e = ns::launch_topk(a.logits, a.ld, nullptr, rows, nullptr, n, k, d_topk_ids, d_topk_vals, cs);
  return e == cudaSuccess ? NS_OK : NS_ERR_CUDA;
}
