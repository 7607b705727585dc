// A dense LM head with top-k that needs no allocation at all.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory pool or a fixed device-memory budget, a plugin that is
// only handed pointers, or a process whose allocator is locked down while it
// serves.  ns_create allocates, so those callers cannot hold a handle.  This
// entry point computes the same dense head as ns_dense_lm_head_topk (the same
// tcgen05 projection and two-launch top-k) using only the caller's inputs and
// outputs plus a fixed scratch array that is part of the library image itself
// (a file-scope __device__ array, so it is reserved on every GPU that loads
// the library and held until the process exits).
#include <mutex>

#include "ns_internal.cuh"

namespace {

// Scratch layout (256-byte aligned pieces; 6,291,456 bytes in all):
//   [0, kCand)                 the top-k slices' lists: order keys
//   [kCand, 2 kCand)           and their columns
//   [2 kCand, + MAX_LOGITS)    logits when the caller passes none
constexpr int kMaxRows = 1 << 19;  // most rows of a head: the slices' lists fit the scratch
constexpr size_t kCand = (size_t)NS_MAX_ROWS * (kMaxRows / ns::kTopkSliceCols) * NS_MAX_TOPK;
constexpr size_t kLogitsOff = 2 * kCand;
constexpr size_t kScratchWords = kLogitsOff + (size_t)NS_NOALLOC_MAX_LOGITS;
static_assert(kScratchWords * 4 == 6291456, "scratch size as documented in nanospec.h");

static __device__ __align__(256) float g_noalloc_scratch[kScratchWords];
static __device__ uint32_t g_noalloc_err;  // where a bounded wait that ran out is recorded (never read back)

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool ready = false;
  float *scratch = nullptr;  // device address of g_noalloc_scratch on this device
  uint32_t *err = nullptr;   // and of g_noalloc_err
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

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
    void *eptr = nullptr;
    e = cudaGetSymbolAddress(&eptr, g_noalloc_err);
    if (e != cudaSuccess) return e;
    e = ns::prepare_dense_kernel();
    if (e != cudaSuccess) return e;
    s.scratch = static_cast<float *>(ptr);
    s.err = static_cast<uint32_t *>(eptr);
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
  if (!d_W_head || (reinterpret_cast<uintptr_t>(d_W_head) & 15u) || rows < 1 || rows > kMaxRows || H < 64 ||
      H > 8192 || H % 64 || !d_hidden || (reinterpret_cast<uintptr_t>(d_hidden) & 15u) || n < 1 ||
      n > NS_MAX_ROWS || k < 1 || k > NS_MAX_TOPK || !d_topk_ids || !d_topk_vals)
    return NS_ERR_ARG;
  if (d_logits && (ld_logits < rows || (reinterpret_cast<uintptr_t>(d_logits) & 3u))) return NS_ERR_ARG;
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
  float *logits = d_logits ? d_logits : base + kLogitsOff;
  const int ld = d_logits ? ld_logits : rows;
  cudaError_t e = ns::launch_dense(d_W_head, rows, d_hidden, n, H, logits, ld, s->err, cs);
  if (e == cudaSuccess)
    e = ns::launch_topk(logits, ld, rows, nullptr, n, k, d_topk_ids, d_topk_vals, reinterpret_cast<uint32_t *>(base),
                        reinterpret_cast<uint32_t *>(base + kCand), cs);
  return e == cudaSuccess ? NS_OK : NS_ERR_CUDA;
}
