// snack_spmm_fwd_noalloc: the forward SpMM for callers that cannot provide a
// workspace.  Some callers may not allocate device memory on their call path
// at all -- a plugin invoked from an inference engine's enqueue step, or a
// real-time loop whose memory is fixed at start-up -- so they cannot hand the
// library the scratch buffer snack_spmm_fwd needs.  This entry point supplies
// that scratch from a file-scope device array instead and allocates nothing.
//
// The array is part of the library's device image: every GPU that loads this
// code holds it (kNoAllocScratchBytes) until the process exits.  All calls
// share it, so two calls that overlap on the GPU (different streams, or
// different host threads) race on it; calls must be ordered.  The array keeps
// whatever the last call left in it; the forward pass writes every scratch
// element before reading it, so nothing needs clearing between calls.
#include <mutex>

#include "internal.hpp"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's name is only a host-side stand-in in host code; its device
// address is looked up per device, with that device current, and kept once
// a lookup succeeds.  A failed lookup (a leftover error from earlier work, or
// a first call made during stream capture) is not remembered: the next call
// on that device tries again.
std::mutex g_mu[kMaxDevices];
void *g_scratch[kMaxDevices];
bool g_have[kMaxDevices];

struct CurrentDevice {
  int prev = -1;
  bool ok = false;
  explicit CurrentDevice(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
  }
  ~CurrentDevice() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" snack_status snack_spmm_fwd_noalloc(snack_handle h, const int32_t *row, const int32_t *col,
                                               const void *val, const void *x, int32_t batch, const float *bias,
                                               void *y, snack_stream_t stream) {
  if (!h) return SNACK_ERR_INVALID_ARG;
  const int dev = h->device;
  if (dev < 0 || dev >= kMaxDevices) return SNACK_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu[dev]);
    if (!g_have[dev]) {
      CurrentDevice cur(dev);
      if (!cur.ok) return SNACK_ERR_CUDA;
      void *ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();  // do not leave the failed lookup's error for the next CUDA call
        return SNACK_ERR_CUDA;
      }
      g_scratch[dev] = ptr;
      g_have[dev] = true;
    }
    scratch = g_scratch[dev];
  }
  // snack_spmm_fwd checks the scratch size this call needs against the
  // array's size and returns SNACK_ERR_WORKSPACE, before any launch, when it
  // does not fit.
  return snack_spmm_fwd(h, row, col, val, x, batch, bias, y, scratch, kNoAllocScratchBytes, stream);
}
