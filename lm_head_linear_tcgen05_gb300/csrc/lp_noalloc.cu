// lp_noalloc.cu - lp_forward_noalloc: the fused forward for callers that cannot
// allocate device memory.
//
// Some hosts cannot hand this library a workspace: plugins that run inside an
// engine whose memory manager owns every device byte, runtimes whose memory budget
// is fixed after start-up, or callers without any binding to a CUDA allocator. For
// them this entry point takes its scratch from one file-scope device array of fixed
// size instead of from a caller workspace, and calls no allocating routine.
//
// The array lives in this module, so every GPU that loads the library holds it
// (LP_NOALLOC_SCRATCH_BYTES) until the process exits. Its device address is looked
// up once per device, on that device's first call, with the device current.
#include <cuda_runtime.h>

#include <mutex>

#include "lp_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[LP_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

extern "C" LP_API lp_status lp_forward_noalloc(const void* X, int64_t T, int64_t H, const void* const* W,
                                               const void* const* bias, const lp_vocab_partition* part,
                                               const int32_t* y, float tau, const lp_outputs* out,
                                               lp_stream_t stream) {
  const size_t need = lp_workspace_size(LP_OP_FORWARD, T, H, part);
  if (need == 0)  // an empty batch, or invalid sizes / partition: lp_forward handles both
    return lp_forward(X, T, H, W, bias, part, y, tau, out, nullptr, 0, stream);
  if (need > size_t(LP_NOALLOC_SCRATCH_BYTES)) return LP_ERR_WORKSPACE_TOO_SMALL;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return LP_ERR_UNSUPPORTED_DEVICE;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
      // host code may not use g_noalloc_scratch directly: its name here is only a
      // host-side stand-in, so ask the runtime for this device's address of it
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return LP_ERR_UNSUPPORTED_DEVICE;
      }
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  return lp_forward(X, T, H, W, bias, part, y, tau, out, scratch, size_t(LP_NOALLOC_SCRATCH_BYTES), stream);
}
