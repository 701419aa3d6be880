// gdn_verify_step_static_scratch: the verify step for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocator) at the point where they
// run the verify step: code inside a memory-pool-managed runtime that forbids allocations on
// its hot path, code paths that must not synchronise the device (cudaMalloc/cudaFree may), or
// embedders that only hand this library the tensors they already own.  This entry point passes
// a fixed array in the library's own device memory as gdn_verify_step's `workspace` argument,
// so such callers never size or allocate one.  The verify kernels need no scratch at all
// (gdn_verify_workspace_size reports 0 bytes), so the array is small; should a shape ever need
// more than it holds, the call returns GDN_ERR_UNSUPPORTED instead of running.
//
// The array is a file-scope __device__ variable, so every GPU on which the library's module is
// loaded holds it until the process exits.  Host code cannot use the array's name as a device
// address (on the host it names a shadow variable), so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the first call made on
// that device, and cached.  Make that first call before any stream capture begins, so the
// lookup does not happen inside a capture.
#include <cstdio>
#include <mutex>

#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace {

// Largest scratch the fixed array provides.
constexpr size_t kStaticScratchBytes = 256;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

gdn_status static_scratch_ptr(void** out) {
  constexpr int kMaxDevices = 64;
  static void* cache[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  char msg[256];
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
    return gdn::report_error(GDN_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof msg, "device ordinal %d out of range", dev);
    return gdn::report_error(GDN_ERR_UNSUPPORTED, msg);
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
      return gdn::report_error(GDN_ERR_CUDA, msg);
    }
    cache[dev] = ptr;
  }
  *out = cache[dev];
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_verify_step_static_scratch(const gdn_dims* dims, const uint16_t* x, const uint16_t* a,
                                                     const uint16_t* b, const float* A_log, const float* dt_bias,
                                                     const float* conv_w, const float* conv_state_in,
                                                     float* conv_state_out, float* conv_inter, const float* state_in,
                                                     float* state_out, float* state_inter, void* out,
                                                     gdn_stream_t stream) {
  uint64_t need = 0;
  gdn_status s = gdn_verify_workspace_size(dims, &need);  // validates dims, sets the error text on failure
  if (s != GDN_OK) return s;
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "gdn_verify_step_static_scratch: these dims need %llu bytes of scratch but the static scratch "
             "holds %zu; call gdn_verify_step with a workspace instead",
             (unsigned long long)need, kStaticScratchBytes);
    return gdn::report_error(GDN_ERR_UNSUPPORTED, msg);
  }
  void* scratch = nullptr;
  s = static_scratch_ptr(&scratch);
  if (s != GDN_OK) return s;
  return gdn_verify_step(dims, x, a, b, A_log, dt_bias, conv_w, conv_state_in, conv_state_out, conv_inter, state_in,
                         state_out, state_inter, out, scratch, kStaticScratchBytes, stream);
}
