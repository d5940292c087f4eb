// ssm_scan_fwd without a caller-provided workspace, for callers that cannot
// allocate device memory (see include/ssm_scan.h, ssm_scan_fwd_noalloc).
//
// The chunk carry of long sequences needs scratch memory.  Here it lives in one
// file-scope device array of SSM_NOALLOC_SCRATCH_BYTES, created when the library
// is loaded on each device and kept until the process exits.  Host code cannot
// use the array's name as a device address (it names a host-side shadow), so the
// first call on each device looks up the real address with
// cudaGetSymbolAddress while that device is current, and caches it.
#include <mutex>

#include "ssm_internal.h"
#include "ssm_scan.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device (nullptr on failure).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" ssm_status ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                                           const void* C, const float* D, const void* z, const float* delta_bias,
                                           void* out, float* final_state, const ssm_dims* dims,
                                           ssm_stream_t stream) {
  // Same validation as ssm_scan_fwd, then the plan decides how much scratch the call needs.
  const size_t need = ssm_scan_workspace_bytes(dims);
  if (need > SSM_NOALLOC_SCRATCH_BYTES) return SSM_ERR_WORKSPACE;
  if (need == 0) return ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, out, final_state, dims, nullptr, 0, stream);
  void* scratch = scratch_address();
  if (!scratch) return SSM_ERR_CUDA;
  return ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, out, final_state, dims, scratch,
                      SSM_NOALLOC_SCRATCH_BYTES, stream);
}
