// ssm_scan_fwd without a caller-provided workspace, for callers that cannot
// allocate device memory (see include/ssm_scan.h, ssm_scan_fwd_noalloc).
//
// The chunk carry of long sequences needs scratch memory.  Here it lives in one
// file-scope device array of SSM_NOALLOC_SCRATCH_BYTES, created when the library
// is loaded on each device and kept until the process exits.  Host code cannot
// use the array's name as a device address (it names a host-side shadow), so the
// first call on each device looks up the real address with
// cudaGetSymbolAddress while that device is current, and caches it together with
// the id of the context it belongs to; a call in another context (after a device
// reset, say) looks it up again.
#include <cuda.h>

#include <mutex>

#include "ssm_internal.h"
#include "ssm_scan.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id;  // the context the address belongs to (0: none yet)
  void* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Unique id of the current context (0 if none is current or the driver cannot say).
// A device reset, or another context made current on the same device, changes it,
// and with it the device address of g_noalloc_scratch.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_scratch in the current context (nullptr on failure),
// looked up with that device current on the first call in each context and cached.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = current_context_id();
  if (id != 0 && g_scratch[dev].ctx_id == id && g_scratch[dev].ptr) return g_scratch[dev].ptr;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
  id = current_context_id();  // the lookup above made the device's context current if none was
  g_scratch[dev] = ScratchEntry{id, ptr};
  return ptr;
}

}  // namespace

extern "C" size_t ssm_noalloc_scratch_bytes(void) { return SSM_NOALLOC_SCRATCH_BYTES; }

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
