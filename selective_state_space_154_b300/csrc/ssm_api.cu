// C ABI of the selective-scan library: argument validation, launch planning,
// status codes.  Declarations and the meaning of every argument are in
// include/ssm_scan.h.
#include <atomic>
#include <climits>
#include <cstdint>
#include <mutex>
#include <cstdlib>
#include <cstring>

#include "ssm_scan.h"
#include "ssm_internal.h"

namespace ssm {

namespace {

// The test hooks (SSM_* environment variables, listed in include/ssm_scan.h) are
// read once, at the first call that needs them, and again only when the
// application calls ssm_test_hooks_reload(): no call reads the environment on
// its own.  Each load publishes an immutable copy.
RuntimeKnobs* load_knobs() {
  RuntimeKnobs* r = new RuntimeKnobs{};
  r->lookback_timeout_ns = 0;  // 0: 1 s + 100 ns per token of a chunk (set at launch)
  if (const char* s = std::getenv("SSM_LOOKBACK_TIMEOUT_MS")) {
    const long long ms = std::atoll(s);
    if (ms > 0) r->lookback_timeout_ns = ms * 1000ll * 1000;
  }
  const char* f = std::getenv("SSM_FAULT");
  r->fault_lookback = f && std::strcmp(f, "lookback") == 0;
  r->fault_step = f && std::strcmp(f, "step") == 0;
  r->fault_ssd = f && std::strcmp(f, "ssd") == 0;
  const char* fs = std::getenv("SSM_FORCE_STEP");
  r->force_step_plain = fs && std::strcmp(fs, "plain") == 0;
  if (const char* c = std::getenv("SSM_FORCE_CHUNKS")) r->force_chunks = std::atoi(c);
  r->force_kind = -1;
  if (const char* k = std::getenv("SSM_FORCE_KERNEL")) {
    if (std::strcmp(k, "tiles") == 0) r->force_kind = kScanTiles;
    if (std::strcmp(k, "rows") == 0) r->force_kind = kScanRows;
    if (std::strcmp(k, "stream") == 0) r->force_kind = kScanStream;
    if (std::strcmp(k, "tiny") == 0) r->force_kind = kScanTiny;
    if (std::strcmp(k, "ssd_walk") == 0) r->force_ssd = 1;
    if (std::strcmp(k, "ssd_chunks") == 0) r->force_ssd = 2;
  }
  if (const char* c = std::getenv("SSM_CTAS_PER_SM")) r->ctas_per_sm = std::atoi(c);
  if (const char* c = std::getenv("SSM_FORCE_TPR")) r->force_tpr = std::atoi(c);
  if (const char* c = std::getenv("SSM_BWD_CHUNKS")) r->bwd_chunks = std::atoi(c);
  if (const char* c = std::getenv("SSM_BWD_FORM")) r->bwd_form = std::strcmp(c, "quad") == 0 ? 1 : 0;
  if (const char* c = std::getenv("SSM_STREAM_ROWS")) {
    const int v = std::atoi(c);
    r->stream_rows = (v == 512 || v == 128) ? v : 0;
  }
  if (const char* c = std::getenv("SSM_STREAM_CTAS")) r->stream_ctas = std::atoi(c);
  if (const char* c = std::getenv("SSM_SSD_SPLIT")) r->ssd_split = std::atoi(c);
  return r;
}

std::atomic<RuntimeKnobs*> g_knobs{nullptr};
std::mutex g_knobs_mu;

}  // namespace

RuntimeKnobs runtime_knobs() {
  RuntimeKnobs* k = g_knobs.load(std::memory_order_acquire);
  if (!k) {
    std::lock_guard<std::mutex> lock(g_knobs_mu);
    k = g_knobs.load(std::memory_order_acquire);
    if (!k) {
      k = load_knobs();
      g_knobs.store(k, std::memory_order_release);
    }
  }
  return *k;
}

void reload_knobs() {
  std::lock_guard<std::mutex> lock(g_knobs_mu);
  // the previous copy stays allocated: a concurrent reader may still hold it
  g_knobs.store(load_knobs(), std::memory_order_release);
}

}  // namespace ssm

namespace {

// The error behind the calling thread's last SSM_ERR_CUDA (see ssm_last_cuda_error).
thread_local int g_last_cuda_error = 0;

ssm_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SSM_OK;
  const int drv = ssm::take_driver_error();
  g_last_cuda_error = drv ? 10000 + drv : (int)e;
  return SSM_ERR_CUDA;
}

bool aligned(const void* p, unsigned bytes) { return (reinterpret_cast<uintptr_t>(p) & (bytes - 1u)) == 0; }
bool aligned16(const void* p) { return aligned(p, 16); }

// Common validation of dims; seqlen is checked only for the scan.
ssm_status check_dims(const ssm_dims* d, bool need_len) {
  if (!d) return SSM_ERR_INVALID_ARG;
  if (d->batch < 1 || d->d_inner < 1 || d->d_state < 1) return SSM_ERR_INVALID_ARG;
  if (need_len && d->seqlen < 1) return SSM_ERR_INVALID_ARG;
  if (d->act != SSM_DTYPE_F32 && d->act != SSM_DTYPE_BF16) return SSM_ERR_INVALID_ARG;
  if (d->d_state > 64) return SSM_ERR_UNSUPPORTED;
  const int64_t lim = int64_t(1) << 62;
  const int64_t len = need_len ? d->seqlen : 1;
  if (d->batch > lim / d->d_inner) return SSM_ERR_UNSUPPORTED;
  const int64_t rows = d->batch * d->d_inner;
  if (len > lim / rows) return SSM_ERR_UNSUPPORTED;
  if (rows > lim / d->d_state) return SSM_ERR_UNSUPPORTED;
  // grid limits: the scan launches nchunks * batch * ctiles CTAs, the step rows * 16 / 256
  if (rows > (int64_t(1) << 35)) return SSM_ERR_UNSUPPORTED;
  return SSM_OK;
}

// Validation of dims for the Conv1D calls (d_state is not used; seqlen only for the sequence form).
ssm_status check_conv(const ssm_dims* d, bool need_len, int32_t width) {
  if (!d) return SSM_ERR_INVALID_ARG;
  if (d->batch < 1 || d->d_inner < 1 || (need_len && d->seqlen < 1)) return SSM_ERR_INVALID_ARG;
  if (d->act != SSM_DTYPE_F32 && d->act != SSM_DTYPE_BF16) return SSM_ERR_INVALID_ARG;
  if (width < 1) return SSM_ERR_INVALID_ARG;
  if (width > ssm::kMaxConvWidth) return SSM_ERR_UNSUPPORTED;
  // d_inner and batch are grid dimensions (at most 65535 each); tokens per row < 2^42
  if (d->d_inner > ssm::kMaxConvGridYZ || d->batch > ssm::kMaxConvGridYZ) return SSM_ERR_UNSUPPORTED;
  if (need_len && d->seqlen > (int64_t(1) << 42)) return SSM_ERR_UNSUPPORTED;
  return SSM_OK;
}

ssm::ConvCall conv_call(const void* x, const float* w, const float* bias, const void* s_in, void* out,
                        void* s_out, const ssm_dims* d, int32_t width, bool seq) {
  ssm::ConvCall k{};
  k.x = x; k.w = w; k.bias = bias; k.state_in = s_in; k.out = out; k.state_out = s_out;
  k.batch = d->batch; k.d_inner = d->d_inner; k.L = seq ? d->seqlen : 1; k.W = width; k.act = d->act;
  return k;
}

ssm::ScanArgs scan_args(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* bias, void* out, float* fs,
                        const ssm_dims* d, void* ws, const float* h0 = nullptr) {
  ssm::ScanArgs a{};
  a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.bias = bias;
  a.out = out; a.final_state = fs; a.h0 = h0;
  a.batch = d->batch; a.d_inner = d->d_inner; a.N = d->d_state; a.L = d->seqlen;
  a.act = d->act;
  a.ws = static_cast<unsigned char*>(ws);
  return a;
}

}  // namespace

namespace {
ssm_status check_ssd_dims(const ssd_dims* d) {
  if (!d) return SSM_ERR_INVALID_ARG;
  if (d->batch < 1 || d->seqlen < 0 || d->nheads < 1 || d->headdim < 1 || d->ngroups < 1 || d->d_state < 1)
    return SSM_ERR_INVALID_ARG;
  if (d->act != SSM_DTYPE_BF16 && d->act != SSM_DTYPE_F32) return SSM_ERR_INVALID_ARG;
  if (d->nheads % d->ngroups != 0) return SSM_ERR_INVALID_ARG;
  if (d->act != SSM_DTYPE_BF16 || d->headdim != ssm::kSsdHeadDim || d->d_state != ssm::kSsdState)
    return SSM_ERR_UNSUPPORTED;
  if (d->nheads > 65535 || d->batch > 65535) return SSM_ERR_UNSUPPORTED;
  return SSM_OK;
}
}  // namespace

extern "C" {

size_t ssm_scan_workspace_bytes(const ssm_dims* dims) {
  if (check_dims(dims, true) != SSM_OK) return 0;
  ssm::ScanArgs a = scan_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                              nullptr, nullptr, dims, nullptr);
  a.z = reinterpret_cast<const void*>(uintptr_t(16));  // the plan does not depend on z for sizing
  ssm::ScanPlan plan;
  if (!ssm::scan_make_plan(a, &plan)) return 0;
  // the z / no-z variants may differ in occupancy; size for the larger plan
  ssm::ScanArgs a2 = a;
  a2.z = nullptr;
  ssm::ScanPlan plan2;
  if (!ssm::scan_make_plan(a2, &plan2)) return 0;
  return plan.ws_bytes > plan2.ws_bytes ? plan.ws_bytes : plan2.ws_bytes;
}

}  // extern "C"

namespace {

ssm_status scan_fwd_impl(const void* u, const void* delta, const float* A, const void* B, const void* C,
                         const float* D, const void* z, const float* delta_bias, const float* h0, void* out,
                         float* final_state, const ssm_dims* dims, void* workspace, size_t workspace_bytes,
                         ssm_stream_t stream) {
  const ssm_status ds = check_dims(dims, true);
  if (ds != SSM_OK) return ds;
  if (!u || !delta || !A || !B || !C || !out) return SSM_ERR_INVALID_ARG;
  // element alignment is required; 16-byte alignment only selects the vector path
  const unsigned esz = dims->act == SSM_DTYPE_BF16 ? 2u : 4u;
  const void* act_ptrs[] = {u, delta, B, C, z, out};
  for (const void* p : act_ptrs)
    if (p && !aligned(p, esz)) return SSM_ERR_ALIGNMENT;
  const void* f32_ptrs[] = {A, D, delta_bias, final_state, h0};
  for (const void* p : f32_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_ALIGNMENT;
  ssm::ScanArgs a = scan_args(u, delta, A, B, C, D, z, delta_bias, out, final_state, dims, workspace, h0);
  ssm::ScanPlan plan;
  if (!ssm::scan_make_plan(a, &plan)) return SSM_ERR_UNSUPPORTED;
  if (plan.ws_bytes > 0) {
    if (!workspace || workspace_bytes < plan.ws_bytes) return SSM_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SSM_ERR_ALIGNMENT;
  }
  if (plan.ws_bytes == 0 && workspace_bytes < sizeof(unsigned) * 2) a.ws = nullptr;  // too small for the error word
  if (plan.ws_bytes == 0 && workspace && workspace_bytes >= sizeof(unsigned) * 2) {
    // clear the error word so ssm_scan_check on this workspace reports this call
    const ssm_status ms =
        cuda_status(cudaMemsetAsync(workspace, 0, sizeof(unsigned) * 2, reinterpret_cast<cudaStream_t>(stream)));
    if (ms != SSM_OK) return ms;
  }
  const cudaError_t e = ssm::scan_launch(a, plan, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

}  // namespace

extern "C" {

ssm_status ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, void* out,
                        float* final_state, const ssm_dims* dims, void* workspace, size_t workspace_bytes,
                        ssm_stream_t stream) {
  return scan_fwd_impl(u, delta, A, B, C, D, z, delta_bias, nullptr, out, final_state, dims, workspace,
                       workspace_bytes, stream);
}

ssm_status ssm_scan_fwd_from_state(const void* u, const void* delta, const float* A, const void* B,
                                   const void* C, const float* D, const void* z, const float* delta_bias,
                                   const float* initial_state, void* out, float* final_state,
                                   const ssm_dims* dims, void* workspace, size_t workspace_bytes,
                                   ssm_stream_t stream) {
  if (!initial_state) return SSM_ERR_INVALID_ARG;
  return scan_fwd_impl(u, delta, A, B, C, D, z, delta_bias, initial_state, out, final_state, dims, workspace,
                       workspace_bytes, stream);
}

ssm_status ssm_step(float* state, const void* x, const void* delta, const float* A, const void* B,
                    const void* C, const float* D, const void* z, const float* delta_bias, void* out,
                    const ssm_dims* dims, ssm_stream_t stream) {
  const ssm_status ds = check_dims(dims, false);
  if (ds != SSM_OK) return ds;
  if (!state || !x || !delta || !A || !B || !C || !out) return SSM_ERR_INVALID_ARG;
  const unsigned esz = dims->act == SSM_DTYPE_BF16 ? 2u : 4u;
  const void* act_ptrs[] = {x, delta, B, C, z, out};
  for (const void* p : act_ptrs)
    if (p && !aligned(p, esz)) return SSM_ERR_ALIGNMENT;
  const void* f32_ptrs[] = {D, delta_bias};
  for (const void* p : f32_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_ALIGNMENT;
  // state and A are read as float4 rows
  if (!aligned16(state) || !aligned16(A)) return SSM_ERR_ALIGNMENT;
  ssm::StepArgs a{};
  a.state = state; a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
  a.bias = delta_bias; a.out = out;
  a.batch = dims->batch; a.d_inner = dims->d_inner; a.N = dims->d_state; a.act = dims->act;
  const ssm::RuntimeKnobs knobs = ssm::runtime_knobs();
  ssm::StepKnobs sk{};
  sk.timeout_ns = knobs.lookback_timeout_ns;
  sk.fault = knobs.fault_step;
  sk.force_plain = knobs.force_step_plain;
  const cudaError_t e = ssm::step_launch(a, sk, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

ssm_status ssm_conv1d_fwd(const void* x, const float* weight, const float* bias, const void* initial_conv_state,
                          void* out, void* final_conv_state, const ssm_dims* dims, int32_t width,
                          ssm_stream_t stream) {
  const ssm_status ds = check_conv(dims, true, width);
  if (ds != SSM_OK) return ds;
  if (!x || !weight || !out) return SSM_ERR_INVALID_ARG;
  const unsigned esz = dims->act == SSM_DTYPE_BF16 ? 2u : 4u;
  const void* act_ptrs[] = {x, out, initial_conv_state, final_conv_state};
  for (const void* p : act_ptrs)
    if (p && !aligned(p, esz)) return SSM_ERR_ALIGNMENT;
  if (!aligned(weight, 4) || (bias && !aligned(bias, 4))) return SSM_ERR_ALIGNMENT;
  const ssm::ConvCall k = conv_call(x, weight, bias, width > 1 ? initial_conv_state : nullptr, out,
                                    width > 1 ? final_conv_state : nullptr, dims, width, true);
  return cuda_status(ssm::conv1d_fwd_launch(k, reinterpret_cast<cudaStream_t>(stream)));
}

ssm_status ssm_conv1d_step(void* conv_state, const void* x, const float* weight, const float* bias, void* out,
                           const ssm_dims* dims, int32_t width, ssm_stream_t stream) {
  const ssm_status ds = check_conv(dims, false, width);
  if (ds != SSM_OK) return ds;
  if (!x || !weight || !out || (width > 1 && !conv_state)) return SSM_ERR_INVALID_ARG;
  const unsigned esz = dims->act == SSM_DTYPE_BF16 ? 2u : 4u;
  const void* act_ptrs[] = {x, out, conv_state};
  for (const void* p : act_ptrs)
    if (p && !aligned(p, esz)) return SSM_ERR_ALIGNMENT;
  if (!aligned(weight, 4) || (bias && !aligned(bias, 4))) return SSM_ERR_ALIGNMENT;
  const ssm::ConvCall k = conv_call(x, weight, bias, nullptr, out, conv_state, dims, width, false);
  return cuda_status(ssm::conv1d_step_launch(k, reinterpret_cast<cudaStream_t>(stream)));
}

size_t ssm_scan_bwd_workspace_bytes(const ssm_dims* dims) {
  if (check_dims(dims, true) != SSM_OK || dims->d_state > 16) return 0;
  return ssm::scan_bwd_workspace_bytes(dims->batch, dims->d_inner, dims->d_state, dims->seqlen, false);
}

size_t ssm_scan_bwd_deterministic_workspace_bytes(const ssm_dims* dims) {
  if (check_dims(dims, true) != SSM_OK || dims->d_state > 16) return 0;
  return ssm::scan_bwd_workspace_bytes(dims->batch, dims->d_inner, dims->d_state, dims->seqlen, true);
}

}  // extern "C"

namespace {

ssm_status scan_bwd_impl(const void* u, const void* delta, const float* A, const void* B, const void* C,
                         const float* D, const void* z, const float* delta_bias, const void* dout, void* du,
                         void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz, float* ddelta_bias,
                         const ssm_dims* dims, void* workspace, size_t workspace_bytes, ssm_stream_t stream,
                         bool det) {
  const ssm_status ds = check_dims(dims, true);
  if (ds != SSM_OK) return ds;
  if (dims->d_state > 16) return SSM_ERR_UNSUPPORTED;
  if (!u || !delta || !A || !B || !C || !dout || !du || !ddelta || !dA || !dB || !dC) return SSM_ERR_INVALID_ARG;
  if ((D && !dD) || (z && !dz)) return SSM_ERR_INVALID_ARG;
  const unsigned esz = dims->act == SSM_DTYPE_BF16 ? 2u : 4u;
  const void* act_ptrs[] = {u, delta, B, C, z, dout, du, ddelta, dz};
  for (const void* p : act_ptrs)
    if (p && !aligned(p, esz)) return SSM_ERR_ALIGNMENT;
  const void* f32_ptrs[] = {A, D, delta_bias, dA, dB, dC, dD, ddelta_bias};
  for (const void* p : f32_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_ALIGNMENT;
  const size_t need = ssm::scan_bwd_workspace_bytes(dims->batch, dims->d_inner, dims->d_state, dims->seqlen, det);
  if (!workspace || workspace_bytes < need) return SSM_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SSM_ERR_ALIGNMENT;
  const int64_t rpc = ssm::scan_bwd_rows_per_cta();
  if (dims->batch * ((dims->d_inner + rpc - 1) / rpc) > INT32_MAX) return SSM_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t b = dims->batch, d = dims->d_inner, N = dims->d_state, L = dims->seqlen;
  if (!det) {
    // accumulated gradients start at zero (the deterministic mode writes them whole)
    cudaError_t me = cudaMemsetAsync(dA, 0, sizeof(float) * d * N, st);
    if (me == cudaSuccess) me = cudaMemsetAsync(dB, 0, sizeof(float) * b * L * N, st);
    if (me == cudaSuccess) me = cudaMemsetAsync(dC, 0, sizeof(float) * b * L * N, st);
    if (me == cudaSuccess && dD) me = cudaMemsetAsync(dD, 0, sizeof(float) * d, st);
    if (me == cudaSuccess && ddelta_bias) me = cudaMemsetAsync(ddelta_bias, 0, sizeof(float) * d, st);
    if (me != cudaSuccess) return cuda_status(me);
  }
  ssm::BwdArgs a{};
  a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.bias = delta_bias; a.dout = dout;
  a.du = du; a.ddelta = ddelta; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dz = dz; a.dbias = ddelta_bias;
  a.ckpt = static_cast<float*>(workspace);
  a.batch = b; a.d_inner = d; a.N = N; a.L = L; a.act = dims->act;
  a.det = det ? 1 : 0;
  a.force_chunks = ssm::runtime_knobs().bwd_chunks;
  a.form = ssm::runtime_knobs().bwd_form;
  return cuda_status(ssm::scan_bwd_launch(a, st));
}

}  // namespace

extern "C" {

ssm_status ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, const void* dout, void* du,
                        void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz, float* ddelta_bias,
                        const ssm_dims* dims, void* workspace, size_t workspace_bytes, ssm_stream_t stream) {
  return scan_bwd_impl(u, delta, A, B, C, D, z, delta_bias, dout, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias, dims,
                       workspace, workspace_bytes, stream, false);
}

ssm_status ssm_scan_bwd_deterministic(const void* u, const void* delta, const float* A, const void* B,
                                      const void* C, const float* D, const void* z, const float* delta_bias,
                                      const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC,
                                      float* dD, void* dz, float* ddelta_bias, const ssm_dims* dims,
                                      void* workspace, size_t workspace_bytes, ssm_stream_t stream) {
  return scan_bwd_impl(u, delta, A, B, C, D, z, delta_bias, dout, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias, dims,
                       workspace, workspace_bytes, stream, true);
}

ssm_status ssm_step_check(ssm_stream_t stream) {
  const ssm_status ss = cuda_status(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  if (ss != SSM_OK) return ss;
  unsigned word = 0;
  const ssm_status fs = cuda_status(ssm::step_error_fetch_clear(&word));
  if (fs != SSM_OK) return fs;
  return word ? SSM_ERR_TIMEOUT : SSM_OK;
}

size_t ssd_scan_workspace_bytes(const ssd_dims* dims) {
  if (check_ssd_dims(dims) != SSM_OK) return 0;
  return ssm::ssd_workspace_bytes(dims->batch, dims->seqlen, dims->nheads);
}

ssm_status ssd_scan_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
                        const void* z, const float* dt_bias, const float* initial_state, void* out,
                        float* final_state, const ssd_dims* dims, void* workspace, size_t workspace_bytes,
                        ssm_stream_t stream) {
  const ssm_status ds = check_ssd_dims(dims);
  if (ds != SSM_OK) return ds;
  // with seqlen = 0 there is nothing to read or write but the state
  if (!A || (dims->seqlen > 0 && (!x || !dt || !B || !C || !out))) return SSM_ERR_INVALID_ARG;
  const void* v16[] = {x, z, out, B, C};
  for (const void* p : v16)
    if (p && !aligned16(p)) return SSM_ERR_ALIGNMENT;
  if (dt && !aligned(dt, 2)) return SSM_ERR_ALIGNMENT;
  const void* f32_ptrs[] = {A, D, dt_bias, initial_state, final_state};
  for (const void* p : f32_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_ALIGNMENT;
  const size_t need = ssm::ssd_workspace_bytes(dims->batch, dims->seqlen, dims->nheads);
  if (!workspace || workspace_bytes < need) return SSM_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SSM_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // clear the error word so ssm_scan_check on this workspace reports this call
  const ssm_status ms = cuda_status(cudaMemsetAsync(workspace, 0, sizeof(unsigned) * 2, st));
  if (ms != SSM_OK) return ms;
  ssm::SsdArgs a{};
  a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.dt_bias = dt_bias;
  a.h0 = initial_state; a.out = out; a.final_state = final_state; a.ws = workspace;
  a.batch = dims->batch; a.L = dims->seqlen; a.H = dims->nheads; a.P = dims->headdim; a.G = dims->ngroups;
  a.N = dims->d_state;
  const ssm::RuntimeKnobs knobs = ssm::runtime_knobs();
  a.timeout_ns = knobs.lookback_timeout_ns;
  a.fault = knobs.fault_ssd ? 1 : 0;
  return cuda_status(ssm::ssd_launch(a, st));
}

ssm_status ssd_step(float* state, const void* x, const void* dt, const float* A, const void* B, const void* C,
                    const float* D, const void* z, const float* dt_bias, void* out, const ssd_dims* dims,
                    ssm_stream_t stream) {
  const ssm_status ds = check_ssd_dims(dims);
  if (ds != SSM_OK) return ds;
  if (!state || !x || !dt || !A || !B || !C || !out) return SSM_ERR_INVALID_ARG;
  const void* v16[] = {state, B, C};
  for (const void* p : v16)
    if (!aligned16(p)) return SSM_ERR_ALIGNMENT;
  const void* v2[] = {x, dt, z, out};
  for (const void* p : v2)
    if (p && !aligned(p, 2)) return SSM_ERR_ALIGNMENT;
  const void* f32_ptrs[] = {A, D, dt_bias};
  for (const void* p : f32_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_ALIGNMENT;
  if (dims->batch * dims->nheads > INT32_MAX) return SSM_ERR_UNSUPPORTED;
  ssm::SsdStepArgs a{};
  a.state = state; a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.dt_bias = dt_bias;
  a.out = out; a.batch = dims->batch; a.H = dims->nheads; a.P = dims->headdim; a.G = dims->ngroups;
  return cuda_status(ssm::ssd_step_launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

ssm_status ssm_scan_check(const void* workspace, size_t workspace_bytes) {
  if (!workspace || workspace_bytes < sizeof(unsigned) * 2) return SSM_OK;
  unsigned word = 0;
  const ssm_status cs = cuda_status(cudaMemcpy(&word, static_cast<const unsigned char*>(workspace) + sizeof(unsigned),
                                                sizeof(word), cudaMemcpyDeviceToHost));
  if (cs != SSM_OK) return cs;
  return (word & ssm::kErrTimeout) ? SSM_ERR_TIMEOUT : SSM_OK;
}

const char* ssm_status_string(ssm_status s) {
  switch (s) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
    case SSM_ERR_ALIGNMENT: return "SSM_ERR_ALIGNMENT";
    case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
    case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
  }
  return "SSM_ERR_UNKNOWN";
}

void ssm_test_hooks_reload(void) { ssm::reload_knobs(); }

int ssm_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
