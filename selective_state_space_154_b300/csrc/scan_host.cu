// ssm_scan_fwd_host: the scan of a sequence held in host memory, its copies to and
// from the device overlapped with the scan (declared in include/ssm_scan.h).
//
// The sequence is cut into pieces of piece_len tokens.  A piece is a scan that
// continues from the previous piece's end state (the affine maps of consecutive
// pieces compose, "Mambaとは？Transformer以外の系列モデル", Selective Scanは選択機構
// そのものではない), so the pieces run one after another on `stream` through
// ssm_scan_fwd_from_state, each on device staging buffers.  Two staging slots
// alternate: while piece k is scanned, piece k+1's inputs arrive on the host-to-device
// stream and piece k-1's output leaves on the device-to-host stream.  Events order
// the three streams; no call here waits on the host.
#include <cstdint>

#include "ssm_internal.h"
#include "ssm_scan.h"

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

// Staging layout: [scan workspace][state][slot 0][slot 1]; a slot holds u, delta, z,
// out ([rows][piece] each) and B, C ([batch][piece][d_state] each).
struct HostLayout {
  size_t ws, state_off, slot_off[2], u, delta, z, out, B, C, total;
};

void host_layout(const ssm_dims* d, int64_t piece, HostLayout* lay) {
  ssm_dims pd = *d;
  pd.seqlen = piece;
  lay->ws = align_up(ssm_scan_workspace_bytes(&pd));
  const size_t e = d->act == SSM_DTYPE_BF16 ? 2 : 4;
  const size_t rows = (size_t)d->batch * (size_t)d->d_inner;
  const size_t act = align_up(rows * (size_t)piece * e);
  const size_t bc = align_up((size_t)d->batch * (size_t)piece * (size_t)d->d_state * e);
  lay->u = 0;
  lay->delta = act;
  lay->z = 2 * act;
  lay->out = 3 * act;
  lay->B = 4 * act;
  lay->C = 4 * act + bc;
  const size_t slot = 4 * act + 2 * bc;
  lay->state_off = lay->ws;
  lay->slot_off[0] = lay->state_off + align_up(rows * (size_t)d->d_state * 4);
  lay->slot_off[1] = lay->slot_off[0] + slot;
  lay->total = lay->slot_off[1] + slot;
}

struct Events {
  cudaEvent_t ev[6] = {};
  int n = 0;
  cudaError_t create() {
    for (; n < 6; ++n) {
      const cudaError_t e = cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  ~Events() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);  // released once their work completes
  }
};

}  // namespace

extern "C" {

size_t ssm_scan_fwd_host_staging_bytes(const ssm_dims* dims, int64_t piece_len) {
  if (!dims || piece_len < 1 || dims->seqlen < 1 || dims->batch < 1 || dims->d_inner < 1 || dims->d_state < 1 ||
      dims->d_state > 64)
    return 0;
  HostLayout lay;
  host_layout(dims, piece_len < dims->seqlen ? piece_len : dims->seqlen, &lay);
  return lay.total;
}

ssm_status ssm_scan_fwd_host(const void* u, const void* delta, const float* A, const void* B, const void* C,
                             const float* D, const void* z, const float* delta_bias, const float* initial_state,
                             void* out, float* final_state, const ssm_dims* dims, int64_t piece_len, void* staging,
                             size_t staging_bytes, ssm_stream_t stream, ssm_stream_t h2d_stream,
                             ssm_stream_t d2h_stream) {
  if (!dims || !u || !delta || !A || !B || !C || !out || piece_len < 1) return SSM_ERR_INVALID_ARG;
  if (dims->batch < 1 || dims->d_inner < 1 || dims->d_state < 1 || dims->seqlen < 1) return SSM_ERR_INVALID_ARG;
  if (dims->act != SSM_DTYPE_F32 && dims->act != SSM_DTYPE_BF16) return SSM_ERR_INVALID_ARG;
  if (dims->d_state > 64) return SSM_ERR_UNSUPPORTED;
  const int64_t L = dims->seqlen;
  const int64_t P = piece_len < L ? piece_len : L;
  HostLayout lay;
  host_layout(dims, P, &lay);
  if (!staging || staging_bytes < lay.total) return SSM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(staging) & (kAlign - 1)) != 0) return SSM_ERR_ALIGNMENT;
  const size_t e = dims->act == SSM_DTYPE_BF16 ? 2 : 4;
  const size_t rows = (size_t)dims->batch * (size_t)dims->d_inner;
  const size_t N = (size_t)dims->d_state;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t hs = reinterpret_cast<cudaStream_t>(h2d_stream);
  cudaStream_t ds = reinterpret_cast<cudaStream_t>(d2h_stream);
  unsigned char* base = static_cast<unsigned char*>(staging);
  float* state = reinterpret_cast<float*>(base + lay.state_off);
  Events evs;
  if (evs.create() != cudaSuccess) return SSM_ERR_CUDA;
  cudaEvent_t* h2d_done = evs.ev;       // [slot]: the slot's inputs arrived
  cudaEvent_t* scan_done = evs.ev + 2;  // [slot]: the slot's scan finished (inputs free, output ready)
  cudaEvent_t* d2h_done = evs.ev + 4;   // [slot]: the slot's output left
  const int64_t npieces = (L + P - 1) / P;
  for (int64_t k = 0; k < npieces; ++k) {
    const int sl = (int)(k & 1);
    unsigned char* slot = base + lay.slot_off[sl];
    const int64_t t0 = k * P;
    const size_t len = (size_t)((L - t0) < P ? (L - t0) : P);
    // inputs of piece k, once the slot's previous scan has read its own
    if (k >= 2 && cudaStreamWaitEvent(hs, scan_done[sl], 0) != cudaSuccess) return SSM_ERR_CUDA;
    const void* rows_src[3] = {u, delta, z};
    const size_t rows_dst[3] = {lay.u, lay.delta, lay.z};
    for (int w = 0; w < 3; ++w) {
      if (!rows_src[w]) continue;
      if (cudaMemcpy2DAsync(slot + rows_dst[w], len * e, static_cast<const unsigned char*>(rows_src[w]) + t0 * e,
                            (size_t)L * e, len * e, rows, cudaMemcpyHostToDevice, hs) != cudaSuccess)
        return SSM_ERR_CUDA;
    }
    const void* bc_src[2] = {B, C};
    const size_t bc_dst[2] = {lay.B, lay.C};
    for (int w = 0; w < 2; ++w) {
      if (cudaMemcpy2DAsync(slot + bc_dst[w], len * N * e, static_cast<const unsigned char*>(bc_src[w]) + t0 * N * e,
                            (size_t)L * N * e, len * N * e, (size_t)dims->batch, cudaMemcpyHostToDevice,
                            hs) != cudaSuccess)
        return SSM_ERR_CUDA;
    }
    if (cudaEventRecord(h2d_done[sl], hs) != cudaSuccess) return SSM_ERR_CUDA;
    // scan of piece k from the state the previous piece left (or the initial state)
    if (cudaStreamWaitEvent(cs, h2d_done[sl], 0) != cudaSuccess) return SSM_ERR_CUDA;
    if (k >= 2 && cudaStreamWaitEvent(cs, d2h_done[sl], 0) != cudaSuccess) return SSM_ERR_CUDA;
    ssm_dims pd = *dims;
    pd.seqlen = (int64_t)len;
    const float* h0 = k == 0 ? initial_state : state;
    ssm_status st;
    if (h0)
      st = ssm_scan_fwd_from_state(slot + lay.u, slot + lay.delta, A, slot + lay.B, slot + lay.C, D,
                                   z ? slot + lay.z : nullptr, delta_bias, h0, slot + lay.out, state, &pd, base,
                                   lay.ws, stream);
    else
      st = ssm_scan_fwd(slot + lay.u, slot + lay.delta, A, slot + lay.B, slot + lay.C, D, z ? slot + lay.z : nullptr,
                        delta_bias, slot + lay.out, state, &pd, base, lay.ws, stream);
    if (st != SSM_OK) return st;
    if (cudaEventRecord(scan_done[sl], cs) != cudaSuccess) return SSM_ERR_CUDA;
    // output of piece k back to the host
    if (cudaStreamWaitEvent(ds, scan_done[sl], 0) != cudaSuccess) return SSM_ERR_CUDA;
    if (cudaMemcpy2DAsync(static_cast<unsigned char*>(out) + t0 * e, (size_t)L * e, slot + lay.out, len * e, len * e,
                          rows, cudaMemcpyDeviceToHost, ds) != cudaSuccess)
      return SSM_ERR_CUDA;
    if (cudaEventRecord(d2h_done[sl], ds) != cudaSuccess) return SSM_ERR_CUDA;
  }
  if (final_state &&
      cudaMemcpyAsync(final_state, state, rows * N * 4, cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
    return SSM_ERR_CUDA;
  // `stream` completes only after the last output copy
  if (cudaStreamWaitEvent(cs, d2h_done[(npieces - 1) & 1], 0) != cudaSuccess) return SSM_ERR_CUDA;
  return SSM_OK;
}

}  // extern "C"
