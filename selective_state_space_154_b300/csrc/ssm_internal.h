// Host/device shared declarations of the selective-scan library (not public).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

// Rows of a scan CTA (channels of one batch) and tokens of one staged tile.
constexpr int kRowsPerCta = 32;
constexpr int kTileTokens = 32;
constexpr int kStatesPerThread = 4;  // G: states of one row held by one thread (tile kernel)
constexpr int kRowsPerRowCta = 128;     // row kernel, small variant: rows per CTA (four CTAs per SM)
constexpr int kRowTokensPerStage = 32;  // row kernel: tokens per stage
// The correction of a chunk's outputs by its carried-in state stops once
// exp(A S) < 2^stop for every state with a nonzero carry-in: 2^-24 (below the
// fp32 rounding of the carry) for fp32 outputs, 2^-12 (1/8 of the half-ulp of a
// bf16 output relative to the carried state) for bf16 outputs.
template <typename T>
__host__ __device__ constexpr float corr_stop_log2() { return sizeof(T) == 2 ? -12.f : -24.f; }

enum ScanKind { kScanTiles = 0, kScanRows = 1, kScanStream = 2, kScanTiny = 3 };

// Small problems (rows × states ≤ kTinyMaxItems, L ≤ kTinyMaxSeq, d_state ≤ 32): the
// token-parallel kernel of scan_tiny.cu.
constexpr int kTinyMaxSeq = 256;
constexpr int64_t kTinyMaxItems = 2048;

// Workspace header (bytes): [0] ticket counter, [1] error word.
constexpr size_t kWsHeaderBytes = 256;

// Error bits in the device error word.
constexpr unsigned kErrTimeout = 1u;

// Launch plan of one scan call, a pure function of the dims and the device.
struct ScanPlan {
  int kind;           // ScanKind
  int npad;           // states per row rounded up to a multiple of 16 (16, 32, 48 or 64)
  int groups;         // npad / kStatesPerThread: threads per row
  int threads;        // threads per CTA: kRowsPerCta * groups (tiles), rows_per_cta * threads per row (rows)
  int rows_per_cta;   // channels per CTA
  int ctiles;         // channel tiles per batch (d_inner / rows_per_cta, rounded up)
  int64_t chunk_len;  // tokens per chunk (multiple of kTileTokens unless one chunk)
  int nchunks;        // chunks along the sequence (1: no carry between chunks)
  size_t smem_bytes;  // dynamic shared memory per CTA
  size_t ws_flags_off, ws_agg_off, ws_bytes;  // workspace layout (0 bytes when nchunks == 1)
};

struct ScanArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* bias;
  void* out;
  float* final_state;
  const float* h0;  // initial state [batch][d_inner][N], or nullptr for h = 0
  int64_t batch, d_inner, N, L;
  int act;  // 0 fp32, 1 bf16
  unsigned char* ws;
};

// Host-side test hooks from the SSM_* environment variables (see ssm_api.cu).
struct RuntimeKnobs {
  long long lookback_timeout_ns;  // device-side wait limit between chunks (0: default)
  bool fault_lookback;            // test hook: chunk waits on a flag nothing sets
  int force_chunks;               // >0: override the chunk count (tests)
  int force_kind;                 // -1: choose by shape; else a ScanKind (tests)
  int ctas_per_sm;                // >0: resident CTAs per SM assumed when splitting into chunks
  int force_tpr;                  // >0: threads per row of the row kernel (1 or 2)
  bool fault_step;                // test hook: the pipelined step's first wait never completes
  bool force_step_plain;          // SSM_FORCE_STEP=plain: the generic step kernel only
  int bwd_chunks;                 // >0: sequence chunks of the backward (tests)
  int bwd_form;                   // 1: the backward's four-threads-per-row gradient pass (tests)
  bool fault_ssd;                 // test hook: the SSD output kernel's first wait never completes
  int stream_rows;                // >0: rows per CTA of the streamed row kernel (512, 256 or 128)
  int stream_ctas;                // >0: work items (CTAs) of the streamed row kernel
  int force_ssd;                  // SSD form: 0 by shape, 1 one CTA per (batch, head), 2 chunk-parallel
  int ssd_split;                  // >0: the walking SSD form cuts every (batch, head) into this many segments
};
RuntimeKnobs runtime_knobs();  // the test hooks as last loaded (first use, or ssm_test_hooks_reload)
void reload_knobs();

bool scan_make_plan(const ScanArgs& a, ScanPlan* plan);  // false: unsupported dims
cudaError_t scan_launch(const ScanArgs& a, const ScanPlan& plan, cudaStream_t stream);
int rows_big_cta_rows(int act);  // rows of the one-CTA-per-SM variant of the row kernel
cudaError_t scan_rows_launch(const ScanArgs& a, const ScanPlan& plan, cudaStream_t stream);

// Streamed row kernel (scan_stream.cu): bf16, d_state 16, tensor-copied stages.
// Workspace: [header][flags: chunks × CTAs × warps][chunk aggregates h: chunks ×
// rows × 16][aggregate ΣΔ': chunks × rows].
struct StreamWs {
  unsigned* hdr;
  unsigned* flags;
  float* agg_h;
  float* agg_s;
  size_t flags_bytes;  // bytes from the start that are cleared per call (header + flags)
};
StreamWs stream_ws_layout(unsigned char* ws, int64_t work_items, int rows_per_cta, size_t* total);
bool stream_supported(const ScanArgs& a);
int take_driver_error();  // CUresult of the calling thread's last failed driver call (then cleared), or 0  // dtype, d_state, alignment and size limits
size_t stream_smem_bytes_for(int rows_per_cta);
constexpr int kStreamTokensPerStage = 32;  // streamed row kernel: tokens per stage
cudaError_t scan_stream_launch(const ScanArgs& a, const ScanPlan& plan, cudaStream_t stream);
bool tiny_supported(const ScanArgs& a);
cudaError_t scan_tiny_launch(const ScanArgs& a, cudaStream_t stream);

struct StepArgs {
  float* state;
  const void* x;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* bias;
  void* out;
  int64_t batch, d_inner, N;
  int act;
};
struct StepKnobs {
  long long timeout_ns;  // wait limit of the pipelined step kernel (0: 1 s)
  bool fault;            // test hook: the pipelined kernel's first wait never completes
  bool force_plain;      // use step_kernel even where the pipelined kernel applies
};
cudaError_t step_launch(const StepArgs& a, const StepKnobs& k, cudaStream_t stream);
// Causal depthwise Conv1D + SiLU (conv1d.cu).  state_in / state_out: [batch][d_inner][W-1]
// in the activation dtype; for the step, state_out is the in-out state and state_in unused.
struct ConvCall {
  const void* x;
  const float* w;
  const float* bias;
  const void* state_in;
  void* out;
  void* state_out;
  int64_t batch, d_inner, L;
  int W;
  int act;
};
constexpr int kMaxConvWidth = 8;
constexpr int64_t kMaxConvGridYZ = 65535;  // d_inner and batch index grid dimensions y / z
cudaError_t conv1d_fwd_launch(const ConvCall& k, cudaStream_t stream);
cudaError_t conv1d_step_launch(const ConvCall& k, cudaStream_t stream);

// Backward of the scan (scan_bwd.cu).  dA, dB, dC, dD, dbias are accumulated
// (zeroed by the caller); ckpt is the workspace of scan_bwd_workspace_bytes().
// force_chunks > 0 fixes the number of sequence chunks (tests); the launcher
// fills nblk, ctiles, nchunks, cblk and kmax.
struct BwdArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* bias;
  const void* dout;
  void* du;
  void* ddelta;
  float* dA;
  float* dB;
  float* dC;
  float* dD;
  void* dz;
  float* dbias;
  float* ckpt;
  // deterministic mode: per-CTA partial sums, reduced in a fixed order by a third launch
  float* part_bc;   // [ctile][batch][L][B | C][N]
  float* part_row;  // [batch][chunk][d_inner][dA 0..N-1 | dD | dbias]
  int64_t batch, d_inner, N, L, nblk, cblk;
  int ctiles, act, nchunks, kmax, force_chunks, det;
  // the chunk pass's chunks: each of the gradient pass's chunks is `sub` of them, of cblk_f
  // blocks (nfine in all); sub = 1 except for the one-thread-per-row form
  int64_t cblk_f;
  int nfine, sub;
  int form;  // gradient pass: 0 by shape, 1 four threads per row (test hook)
};
// deterministic = false: the checkpoints and chunk summaries; true: those plus the partial sums
size_t scan_bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t N, int64_t L, bool deterministic);
int scan_bwd_rows_per_cta();
cudaError_t scan_bwd_launch(BwdArgs p, cudaStream_t stream);

// Mamba-2 (SSD) layer scan (ssd.cu): x, z, out [batch][L][H][P]; dt [batch][L][H];
// B, C [batch][L][G][N] (bf16); A, D, dt_bias [H]; h0, final_state [batch][H][P][N]
// (fp32).  ws: the workspace of ssd_workspace_bytes() (error word at byte 4).
struct SsdArgs {
  const void* x;
  const void* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* dt_bias;
  const float* h0;
  void* out;
  float* final_state;
  void* ws;
  int64_t batch, L, H, P, G, N, nchunks;
  long long timeout_ns;
  int heads_per_cta;  // set by the launcher
  int fault;          // test hook: the output kernel waits on an mbarrier nothing arrives on
};
constexpr int kSsdChunk = 128;    // tokens per chunk
constexpr int kSsdHeadDim = 64;   // supported headdim
constexpr int kSsdState = 128;    // supported d_state
constexpr int kSsdWalkMinPairs = 64;  // batch · heads from which one CTA walks each (batch, head)
size_t ssd_workspace_bytes(int64_t batch, int64_t L, int64_t H);
cudaError_t ssd_launch(SsdArgs p, cudaStream_t stream);
// the sequence-walking form (ssd_walk.cu): one CTA per (batch, head), no workspace
// beyond the error word
bool ssd_use_walk(int64_t batch, int64_t L, int64_t H);
// How the walking form splits the work: units [0, full_units) whole, the rest in seg_k
// segments each, handing states over through `slots` workspace slots.
struct WalkSplit {
  int64_t full_units;
  int seg_k;
  int64_t slots;
};
WalkSplit ssd_walk_split(int64_t batch, int64_t H, int64_t L);
size_t ssd_walk_workspace_bytes(const WalkSplit& sp);
cudaError_t ssd_walk_launch(SsdArgs p, void* ws, cudaStream_t stream);

// One decode token of the Mamba-2 layer (ssd.cu): state [batch][H][P][N] fp32 in place;
// x, z, out [batch][H][P], dt [batch][H], B, C [batch][G][N] (bf16); A, D, dt_bias [H].
struct SsdStepArgs {
  float* state;
  const void* x;
  const void* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* dt_bias;
  void* out;
  int64_t batch, H, P, G;
};
cudaError_t ssd_step_launch(const SsdStepArgs& p, cudaStream_t stream);

// Reads and clears the sticky error word of the pipelined step kernel (current device).
cudaError_t step_error_fetch_clear(unsigned* word);

}  // namespace ssm
