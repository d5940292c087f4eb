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

enum ScanKind { kScanTiles = 0, kScanRows = 1 };

// Workspace header (bytes): [0] ticket counter, [1] error word.
constexpr size_t kWsHeaderBytes = 256;

// Error bits in the device error word.
constexpr unsigned kErrTimeout = 1u;

// Launch plan of one scan call, a pure function of the dims and the device.
struct ScanPlan {
  int kind;           // ScanKind
  int npad;           // states per row rounded up to a multiple of 16 (16, 32, 48 or 64)
  int groups;         // npad / kStatesPerThread: threads per row
  int threads;        // kRowsPerCta * groups
  int ctiles;         // channel tiles per batch (32 channels for kScanTiles, 128 for kScanRows)
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
  int64_t batch, d_inner, N, L;
  int act;  // 0 fp32, 1 bf16
  unsigned char* ws;
};

// Host-side knobs read from the environment at every call (see ssm_api.cu).
struct RuntimeKnobs {
  long long lookback_timeout_ns;  // device-side wait limit between chunks (0: default)
  bool fault_lookback;            // test hook: chunk waits on a flag nothing sets
  int force_chunks;               // >0: override the chunk count (tests)
  int force_kind;                 // -1: choose by shape; else a ScanKind (tests)
  int ctas_per_sm;                // >0: resident CTAs per SM assumed when splitting into chunks
};
RuntimeKnobs runtime_knobs();

bool scan_make_plan(const ScanArgs& a, ScanPlan* plan);  // false: unsupported dims
cudaError_t scan_launch(const ScanArgs& a, const ScanPlan& plan, cudaStream_t stream);
int rows_big_cta_rows(int act);  // rows of the one-CTA-per-SM variant of the row kernel
cudaError_t scan_rows_launch(const ScanArgs& a, const ScanPlan& plan, cudaStream_t stream);

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
cudaError_t step_launch(const StepArgs& a, cudaStream_t stream);

}  // namespace ssm
