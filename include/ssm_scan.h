/*
 * ssm_scan.h — C ABI of a B300 (sm_103a) selective state-space scan (S6).
 *
 * The operation (per batch b, channel c, state n; diagonal A):
 *
 *   Δ_t   = softplus(Δraw[b,c,t] + bias[c])
 *   Ā_t   = exp(Δ_t · A[c,n])                                  zero-order hold
 *   B̄_t   = (Δ_t A)^-1 (exp(Δ_t A) - 1) Δ_t B[b,t,n]
 *         = expm1(Δ_t A[c,n]) / A[c,n] · B[b,t,n]   (Δ_t · B[b,t,n] when A[c,n] = 0)
 *   h_t   = Ā_t h_{t-1} + B̄_t u[b,c,t]                           h_0 = 0
 *   y_t   = Σ_n C[b,t,n] h_t[n] + D[c] u[b,c,t]
 *   out   = y_t · silu(z[b,c,t])          silu(z) = z / (1 + exp(-z))
 *
 * Sources: "State Space Models（SSM）とMamba" §2.2 離散化 (ZOH formulas, the
 * discrete recurrence), §2.4 二つのモード (parallel training mode, recurrent
 * fixed-memory inference mode), §4.2 Selective SSM (Δ, B, C per token, A fixed);
 * "Mambaとは？Transformer以外の系列モデル", sections 状態空間モデルを一つの式から
 * 理解する (readout with the D skip term), Mamba blockのarchitecture (SiLU gate
 * multiplies the SSM branch) and training、prefill、decodeでは計算の姿が違う
 * (prefill runs the scan over the prompt, decode updates the state once per
 * token).  softplus(Δraw + bias) is this library's parameterisation of the
 * positive step size, which the pages leave open.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates nothing and never frees caller memory.  Its only global state:
 *    the decode step's device error word (read and cleared by ssm_step_check),
 *    the static scratch array of ssm_scan_fwd_noalloc with its cached device
 *    address, and the test hooks read from the environment (see the end of
 *    this header).  Every other call works only on the memory it is given.
 *  - Layouts are dense row-major:
 *        u, delta, z, out          [batch][d_inner][seqlen]   (act dtype)
 *        B, C                      [batch][seqlen][d_state]   (act dtype)
 *        A                         [d_inner][d_state]         (float32)
 *        D, delta_bias             [d_inner]                  (float32)
 *        final_state / state       [batch][d_inner][d_state]  (float32)
 *    (for ssm_step, seqlen is 1: x, delta, z, out are [batch][d_inner] and
 *    B, C are [batch][d_state].)
 *  - act dtype is float32 or bfloat16 (ssm_dims.act); outputs of the act dtype
 *    are rounded to nearest even.  State and all arithmetic are float32.
 *  - Work is enqueued on `stream` and runs asynchronously; the call returns
 *    once the work is queued.  Arguments are validated on the host before any
 *    launch, and a failed validation queues nothing.
 *  - Inputs are never written.  out must not overlap any input.
 *  - NaN / Inf inputs are not checked and propagate.
 *  - Limits: 1 ≤ d_state ≤ 64; batch, d_inner, seqlen ≥ 1;
 *    batch·d_inner·seqlen < 2^62.
 *  - Alignment: every pointer must be aligned to its element (2 bytes for bf16,
 *    4 for float32 arrays), else SSM_ERR_ALIGNMENT.  16-byte alignment of u,
 *    delta, z, B, C and out, with rows whose byte length is a multiple of 16,
 *    selects the vectorised kernels (for bf16 with d_state 16 and seqlen a
 *    multiple of 8, the tensor-copy kernel); other inputs take element copies.
 *    The Mamba-2 calls below state their own, stricter, alignment.
 */
#ifndef SSM_SCAN_H_
#define SSM_SCAN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* ssm_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  SSM_OK = 0,
  SSM_ERR_INVALID_ARG = 1, /* null required pointer, non-positive size, bad dtype */
  SSM_ERR_UNSUPPORTED = 2, /* d_state > 64, or a size beyond the limits above */
  SSM_ERR_ALIGNMENT = 3,   /* a pointer not aligned as required (see Conventions) */
  SSM_ERR_WORKSPACE = 4,   /* workspace missing or smaller than ssm_scan_workspace_bytes() */
  SSM_ERR_CUDA = 5,        /* a CUDA runtime call or a launch failed */
  SSM_ERR_TIMEOUT = 6      /* a device-side wait between chunks gave up (see ssm_scan_check) */
} ssm_status;

typedef enum { SSM_DTYPE_F32 = 0, SSM_DTYPE_BF16 = 1 } ssm_dtype;

typedef struct {
  int64_t batch;
  int64_t d_inner;
  int64_t d_state; /* N */
  int64_t seqlen;  /* L; ignored by ssm_step */
  int32_t act;     /* ssm_dtype of u, delta, z, B, C, out */
  int32_t reserved;
} ssm_dims;

/*
 * Bytes of device workspace ssm_scan_fwd needs for `dims` on the current
 * device (0 means none is needed and workspace may be NULL).  Long sequences
 * with few (batch, channel) rows are split into chunks along the sequence;
 * the workspace then carries each chunk's state summary to the next chunk.
 * Returns 0 for invalid dims as well (ssm_scan_fwd reports those).
 */
SSM_API size_t ssm_scan_workspace_bytes(const ssm_dims* dims);

/*
 * Parallel (training / prefill) mode over the whole sequence, initial state 0.
 *   u, delta (= Δraw), A, B, C, out, dims: required.
 *   D, z, delta_bias: may be NULL (no skip term / no gate / zero bias).
 *   final_state: may be NULL; otherwise receives h_L.
 *   workspace: device memory of at least ssm_scan_workspace_bytes(dims) bytes,
 *     16-byte aligned when any is needed, caller-owned, contents on entry
 *     irrelevant, not shared with a concurrent call.  It also holds a device
 *     error word read by ssm_scan_check.
 * Returns SSM_OK when the work was queued.
 */
SSM_API ssm_status ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                        const void* C, const float* D, const void* z, const float* delta_bias,
                        void* out, float* final_state, const ssm_dims* dims, void* workspace,
                        size_t workspace_bytes, ssm_stream_t stream);

/*
 * ssm_scan_fwd starting from a given state instead of h = 0: the scan of a
 * sequence that continues an earlier one (a prompt processed in pieces, or a
 * prefill resumed from a decode state), the state being carried between the
 * two modes as "State Space Models（SSM）とMamba" §2.4 二つのモード and
 * "Mambaとは？Transformer以外の系列モデル", section training、prefill、decodeでは
 * 計算の姿が違う describe.  Scanning [0, L) equals scanning [0, k) and then
 * [k, L) from the first call's final_state.
 *   initial_state: [batch][d_inner][d_state] float32, required, 4-byte aligned,
 *     read only.  final_state may be the same array (the state is then updated
 *     in place); any other overlap with an output is not allowed.
 *   All other arguments, the workspace and the errors as for ssm_scan_fwd.
 */
SSM_API ssm_status ssm_scan_fwd_from_state(const void* u, const void* delta, const float* A, const void* B,
                                   const void* C, const float* D, const void* z, const float* delta_bias,
                                   const float* initial_state, void* out, float* final_state,
                                   const ssm_dims* dims, void* workspace, size_t workspace_bytes,
                                   ssm_stream_t stream);

/*
 * ssm_scan_fwd for a sequence held in HOST memory, the copies to and from the
 * device overlapped with the scan: the sequence is cut into pieces of piece_len
 * tokens; each piece's u, delta, z, B and C are copied to device staging memory on
 * h2d_stream, scanned on `stream` from the state the previous piece left
 * (initial_state, or 0, for the first), and its output copied back on d2h_stream.
 * Two staging slots alternate, so one piece's copies run while another is scanned.
 * Scanning in pieces equals one scan of the whole sequence (the state carries
 * across, as for ssm_scan_fwd_from_state).
 *   u, delta, z, out: [batch][d_inner][seqlen] and B, C: [batch][seqlen][d_state]
 *     in HOST memory (page-locked for the copies to overlap); z may be NULL.
 *   A, D, delta_bias, initial_state (NULL: h = 0), final_state (NULL: not
 *     written): DEVICE memory, as for ssm_scan_fwd_from_state.
 *   staging: device memory of ssm_scan_fwd_host_staging_bytes(dims, piece_len)
 *     bytes, 256-byte aligned, caller-owned; its first bytes are the pieces' scan
 *     workspace, so ssm_scan_check(staging, bytes) reports their device-side waits.
 *   stream, h2d_stream, d2h_stream: may be the same stream (then nothing overlaps).
 *     The call returns once everything is queued; `stream` is made to wait for the
 *     last output copy, so synchronising `stream` completes the call.
 * Errors: as for ssm_scan_fwd, plus SSM_ERR_INVALID_ARG for piece_len < 1 and
 * SSM_ERR_WORKSPACE for missing or small staging memory.
 */
SSM_API size_t ssm_scan_fwd_host_staging_bytes(const ssm_dims* dims, int64_t piece_len);
SSM_API ssm_status ssm_scan_fwd_host(const void* u, const void* delta, const float* A, const void* B, const void* C,
                                     const float* D, const void* z, const float* delta_bias,
                                     const float* initial_state, void* out, float* final_state,
                                     const ssm_dims* dims, int64_t piece_len, void* staging, size_t staging_bytes,
                                     ssm_stream_t stream, ssm_stream_t h2d_stream, ssm_stream_t d2h_stream);

/*
 * Backward of ssm_scan_fwd (from h = 0): the gradients of ℓ = Σ dout·out with
 * respect to every input, the states being recomputed from checkpoints in the
 * workspace instead of stored ("Mambaとは？Transformer以外の系列モデル", section
 * Selective Scanは選択機構そのものではない: recomputation as the third
 * hardware-aware ingredient).  d_state ≤ 16 (SSM_ERR_UNSUPPORTED above).
 *   Inputs as for ssm_scan_fwd, plus dout [batch][d_inner][seqlen] (act dtype).
 *   du, ddelta: [batch][d_inner][seqlen], act dtype (ddelta is dℓ/dΔraw).
 *   dz: same shape, required when z is given (else ignored and may be NULL).
 *   dA: [d_inner][d_state] float32; dB, dC: [batch][seqlen][d_state] float32.
 *   dD: [d_inner] float32, required when D is given; ddelta_bias: [d_inner]
 *     float32 or NULL (dℓ/dbias, whether or not delta_bias is given).
 *   The call zeroes dA, dB, dC, dD and ddelta_bias, then accumulates into them
 *   (the sums over batch and channels use atomic adds, so their last bits may
 *   differ from call to call; ssm_scan_bwd_deterministic below does not).
 *   workspace: at least ssm_scan_bwd_workspace_bytes(dims) bytes, 16-byte
 *   aligned, caller-owned; it holds the state every 8 tokens of every row and,
 *   the sequence being split into chunks that run in parallel, each chunk's
 *   end state, Δ sum and outgoing adjoint (at most 32 chunks of ≥ 16 tokens).
 * Two kernel launches on `stream` after the zeroing copies; no host sync.
 * Outputs must not overlap inputs or each other.
 */
SSM_API size_t ssm_scan_bwd_workspace_bytes(const ssm_dims* dims);
SSM_API ssm_status ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z, const float* delta_bias,
                                const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC,
                                float* dD, void* dz, float* ddelta_bias, const ssm_dims* dims, void* workspace,
                                size_t workspace_bytes, ssm_stream_t stream);

/*
 * The same gradients, bitwise reproducible: the sums over channels (dB, dC) and over
 * batch rows and sequence chunks (dA, dD, ddelta_bias) are not accumulated by atomic
 * adds but written as per-CTA partial sums into the workspace and added by a third
 * launch in a fixed order.  Arguments as for ssm_scan_bwd; the workspace must hold
 * ssm_scan_bwd_deterministic_workspace_bytes(dims) bytes (the checkpoints, plus
 * 4·2·d_state bytes per (64-channel tile, batch, token) and 4·(d_state + 2) bytes
 * per (batch, chunk, channel) of partials).  dA, dB, dC, dD, ddelta_bias need not be
 * zeroed.  Three kernel launches on `stream`; no host sync.  Repeated calls on the same
 * inputs, device and dims return identical bits, provided the input arrays keep their
 * 16-byte alignment or lack of it (bf16 rows at d_state 16 with L a multiple of 8 take a
 * kernel with one thread per row when u, delta, dout, z, B and C are 16-byte aligned,
 * else one with four, and the two add in different orders).
 */
SSM_API size_t ssm_scan_bwd_deterministic_workspace_bytes(const ssm_dims* dims);
SSM_API ssm_status ssm_scan_bwd_deterministic(const void* u, const void* delta, const float* A, const void* B,
                                              const void* C, const float* D, const void* z,
                                              const float* delta_bias, const void* dout, void* du, void* ddelta,
                                              float* dA, float* dB, float* dC, float* dD, void* dz,
                                              float* ddelta_bias, const ssm_dims* dims, void* workspace,
                                              size_t workspace_bytes, ssm_stream_t stream);

/*
 * Recurrent (decode) mode: one token for every (batch, channel) row, updating
 * `state` in place (h ← Ā h + B̄ x) and writing out = (C·h + D x) · silu(z).
 *   state, x, delta, A, B, C, out, dims: required (dims->seqlen is ignored).
 *   D, z, delta_bias: may be NULL.
 * A and delta_bias are needed to discretise (A enters Ā and B̄; the bias is
 * part of the step size), so they are arguments of the step as of the scan.
 */
SSM_API ssm_status ssm_step(float* state, const void* x, const void* delta, const float* A,
                    const void* B, const void* C, const float* D, const void* z,
                    const float* delta_bias, void* out, const ssm_dims* dims,
                    ssm_stream_t stream);

/*
 * After the stream that ran ssm_scan_fwd has been synchronised: reads the
 * device error word in `workspace` (synchronous device-to-host copy of 4
 * bytes) and returns SSM_ERR_TIMEOUT if a wait between chunks gave up,
 * SSM_OK otherwise (also when workspace is NULL).  Each ssm_scan_fwd call
 * clears the word before its kernel runs.
 */
SSM_API ssm_status ssm_scan_check(const void* workspace, size_t workspace_bytes);

/*
 * Causal depthwise Conv1D + SiLU over whole sequences: the short convolution of
 * the Mamba block's main branch that feeds the selective SSM
 * ("Mambaとは？Transformer以外の系列モデル", section Mamba blockのarchitecture,
 * steps 2 and 3).  For every (batch, channel) row, with W = width:
 *   out[t] = silu(bias[c] + Σ_{k<W} weight[c][k] · x̃[t - (W-1) + k])
 * where x̃ is the row prefixed by the W-1 inputs before it, initial_conv_state
 * (oldest first), or zeros when it is NULL.  final_conv_state (may be NULL)
 * receives the last W-1 entries of x̃: the state ssm_conv1d_step continues from.
 *   x, out: [batch][d_inner][seqlen], act dtype (ssm_dims.act; d_state ignored).
 *   weight: [d_inner][width] float32; bias: [d_inner] float32 or NULL.
 *   initial_conv_state, final_conv_state: [batch][d_inner][width-1], act dtype
 *     (the raw inputs, so they are exact), or NULL; unused when width is 1.
 *   1 <= width <= 8, batch and d_inner <= 65535 (SSM_ERR_UNSUPPORTED otherwise).
 *   Element alignment as for the scan.
 *   out and final_conv_state must not overlap x, initial_conv_state or each
 *   other.  No workspace; stream-ordered and asynchronous like ssm_scan_fwd.
 */
SSM_API ssm_status ssm_conv1d_fwd(const void* x, const float* weight, const float* bias,
                                  const void* initial_conv_state, void* out, void* final_conv_state,
                                  const ssm_dims* dims, int32_t width, ssm_stream_t stream);

/*
 * One decode token of the same convolution ("Mambaとは？…", section training、
 * prefill、decodeでは計算の姿が違う: each layer keeps a state for its short causal
 * Conv1D next to the SSM state).  For every row: window = (conv_state, x);
 * out = silu(bias + Σ_k weight[c][k] · window[k]); conv_state ← window[1..W-1].
 *   conv_state: [batch][d_inner][width-1], act dtype, updated in place
 *     (required unless width is 1).
 *   x, out: [batch][d_inner], act dtype; weight, bias as for ssm_conv1d_fwd.
 */
SSM_API ssm_status ssm_conv1d_step(void* conv_state, const void* x, const float* weight, const float* bias,
                                   void* out, const ssm_dims* dims, int32_t width, ssm_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears this library's device-side step
 * error word on the current device: SSM_ERR_TIMEOUT if, since the last check,
 * an ssm_step on this device gave up waiting for its state to arrive in shared
 * memory (bounded at 1 s, or SSM_LOOKBACK_TIMEOUT_MS), in which case the state
 * rows of the affected tiles were left unchanged and their outputs are
 * undefined; SSM_OK otherwise.  The word is shared by all streams of the device.
 */
SSM_API ssm_status ssm_step_check(ssm_stream_t stream);

/* Static, human-readable name of a status. */
SSM_API const char* ssm_status_string(ssm_status s);

/*
 * The error behind the calling thread's most recent SSM_ERR_CUDA: the CUDA
 * runtime's cudaError_t code, or 10000 + the driver's CUresult when a driver
 * call failed (the encoding of a tensor-copy descriptor).  0 if none occurred.
 */
SSM_API int ssm_last_cuda_error(void);

/*
 * ssm_scan_fwd for callers that cannot allocate device memory: a plug-in whose
 * host framework owns every allocation, a serving loop that may not call
 * cudaMalloc after start-up, or any caller with a fixed device-memory budget.
 * (This entry point has no counterpart in the pages; it is a property of the
 * library, not of the method.)
 *
 * Same arguments and results as ssm_scan_fwd without the workspace.  The scratch
 * that long sequences need (the carry between chunks) comes from one static
 * device array of SSM_NOALLOC_SCRATCH_BYTES inside this library, which exists
 * on every device that loads the library until the process exits.  The call
 * allocates nothing and frees nothing.
 *  - Returns SSM_ERR_WORKSPACE when ssm_scan_workspace_bytes(dims) exceeds
 *    SSM_NOALLOC_SCRATCH_BYTES; use ssm_scan_fwd with your own workspace then.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it with the id of the current context;
 *    make that first call before any stream capture.  After cudaDeviceReset, or
 *    under another context on the same device, the next call looks the address
 *    up again (that call, too, must not be captured).
 *  - All calls share the one array, and each call resets what must start at
 *    zero.  Calls whose work overlaps on the GPU (concurrent streams, or other
 *    threads) race on the array: serialise them.
 *  - A wait between chunks that gives up sets its error bit in the shared
 *    array, where ssm_scan_check cannot see it; callers who need that report
 *    use ssm_scan_fwd.
 */
#define SSM_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
/* SSM_NOALLOC_SCRATCH_BYTES as built into this library (for callers without the header). */
SSM_API size_t ssm_noalloc_scratch_bytes(void);
SSM_API ssm_status ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z, const float* delta_bias,
                                void* out, float* final_state, const ssm_dims* dims, ssm_stream_t stream);

/*
 * Mamba-2 layer scan (state space duality, SSD): each head's state matrix is a
 * scalar a_h times the identity, so the layer equals causal linear attention
 * with queries C, keys B, values φ·x and the decay mask e^{Σ Δa}
 * ("Mambaとは？Transformer以外の系列モデル", section Mamba-2とTransformerとの関係性;
 * "State Space Models（SSM）とMamba" §4.6 Mamba-2).  Per head h, with
 * Δ_t = softplus(dt[t,h] + dt_bias[h]), Ā_t = e^{Δ_t a_h}, φ_t = (Ā_t − 1)/a_h
 * (Δ_t when a_h = 0), the state (headdim × d_state) follows
 *   H_t = Ā_t H_{t-1} + φ_t x_t B_tᵀ,   out_t = (H_t C_t + D_h x_t) · silu(z_t)
 * from H_0 = initial_state (zero when NULL).  Evaluated in chunks of 128
 * tokens on the tensor cores (bf16 operands, fp32 accumulation; the operands
 * the library computes — the masked decay-weighted C·Bᵀ, the weighted x of a
 * chunk's state and the state entering a chunk — go in as two bf16 terms each,
 * and the state is carried between chunks in fp32).  With batch · nheads ≥ 64
 * one CTA walks the whole sequence of each (batch, head), the state in
 * registers; below that the chunks run in parallel with a chunk-state pass
 * through the workspace.
 *   x, z, out: [batch][seqlen][nheads][headdim] bf16, 16-byte aligned (z may be NULL).
 *   dt: [batch][seqlen][nheads] bf16 (Δraw).
 *   B, C: [batch][seqlen][ngroups][d_state] bf16, 16-byte aligned; head h
 *     reads group h / (nheads / ngroups).
 *   A, D, dt_bias: [nheads] float32 (D, dt_bias may be NULL).
 *   initial_state, final_state: [batch][nheads][headdim][d_state] float32, or NULL.
 *   workspace: at least ssd_scan_workspace_bytes(dims) bytes, 16-byte aligned,
 *     caller-owned; its error word is read by ssm_scan_check (a tensor-core
 *     wait that ran out of time).  256 bytes (the error words) for the
 *     sequence-walking form; the chunk states besides for the chunk-parallel one.
 * seqlen may be 0: x, dt, B, C, z and out may then be NULL and final_state
 * receives the initial state.
 * Supported: act = SSM_DTYPE_BF16, headdim = 64, d_state = 128, nheads and batch
 * ≤ 65535 (else SSM_ERR_UNSUPPORTED); nheads a multiple of ngroups (else
 * SSM_ERR_INVALID_ARG).  One kernel launch on `stream` (three in the
 * chunk-parallel form); no host sync.
 */
typedef struct {
  int64_t batch;
  int64_t seqlen;
  int64_t nheads;
  int64_t headdim;  /* P */
  int64_t ngroups;  /* G: heads share B and C within a group */
  int64_t d_state;  /* N */
  int32_t act;      /* ssm_dtype of x, dt, z, B, C, out */
  int32_t reserved;
} ssd_dims;

SSM_API size_t ssd_scan_workspace_bytes(const ssd_dims* dims);
SSM_API ssm_status ssd_scan_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                                const float* D, const void* z, const float* dt_bias, const float* initial_state,
                                void* out, float* final_state, const ssd_dims* dims, void* workspace,
                                size_t workspace_bytes, ssm_stream_t stream);

/*
 * Recurrent (decode) mode of the Mamba-2 layer: one token for every (batch, head),
 * with `state` updated in place:
 *   H ← Ā H + φ x Bᵀ,   out = (H C + D x) · silu(z)
 * (Ā, φ and the step size as for ssd_scan_fwd; the two modes of the pages,
 * "State Space Models（SSM）とMamba" §2.4 二つのモード).  Continues a prefill whose
 * final_state it is given.
 *   state: [batch][nheads][headdim][d_state] float32, 16-byte aligned (in-out).
 *   x, z, out: [batch][nheads][headdim] bf16 (z may be NULL).
 *   dt: [batch][nheads] bf16 (Δraw).
 *   B, C: [batch][ngroups][d_state] bf16, 16-byte aligned.
 *   A, D, dt_bias: [nheads] float32 (D, dt_bias may be NULL).
 *   dims: as for ssd_scan_fwd (seqlen is ignored), with the same supported sizes.
 * One kernel launch on `stream`; no workspace; out must not alias an input.
 */
SSM_API ssm_status ssd_step(float* state, const void* x, const void* dt, const float* A, const void* B,
                            const void* C, const float* D, const void* z, const float* dt_bias, void* out,
                            const ssd_dims* dims, ssm_stream_t stream);

/*
 * Test hooks.  The library reads these environment variables once, at the first
 * call that needs them, and again only inside ssm_test_hooks_reload(); no other
 * call reads the environment.  They exist for the test suite (forcing a kernel,
 * a chunk count, or a device-side wait that never completes) and are not part of
 * the supported interface:
 *   SSM_FORCE_KERNEL = tiles | rows | stream | tiny   scan kernel, where the shape allows it
 *   SSM_FORCE_KERNEL = ssd_walk | ssd_chunks           form of ssd_scan_fwd (and its workspace size)
 *   SSM_SSD_SPLIT = k           the walking form cuts every (batch, head) into k segments
 *   SSM_FORCE_CHUNKS = n        sequence chunks of the scan
 *   SSM_FORCE_TPR = 2           two threads per row in the row kernel
 *   SSM_CTAS_PER_SM = n         resident CTAs per SM assumed by the row kernel's planner
 *   SSM_STREAM_ROWS = 512 | 128 rows per CTA of the streamed row kernel
 *   SSM_STREAM_CTAS = n         work items (CTAs) of the streamed row kernel
 *   SSM_BWD_CHUNKS = n          sequence chunks of ssm_scan_bwd
 *   SSM_BWD_FORM = quad         ssm_scan_bwd with four threads per row where it would take one
 *   SSM_FORCE_STEP = plain      the generic decode-step kernel only
 *   SSM_FAULT = lookback | step | ssd   the named device-side wait never completes
 *                               (the call reports SSM_ERR_TIMEOUT; nothing faults)
 *   SSM_LOOKBACK_TIMEOUT_MS = n limit of the device-side waits
 */
SSM_API void ssm_test_hooks_reload(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H_ */
