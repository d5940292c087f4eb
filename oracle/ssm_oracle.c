/*
 * Double-precision CPU oracle for the selective state-space scan (S6).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code with the CUDA path.
 *
 * It is the plain definition written out as loops, in the order the sources
 * state it, with no blocking, fusion or reordering:
 *
 *   Δ_t  = softplus(Δraw_t + bias)                       (step size, kept > 0)
 *   Ā    = exp(Δ_t A)                                    [1]
 *   B̄    = (Δ_t A)^-1 (exp(Δ_t A) - I) Δ_t B_t           [1]
 *        = expm1(Δ_t a_n) / a_n · B_t[n]   for diagonal A (a_n ≠ 0)
 *        = Δ_t · B_t[n]                    in the limit a_n → 0
 *   h_t  = Ā h_{t-1} + B̄ x_t,   h_0 = 0                  [1] [2]
 *   y_t  = C_t h_t + D x_t                                [2]
 *   out_t = y_t · silu(z_t)                               [3]
 *
 * [1] "State Space Models（SSM）とMamba", §2.2 離散化 (zero-order hold), and
 *     "Mambaとは？Transformer以外の系列モデル", section 状態空間モデルを一つの式から理解する.
 * [2] "Mambaとは？Transformer以外の系列モデル", same section (readout with the
 *     D skip term), and section 固定SSMには「再帰」と「畳み込み」の二つの顔がある
 *     (the initial state is zero).
 * [3] "Mambaとは？Transformer以外の系列モデル", section Mamba blockのarchitecture,
 *     step 4: the gate branch passes through SiLU and multiplies the SSM branch
 *     output element-wise.
 *
 * Δ_t, B_t and C_t are per token ("State Space Models（SSM）とMamba" §4.2
 * Selective SSM; "Mambaとは？…" section Mambaの核心は入力依存のDelta、B、C);
 * A is diagonal (S4D, §3.4) and not input dependent.  The positive step size is
 * formed as softplus(Δraw + bias): the pages leave the map f_Δ open; this is
 * the library's interface, and softplus is evaluated here in its stable form
 * max(r, 0) + log1p(exp(-|r|)).
 *
 * Layouts (row-major, all double):
 *   u, delta, z, out : [batch][d_inner][L]
 *   B, C             : [batch][L][N]
 *   A                : [d_inner][N]
 *   D, bias          : [d_inner]          (may be NULL: treated as 0)
 *   h0, hT, state    : [batch][d_inner][N] (h0 may be NULL: zero state)
 * z NULL means no gate.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

static double softplus(double r) { return fmax(r, 0.0) + log1p(exp(-fabs(r))); }

/* logistic sigmoid in the form that never overflows */
static double sigmoid(double z) {
  if (z >= 0.0) return 1.0 / (1.0 + exp(-z));
  double e = exp(z);
  return e / (1.0 + e);
}

static double silu(double z) { return z * sigmoid(z); }

/*
 * One token of one (batch, channel) row: discretise, update the N states in
 * place, read out, add the skip term, apply the gate.  Returns the output.
 */
static double token(int64_t N, double* h, double x, double delta_raw, double bias,
                    const double* a, const double* Bt, const double* Ct,
                    int has_D, double D, int has_z, double z) {
  const double dt = softplus(delta_raw + bias);
  double y = 0.0;
  for (int64_t n = 0; n < N; ++n) {
    const double abar = exp(dt * a[n]);
    const double bbar = (a[n] != 0.0) ? expm1(dt * a[n]) / a[n] * Bt[n] : dt * Bt[n];
    h[n] = abar * h[n] + bbar * x;
    y += Ct[n] * h[n];
  }
  if (has_D) y += D * x;
  if (has_z) y *= silu(z);
  return y;
}

/*
 * Parallel (training / prefill) mode, computed here as the plain sequential
 * loop over t.  Processes rows r = b*d_inner + c for r in [row_begin, row_end),
 * so independent callers may split the rows between threads.
 */
void oracle_scan(int64_t batch, int64_t d_inner, int64_t N, int64_t L,
                 const double* u, const double* delta, const double* A,
                 const double* B, const double* C, const double* D,
                 const double* z, const double* bias, const double* h0,
                 double* out, double* hT, int64_t row_begin, int64_t row_end) {
  double h[1024];
  if (N > 1024) return;
  if (row_end > batch * d_inner) row_end = batch * d_inner;
  for (int64_t r = row_begin; r < row_end; ++r) {
    const int64_t b = r / d_inner, c = r % d_inner;
    for (int64_t n = 0; n < N; ++n) h[n] = h0 ? h0[r * N + n] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
      const int64_t i = r * L + t;
      out[i] = token(N, h, u[i], delta[i], bias ? bias[c] : 0.0, A + c * N,
                     B + (b * L + t) * N, C + (b * L + t) * N,
                     D != NULL, D ? D[c] : 0.0, z != NULL, z ? z[i] : 0.0);
    }
    if (hT)
      for (int64_t n = 0; n < N; ++n) hT[r * N + n] = h[n];
  }
}

/*
 * Recurrent (decode) mode: one token for every row, state updated in place
 * ("Mambaとは？…", section training、prefill、decodeでは計算の姿が違う).
 * Layouts: state [batch][d_inner][N]; x, delta, z, out [batch][d_inner];
 * B, C [batch][N].
 */
void oracle_step(int64_t batch, int64_t d_inner, int64_t N, double* state,
                 const double* x, const double* delta, const double* A,
                 const double* B, const double* C, const double* D,
                 const double* z, const double* bias, double* out,
                 int64_t row_begin, int64_t row_end) {
  if (row_end > batch * d_inner) row_end = batch * d_inner;
  for (int64_t r = row_begin; r < row_end; ++r) {
    const int64_t b = r / d_inner, c = r % d_inner;
    out[r] = token(N, state + r * N, x[r], delta[r], bias ? bias[c] : 0.0, A + c * N,
                   B + b * N, C + b * N, D != NULL, D ? D[c] : 0.0, z != NULL,
                   z ? z[r] : 0.0);
  }
}

/*
 * Causal depthwise Conv1D followed by SiLU: the short convolution of the Mamba
 * block's main branch, in front of the selective SSM ("Mambaとは？Transformer以外の
 * 系列モデル", section Mamba blockのarchitecture, steps 2 and 3: a short causal
 * Conv1D mixes neighbouring tokens, then SiLU).  Per (batch, channel) row and
 * width W (the pages give no width or formula; this is the plain reading):
 *
 *   pre[t] = bias + Σ_{k=0}^{W-1} w[k] · x̃[t - (W-1) + k]
 *   out[t] = silu(pre[t])
 *
 * where x̃ is x extended to the left by the W-1 inputs that came before it:
 * state0[0..W-2] (oldest first), or zeros when state0 is NULL.  The state after
 * the sequence is the last W-1 entries of x̃ ("Mambaとは？…", section
 * training、prefill、decodeでは計算の姿が違う: in decode each layer keeps its
 * SSM state and a state for the short causal Conv1D).
 *
 * Layouts (row-major, all double): x, out [batch][d_inner][L]; w [d_inner][W];
 * bias [d_inner] (NULL: 0); state0, stateT [batch][d_inner][W-1].
 */
static double conv_input(const double* xr, const double* s0r, int64_t W, int64_t p) {
  if (p >= 0) return xr[p];
  return s0r ? s0r[(W - 1) + p] : 0.0;
}

void oracle_conv1d(int64_t batch, int64_t d_inner, int64_t L, int64_t W, const double* x, const double* w,
                   const double* bias, const double* state0, double* out, double* stateT, int64_t row_begin,
                   int64_t row_end) {
  (void)batch;
  for (int64_t r = row_begin; r < row_end; ++r) {
    const int64_t c = r % d_inner;
    const double* xr = x + r * L;
    const double* s0r = state0 ? state0 + r * (W - 1) : NULL;
    for (int64_t t = 0; t < L; ++t) {
      double pre = bias ? bias[c] : 0.0;
      for (int64_t k = 0; k < W; ++k) pre += w[c * W + k] * conv_input(xr, s0r, W, t - (W - 1) + k);
      out[r * L + t] = silu(pre);
    }
    if (stateT)
      for (int64_t j = 0; j < W - 1; ++j) stateT[r * (W - 1) + j] = conv_input(xr, s0r, W, L - (W - 1) + j);
  }
}

/* One decode token: window = (state[0..W-2], x); out = silu(bias + Σ w·window);
 * state ← window[1..W-1].  state [batch][d_inner][W-1] is updated in place. */
void oracle_conv1d_step(int64_t batch, int64_t d_inner, int64_t W, double* state, const double* x,
                        const double* w, const double* bias, double* out, int64_t row_begin, int64_t row_end) {
  (void)batch;
  double win[64];
  for (int64_t r = row_begin; r < row_end; ++r) {
    const int64_t c = r % d_inner;
    for (int64_t k = 0; k < W - 1; ++k) win[k] = state[r * (W - 1) + k];
    win[W - 1] = x[r];
    double pre = bias ? bias[c] : 0.0;
    for (int64_t k = 0; k < W; ++k) pre += w[c * W + k] * win[k];
    out[r] = silu(pre);
    for (int64_t k = 0; k < W - 1; ++k) state[r * (W - 1) + k] = win[k + 1];
  }
}
