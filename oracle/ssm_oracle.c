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

/*
 * Backward of the scan: the gradients of the scalar loss
 *   ℓ = Σ_{b,c,t} dout[b,c,t] · out[b,c,t]  +  Σ_{b,c,n} dhT[b,c,n] · h_L[b,c,n]
 * with respect to every input, by reverse-mode differentiation of the loop of
 * oracle_scan written out: the forward states h_0..h_L of a row are kept, then
 * t runs backwards carrying dℓ/dh_t.  Per token (a = A[c,n], Ā = exp(Δa),
 * φ = expm1(Δa)/a, or Δ when a = 0, q = φ B x, h_t = Ā h_{t-1} + q):
 *   dy = dout·silu(z), dz = dout·y·silu'(z), dD += dy x, dx = dy D
 *   dh_t += dy C_t;  dC_t += dy h_t
 *   dĀ = dh_t h_{t-1}, dφ = dh_t B x;  dB_t += dh_t φ x;  dx += dh_t φ B
 *   dΔ += dĀ a Ā + dφ Ā;  da += dĀ Δ Ā + dφ (Δ Ā − φ)/a   (a = 0: dΔ += dφ, da += dĀ Δ + dφ Δ²/2)
 *   dh_{t-1} = Ā dh_t
 *   dΔraw = dΔ · sigmoid(Δraw + bias);  dbias += dΔraw
 * and dh0 = dℓ/dh_0.  This is the plain chain rule on the definition of
 * oracle_scan; the pages describe the backward only as recomputing the states
 * instead of storing them ("Mambaとは？…", section Selective Scanは選択機構そのもの
 * ではない, hardware-aware parallel scan).
 *
 * du, ddelta, dz, dh0 are written; dA [d_inner][N], dB, dC [batch][L][N], dD and
 * dbias [d_inner] are accumulated (the caller zeroes them).  z, D, bias, h0, dhT
 * and the matching outputs may be NULL.  work: (L + 1) * N doubles.
 * Rows are processed in order (the accumulations are shared).
 */
static double dsilu(double z) {
  const double s = sigmoid(z);
  return s * (1.0 + z * (1.0 - s));
}

void oracle_scan_bwd(int64_t batch, int64_t d_inner, int64_t N, int64_t L, const double* u, const double* delta,
                     const double* A, const double* B, const double* C, const double* D, const double* z,
                     const double* bias, const double* h0, const double* dout, const double* dhT, double* du,
                     double* ddelta, double* dA, double* dB, double* dC, double* dD, double* dz, double* dbias,
                     double* dh0, double* work) {
  double dh[1024];
  if (N > 1024) return;
  for (int64_t r = 0; r < batch * d_inner; ++r) {
    const int64_t b = r / d_inner, c = r % d_inner;
    const double bc = bias ? bias[c] : 0.0;
    double* H = work;  // H[t * N + n] = h_t[n], t = 0..L
    for (int64_t n = 0; n < N; ++n) H[n] = h0 ? h0[r * N + n] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
      const int64_t i = r * L + t;
      const double dtv = softplus(delta[i] + bc);
      for (int64_t n = 0; n < N; ++n) {
        const double a = A[c * N + n];
        const double abar = exp(dtv * a);
        const double phi = (a != 0.0) ? expm1(dtv * a) / a : dtv;
        H[(t + 1) * N + n] = abar * H[t * N + n] + phi * B[(b * L + t) * N + n] * u[i];
      }
    }
    for (int64_t n = 0; n < N; ++n) dh[n] = dhT ? dhT[r * N + n] : 0.0;
    for (int64_t t = L - 1; t >= 0; --t) {
      const int64_t i = r * L + t;
      const double* Bt = B + (b * L + t) * N;
      const double* Ct = C + (b * L + t) * N;
      const double x = u[i];
      const double rr = delta[i] + bc;
      const double dtv = softplus(rr);
      double y = 0.0;
      for (int64_t n = 0; n < N; ++n) y += Ct[n] * H[(t + 1) * N + n];
      if (D) y += D[c] * x;
      double dy = dout[i];
      if (z) {
        dy = dout[i] * silu(z[i]);
        if (dz) dz[i] = dout[i] * y * dsilu(z[i]);
      }
      double dx = 0.0, ddt = 0.0;
      if (D) {
        if (dD) dD[c] += dy * x;
        dx = dy * D[c];
      }
      for (int64_t n = 0; n < N; ++n) {
        const double a = A[c * N + n];
        const double abar = exp(dtv * a);
        const double phi = (a != 0.0) ? expm1(dtv * a) / a : dtv;
        dh[n] += dy * Ct[n];
        dC[(b * L + t) * N + n] += dy * H[(t + 1) * N + n];
        const double dabar = dh[n] * H[t * N + n];
        const double dphi = dh[n] * Bt[n] * x;
        dB[(b * L + t) * N + n] += dh[n] * phi * x;
        dx += dh[n] * phi * Bt[n];
        if (a != 0.0) {
          ddt += dabar * a * abar + dphi * abar;
          dA[c * N + n] += dabar * dtv * abar + dphi * (dtv * abar - phi) / a;
        } else {
          ddt += dphi;
          dA[c * N + n] += dabar * dtv + dphi * dtv * dtv / 2.0;
        }
        dh[n] *= abar;
      }
      du[i] = dx;
      const double dr = ddt * sigmoid(rr);
      ddelta[i] = dr;
      if (dbias) dbias[c] += dr;
    }
    if (dh0)
      for (int64_t n = 0; n < N; ++n) dh0[r * N + n] = dh[n];
  }
}
