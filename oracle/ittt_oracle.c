/*
 * ittt_oracle.c -- plain, slow, fp64 CPU oracle for the In-Place Test-Time
 * Training fast-weight layer (chunk-wise apply/update of a gated MLP's W_down).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Sources (web pages on In-Place TTT):
 *   [P1] "[논문리뷰] In-Place Test-Time Training" (kimjy99 blog review)
 *        Method §1 eq. (1)-(4), Method §2 eq. (5)-(6), Method §3
 *        "Implementation Details" (context parallelism, causality and
 *        boundary handling).
 *   [P3] "In-Place Test-Time Training" reading notes (gitcode.csdn.net),
 *        sections "整体框架" (apply / update) and "实现细节" (prefix sum).
 *
 * Notation: B batch, T tokens per sequence, d = d_model, f = d_ff, C chunk,
 * n = ceil(T / C) chunks; chunk i holds tokens [iC, min((i+1)C, T)).
 * Weights use the [out, in] row-major layout:
 *   W_gate, W_up : [f, d]      W_down (fast weight) : [d, f]
 *   W_target     : [d, d]      conv_w               : [d, 3]
 * Activations are [B, T, ...] row-major.  Inputs arrive as float (they hold
 * bf16 or fp32 values exactly); every operation is done in double.
 *
 * Readings where the pages are silent (stated once here, used throughout):
 *   - phi = SiLU(x) = x / (1 + exp(-x)).
 *   - Conv1D is depthwise with three taps, cross-correlation order:
 *     conv_w[c,0] multiplies X0[t-1,c], conv_w[c,1] X0[t,c], conv_w[c,2]
 *     X0[t+1,c]; no bias.
 *   - Boundary ("causal padding" in [P1] Method §3): in pad mode
 *     ORACLE_PAD_CHUNK a tap that reaches outside the current chunk reads 0,
 *     so each chunk's update delta depends on that chunk's tokens alone.  In
 *     ORACLE_PAD_SEQUENCE only taps outside the sequence read 0.
 *   - Chunks are 0-based; the state applied to chunk i holds the updates of
 *     chunks 0..i-1 exactly (exclusive prefix, [P3] 实现细节).
 *   - The update is W <- W + eta * Vhat_[i]^T Z_[i] ([P1] eq. (6)): the
 *     gradient step on L = -<Z W^T, Vhat>_F, with no 1/C averaging.
 *   - Per-token learning rate (optional): with eta_tok given, token t's term
 *     of the chunk gradient is weighted by eta_tok[t], i.e. the step uses
 *     grad sum_t eta_tok[t] L_t as in the large-chunk update of [P2]
 *     ("[논문리뷰] Test-Time Training Done Right", Large-Chunk TTT Layer,
 *     per-token eta_i); eta_tok == 1 is the plain update.
 *   - Fast-weight L2 normalisation (optional, oracle_forward_l2norm): the
 *     normalised update of [P2] (Non-Linear Update of Fast-Weight),
 *     W <- L2-Normalize(W + eta * dW), each row of W_down divided by its
 *     norm over the f inputs (floor 1e-12); W_down0 itself is used as given.
 *   - When C does not divide T the last chunk is the shorter remainder
 *     (the pages only use equal chunks; a stream whose length is not a
 *     multiple of C ends with a partial chunk).  Chunk-edge padding then
 *     also pads at T.
 *
 * Parity pins: every function below is checked by tests/test_oracle_pins.py
 * against library routines, closed forms, invariants and finite differences.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_PAD_CHUNK 0
#define ORACLE_PAD_SEQUENCE 1

static double silu(double x) { return x / (1.0 + exp(-x)); }

/*
 * Intermediate activation of the gated MLP, [P1] eq. (2) / [P3] 整体框架:
 *   Z = phi(H W_gate^T) (.) (H W_up^T),  Z in R^{T x f}.
 * H: [T, d], W_gate / W_up: [f, d], Z: [T, f].
 */
void oracle_gated_activation(int64_t T, int64_t d, int64_t f, const float* H,
                             const float* W_gate, const float* W_up,
                             double* Z) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t j = 0; j < f; ++j) {
      double g = 0.0, u = 0.0;
      for (int64_t k = 0; k < d; ++k) {
        g += (double)H[t * d + k] * (double)W_gate[j * d + k];
        u += (double)H[t * d + k] * (double)W_up[j * d + k];
      }
      Z[t * f + j] = silu(g) * u;
    }
  }
}

/*
 * Depthwise three-tap Conv1D over the token embeddings X0 ([P1] eq. (5)),
 * with the boundary reading stated in the header.  X0, Xc: [T, d].
 */
void oracle_conv1d(int64_t T, int64_t d, int64_t C, int pad_mode,
                   const float* X0, const float* conv_w, double* Xc) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    int64_t lo, hi; /* first and one-past-last token a tap may read */
    if (pad_mode == ORACLE_PAD_SEQUENCE) {
      lo = 0;
      hi = T;
    } else {
      lo = (t / C) * C;
      hi = lo + C < T ? lo + C : T;
    }
    for (int64_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int64_t k = -1; k <= 1; ++k) {
        int64_t s = t + k;
        if (s < lo || s >= hi) continue; /* zero padding */
        acc += (double)conv_w[c * 3 + (k + 1)] * (double)X0[s * d + c];
      }
      Xc[t * d + c] = acc;
    }
  }
}

/*
 * NTP-aligned value target, [P1] eq. (5):  Vhat = Conv1D(X0) W_target^T.
 * W_target is stored [d_out, d_in].  X0, Vhat: [T, d].
 */
void oracle_value_target(int64_t T, int64_t d, int64_t C, int pad_mode,
                         const float* X0, const float* conv_w,
                         const float* W_target, double* Vhat) {
  double* Xc = (double*)malloc((size_t)(T * d) * sizeof(double));
  oracle_conv1d(T, d, C, pad_mode, X0, conv_w, Xc);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t m = 0; m < d; ++m) {
      double acc = 0.0;
      for (int64_t c = 0; c < d; ++c)
        acc += Xc[t * d + c] * (double)W_target[m * d + c];
      Vhat[t * d + m] = acc;
    }
  }
  free(Xc);
}

/* Apply, [P1] eq. (3): O_[i] = Z_[i] W^T for the Cn rows starting at row t0. */
static void apply_chunk(int64_t t0, int64_t Cn, int64_t d, int64_t f,
                        const double* Z, const double* W, double* O) {
#pragma omp parallel for schedule(static)
  for (int64_t t = t0; t < t0 + Cn; ++t) {
    for (int64_t m = 0; m < d; ++m) {
      double acc = 0.0;
      for (int64_t j = 0; j < f; ++j) acc += Z[t * f + j] * W[m * f + j];
      O[t * d + m] = acc;
    }
  }
}

/* Per-token weight of the chunk gradient ([P2] per-token eta_i): 1 when no
 * per-token rates are given. */
static double token_rate(const float* eta_tok, int64_t t) {
  return eta_tok ? (double)eta_tok[t] : 1.0;
}

/* Per-chunk delta, [P1] eq. (6) and Method §3 stage 1:
 *   dW = sum_t eta_tok[t] Vhat_t^T Z_t   ([d, f]) over the Cn rows starting
 * at row t0 (eta_tok == NULL: all weights 1, dW = Vhat_[i]^T Z_[i]). */
static void chunk_delta(int64_t t0, int64_t Cn, int64_t d, int64_t f,
                        const double* Vhat, const double* Z, const float* eta_tok,
                        double* dW) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < d; ++m) {
    for (int64_t j = 0; j < f; ++j) {
      double acc = 0.0;
      for (int64_t t = t0; t < t0 + Cn; ++t)
        acc += token_rate(eta_tok, t) * Vhat[t * d + m] * Z[t * f + j];
      dW[m * f + j] = acc;
    }
  }
}

/* Number of chunks and the length of chunk i. */
static int64_t num_chunks(int64_t T, int64_t C) { return (T + C - 1) / C; }
static int64_t chunk_len(int64_t T, int64_t C, int64_t i) {
  return (i + 1) * C <= T ? C : T - i * C;
}

/* Per-sequence intermediates shared by the three forms below. */
static void sequence_intermediates(int64_t T, int64_t d, int64_t f, int64_t C,
                                   int pad_mode, const float* H,
                                   const float* X0, const float* W_gate,
                                   const float* W_up, const float* W_target,
                                   const float* conv_w, double* Z,
                                   double* Vhat) {
  oracle_gated_activation(T, d, f, H, W_gate, W_up, Z);
  oracle_value_target(T, d, C, pad_mode, X0, conv_w, W_target, Vhat);
}

/*
 * The layer as the pages define it: a sequential loop over chunks, each one
 * first applied with the current fast weight ([P1] eq. (3)), then used to
 * update it ([P1] eq. (4) specialised by eq. (6)):
 *     W^(0) = W_down0
 *     O_[i] = Z_[i] (W^(i))^T
 *     W^(i+1) = W^(i) + eta * Vhat_[i]^T Z_[i]
 * Every sequence starts from W_down0 (reset at document boundaries, [P1]
 * Method §3).
 *
 * Inputs (float, row-major): H, X0 [B,T,d]; W_gate, W_up [f,d];
 * W_down0 [d,f] if w0_batch_stride == 0, else [B,d,f] with that stride
 * (per-sequence initial state); W_target [d,d]; conv_w [d,3]; eta_tok
 * [B,T] per-token rates or NULL.
 * Outputs (double): O [B,T,d].  Optional (may be NULL): Z [B,T,f],
 * Vhat [B,T,d], states [B, n+1, d, f] holding W^(0) .. W^(n).
 */
void oracle_forward_sequential(int64_t B, int64_t T, int64_t d, int64_t f,
                               int64_t C, double eta, int pad_mode,
                               const float* H, const float* X0,
                               const float* W_gate, const float* W_up,
                               const float* W_down0, int64_t w0_batch_stride,
                               const float* W_target, const float* conv_w,
                               const float* eta_tok, double* O, double* Z_out,
                               double* Vhat_out, double* states_out) {
  const int64_t n = num_chunks(T, C);
  double* Z = (double*)malloc((size_t)(T * f) * sizeof(double));
  double* Vhat = (double*)malloc((size_t)(T * d) * sizeof(double));
  double* W = (double*)malloc((size_t)(d * f) * sizeof(double));
  double* dW = (double*)malloc((size_t)(d * f) * sizeof(double));
  for (int64_t b = 0; b < B; ++b) {
    sequence_intermediates(T, d, f, C, pad_mode, H + b * T * d, X0 + b * T * d,
                           W_gate, W_up, W_target, conv_w, Z, Vhat);
    const float* W0 = W_down0 + b * w0_batch_stride;
    const float* et = eta_tok ? eta_tok + b * T : NULL;
    for (int64_t e = 0; e < d * f; ++e) W[e] = (double)W0[e];
    if (states_out)
      memcpy(states_out + (b * (n + 1)) * d * f, W,
             (size_t)(d * f) * sizeof(double));
    for (int64_t i = 0; i < n; ++i) {
      const int64_t Cn = chunk_len(T, C, i);
      apply_chunk(i * C, Cn, d, f, Z, W, O + b * T * d);         /* apply  */
      chunk_delta(i * C, Cn, d, f, Vhat, Z, et, dW);             /* update */
      for (int64_t e = 0; e < d * f; ++e) W[e] += eta * dW[e];
      if (states_out)
        memcpy(states_out + (b * (n + 1) + i + 1) * d * f, W,
               (size_t)(d * f) * sizeof(double));
    }
    if (Z_out) memcpy(Z_out + b * T * f, Z, (size_t)(T * f) * sizeof(double));
    if (Vhat_out)
      memcpy(Vhat_out + b * T * d, Vhat, (size_t)(T * d) * sizeof(double));
  }
  free(Z);
  free(Vhat);
  free(W);
  free(dW);
}

/*
 * Fast-weight L2 normalisation ([P2] "[논문리뷰] Test-Time Training Done
 * Right", Non-Linear Update of Fast-Weight, fast-weight normalisation:
 * weight-update(W, g) = L2-Normalize(W - g), taken along the weight's input
 * dimension).  W_down maps the f-dimensional Z to the d-dimensional output,
 * so its input dimension is f: each row m is divided by its L2 norm over
 * the f inputs.  A zero row is divided by 1e-12 instead (the usual floor).
 */
static void l2_normalize_rows(int64_t d, int64_t f, double* W) {
  for (int64_t m = 0; m < d; ++m) {
    double ss = 0.0;
    for (int64_t j = 0; j < f; ++j) ss += W[m * f + j] * W[m * f + j];
    double norm = sqrt(ss);
    if (norm < 1e-12) norm = 1e-12;
    for (int64_t j = 0; j < f; ++j) W[m * f + j] /= norm;
  }
}

/*
 * The sequential layer with the normalised update rule of [P2] applied to
 * In-Place TTT's fast weight: every updated state is normalised row by row,
 *     W^(0)   = W_down0                      (used as given)
 *     O_[i]   = Z_[i] (W^(i))^T
 *     W^(i+1) = L2-Normalize(W^(i) + eta * Vhat_[i]^T Z_[i]).
 * The gradient step inside is the one of oracle_forward_sequential (the
 * pages' L2-Normalize(W - g) with g the gradient of L = -<Z W^T, Vhat>_F).
 * The normalisation makes the update non-additive: there is no prefix or
 * dual form.  Same arguments as oracle_forward_sequential, without the Z
 * and Vhat outputs.
 */
void oracle_forward_l2norm(int64_t B, int64_t T, int64_t d, int64_t f, int64_t C,
                           double eta, int pad_mode, const float* H, const float* X0,
                           const float* W_gate, const float* W_up, const float* W_down0,
                           int64_t w0_batch_stride, const float* W_target,
                           const float* conv_w, const float* eta_tok, double* O,
                           double* states_out) {
  const int64_t n = num_chunks(T, C);
  const int64_t df = d * f;
  double* Z = (double*)malloc((size_t)(T * f) * sizeof(double));
  double* Vhat = (double*)malloc((size_t)(T * d) * sizeof(double));
  double* W = (double*)malloc((size_t)df * sizeof(double));
  double* dW = (double*)malloc((size_t)df * sizeof(double));
  for (int64_t b = 0; b < B; ++b) {
    sequence_intermediates(T, d, f, C, pad_mode, H + b * T * d, X0 + b * T * d,
                           W_gate, W_up, W_target, conv_w, Z, Vhat);
    const float* et = eta_tok ? eta_tok + b * T : NULL;
    for (int64_t e = 0; e < df; ++e) W[e] = (double)W_down0[b * w0_batch_stride + e];
    if (states_out) memcpy(states_out + (b * (n + 1)) * df, W, (size_t)df * sizeof(double));
    for (int64_t i = 0; i < n; ++i) {
      const int64_t Cn = chunk_len(T, C, i);
      apply_chunk(i * C, Cn, d, f, Z, W, O + b * T * d);
      chunk_delta(i * C, Cn, d, f, Vhat, Z, et, dW);
      for (int64_t e = 0; e < df; ++e) W[e] = W[e] + eta * dW[e];
      l2_normalize_rows(d, f, W);
      if (states_out)
        memcpy(states_out + (b * (n + 1) + i + 1) * df, W, (size_t)df * sizeof(double));
    }
  }
  free(Z);
  free(Vhat);
  free(W);
  free(dW);
}

/*
 * The same layer in the three-stage parallel form of [P1] Method §3
 * ("Implementation Details", context parallelism) and [P3] 实现细节:
 *   stage 1: dW_i = Vhat_[i]^T Z_[i] for every chunk;
 *   stage 2: one exclusive prefix sum S_i = sum_{j<i} dW_j;
 *   stage 3: W^(i) = W_down0 + eta * S_i and O_[i] = Z_[i] (W^(i))^T.
 * Same arguments as oracle_forward_sequential; states_out (optional) gets
 * W^(0) .. W^(n) as [B, n+1, d, f].
 */
void oracle_forward_prefix(int64_t B, int64_t T, int64_t d, int64_t f,
                           int64_t C, double eta, int pad_mode, const float* H,
                           const float* X0, const float* W_gate,
                           const float* W_up, const float* W_down0,
                           int64_t w0_batch_stride, const float* W_target,
                           const float* conv_w, const float* eta_tok, double* O,
                           double* states_out) {
  const int64_t n = num_chunks(T, C);
  const int64_t df = d * f;
  double* Z = (double*)malloc((size_t)(T * f) * sizeof(double));
  double* Vhat = (double*)malloc((size_t)(T * d) * sizeof(double));
  double* dWs = (double*)malloc((size_t)(n * df) * sizeof(double));
  double* S = (double*)malloc((size_t)((n + 1) * df) * sizeof(double));
  double* W = (double*)malloc((size_t)df * sizeof(double));
  for (int64_t b = 0; b < B; ++b) {
    sequence_intermediates(T, d, f, C, pad_mode, H + b * T * d, X0 + b * T * d,
                           W_gate, W_up, W_target, conv_w, Z, Vhat);
    const float* et = eta_tok ? eta_tok + b * T : NULL;
    /* stage 1 */
    for (int64_t i = 0; i < n; ++i)
      chunk_delta(i * C, chunk_len(T, C, i), d, f, Vhat, Z, et, dWs + i * df);
    /* stage 2: exclusive scan, S_0 = 0 */
    for (int64_t e = 0; e < df; ++e) S[e] = 0.0;
    for (int64_t i = 1; i <= n; ++i)
      for (int64_t e = 0; e < df; ++e)
        S[i * df + e] = S[(i - 1) * df + e] + dWs[(i - 1) * df + e];
    /* stage 3 */
    const float* W0 = W_down0 + b * w0_batch_stride;
    for (int64_t i = 0; i <= n; ++i) {
      for (int64_t e = 0; e < df; ++e) W[e] = (double)W0[e] + eta * S[i * df + e];
      if (i < n) apply_chunk(i * C, chunk_len(T, C, i), d, f, Z, W, O + b * T * d);
      if (states_out)
        memcpy(states_out + (b * (n + 1) + i) * df, W, (size_t)df * sizeof(double));
    }
  }
  free(Z);
  free(Vhat);
  free(dWs);
  free(S);
  free(W);
}

/*
 * The dual (attention-like) form obtained by expanding W^(i) in the apply:
 *   O_[i] = Z_[i] W_down0^T + eta * sum_{j<i} (Z_[i] Z_[j]^T) Vhat_[j]
 * (per-token rates weight each token s of the earlier chunks).
 * ([P1] eq. (3) with W^(i) = W_down0 + eta * sum_{j<i} Vhat_[j]^T Z_[j].)
 * Output O [B,T,d] only.
 */
void oracle_forward_dual(int64_t B, int64_t T, int64_t d, int64_t f, int64_t C,
                         double eta, int pad_mode, const float* H,
                         const float* X0, const float* W_gate,
                         const float* W_up, const float* W_down0,
                         int64_t w0_batch_stride, const float* W_target,
                         const float* conv_w, const float* eta_tok, double* O) {
  const int64_t n = num_chunks(T, C);
  double* Z = (double*)malloc((size_t)(T * f) * sizeof(double));
  double* Vhat = (double*)malloc((size_t)(T * d) * sizeof(double));
  double* W0d = (double*)malloc((size_t)(d * f) * sizeof(double));
  for (int64_t b = 0; b < B; ++b) {
    sequence_intermediates(T, d, f, C, pad_mode, H + b * T * d, X0 + b * T * d,
                           W_gate, W_up, W_target, conv_w, Z, Vhat);
    const float* W0 = W_down0 + b * w0_batch_stride;
    const float* et = eta_tok ? eta_tok + b * T : NULL;
    for (int64_t e = 0; e < d * f; ++e) W0d[e] = (double)W0[e];
    double* Ob = O + b * T * d;
    for (int64_t i = 0; i < n; ++i) {
      const int64_t Cn = chunk_len(T, C, i);
      apply_chunk(i * C, Cn, d, f, Z, W0d, Ob); /* Z_[i] W_down0^T */
#pragma omp parallel for schedule(static)
      for (int64_t t = i * C; t < i * C + Cn; ++t) {
        for (int64_t s = 0; s < i * C; ++s) { /* every token of chunks j < i */
          double a = 0.0;                     /* (Z_[i] Z_[j]^T)[t, s] */
          for (int64_t k = 0; k < f; ++k) a += Z[t * f + k] * Z[s * f + k];
          const double w = eta * token_rate(et, s) * a;
          for (int64_t m = 0; m < d; ++m) Ob[t * d + m] += w * Vhat[s * d + m];
        }
      }
    }
  }
  free(Z);
  free(Vhat);
  free(W0d);
}

/* ---------------------------------------------------------------------------
 * Entry-wise evaluators for the full-size workloads, where the whole layer is
 * too slow for a CPU.  Each computes single entries straight from the
 * definitions above, reading only the rows it needs.
 * ------------------------------------------------------------------------- */

/* Z[t, j] for `count` (t, j) pairs of one sequence ([P1] eq. (2)). */
void oracle_z_entries(int64_t d, const float* H, const float* W_gate,
                      const float* W_up, int64_t count, const int64_t* t_idx,
                      const int64_t* j_idx, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t q = 0; q < count; ++q) {
    const int64_t t = t_idx[q], j = j_idx[q];
    double g = 0.0, u = 0.0;
    for (int64_t k = 0; k < d; ++k) {
      g += (double)H[t * d + k] * (double)W_gate[j * d + k];
      u += (double)H[t * d + k] * (double)W_up[j * d + k];
    }
    out[q] = silu(g) * u;
  }
}

/* Vhat[t, m] of one sequence at token t and column m ([P1] eq. (5)). */
static double vhat_entry(int64_t T, int64_t d, int64_t C, int pad_mode,
                         const float* X0, const float* conv_w,
                         const float* W_target, int64_t t, int64_t m) {
  int64_t lo = 0, hi = T;
  if (pad_mode != ORACLE_PAD_SEQUENCE) {
    lo = (t / C) * C;
    hi = lo + C < T ? lo + C : T;
  }
  double acc = 0.0;
  for (int64_t c = 0; c < d; ++c) {
    double xc = 0.0;
    for (int64_t k = -1; k <= 1; ++k) {
      int64_t s = t + k;
      if (s < lo || s >= hi) continue;
      xc += (double)conv_w[c * 3 + (k + 1)] * (double)X0[s * d + c];
    }
    acc += xc * (double)W_target[m * d + c];
  }
  return acc;
}

/* Vhat[t, m] for `count` (t, m) pairs of one sequence. */
void oracle_vhat_entries(int64_t T, int64_t d, int64_t C, int pad_mode,
                         const float* X0, const float* conv_w,
                         const float* W_target, int64_t count,
                         const int64_t* t_idx, const int64_t* m_idx,
                         double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t q = 0; q < count; ++q)
    out[q] = vhat_entry(T, d, C, pad_mode, X0, conv_w, W_target, t_idx[q],
                        m_idx[q]);
}

/*
 * Fast-weight state entries W^(i)[m, j] for i = 0..n of one sequence, for
 * `count` (m, j) pairs ([P1] eq. (6) summed over chunks; [P3] 实现细节).
 * W^(i)[m, j] = W_down0[m, j] + eta * sum_{s < iC} eta_tok[s] Vhat[s, m] Z[s, j]
 * (eta_tok NULL: weights 1).  out: [count, n+1].  w0 is this sequence's
 * initial state [d, f].
 */
void oracle_state_entries(int64_t T, int64_t d, int64_t f, int64_t C,
                          double eta, int pad_mode, const float* H,
                          const float* X0, const float* W_gate,
                          const float* W_up, const float* w0,
                          const float* W_target, const float* conv_w,
                          const float* eta_tok, int64_t count,
                          const int64_t* m_idx, const int64_t* j_idx,
                          double* out) {
  const int64_t n = num_chunks(T, C);
#pragma omp parallel for schedule(dynamic)
  for (int64_t q = 0; q < count; ++q) {
    const int64_t m = m_idx[q], j = j_idx[q];
    double sum = 0.0;
    out[q * (n + 1)] = (double)w0[m * f + j];
    for (int64_t i = 0; i < n; ++i) {
      for (int64_t s = i * C; s < i * C + chunk_len(T, C, i); ++s) {
        double g = 0.0, u = 0.0;
        for (int64_t k = 0; k < d; ++k) {
          g += (double)H[s * d + k] * (double)W_gate[j * d + k];
          u += (double)H[s * d + k] * (double)W_up[j * d + k];
        }
        sum += token_rate(eta_tok, s) *
               vhat_entry(T, d, C, pad_mode, X0, conv_w, W_target, s, m) * (silu(g) * u);
      }
      out[q * (n + 1) + i + 1] = (double)w0[m * f + j] + eta * sum;
    }
  }
}

/*
 * Output rows of the first chunk of one sequence: O[t, :] = Z[t, :] W_down0^T
 * for tokens t < C, where no update has been applied yet ([P1] eq. (3) with
 * W^(0) = W_down0).  rows: `count` token indices, all < C.  out: [count, d].
 */
void oracle_first_chunk_rows(int64_t d, int64_t f, const float* H,
                             const float* W_gate, const float* W_up,
                             const float* w0, int64_t count,
                             const int64_t* rows, double* out) {
  double* z = (double*)malloc((size_t)(count * f) * sizeof(double));
#pragma omp parallel for schedule(static)
  for (int64_t q = 0; q < count; ++q) {
    const int64_t t = rows[q];
    for (int64_t j = 0; j < f; ++j) {
      double g = 0.0, u = 0.0;
      for (int64_t k = 0; k < d; ++k) {
        g += (double)H[t * d + k] * (double)W_gate[j * d + k];
        u += (double)H[t * d + k] * (double)W_up[j * d + k];
      }
      z[q * f + j] = silu(g) * u;
    }
    for (int64_t m = 0; m < d; ++m) {
      double acc = 0.0;
      for (int64_t j = 0; j < f; ++j) acc += z[q * f + j] * (double)w0[m * f + j];
      out[q * d + m] = acc;
    }
  }
  free(z);
}

/* Threads OpenMP will use (reported with CPU baseline timings). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the OpenMP loops use from now on (n >= 1; a single-threaded timing
 * of the baseline sets 1, then restores the previous count).  No effect on
 * any result: every parallel loop writes disjoint outputs. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
