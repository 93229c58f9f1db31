/*
 * kda_oracle.c -- plain, slow, float64 CPU oracle for the KDA token-generation
 * recurrence and the fused KDA block.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; the two are compared element by element on the same inputs.
 *
 * Everything is computed in double.  Inputs arrive already widened to double
 * (bf16 and fp32 values widen exactly), so the only rounding is this file's own
 * float64 arithmetic.  Loops follow the order in which the pages state the
 * method; no blocking, fusion or reordering is applied.
 *
 * Sources (page title, then section):
 *   [DR]  "Delta-rule write" (Kimi K3 model atlas): the prose above the code
 *         and the naive_recurrent_kda excerpt (flash-linear-attention
 *         fla/ops/kda/naive.py): decay the state per key channel, write
 *         beta*k (x) (v - k^T S), then read o = q^T S with the scaled query.
 *   [KD]  "KdaDecode" (MAX Mojo builtin kernel): "Default parameters" (gate_mode
 *         original = stable softplus gate, beta_mode logits = sigmoid,
 *         state_layout K_FIRST = pool [N, HV, K, V]) and "Tensor Shapes".
 *   [BT]  "KDA Block TKG Kernel API Reference" (AWS Neuron NKI): the
 *         kda_block_tkg signature, Background and each :param: entry.
 *
 * Parity status of each function is stated in its header comment.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Bits reported through *status; the values are the oracle's own and are
 * matched against the library's by the tests, not shared with it. */
#define ORACLE_BAD_SLOT 1
#define ORACLE_BAD_SEQLEN 2

#define ORACLE_GATE_SOFTPLUS 0
#define ORACLE_GATE_LOWER_BOUND 1

/* Output-gate activations of the block (a reading, see output_gate). */
#define ORACLE_OUT_GATE_SIGMOID 0
#define ORACLE_OUT_GATE_SWISH 1

/* ---------------------------------------------------------------- scalars */

/* Logistic sigmoid 1 / (1 + e^-x).  [KD] beta_mode "logits"; [BT] :param
 * lower_bound: (activated gate = lower_bound * sigmoid(...)). */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Softplus log(1 + e^x) in its overflow-free ("stable") form
 * max(x, 0) + log1p(e^-|x|).  [KD] gate_mode "original (stable-softplus)". */
static double softplus(double x) { return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x))); }

/* Per-channel log-decay g for one key channel.
 *   softplus mode: g = -exp(A_log) * softplus(raw + dt_bias)
 *   lower-bound mode: g = lower_bound * sigmoid(exp(A_log) * (raw + dt_bias))
 * [KD] gate_mode; [BT] :param A_log: (exp(A_log) scales the gate
 * pre-activation), :param dt_bias: (added before the activation),
 * :param lower_bound:.  The pages give these in words, not as a printed
 * formula.  The reading: dt_bias joins the raw gate first, and exp(A_log)
 * scales that whole pre-activation.  The test suite pins what the words fix:
 * at raw = -dt_bias the pre-activation is 0, so the lower-bound gate is
 * exactly lower_bound / 2 and the softplus gate exactly -exp(A_log) ln 2 for
 * every A_log; the softplus gate's asymptote for large raw is
 * -exp(A_log) (raw + dt_bias); the lower-bound gate's slope at that point is
 * lower_bound exp(A_log) / 4; g <= 0 and g in [lower_bound, 0]. */
static double gate_value(double raw, double dt_bias, double a_log, int gate_mode,
                         double lower_bound) {
  double x = raw + dt_bias;
  if (gate_mode == ORACLE_GATE_SOFTPLUS) return -exp(a_log) * softplus(x);
  return lower_bound * sigmoid(exp(a_log) * x);
}

/* Activation of the block's output gate z.  [BT] Background: the recurrence
 * read goes through a "gated" output RMSNorm; the page names no activation
 * for the gate.  Reading: the logistic sigmoid (the same squashing the page
 * uses for the forget gate), with z * sigmoid(z) (swish) as the documented
 * alternative.  Pinned per setting by closed forms at z = 0 and z >> 0 in
 * the test suite; which of the two the page means is a reading the page
 * leaves open (sigmoid is the default). */
static double output_gate(double z, int out_gate) {
  if (out_gate == ORACLE_OUT_GATE_SWISH) return z * sigmoid(z);
  return sigmoid(z);
}

/* x / sqrt(sum x^2 + eps) over n entries, times mul.  [DR] Code
 * (use_qk_l2norm_in_kernel=True); [BT] l2_eps and :param scale: (the scale is
 * folded into the normalised query). */
static void l2_normalise(double* out, const double* x, int n, double eps, double mul) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * inv * mul;
}

/* One token of the delta rule on a [K, V] state S (row k contiguous over v).
 * [DR] naive_recurrent_kda loop body, in its order:
 *   S <- S * exp(g)[:, None]              decay, channel by channel
 *   u  = v - (k^T S)                      what the key does not yet return
 *   S <- S + (beta * k) outer u           delta write
 *   o  = q^T S                            read, after the write
 * kh and qh are the normalised key and (scaled) query. */
static void delta_rule_token(double* S, double* o, const double* qh, const double* kh,
                             const double* v, const double* g, double beta, int K, int V,
                             double* u /* scratch [V] */) {
  for (int i = 0; i < K; ++i) {
    double d = exp(g[i]);
    for (int j = 0; j < V; ++j) S[i * V + j] *= d;
  }
  for (int j = 0; j < V; ++j) {
    double ks = 0.0;
    for (int i = 0; i < K; ++i) ks += kh[i] * S[i * V + j];
    u[j] = v[j] - ks;
  }
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j) S[i * V + j] += beta * kh[i] * u[j];
  for (int j = 0; j < V; ++j) {
    double acc = 0.0;
    for (int i = 0; i < K; ++i) acc += qh[i] * S[i * V + j];
    o[j] = acc;
  }
}

/* ------------------------------------------------------------- kda_decode */

/* oracle_kda_decode: the decode recurrence over a slot-indexed state pool.
 *
 * [KD] Tensor Shapes: output [T, HV, V]; q, k [T, H, K]; v [T, HV, V];
 * raw_gate [T, HV, K]; beta_logits [T, HV]; a_log [HV]; dt_bias [HV, K];
 * cu_seqlens [B + 1]; state_pool [max_slots, HV, K, V] (K_FIRST, mutated);
 * state_indices [B].  (The leading batch dimension of 1 is dropped.)
 * [DR] Code: value head hv uses key head hv / G with G = HV / H
 * (repeat_interleave), scale defaults to K^-1/2, the state starts from the
 * kept state and the final state is returned (here: written back to the
 * pool).
 *
 * Requests are processed one after another, b = 0 .. B-1, value heads in
 * order.  Slot and range handling (the pages are silent; this is the
 * library's documented contract):
 *   state_indices[b] < 0          padded request: output rows zeroed, no state
 *                                 touched, no error;
 *   state_indices[b] >= max_slots ORACLE_BAD_SLOT, output rows zeroed;
 *   a range outside 0 <= cu[b] <= cu[b+1] <= T sets ORACLE_BAD_SEQLEN and the
 *   request is skipped (its rows are unknown, so nothing is written);
 *   cu[0] != 0 or cu[B] != T sets ORACLE_BAD_SEQLEN only.
 *
 * Parity: pinned by the delta-rule properties, closed forms and brute force in
 * the test suite; the gate formula by the closed forms its wording fixes (see
 * gate_value). */
int oracle_kda_decode(double* output, const double* q, const double* k, const double* v,
                      const double* raw_gate, const double* beta_logits, const double* a_log,
                      const double* dt_bias, const int32_t* cu_seqlens, double* state_pool,
                      const int32_t* state_indices, int gate_mode, double lower_bound,
                      double scale, double l2_eps, int B, int T, int H, int HV, int K, int V,
                      int max_slots, int32_t* status) {
  if (H <= 0 || HV % H != 0) return -1;
  int G = HV / H;
  int32_t st = 0;
  if (cu_seqlens[0] != 0 || cu_seqlens[B] != T) st |= ORACLE_BAD_SEQLEN;

  double* S = (double*)malloc(sizeof(double) * (size_t)K * V);
  double* qh = (double*)malloc(sizeof(double) * K);
  double* kh = (double*)malloc(sizeof(double) * K);
  double* g = (double*)malloc(sizeof(double) * K);
  double* vv = (double*)malloc(sizeof(double) * V);
  double* u = (double*)malloc(sizeof(double) * V);

  for (int b = 0; b < B; ++b) {
    int t0 = cu_seqlens[b], t1 = cu_seqlens[b + 1];
    if (t0 < 0 || t1 < t0 || t1 > T) {
      st |= ORACLE_BAD_SEQLEN;
      continue;
    }
    int slot = state_indices[b];
    if (slot < 0 || slot >= max_slots) {
      if (slot >= max_slots) st |= ORACLE_BAD_SLOT;
      for (int t = t0; t < t1; ++t)
        for (int hv = 0; hv < HV; ++hv)
          for (int j = 0; j < V; ++j) output[((size_t)t * HV + hv) * V + j] = 0.0;
      continue;
    }
    for (int hv = 0; hv < HV; ++hv) {
      int h = hv / G;
      double* Sp = state_pool + ((size_t)slot * HV + hv) * (size_t)K * V;
      memcpy(S, Sp, sizeof(double) * (size_t)K * V);
      for (int t = t0; t < t1; ++t) {
        l2_normalise(qh, q + ((size_t)t * H + h) * K, K, l2_eps, scale);
        l2_normalise(kh, k + ((size_t)t * H + h) * K, K, l2_eps, 1.0);
        for (int i = 0; i < K; ++i)
          g[i] = gate_value(raw_gate[((size_t)t * HV + hv) * K + i], dt_bias[(size_t)hv * K + i],
                            a_log[hv], gate_mode, lower_bound);
        double beta = sigmoid(beta_logits[(size_t)t * HV + hv]);
        for (int j = 0; j < V; ++j) vv[j] = v[((size_t)t * HV + hv) * V + j];
        delta_rule_token(S, output + ((size_t)t * HV + hv) * V, qh, kh, vv, g, beta, K, V, u);
      }
      if (t1 > t0) memcpy(Sp, S, sizeof(double) * (size_t)K * V);
    }
  }
  free(S); free(qh); free(kh); free(g); free(vv); free(u);
  if (status) *status |= st;
  return 0;
}

/* --------------------------------------------------------- kda_block_tkg */

/* Optional intermediates of the block, for the layout and stage pins in the
 * test suite.  Any pointer may be NULL.  Shapes use r = b * n + j. */
typedef struct {
  double* xhat;  /* [B*n, Hd]    input RMSNorm output                       */
  double* proj;  /* [B*n, I]     fused projection, I = 2*K*nh + V*nh + 2*K + nh */
  double* qc;    /* [B*n, nh, K] q after short conv + SiLU, head-major      */
  double* kc;    /* [B*n, nh, K]                                             */
  double* vc;    /* [B*n, nh, V]                                             */
  double* graw;  /* [B*n, nh, K] forget-gate pre-activation (f_a . W_fb)    */
  double* g;     /* [B*n, nh, K] activated log-decay                         */
  double* beta;  /* [B*n, nh]    sigmoid(beta column)                        */
  double* o;     /* [B*n, nh, V] recurrence read                             */
  double* z;     /* [B*n, nh, V] output-gate pre-activation (g_a . W_gb)    */
  double* on;    /* [B*n, nh, V] gated output RMSNorm                        */
} oracle_block_trace;

/* oracle_kda_block_tkg: the fused KDA block for token generation.
 *
 * [BT] signature and :param: entries, in the Background's order:
 *   1. input RMSNorm: xhat = hidden * (mean(hidden^2) + rms_norm_eps)^-1/2 * gamma_in
 *   2. fused projection P = xhat . W_in, W_in [Hd, I] contraction-first, columns
 *      q | k | v | g_a | beta | f_a with widths K*nh, K*nh, V*nh, K, nh, K;
 *      q and k channel-outer (column d*nh + h), v head-outer (h*V + d);
 *   3. depthwise causal short conv over the q, k, v streams: window =
 *      conv_state[b, s, c, 0..Kc-2] (oldest first) then the new input;
 *      y = sum_j conv_w[s, j, c] * window[j] (tap 0 oldest); y <- SiLU(y);
 *      conv_state keeps the last Kc-1 PRE-convolution inputs;
 *   4. forget gate: graw[h*K + d] = f_a . W_fb[:, h*K + d] (W_fb head-outer),
 *      g = lower_bound * sigmoid(exp(A_log[h]) * (graw + dt_bias[d, h]));
 *   5. beta = sigmoid(beta column); q, k L2-normalised with l2_eps, q * scale;
 *   6. delta-rule recurrence on S[b, h] ([B, nh, K, V], K_FIRST), in place;
 *   7. gated output RMSNorm over V per head: z[d*nh + h] = g_a . W_gb[:, d*nh + h]
 *      (W_gb channel-outer); on = o * (mean_d o^2 + rms_norm_eps)^-1/2 *
 *      gamma_o[d] * act(z), act = sigmoid (out_gate ORACLE_OUT_GATE_SIGMOID,
 *      the default) or swish (ORACLE_OUT_GATE_SWISH): see output_gate;
 *   8. out[b, j, :] = sum_{h, d} on[h, d] * W_o[h*V + d, :]  (W_o rows taken
 *      head-outer, a reading of "dv * num_head on the partition axis").
 * Tokens j = 0 .. n-1 of a request are processed in order, the conv window and
 * S carried from one to the next.  No activation sits between f_a and W_fb.
 *
 * Parity: every stage pinned by closed forms and layout probes in the test
 * suite (the forget gate by the same closed forms as gate_value, the output
 * gate per setting by its values at z = 0 and z >> 0).  Which output-gate
 * activation the page means stays a reading. */
int oracle_kda_block_tkg(double* out, const double* hidden, const double* gamma_in,
                         const double* W_in, const double* W_fb, const double* W_gb,
                         const double* conv_w, const double* A_log, const double* dt_bias,
                         const double* gamma_o, const double* W_o, double* S,
                         double* conv_state, double scale, double lower_bound,
                         double rms_norm_eps, double l2_eps, int B, int n, int Hd, int nh,
                         int K, int V, int Kc, int out_gate, oracle_block_trace* tr) {
  if (B < 0 || n < 1 || Kc < 1) return -1;
  if (out_gate != ORACLE_OUT_GATE_SIGMOID && out_gate != ORACLE_OUT_GATE_SWISH) return -1;
  const int CQ = K * nh, CV = V * nh;
  const int I = CQ + CQ + CV + K + nh + K;
  const int off_q = 0, off_k = CQ, off_v = 2 * CQ, off_ga = 2 * CQ + CV;
  const int off_beta = off_ga + K, off_fa = off_beta + nh;
  const int CS = CQ > CV ? CQ : CV; /* channels per conv stream (conv_w inner dim) */

  double* xh = (double*)malloc(sizeof(double) * Hd);
  double* P = (double*)malloc(sizeof(double) * I);
  double* y = (double*)malloc(sizeof(double) * 3 * CS); /* conv outputs, per stream */
  double* qh = (double*)malloc(sizeof(double) * K);
  double* kh = (double*)malloc(sizeof(double) * K);
  double* g = (double*)malloc(sizeof(double) * K);
  double* vv = (double*)malloc(sizeof(double) * V);
  double* u = (double*)malloc(sizeof(double) * V);
  double* o = (double*)malloc(sizeof(double) * V);
  double* on = (double*)malloc(sizeof(double) * (size_t)nh * V);
  double* tmpq = (double*)malloc(sizeof(double) * K);
  double* tmpk = (double*)malloc(sizeof(double) * K);
  double* graw = (double*)malloc(sizeof(double) * CQ);
  double* zall = (double*)malloc(sizeof(double) * CV);

  for (int b = 0; b < B; ++b) {
    for (int j = 0; j < n; ++j) {
      const size_t r = (size_t)b * n + j;
      const double* x = hidden + r * Hd;
      /* 1. input RMSNorm */
      double ms = 0.0;
      for (int i = 0; i < Hd; ++i) ms += x[i] * x[i];
      ms /= Hd;
      double rinv = 1.0 / sqrt(ms + rms_norm_eps);
      for (int i = 0; i < Hd; ++i) xh[i] = x[i] * rinv * gamma_in[i];
      /* 2. fused projection.  Each P[c] is summed over i = 0 .. Hd-1 in order;
       * the i-outer loop only walks W_in row by row. */
      for (int c = 0; c < I; ++c) P[c] = 0.0;
      for (int i = 0; i < Hd; ++i) {
        const double* w = W_in + (size_t)i * I;
        for (int c = 0; c < I; ++c) P[c] += xh[i] * w[c];
      }
      /* 4a/7a. the two low-rank up-projections of the gate latents (same
       * summation order, r = 0 .. K-1, for every output column) */
      for (int c = 0; c < CQ; ++c) graw[c] = 0.0;
      for (int c = 0; c < CV; ++c) zall[c] = 0.0;
      for (int rr = 0; rr < K; ++rr) {
        const double* wf = W_fb + (size_t)rr * CQ;
        const double* wg = W_gb + (size_t)rr * CV;
        for (int c = 0; c < CQ; ++c) graw[c] += P[off_fa + rr] * wf[c];
        for (int c = 0; c < CV; ++c) zall[c] += P[off_ga + rr] * wg[c];
      }
      /* 3. short conv + SiLU per stream and channel, then the window shift */
      for (int s = 0; s < 3; ++s) {
        const int nch = (s == 2) ? CV : CQ;
        const int off = (s == 0) ? off_q : (s == 1) ? off_k : off_v;
        for (int c = 0; c < nch; ++c) {
          double* cs = conv_state + (((size_t)b * 3 + s) * CS + c) * (Kc - 1);
          double acc = 0.0;
          for (int t = 0; t < Kc - 1; ++t) acc += conv_w[((size_t)s * Kc + t) * CS + c] * cs[t];
          double xnew = P[off + c];
          acc += conv_w[((size_t)s * Kc + (Kc - 1)) * CS + c] * xnew;
          y[(size_t)s * CS + c] = acc * sigmoid(acc);
          for (int t = 0; t + 1 < Kc - 1; ++t) cs[t] = cs[t + 1];
          if (Kc > 1) cs[Kc - 2] = xnew;
        }
      }
      /* 4-7 per head */
      for (int h = 0; h < nh; ++h) {
        for (int d = 0; d < K; ++d) {
          tmpq[d] = y[0 * (size_t)CS + (size_t)d * nh + h];
          tmpk[d] = y[1 * (size_t)CS + (size_t)d * nh + h];
        }
        for (int d = 0; d < V; ++d) vv[d] = y[2 * (size_t)CS + (size_t)h * V + d];
        for (int d = 0; d < K; ++d) {
          double acc = graw[(size_t)h * K + d]; /* W_fb columns are head-outer */
          if (tr && tr->graw) tr->graw[(r * nh + h) * K + d] = acc;
          g[d] = lower_bound * sigmoid(exp(A_log[h]) * (acc + dt_bias[(size_t)d * nh + h]));
        }
        double beta = sigmoid(P[off_beta + h]);
        l2_normalise(qh, tmpq, K, l2_eps, scale);
        l2_normalise(kh, tmpk, K, l2_eps, 1.0);
        double* Sh = S + ((size_t)b * nh + h) * (size_t)K * V;
        delta_rule_token(Sh, o, qh, kh, vv, g, beta, K, V, u);
        /* 7. gated output RMSNorm */
        double m2 = 0.0;
        for (int d = 0; d < V; ++d) m2 += o[d] * o[d];
        m2 /= V;
        double oinv = 1.0 / sqrt(m2 + rms_norm_eps);
        for (int d = 0; d < V; ++d) {
          double zz = zall[(size_t)d * nh + h]; /* W_gb columns are channel-outer */
          if (tr && tr->z) tr->z[(r * nh + h) * V + d] = zz;
          on[(size_t)h * V + d] = o[d] * oinv * gamma_o[d] * output_gate(zz, out_gate);
        }
        if (tr) {
          for (int d = 0; d < K; ++d) {
            if (tr->qc) tr->qc[(r * nh + h) * K + d] = tmpq[d];
            if (tr->kc) tr->kc[(r * nh + h) * K + d] = tmpk[d];
            if (tr->g) tr->g[(r * nh + h) * K + d] = g[d];
          }
          for (int d = 0; d < V; ++d) {
            if (tr->vc) tr->vc[(r * nh + h) * V + d] = vv[d];
            if (tr->o) tr->o[(r * nh + h) * V + d] = o[d];
            if (tr->on) tr->on[(r * nh + h) * V + d] = on[(size_t)h * V + d];
          }
          if (tr->beta) tr->beta[r * nh + h] = beta;
        }
      }
      /* 8. output projection (each out column summed over i in order) */
      double* orow = out + r * Hd;
      for (int c = 0; c < Hd; ++c) orow[c] = 0.0;
      for (int i = 0; i < nh * V; ++i) {
        const double* w = W_o + (size_t)i * Hd;
        for (int c = 0; c < Hd; ++c) orow[c] += on[i] * w[c];
      }
      if (tr) {
        if (tr->xhat) memcpy(tr->xhat + r * Hd, xh, sizeof(double) * Hd);
        if (tr->proj) memcpy(tr->proj + r * I, P, sizeof(double) * I);
      }
    }
  }
  free(xh); free(P); free(y); free(qh); free(kh); free(g); free(vv); free(u); free(o);
  free(on); free(tmpq); free(tmpk); free(graw); free(zall);
  return 0;
}
