/*
 * gdn_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, sequential fp64 CPU statement of the batched Gated DeltaNet
 * (GDN) speculative transaction: causal short convolution over the verify
 * positions, L2 normalisation of q and k, the gated delta rule, and the
 * per-row accepted-prefix commit.  It exists only to check the CUDA library;
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header or constant with the CUDA sources.
 *
 * Sources followed (page title, section):
 *  - "MTP inference: review and commit structure", Functional commits, item 2
 *    (GDN speculative transactions: verifier buffers, accepted-prefix state
 *    replay, compiled short convolution) and Verification and limits (partial
 *    GDN commits replay only the accepted recurrent prefix; chunked and
 *    sequential recurrences differ only in rounding).
 *  - "Add request-owned eight-way MTP serving for Qwen 35B", sections 2 and 4
 *    (per-row committed offsets; inactive rows use keep=0; the commit handles
 *    keep = 0, 1, 2 and keep=0 restores the pre-verification state).
 *  - "perf(qwen): full-context MTP draft prefill and replay-free rewind",
 *    Summary item 4 (the GDN mixer is rerun from the pre-verification state,
 *    no full-model replay).
 *  - The gated delta rule itself, S_t = a_t S_{t-1} (I - b_t k_t k_t^T)
 *    + b_t v_t k_t^T with a_t = exp(g_t) and o_t = S_t q_t / sqrt(d_k)
 *    (Yang, Kautz & Hatamizadeh, "Gated Delta Networks", ICLR 2025, the gated
 *    delta rule), with the state stored as S[j][i], j over d_v, i over d_k,
 *    so that v ~ S k.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - conv: depthwise, width 4, no bias; w[c][3] multiplies the current token,
 *    w[c][0] the token three positions back; activation SiLU (act=1) or none;
 *  - L2 norm: x / sqrt(sum x^2 + 1e-6); q is further scaled by 1/sqrt(d_k);
 *  - channel order of the conv input: q [H_k][d_k] | k [H_k][d_k] | v [H_v][d_v];
 *  - value head h reads key head floor(h * H_k / H_v);
 *  - the state is fp32 between calls and fp64 inside a call; outputs are fp64.
 *
 * Everything is fp64 with IEEE semantics; build with -ffp-contract=off so the
 * result does not depend on the host's fused multiply-add.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_W 4        /* conv width */
#define OR_HIST 3     /* inputs kept in the committed conv window */
#define OR_EPS 1e-6   /* L2-norm epsilon */

#define OR_EXPORT __attribute__((visibility("default")))

static double or_act(double z, int act) { return act ? z / (1.0 + exp(-z)) : z; }

/*
 * Causal depthwise convolution of one row over n new tokens.
 *   hist [C][3]  the three inputs before the first new token, oldest first
 *   x    [n][C]  the new raw inputs
 *   w    [C][4]  taps; w[c][3] multiplies the current token
 *   y    [n][C]  act(sum_j w[c][j] * xt[t - 3 + j]) where xt is hist ++ x
 */
OR_EXPORT void oracle_causal_conv(int n, int C, int act, const double *hist,
                                  const double *x, const double *w, double *y) {
  for (int t = 0; t < n; ++t) {
    for (int c = 0; c < C; ++c) {
      double acc = 0.0;
      for (int j = 0; j < OR_W; ++j) {
        int p = t - (OR_W - 1) + j; /* index into x; negative reaches hist */
        double v = p < 0 ? hist[(size_t)c * OR_HIST + (OR_HIST + p)] : x[(size_t)p * C + c];
        acc += w[(size_t)c * OR_W + j] * v;
      }
      y[(size_t)t * C + c] = or_act(acc, act);
    }
  }
}

/* out = a / sqrt(sum a^2 + eps) * scale */
static void or_l2norm(int d, const double *a, double scale, double *out) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += a[i] * a[i];
  double inv = 1.0 / sqrt(ss + OR_EPS);
  for (int i = 0; i < d; ++i) out[i] = a[i] * inv * scale;
}

/*
 * One gated delta-rule step on one head, in place.
 *   S [dv][dk]; k, q length dk (already normalised); v length dv.
 * For each value row j: u = S_j . k;  S_j <- a S_j + b (v_j - a u) k;
 * o_j = S_j . q  (with the updated S_j).  This is row j of
 * S <- a S (I - b k k^T) + b v k^T, o = S q.
 */
static void or_delta_step(int dk, int dv, double *S, const double *k, const double *q,
                          const double *v, double g, double beta, double *o) {
  double a = exp(g);
  for (int j = 0; j < dv; ++j) {
    double *row = S + (size_t)j * dk;
    double u = 0.0;
    for (int i = 0; i < dk; ++i) u += row[i] * k[i];
    double e = beta * (v[j] - a * u);
    for (int i = 0; i < dk; ++i) row[i] = a * row[i] + e * k[i];
    double oj = 0.0;
    for (int i = 0; i < dk; ++i) oj += row[i] * q[i];
    o[j] = oj;
  }
}

/*
 * Run n tokens of one row through conv, normalisation and the recurrence.
 *   hist [C][3], x [n][C], w [C][4], g/beta [n][Hv]
 *   S    [Hv][dv][dk] fp64, advanced in place over all n tokens
 *   o    [n][Hv][dv]
 *   Sall [n][Hv][dv][dk] state after each token, or NULL
 */
static int or_row(int n, int Hk, int Hv, int dk, int dv, int act, const double *hist,
                  const double *x, const double *w, const double *g, const double *beta,
                  double *S, double *o, double *Sall) {
  const int C = 2 * Hk * dk + Hv * dv;
  double *y = (double *)malloc(sizeof(double) * (size_t)n * C);
  double *kh = (double *)malloc(sizeof(double) * dk);
  double *qh = (double *)malloc(sizeof(double) * dk);
  if (!y || !kh || !qh) { free(y); free(kh); free(qh); return -1; }
  oracle_causal_conv(n, C, act, hist, x, w, y);
  const size_t Shead = (size_t)dv * dk;
  for (int t = 0; t < n; ++t) {
    const double *yt = y + (size_t)t * C;
    for (int h = 0; h < Hv; ++h) {
      int hk = (int)(((long long)h * Hk) / Hv);
      or_l2norm(dk, yt + (size_t)hk * dk, 1.0 / sqrt((double)dk), qh);
      or_l2norm(dk, yt + (size_t)Hk * dk + (size_t)hk * dk, 1.0, kh);
      const double *v = yt + (size_t)2 * Hk * dk + (size_t)h * dv;
      or_delta_step(dk, dv, S + h * Shead, kh, qh, v, g[(size_t)t * Hv + h],
                    beta[(size_t)t * Hv + h], o + ((size_t)t * Hv + h) * dv);
      if (Sall) memcpy(Sall + ((size_t)t * Hv + h) * Shead, S + h * Shead, sizeof(double) * Shead);
    }
  }
  free(y); free(kh); free(qh);
  return 0;
}

/*
 * Verify: run the T draft-plus-verify positions of every active row from the
 * pre-verification state S0, without changing S0 or the window.
 *   x    [B][T][C] raw inputs;  w [C][4];  win [B][C][3] committed window
 *   g, beta [B][T][Hv];  S0 [B][Hv][dv][dk] fp32;  active [B]
 *   o    [B][T][Hv][dv] out; inactive rows get 0
 *   Sall [B][T][Hv][dv][dk] out (state after each position), or NULL
 * Returns 0, or -1 on allocation failure.
 */
OR_EXPORT int oracle_verify(int B, int T, int Hk, int Hv, int dk, int dv, int act,
                            const double *x, const double *w, const double *win,
                            const double *g, const double *beta, const float *S0,
                            const uint8_t *active, double *o, double *Sall) {
  const int C = 2 * Hk * dk + Hv * dv;
  const size_t nS = (size_t)Hv * dv * dk;
  double *S = (double *)malloc(sizeof(double) * nS);
  if (!S) return -1;
  for (int b = 0; b < B; ++b) {
    double *ob = o + (size_t)b * T * Hv * dv;
    double *Sb = Sall ? Sall + (size_t)b * T * nS : NULL;
    if (!active[b]) {
      memset(ob, 0, sizeof(double) * (size_t)T * Hv * dv);
      if (Sb)
        for (int t = 0; t < T; ++t)
          for (size_t i = 0; i < nS; ++i) Sb[t * nS + i] = S0[(size_t)b * nS + i];
      continue;
    }
    for (size_t i = 0; i < nS; ++i) S[i] = S0[(size_t)b * nS + i];
    if (or_row(T, Hk, Hv, dk, dv, act, win + (size_t)b * C * OR_HIST, x + (size_t)b * T * C, w,
               g + (size_t)b * T * Hv, beta + (size_t)b * T * Hv, S, ob, Sb)) {
      free(S);
      return -1;
    }
  }
  free(S);
  return 0;
}

/*
 * Commit the accepted prefix of each row.
 *   keep' = keep if the row is active and 0 <= keep <= T, else 0; an active
 *   row with keep outside [0, T] also sets bit 0 of *status.
 *   keep' >= 1: S[b] <- fp32(state after keep' positions), the window becomes
 *              the last three of (window ++ x_0 .. x_{keep'-1}), offsets += keep'.
 *   keep' == 0: nothing changes (exact restore of the pre-verification state).
 *   Sall [B][T][Hv][dv][dk] from oracle_verify; x [B][T][C];
 *   S [B][Hv][dv][dk] fp32 in/out; win [B][C][3] in/out; offsets [B] in/out.
 */
OR_EXPORT void oracle_commit(int B, int T, int Hv, int dk, int dv, int C, const int32_t *keep,
                             const uint8_t *active, const double *Sall, const double *x,
                             float *S, double *win, int32_t *offsets, int32_t *status) {
  const size_t nS = (size_t)Hv * dv * dk;
  for (int b = 0; b < B; ++b) {
    int kp = 0;
    if (active[b]) {
      if (keep[b] >= 0 && keep[b] <= T) kp = keep[b];
      else *status |= 1;
    }
    if (kp == 0) continue;
    const double *src = Sall + ((size_t)b * T + (kp - 1)) * nS;
    for (size_t i = 0; i < nS; ++i) S[(size_t)b * nS + i] = (float)src[i];
    for (int c = 0; c < C; ++c) {
      double *wc = win + ((size_t)b * C + c) * OR_HIST;
      double tail[OR_HIST];
      for (int i = 0; i < OR_HIST; ++i) {
        int p = kp - OR_HIST + i; /* index into x; negative reaches the old window */
        tail[i] = p < 0 ? wc[OR_HIST + p] : x[((size_t)b * T + p) * C + c];
      }
      for (int i = 0; i < OR_HIST; ++i) wc[i] = tail[i];
    }
    offsets[b] += kp;
  }
}

/*
 * Prime the state over a prompt of L tokens per row: the same sequential
 * recurrence as verify, over all L tokens, followed by a full commit.
 *   x [B][L][C]; g, beta [B][L][Hv]; win [B][C][3] in/out; S fp32 in/out;
 *   o [B][L][Hv][dv] out; offsets [B] += L.
 */
OR_EXPORT int oracle_prefill(int B, int L, int Hk, int Hv, int dk, int dv, int act,
                             const double *x, const double *w, double *win, const double *g,
                             const double *beta, float *S, double *o, int32_t *offsets) {
  const int C = 2 * Hk * dk + Hv * dv;
  const size_t nS = (size_t)Hv * dv * dk;
  double *Sd = (double *)malloc(sizeof(double) * nS);
  if (!Sd) return -1;
  for (int b = 0; b < B; ++b) {
    for (size_t i = 0; i < nS; ++i) Sd[i] = S[(size_t)b * nS + i];
    double *wb = win + (size_t)b * C * OR_HIST;
    const double *xb = x + (size_t)b * L * C;
    if (or_row(L, Hk, Hv, dk, dv, act, wb, xb, w, g + (size_t)b * L * Hv,
               beta + (size_t)b * L * Hv, Sd, o + (size_t)b * L * Hv * dv, NULL)) {
      free(Sd);
      return -1;
    }
    for (size_t i = 0; i < nS; ++i) S[(size_t)b * nS + i] = (float)Sd[i];
    for (int c = 0; c < C; ++c) {
      double tail[OR_HIST];
      for (int i = 0; i < OR_HIST; ++i) {
        int p = L - OR_HIST + i; /* position in the prompt; negative reaches the old window */
        tail[i] = p < 0 ? wb[(size_t)c * OR_HIST + (OR_HIST + p)] : xb[(size_t)p * C + c];
      }
      for (int i = 0; i < OR_HIST; ++i) wb[(size_t)c * OR_HIST + i] = tail[i];
    }
    offsets[b] += L;
  }
  free(Sd);
  return 0;
}

/*
 * Greedy acceptance of one verify cycle, the decision that "Add request-owned
 * eight-way MTP serving for Qwen 35B" takes off the host so that a decode
 * cycle needs no host synchronisation.  Position 0 of a row's verify holds the
 * last accepted token; positions 1..T-1 hold the draft tokens.  For an active
 * row b:
 *   target_t = argmax_v logits[b][t][v]   (the first index of the maximum;
 *                                          NaN never wins; an all-NaN row gives 0)
 *   keep[b]  = 1 + the number of leading t in 1..T-1 with draft[b][t] == target_{t-1}
 *   next[b]  = target_{keep[b] - 1}       (the token the next cycle feeds)
 * Inactive rows: keep 0, next -1.  logits [B][T][V] as fp64 (the bf16 values,
 * exactly); draft [B][T] (draft[b][0] is not read).
 */
OR_EXPORT int oracle_accept(int B, int T, int V, const double *logits, const int32_t *draft,
                            const uint8_t *active, int32_t *keep, int32_t *next) {
  int32_t *target = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
  if (!target) return -1;
  for (int b = 0; b < B; ++b) {
    if (!active[b]) {
      keep[b] = 0;
      next[b] = -1;
      continue;
    }
    for (int t = 0; t < T; ++t) {
      const double *row = logits + ((size_t)b * T + t) * V;
      int best = -1;
      double best_v = 0.0;
      for (int v = 0; v < V; ++v) {
        const double x = row[v];
        if (x != x) continue; /* NaN */
        if (best < 0 || x > best_v) {
          best = v;
          best_v = x;
        }
      }
      target[t] = best < 0 ? 0 : best;
    }
    int k = 1;
    while (k < T && draft[(size_t)b * T + k] == target[k - 1]) ++k;
    keep[b] = k;
    next[b] = target[k - 1];
  }
  free(target);
  return 0;
}

/*
 * Gated RMSNorm of the GDN output, the step that follows the mixer in the
 * hybrid-Qwen GDN layer ("MTP inference: review and commit structure",
 * Functional commits item 4, names it beside the conv-cache mutation as a
 * custom-operator boundary).  Per (row, position, value head) vector o of d
 * values with gate z and weight w [d]:
 *   y[j] = o[j] / sqrt(mean_j o[j]^2 + eps) * w[j] * silu(z[j]),  silu(z) = z / (1 + e^-z)
 * o, z, y [n][d]; w [d].
 */
OR_EXPORT void oracle_gated_rmsnorm(int n, int d, const double *o, const double *z, const double *w, double eps,
                                    double *y) {
  for (int r = 0; r < n; ++r) {
    const double *orow = o + (size_t)r * d, *zrow = z + (size_t)r * d;
    double ss = 0.0;
    for (int j = 0; j < d; ++j) ss += orow[j] * orow[j];
    const double inv = 1.0 / sqrt(ss / d + eps);
    for (int j = 0; j < d; ++j) {
      const double gate = zrow[j] / (1.0 + exp(-zrow[j]));
      y[(size_t)r * d + j] = orow[j] * inv * w[j] * gate;
    }
  }
}
