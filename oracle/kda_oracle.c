/*
 * kda_oracle.c -- float64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the GPU library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (one head at a time, token by token, in float64):
 *
 *   a_t  = exp(-exp(log_alpha_t))     per key channel (vector over dk),
 *                                     one scalar per token, or 1 (no decay)
 *   S    = Diag(a_t) S                decay first: row i of S is scaled by a_t[i]
 *   u_t  = beta_t (v_t - S^T k_t)     read the decayed memory at key k_t
 *   S    = S + k_t u_t^T              write the correction along k_t
 *   o_t  = S^T q_t                    read-out after the write
 *
 * Sources, by page title and section:
 *  - "22,580: From GPT-2 to Kimi K3" (yichencityu.github.io), section 5.2
 *    "The delta rule: erase first, then write": v_old = k S, u = beta (v - v_old),
 *    S <- S + k^T u, o = q S (row-vector form; S^T q above is the same product
 *    written for column vectors, with S stored [dk][dv]).
 *  - same page, section 6.1: the token-by-token prefill loop that collects
 *    q_t S_t after each write, so the output includes the current token.
 *  - "22580: From GPT-2 to Kimi3, Explained" (zharfai.com), "Gated DeltaNet
 *    adds controlled forgetting": S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T.
 *    With a per-channel a_t the decay is applied first, as Diag(a_t) S_{t-1},
 *    and the delta read and write act on the decayed state.
 *  - "22580: From GPT-2 to Kimi K3, Explained" (lukebest.github.io),
 *    "KDA (per-channel alpha)": alpha = exp(-exp(log_alpha)), one value per
 *    channel; the channel is the key axis (rows of S).
 *
 * Inputs are float32 arrays (bf16 inputs arrive already widened, which is
 * exact); every value is widened to double on read and nothing is rounded
 * back.  Layout per head: q,k [T][dk], v [T][dv], beta [T],
 * log_alpha [T][dk] (mode 2) or [T] (mode 1) or unused (mode 0),
 * h0 and hT [dk][dv] (double), o [T][dv] (double).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ALPHA_NONE 0
#define ORACLE_ALPHA_SCALAR 1
#define ORACLE_ALPHA_CHANNEL 2

/* Returns 0 on success, -1 on bad arguments, -2 if scratch allocation fails. */
int kda_oracle_recurrent(const float *q, const float *k, const float *v,
                         const float *beta, const float *log_alpha,
                         int alpha_mode, const double *h0, long T, int dk,
                         int dv, double *o, double *hT) {
  if (T < 0 || dk <= 0 || dv <= 0 || !o || !hT) return -1;
  if (alpha_mode < 0 || alpha_mode > 2) return -1;
  if (alpha_mode != ORACLE_ALPHA_NONE && !log_alpha) return -1;
  if (T > 0 && (!q || !k || !v || !beta)) return -1;

  double *S = hT; /* the state lives in the output buffer */
  double *a = (double *)malloc(sizeof(double) * (size_t)dk);
  double *kd = (double *)malloc(sizeof(double) * (size_t)dk);
  double *u = (double *)malloc(sizeof(double) * (size_t)dv);
  if (!a || !kd || !u) {
    free(a); free(kd); free(u);
    return -2;
  }
  if (h0)
    memcpy(S, h0, sizeof(double) * (size_t)dk * (size_t)dv);
  else
    memset(S, 0, sizeof(double) * (size_t)dk * (size_t)dv);

  for (long t = 0; t < T; ++t) {
    const float *qt = q + t * dk;
    const float *kt = k + t * dk;
    const float *vt = v + t * dv;
    const double bt = (double)beta[t];

    /* decay: a = exp(-exp(log_alpha)) */
    for (int i = 0; i < dk; ++i) {
      if (alpha_mode == ORACLE_ALPHA_CHANNEL)
        a[i] = exp(-exp((double)log_alpha[t * dk + i]));
      else if (alpha_mode == ORACLE_ALPHA_SCALAR)
        a[i] = exp(-exp((double)log_alpha[t]));
      else
        a[i] = 1.0;
      kd[i] = (double)kt[i];
    }
    /* S <- Diag(a) S */
    for (int i = 0; i < dk; ++i) {
      double *row = S + (size_t)i * dv;
      for (int j = 0; j < dv; ++j) row[j] *= a[i];
    }
    /* u = beta (v - S^T k) */
    for (int j = 0; j < dv; ++j) u[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
      const double *row = S + (size_t)i * dv;
      for (int j = 0; j < dv; ++j) u[j] += kd[i] * row[j];
    }
    for (int j = 0; j < dv; ++j) u[j] = bt * ((double)vt[j] - u[j]);
    /* S <- S + k u^T */
    for (int i = 0; i < dk; ++i) {
      double *row = S + (size_t)i * dv;
      for (int j = 0; j < dv; ++j) row[j] += kd[i] * u[j];
    }
    /* o_t = S^T q */
    double *ot = o + t * dv;
    for (int j = 0; j < dv; ++j) ot[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
      const double *row = S + (size_t)i * dv;
      const double qi = (double)qt[i];
      for (int j = 0; j < dv; ++j) ot[j] += qi * row[j];
    }
  }
  free(a); free(kd); free(u);
  return 0;
}

/*
 * Linear attention, one head, float64, token by token:
 *
 *   S   = Diag(a_t) S + k_t v_t^T      decay first (rows = key channels), then add
 *   o_t = S^T q_t                      read-out after the write
 *
 * Source: "22,580: From GPT-2 to Kimi K3" (yichencityu.github.io), section
 * 6.2: the state accumulates k^T v chunk after chunk and each query reads the
 * state of all earlier chunks plus the masked (diagonal included) scores of
 * its own chunk, i.e. the token loop above with a_t = 1.  The decayed form
 * (a_t as in kda_oracle_recurrent) is the same decay applied before each
 * write; the pages print only a_t = 1.  No normaliser (the pages' section 6.2
 * form, not the feature-map-with-denominator variant of section 04; that one
 * is kda_oracle_linear_norm).
 * Same layouts and return codes as kda_oracle_recurrent; there is no beta.
 */
int kda_oracle_linear(const float *q, const float *k, const float *v,
                      const float *log_alpha, int alpha_mode, const double *h0,
                      long T, int dk, int dv, double *o, double *hT) {
  if (T < 0 || dk <= 0 || dv <= 0 || !o || !hT) return -1;
  if (alpha_mode < 0 || alpha_mode > 2) return -1;
  if (alpha_mode != ORACLE_ALPHA_NONE && !log_alpha) return -1;
  if (T > 0 && (!q || !k || !v)) return -1;
  double *state = hT;
  if (h0)
    memcpy(state, h0, sizeof(double) * (size_t)dk * (size_t)dv);
  else
    memset(state, 0, sizeof(double) * (size_t)dk * (size_t)dv);
  for (long t = 0; t < T; ++t) {
    for (int c = 0; c < dk; ++c) {
      double decay = 1.0;
      if (alpha_mode == ORACLE_ALPHA_CHANNEL)
        decay = exp(-exp((double)log_alpha[t * dk + c]));
      else if (alpha_mode == ORACLE_ALPHA_SCALAR)
        decay = exp(-exp((double)log_alpha[t]));
      const double kc = (double)k[t * dk + c];
      double *srow = state + (size_t)c * dv;
      for (int e = 0; e < dv; ++e) srow[e] = decay * srow[e] + kc * (double)v[t * dv + e];
    }
    for (int e = 0; e < dv; ++e) {
      double acc = 0.0;
      for (int c = 0; c < dk; ++c) acc += (double)q[t * dk + c] * state[(size_t)c * dv + e];
      o[t * dv + e] = acc;
    }
  }
  return 0;
}

/*
 * Normalised linear attention, one head, float64, token by token, from a
 * zero state:
 *
 *   S   = Diag(a_t) S + k_t v_t^T      as kda_oracle_linear
 *   z   = a_t * z + k_t                the normaliser accumulator (per key channel)
 *   o_t = (S^T q_t) / (q_t . z)        read-out after the write, divided
 *
 * Source: "22,580: From GPT-2 to Kimi K3" (yichencityu.github.io), section 04
 * ("Linear Attention: Bring Back the RNN"): the state gathers k v^T and a
 * normaliser z gathers k, the read-out q S is divided by q z (with q and k
 * passed through a positive feature map first, e.g. ELU + 1; the caller
 * applies it).  The decayed form applies a_t to z exactly as to the rows of S
 * (z is the state's column for a value of all ones); the pages print a_t = 1.
 * A zero denominator is left to IEEE arithmetic.  Writes o [T][dv] and the
 * final S to hT and the final z to zT.  Returns 0, or -1 on bad arguments.
 */
int kda_oracle_linear_norm(const float *q, const float *k, const float *v,
                           const float *log_alpha, int alpha_mode, long T, int dk, int dv,
                           double *o, double *hT, double *zT) {
  if (T < 0 || dk <= 0 || dv <= 0 || !o || !hT || !zT) return -1;
  if (alpha_mode < 0 || alpha_mode > 2) return -1;
  if (alpha_mode != ORACLE_ALPHA_NONE && !log_alpha) return -1;
  if (T > 0 && (!q || !k || !v)) return -1;
  memset(hT, 0, sizeof(double) * (size_t)dk * (size_t)dv);
  memset(zT, 0, sizeof(double) * (size_t)dk);
  for (long t = 0; t < T; ++t) {
    const float *qt = q + t * dk, *kt = k + t * dk, *vt = v + t * dv;
    for (int i = 0; i < dk; ++i) {
      double ai = 1.0;  /* a_t of key channel i */
      if (alpha_mode == ORACLE_ALPHA_CHANNEL)
        ai = exp(-exp((double)log_alpha[t * dk + i]));
      else if (alpha_mode == ORACLE_ALPHA_SCALAR)
        ai = exp(-exp((double)log_alpha[t]));
      double *Si = hT + (size_t)i * dv;
      for (int j = 0; j < dv; ++j) Si[j] = ai * Si[j] + (double)kt[i] * (double)vt[j];
      zT[i] = ai * zT[i] + (double)kt[i];
    }
    double den = 0.0;
    for (int i = 0; i < dk; ++i) den += (double)qt[i] * zT[i];
    for (int j = 0; j < dv; ++j) {
      double num = 0.0;
      for (int i = 0; i < dk; ++i) num += (double)qt[i] * hT[(size_t)i * dv + j];
      o[t * dv + j] = num / den;
    }
  }
  return 0;
}

/* Interface version, so the Python side can refuse a stale build. */
int kda_oracle_version(void) { return 3; }
