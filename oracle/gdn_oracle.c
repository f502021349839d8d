/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet (GDN) core.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this code.  It shares nothing with the CUDA
 * library: no headers, helpers, tables or constants.
 *
 * What it computes (definition, not the chunked method):
 *
 *   The pages ("linear attention cp #1035", section "What does this PR do";
 *   "Linear Attention CP 融合算子 PR #1114 测试报告", section 4.1) name the
 *   operator -- the Gated DeltaNet core of Qwen3.5's linear-attention layers --
 *   and its interface: inputs q, k, v, g, beta and an initial state; outputs the
 *   token output and the final state; gradients dq, dk, dv, dg, dbeta, dH0.  They
 *   do not print the recurrence.  This file writes out the standard gated delta
 *   rule, per batch row b and V head h, with S in R^{dk x dv}:
 *
 *     q_hat = scale * q / sqrt(|q|^2 + eps)      (L2 norm over dk; flag l2norm)
 *     k_hat =         k / sqrt(|k|^2 + eps)
 *     g     = -exp(A_log[h]) * softplus(a + dt_bias[h]),   alpha = exp(g)
 *     beta  = sigmoid(b)
 *     S_t   = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t   = S_t^T q_t
 *
 *   V head h reads Q/K head h / r, r = H / Hqk (section 4.1 of the test report:
 *   the 16 Q/K heads are copied "by grouping" onto the 32 V heads).
 *
 *   Trailing padding (test report section 5.2, B=2 / valid_length 7777): a token
 *   t >= valid_len[b] has output 0, leaves the state unchanged (it acts as g=0,
 *   beta=0) and receives zero gradients.
 *
 *   Segment summary (PR #1035, "p2p" mode: each rank computes the affine map
 *   H_out = M @ H_in + S of its local segment; "all_gather" mode: the summaries
 *   of earlier ranks are merged into the initial state):
 *     M = A_T ... A_1 with A_t = alpha_t (I - beta_t k_t k_t^T)   (dk x dk)
 *     S = the state reached from a zero initial state             (dk x dv)
 *   composition (M2,S2) o (M1,S1) = (M2 M1, M2 S1 + S2), exclusive prefix
 *   H_in[0] = h0, H_in[i] = M_{i-1} H_in[i-1] + S_{i-1}.
 *
 *   Backward: back-propagation through time of the recurrence above for the
 *   scalar L = sum_t <dO_t, o_t> + <dH_T, S_T>, then through the L2 norm and
 *   the scale to the raw q and k, summed over the V heads that share a Q/K head.
 *   PR #1035 passes the state gradient backward across segments ("p2p": the
 *   custom autograd boundary sends the state gradient in the reverse direction);
 *   the gradient summary D of a segment is dL/dH_in for its token outputs alone,
 *   so dH_in = M^T dH_out + D.
 *
 * Layouts (all contiguous, fp64):
 *   q, k [B,T,Hqk,dk]   v, o, dO [B,T,H,dv]   a, b, g, beta [B,T,H]
 *   A_log, dt_bias [H]  states h0, hT, S, D [B,H,dk,dv]   M [B,H,dk,dk]
 *   valid_len int32 [B] or NULL (NULL: every token valid)
 *
 * Every entry point returns 0 on success and a negative number on a bad
 * argument.  Parallel over (b, head) with OpenMP; nthreads <= 0 uses the
 * OpenMP default.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int64_t B, T, Hqk, H, dk, dv;
  int32_t l2norm;
  int32_t reserved;
  double eps;
  double scale;
} oracle_problem;

static int check_problem(const oracle_problem* p) {
  if (!p) return -1;
  if (p->B < 0 || p->T < 0 || p->Hqk <= 0 || p->H <= 0 || p->dk <= 0 || p->dv <= 0) return -2;
  if (p->H % p->Hqk != 0) return -3;
  if (!(p->scale > 0.0)) return -4;
  return 0;
}

static int64_t valid_length(const oracle_problem* p, const int32_t* valid_len, int64_t b) {
  if (!valid_len) return p->T;
  int64_t L = valid_len[b];
  if (L < 0) L = 0;
  if (L > p->T) L = p->T;
  return L;
}

static int check_valid_len(const oracle_problem* p, const int32_t* valid_len) {
  if (!valid_len) return 0;
  for (int64_t b = 0; b < p->B; ++b)
    if (valid_len[b] < 0 || valid_len[b] > p->T) return -5;
  return 0;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

static double softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* index helpers */
#define QK_IDX(p, b, t, hq) ((((b) * (p)->T + (t)) * (p)->Hqk + (hq)) * (p)->dk)
#define V_IDX(p, b, t, h) ((((b) * (p)->T + (t)) * (p)->H + (h)) * (p)->dv)
#define G_IDX(p, b, t, h) (((b) * (p)->T + (t)) * (p)->H + (h))
#define ST_IDX(p, b, h) (((b) * (p)->H + (h)) * (p)->dk * (p)->dv)
#define M_IDX(p, b, h) (((b) * (p)->H + (h)) * (p)->dk * (p)->dk)

/* ------------------------------------------------------------------ prologue */

/* x_hat = s * x / sqrt(|x|^2 + eps) (or s * x without the norm). */
static void normalise_row(const oracle_problem* p, const double* x, double s, double* out) {
  double r = 1.0;
  if (p->l2norm) {
    double ss = 0.0;
    for (int64_t i = 0; i < p->dk; ++i) ss += x[i] * x[i];
    r = 1.0 / sqrt(ss + p->eps);
  }
  for (int64_t i = 0; i < p->dk; ++i) out[i] = x[i] * r * s;
}

/* Gate and write strength of every token; padded tokens get g = 0, beta = 0. */
int oracle_prologue(const oracle_problem* p, const double* q, const double* k, const double* a,
                    const double* b, const double* A_log, const double* dt_bias,
                    const int32_t* valid_len, double* qh, double* kh, double* g, double* beta) {
  int rc = check_problem(p);
  if (rc) return rc;
  if ((rc = check_valid_len(p, valid_len))) return rc;
  for (int64_t bb = 0; bb < p->B; ++bb) {
    int64_t L = valid_length(p, valid_len, bb);
    for (int64_t t = 0; t < p->T; ++t) {
      for (int64_t hq = 0; hq < p->Hqk; ++hq) {
        if (qh) normalise_row(p, q + QK_IDX(p, bb, t, hq), p->scale, qh + QK_IDX(p, bb, t, hq));
        if (kh) normalise_row(p, k + QK_IDX(p, bb, t, hq), 1.0, kh + QK_IDX(p, bb, t, hq));
      }
      for (int64_t h = 0; h < p->H; ++h) {
        int64_t gi = G_IDX(p, bb, t, h);
        if (t < L) {
          g[gi] = -exp(A_log[h]) * softplus(a[gi] + dt_bias[h]);
          beta[gi] = sigmoid(b[gi]);
        } else {
          g[gi] = 0.0;
          beta[gi] = 0.0;
        }
      }
    }
  }
  return 0;
}

/* -------------------------------------------------------------- recurrence */

/* One token: S <- alpha (S - beta k (k^T S)) + beta k v^T.  kS is scratch [dv]. */
static void token_step(int64_t dk, int64_t dv, double* S, const double* kt, const double* vt,
                       double alpha, double beta, double* kS) {
  for (int64_t j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int64_t i = 0; i < dk; ++i) acc += kt[i] * S[i * dv + j];
    kS[j] = acc;
  }
  for (int64_t i = 0; i < dk; ++i)
    for (int64_t j = 0; j < dv; ++j)
      S[i * dv + j] = alpha * (S[i * dv + j] - beta * kt[i] * kS[j]) + beta * kt[i] * vt[j];
}

/* Core forward over prepared q_hat, k_hat, g, beta. */
int oracle_core_fwd(const oracle_problem* p, const double* qh, const double* kh, const double* v,
                    const double* g, const double* beta, const double* h0,
                    const int32_t* valid_len, double* o, double* hT, int nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  if ((rc = check_valid_len(p, valid_len))) return rc;
  const int64_t r = p->H / p->Hqk, dk = p->dk, dv = p->dv;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < p->B * p->H; ++bh) {
    const int64_t bb = bh / p->H, h = bh % p->H, hq = h / r;
    const int64_t L = valid_length(p, valid_len, bb);
    double* S = (double*)malloc(sizeof(double) * (size_t)(dk * dv));
    double* kS = (double*)malloc(sizeof(double) * (size_t)dv);
    if (h0) memcpy(S, h0 + ST_IDX(p, bb, h), sizeof(double) * (size_t)(dk * dv));
    else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
    for (int64_t t = 0; t < p->T; ++t) {
      double* ot = o ? o + V_IDX(p, bb, t, h) : NULL;
      if (t >= L) {
        if (ot) for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
        continue;
      }
      const int64_t gi = G_IDX(p, bb, t, h);
      token_step(dk, dv, S, kh + QK_IDX(p, bb, t, hq), v + V_IDX(p, bb, t, h), exp(g[gi]),
                 beta[gi], kS);
      if (ot) {
        const double* qt = qh + QK_IDX(p, bb, t, hq);
        for (int64_t j = 0; j < dv; ++j) {
          double acc = 0.0;
          for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * qt[i];
          ot[j] = acc;
        }
      }
    }
    if (hT) memcpy(hT + ST_IDX(p, bb, h), S, sizeof(double) * (size_t)(dk * dv));
    free(S);
    free(kS);
  }
  return 0;
}

/*
 * Core backward: BPTT of L = sum_t <dO_t, o_t> + <dH_T, S_T>.
 * States are checkpointed every 64 tokens and recomputed per block in reverse.
 * dqh and dkh are accumulated at Q/K-head granularity (sum over the r V heads).
 * With S_t = alpha S_{t-1} + beta k r^T, r = v - alpha S_{t-1}^T k:
 *   dv     = beta dS^T k
 *   dbeta  = k^T dS r
 *   dalpha = <dS, S_{t-1}> - beta (dS^T k).(S_{t-1}^T k),  dg = alpha dalpha
 *   dk    += beta dS r - alpha beta S_{t-1} (dS^T k)
 *   dS    <- alpha (dS - beta k (k^T dS))
 * and the output term adds q dO^T to dS and S_t dO to dq first.
 */
int oracle_core_bwd(const oracle_problem* p, const double* qh, const double* kh, const double* v,
                    const double* g, const double* beta, const double* h0,
                    const int32_t* valid_len, const double* dO, const double* dHT, double* dqh,
                    double* dkh, double* dv_out, double* dg, double* dbeta, double* dH0,
                    int nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  if ((rc = check_valid_len(p, valid_len))) return rc;
  const int64_t r = p->H / p->Hqk, dk = p->dk, dv = p->dv, T = p->T;
  const int64_t CK = 64;
  const int64_t nblk = (T + CK - 1) / CK;
  memset(dqh, 0, sizeof(double) * (size_t)(p->B * T * p->Hqk * dk));
  memset(dkh, 0, sizeof(double) * (size_t)(p->B * T * p->Hqk * dk));
  set_threads(nthreads);
  /* parallel over (b, Q/K head): the r V heads of a group write the same dq/dk rows */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bq = 0; bq < p->B * p->Hqk; ++bq) {
    const int64_t bb = bq / p->Hqk, hq = bq % p->Hqk;
    const int64_t L = valid_length(p, valid_len, bb);
    const size_t SS = (size_t)(dk * dv);
    double* ck = (double*)malloc(sizeof(double) * SS * (size_t)(nblk > 0 ? nblk : 1));
    double* blk = (double*)malloc(sizeof(double) * SS * (size_t)(CK + 1));
    double* dS = (double*)malloc(sizeof(double) * SS);
    double* kS = (double*)malloc(sizeof(double) * (size_t)dv);
    double* dSk = (double*)malloc(sizeof(double) * (size_t)dv);
    double* rr = (double*)malloc(sizeof(double) * (size_t)dv);
    double* kdS = (double*)malloc(sizeof(double) * (size_t)dv);
    for (int64_t h = hq * r; h < (hq + 1) * r; ++h) {
      /* forward with checkpoints */
      double* S = blk; /* reuse slot 0 as the running state */
      if (h0) memcpy(S, h0 + ST_IDX(p, bb, h), sizeof(double) * SS);
      else memset(S, 0, sizeof(double) * SS);
      for (int64_t c = 0; c < nblk; ++c) {
        memcpy(ck + (size_t)c * SS, S, sizeof(double) * SS);
        for (int64_t t = c * CK; t < T && t < (c + 1) * CK; ++t) {
          if (t >= L) continue;
          const int64_t gi = G_IDX(p, bb, t, h);
          token_step(dk, dv, S, kh + QK_IDX(p, bb, t, hq), v + V_IDX(p, bb, t, h), exp(g[gi]),
                     beta[gi], kS);
        }
      }
      if (dHT) memcpy(dS, dHT + ST_IDX(p, bb, h), sizeof(double) * SS);
      else memset(dS, 0, sizeof(double) * SS);
      for (int64_t c = nblk - 1; c >= 0; --c) {
        const int64_t t0 = c * CK, t1 = (c + 1) * CK < T ? (c + 1) * CK : T;
        /* blk[i] = state before token t0+i; blk[i+1] = state after it */
        memcpy(blk, ck + (size_t)c * SS, sizeof(double) * SS);
        for (int64_t t = t0; t < t1; ++t) {
          double* Sn = blk + (size_t)(t - t0 + 1) * SS;
          memcpy(Sn, blk + (size_t)(t - t0) * SS, sizeof(double) * SS);
          if (t >= L) continue;
          const int64_t gi = G_IDX(p, bb, t, h);
          token_step(dk, dv, Sn, kh + QK_IDX(p, bb, t, hq), v + V_IDX(p, bb, t, h), exp(g[gi]),
                     beta[gi], kS);
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
          const int64_t gi = G_IDX(p, bb, t, h);
          const double* Sp = blk + (size_t)(t - t0) * SS;
          const double* Sc = blk + (size_t)(t - t0 + 1) * SS;
          if (t >= L) {
            for (int64_t j = 0; j < dv; ++j) dv_out[V_IDX(p, bb, t, h) + j] = 0.0;
            dg[gi] = 0.0;
            dbeta[gi] = 0.0;
            continue;
          }
          const double al = exp(g[gi]), be = beta[gi];
          const double* kt = kh + QK_IDX(p, bb, t, hq);
          const double* qt = qh + QK_IDX(p, bb, t, hq);
          const double* vt = v + V_IDX(p, bb, t, h);
          const double* dOt = dO ? dO + V_IDX(p, bb, t, h) : NULL;
          double* dqt = dqh + QK_IDX(p, bb, t, hq);
          double* dkt = dkh + QK_IDX(p, bb, t, hq);
          /* output term: o_t = S_t^T q_t */
          if (dOt) {
            for (int64_t i = 0; i < dk; ++i) {
              double acc = 0.0;
              for (int64_t j = 0; j < dv; ++j) {
                dS[i * dv + j] += qt[i] * dOt[j];
                acc += Sc[i * dv + j] * dOt[j];
              }
              dqt[i] += acc;
            }
          }
          /* kS = S_{t-1}^T k, r = v - alpha kS, dSk = dS^T k */
          for (int64_t j = 0; j < dv; ++j) {
            double a1 = 0.0, a2 = 0.0;
            for (int64_t i = 0; i < dk; ++i) {
              a1 += kt[i] * Sp[i * dv + j];
              a2 += kt[i] * dS[i * dv + j];
            }
            kS[j] = a1;
            dSk[j] = a2;
            rr[j] = vt[j] - al * a1;
          }
          double dbe = 0.0, dal = 0.0, kSdSk = 0.0;
          for (int64_t j = 0; j < dv; ++j) {
            dv_out[V_IDX(p, bb, t, h) + j] = be * dSk[j];
            kSdSk += dSk[j] * kS[j];
          }
          for (int64_t i = 0; i < dk; ++i) {
            double dSr = 0.0, SpdSk = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
              dSr += dS[i * dv + j] * rr[j];
              SpdSk += Sp[i * dv + j] * dSk[j];
              dal += dS[i * dv + j] * Sp[i * dv + j];
            }
            dbe += kt[i] * dSr;
            dkt[i] += be * dSr - al * be * SpdSk;
          }
          dal -= be * kSdSk;
          dbeta[gi] = dbe;
          dg[gi] = al * dal;
          /* dS <- alpha (dS - beta k (k^T dS)) */
          for (int64_t j = 0; j < dv; ++j) kdS[j] = dSk[j];
          for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j)
              dS[i * dv + j] = al * (dS[i * dv + j] - be * kt[i] * kdS[j]);
        }
      }
      if (dH0) memcpy(dH0 + ST_IDX(p, bb, h), dS, sizeof(double) * SS);
    }
    free(ck);
    free(blk);
    free(dS);
    free(kS);
    free(dSk);
    free(rr);
    free(kdS);
  }
  return 0;
}

/* ------------------------------------------------------- full forward/backward */

static size_t qk_count(const oracle_problem* p) { return (size_t)(p->B * p->T * p->Hqk * p->dk); }
static size_t gate_count(const oracle_problem* p) { return (size_t)(p->B * p->T * p->H); }

/* Forward from the raw inputs: prologue, then the recurrence. */
int oracle_fwd(const oracle_problem* p, const double* q, const double* k, const double* v,
               const double* a, const double* b, const double* A_log, const double* dt_bias,
               const double* h0, const int32_t* valid_len, double* o, double* hT, int nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  double* qh = (double*)malloc(sizeof(double) * (qk_count(p) + 1));
  double* kh = (double*)malloc(sizeof(double) * (qk_count(p) + 1));
  double* g = (double*)malloc(sizeof(double) * (gate_count(p) + 1));
  double* be = (double*)malloc(sizeof(double) * (gate_count(p) + 1));
  rc = oracle_prologue(p, q, k, a, b, A_log, dt_bias, valid_len, qh, kh, g, be);
  if (!rc) rc = oracle_core_fwd(p, qh, kh, v, g, be, h0, valid_len, o, hT, nthreads);
  free(qh);
  free(kh);
  free(g);
  free(be);
  return rc;
}

/* d/dx of x_hat = s x / sqrt(|x|^2 + eps):  dx = s (dxh - u (u . dxh)) / n, u = x / n. */
static void normalise_row_bwd(const oracle_problem* p, const double* x, double s,
                              const double* dxh, double* dx) {
  if (!p->l2norm) {
    for (int64_t i = 0; i < p->dk; ++i) dx[i] = s * dxh[i];
    return;
  }
  double ss = 0.0;
  for (int64_t i = 0; i < p->dk; ++i) ss += x[i] * x[i];
  const double n = sqrt(ss + p->eps);
  double ud = 0.0;
  for (int64_t i = 0; i < p->dk; ++i) ud += (x[i] / n) * dxh[i];
  for (int64_t i = 0; i < p->dk; ++i) dx[i] = s * (dxh[i] - (x[i] / n) * ud) / n;
}

/* Backward from the raw inputs: gradients w.r.t. raw q, k (Q/K heads), v, g, beta, h0. */
int oracle_bwd(const oracle_problem* p, const double* q, const double* k, const double* v,
               const double* a, const double* b, const double* A_log, const double* dt_bias,
               const double* h0, const int32_t* valid_len, const double* dO, const double* dHT,
               double* dq, double* dk, double* dv, double* dg, double* dbeta, double* dH0,
               int nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  const size_t nqk = qk_count(p), ng = gate_count(p);
  double* qh = (double*)malloc(sizeof(double) * (nqk + 1));
  double* kh = (double*)malloc(sizeof(double) * (nqk + 1));
  double* g = (double*)malloc(sizeof(double) * (ng + 1));
  double* be = (double*)malloc(sizeof(double) * (ng + 1));
  double* dqh = (double*)malloc(sizeof(double) * (nqk + 1));
  double* dkh = (double*)malloc(sizeof(double) * (nqk + 1));
  rc = oracle_prologue(p, q, k, a, b, A_log, dt_bias, valid_len, qh, kh, g, be);
  if (!rc)
    rc = oracle_core_bwd(p, qh, kh, v, g, be, h0, valid_len, dO, dHT, dqh, dkh, dv, dg, dbeta,
                         dH0, nthreads);
  if (!rc) {
    for (int64_t bb = 0; bb < p->B; ++bb)
      for (int64_t t = 0; t < p->T; ++t)
        for (int64_t hq = 0; hq < p->Hqk; ++hq) {
          const int64_t off = QK_IDX(p, bb, t, hq);
          normalise_row_bwd(p, q + off, p->scale, dqh + off, dq + off);
          normalise_row_bwd(p, k + off, 1.0, dkh + off, dk + off);
        }
  }
  free(qh);
  free(kh);
  free(g);
  free(be);
  free(dqh);
  free(dkh);
  return rc;
}

/* ---------------------------------------------------------- segment summaries */

/*
 * Summary (M, S) of the whole [0, T) of each (b, h):
 *   M <- A_t M with A_t = alpha_t (I - beta_t k_t k_t^T), i.e. M = A_T ... A_1,
 *   S <- A_t S + beta_t k_t v_t^T from S = 0.
 * A_t M is applied as alpha (M - beta k (k^T M)), the same product without
 * forming A_t.
 */
int oracle_summary(const oracle_problem* p, const double* k, const double* v, const double* a,
                   const double* b, const double* A_log, const double* dt_bias,
                   const int32_t* valid_len, double* M, double* S, int nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  const size_t nqk = qk_count(p), ng = gate_count(p);
  double* kh = (double*)malloc(sizeof(double) * (nqk + 1));
  double* g = (double*)malloc(sizeof(double) * (ng + 1));
  double* be = (double*)malloc(sizeof(double) * (ng + 1));
  oracle_problem pk = *p;
  rc = oracle_prologue(&pk, k, k, a, b, A_log, dt_bias, valid_len, NULL, kh, g, be);
  if (rc) goto done;
  {
    const int64_t r = p->H / p->Hqk, dk = p->dk, dv = p->dv;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < p->B * p->H; ++bh) {
      const int64_t bb = bh / p->H, h = bh % p->H, hq = h / r;
      double* Mh = M + M_IDX(p, bb, h);
      double* Sh = S + ST_IDX(p, bb, h);
      double* kM = (double*)malloc(sizeof(double) * (size_t)(dk > dv ? dk : dv));
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dk; ++j) Mh[i * dk + j] = (i == j) ? 1.0 : 0.0;
      memset(Sh, 0, sizeof(double) * (size_t)(dk * dv));
      for (int64_t t = 0; t < p->T; ++t) {
        const int64_t gi = G_IDX(p, bb, t, h);
        const double al = exp(g[gi]), bt = be[gi];
        const double* kt = kh + QK_IDX(p, bb, t, hq);
        /* padded tokens have g = 0, beta = 0: A_t = I, no write */
        for (int64_t j = 0; j < dk; ++j) {
          double acc = 0.0;
          for (int64_t i = 0; i < dk; ++i) acc += kt[i] * Mh[i * dk + j];
          kM[j] = acc;
        }
        for (int64_t i = 0; i < dk; ++i)
          for (int64_t j = 0; j < dk; ++j)
            Mh[i * dk + j] = al * (Mh[i * dk + j] - bt * kt[i] * kM[j]);
        token_step(dk, dv, Sh, kt, v + V_IDX(p, bb, t, h), al, bt, kM);
      }
      free(kM);
    }
  }
done:
  free(kh);
  free(g);
  free(be);
  return rc;
}

/*
 * Gradient summary D = d/dH_in sum_t <dO_t, o_t> of the run of [0, T) started
 * from H_in (it does not depend on H_in or v):  dS = 0; for t = T-1 .. 0:
 * dS += q_t dO_t^T;  dS <- A_t^T dS  (A_t is symmetric).  D = dS.
 */
int oracle_summary_bwd(const oracle_problem* p, const double* q, const double* k,
                       const double* a, const double* b, const double* A_log,
                       const double* dt_bias, const int32_t* valid_len, const double* dO,
                       double* D, int nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  const size_t nqk = qk_count(p), ng = gate_count(p);
  double* qh = (double*)malloc(sizeof(double) * (nqk + 1));
  double* kh = (double*)malloc(sizeof(double) * (nqk + 1));
  double* g = (double*)malloc(sizeof(double) * (ng + 1));
  double* be = (double*)malloc(sizeof(double) * (ng + 1));
  rc = oracle_prologue(p, q, k, a, b, A_log, dt_bias, valid_len, qh, kh, g, be);
  if (rc) goto done;
  {
    const int64_t r = p->H / p->Hqk, dk = p->dk, dv = p->dv;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < p->B * p->H; ++bh) {
      const int64_t bb = bh / p->H, h = bh % p->H, hq = h / r;
      const int64_t L = valid_length(p, valid_len, bb);
      double* dS = D + ST_IDX(p, bb, h);
      double* kd = (double*)malloc(sizeof(double) * (size_t)dv);
      memset(dS, 0, sizeof(double) * (size_t)(dk * dv));
      for (int64_t t = p->T - 1; t >= 0; --t) {
        if (t >= L) continue;
        const int64_t gi = G_IDX(p, bb, t, h);
        const double al = exp(g[gi]), bt = be[gi];
        const double* kt = kh + QK_IDX(p, bb, t, hq);
        const double* qt = qh + QK_IDX(p, bb, t, hq);
        const double* dOt = dO + V_IDX(p, bb, t, h);
        for (int64_t i = 0; i < dk; ++i)
          for (int64_t j = 0; j < dv; ++j) dS[i * dv + j] += qt[i] * dOt[j];
        for (int64_t j = 0; j < dv; ++j) {
          double acc = 0.0;
          for (int64_t i = 0; i < dk; ++i) acc += kt[i] * dS[i * dv + j];
          kd[j] = acc;
        }
        for (int64_t i = 0; i < dk; ++i)
          for (int64_t j = 0; j < dv; ++j) dS[i * dv + j] = al * (dS[i * dv + j] - bt * kt[i] * kd[j]);
      }
      free(kd);
    }
  }
done:
  free(qh);
  free(kh);
  free(g);
  free(be);
  return rc;
}

/* (M, S) = (M2 M1, M2 S1 + S2) for n independent pairs. */
int oracle_compose(int64_t n, int64_t dk, int64_t dv, const double* M2, const double* S2,
                   const double* M1, const double* S1, double* M, double* S) {
  if (n < 0 || dk <= 0 || dv <= 0) return -2;
  for (int64_t e = 0; e < n; ++e) {
    const double* m2 = M2 + e * dk * dk;
    const double* m1 = M1 + e * dk * dk;
    const double* s1 = S1 + e * dk * dv;
    const double* s2 = S2 + e * dk * dv;
    double* m = M + e * dk * dk;
    double* s = S + e * dk * dv;
    for (int64_t i = 0; i < dk; ++i) {
      for (int64_t j = 0; j < dk; ++j) {
        double acc = 0.0;
        for (int64_t l = 0; l < dk; ++l) acc += m2[i * dk + l] * m1[l * dk + j];
        m[i * dk + j] = acc;
      }
      for (int64_t j = 0; j < dv; ++j) {
        double acc = s2[i * dv + j];
        for (int64_t l = 0; l < dk; ++l) acc += m2[i * dk + l] * s1[l * dv + j];
        s[i * dv + j] = acc;
      }
    }
  }
  return 0;
}

/*
 * Exclusive prefix over P segments, n = B*H maps each:
 *   H_in[0] = h0 (or 0),  H_in[i] = M[i-1] H_in[i-1] + S[i-1];
 *   H_out (optional) = M[P-1] H_in[P-1] + S[P-1].
 * M [P,n,dk,dk], S/H_in [P,n,dk,dv], h0/H_out [n,dk,dv].
 */
int oracle_prefix(int64_t n, int64_t P, int64_t dk, int64_t dv, const double* M, const double* S,
                  const double* h0, double* Hin, double* Hout) {
  if (n < 0 || P <= 0 || dk <= 0 || dv <= 0) return -2;
  const int64_t MS = dk * dk, SS = dk * dv;
  for (int64_t e = 0; e < n; ++e) {
    double* cur = (double*)malloc(sizeof(double) * (size_t)SS);
    double* nxt = (double*)malloc(sizeof(double) * (size_t)SS);
    if (h0) memcpy(cur, h0 + e * SS, sizeof(double) * (size_t)SS);
    else memset(cur, 0, sizeof(double) * (size_t)SS);
    for (int64_t s = 0; s < P; ++s) {
      memcpy(Hin + (s * n + e) * SS, cur, sizeof(double) * (size_t)SS);
      const double* m = M + (s * n + e) * MS;
      const double* sv = S + (s * n + e) * SS;
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j) {
          double acc = sv[i * dv + j];
          for (int64_t l = 0; l < dk; ++l) acc += m[i * dk + l] * cur[l * dv + j];
          nxt[i * dv + j] = acc;
        }
      memcpy(cur, nxt, sizeof(double) * (size_t)SS);
    }
    if (Hout) memcpy(Hout + e * SS, cur, sizeof(double) * (size_t)SS);
    free(cur);
    free(nxt);
  }
  return 0;
}

/*
 * Reverse exclusive prefix of state gradients:
 *   dH_out[P-1] = dHT (or 0),  dH_out[i] = M[i+1]^T dH_out[i+1] + D[i+1];
 *   dH0 (optional) = M[0]^T dH_out[0] + D[0].
 */
int oracle_prefix_bwd(int64_t n, int64_t P, int64_t dk, int64_t dv, const double* M,
                      const double* D, const double* dHT, double* dHout, double* dH0) {
  if (n < 0 || P <= 0 || dk <= 0 || dv <= 0) return -2;
  const int64_t MS = dk * dk, SS = dk * dv;
  for (int64_t e = 0; e < n; ++e) {
    double* cur = (double*)malloc(sizeof(double) * (size_t)SS);
    double* nxt = (double*)malloc(sizeof(double) * (size_t)SS);
    if (dHT) memcpy(cur, dHT + e * SS, sizeof(double) * (size_t)SS);
    else memset(cur, 0, sizeof(double) * (size_t)SS);
    for (int64_t s = P - 1; s >= 0; --s) {
      memcpy(dHout + (s * n + e) * SS, cur, sizeof(double) * (size_t)SS);
      const double* m = M + (s * n + e) * MS;
      const double* d = D + (s * n + e) * SS;
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j) {
          double acc = d[i * dv + j];
          for (int64_t l = 0; l < dk; ++l) acc += m[l * dk + i] * cur[l * dv + j];
          nxt[i * dv + j] = acc;
        }
      memcpy(cur, nxt, sizeof(double) * (size_t)SS);
    }
    if (dH0) memcpy(dH0 + e * SS, cur, sizeof(double) * (size_t)SS);
    free(cur);
    free(nxt);
  }
  return 0;
}

/* ------------------------------------------------- gate parameter gradients */

/* Chain of dg, dbeta [B,T,H] to the gate parameters, from the prologue's
 * definitions g = -exp(A_log[h]) softplus(a + dt_bias[h]), beta = sigmoid(b)
 * (softplus' = sigmoid):
 *   da_t       = dg_t * (-exp(A_log[h])) * sigmoid(a_t + dt_bias[h])
 *   db_t       = dbeta_t * beta_t (1 - beta_t)
 *   ddt_bias_h = sum_{b,t} da_t            dA_log_h = sum_{b,t} dg_t * g_t
 * Padded tokens (t >= valid_len[b]) have g and beta fixed at 0, independent of
 * a, b and the parameters: their da, db are 0 and they add nothing to the sums.
 * Softplus is x for x > 20 in the forward; its derivative there is taken as 1. */
int oracle_gate_param_bwd(const oracle_problem* p, const double* a, const double* b,
                          const double* A_log, const double* dt_bias, const int32_t* valid_len,
                          const double* dg, const double* dbeta, double* da, double* db,
                          double* dA_log, double* ddt_bias) {
  int rc = check_problem(p);
  if (rc) return rc;
  if ((rc = check_valid_len(p, valid_len))) return rc;
  for (int64_t h = 0; h < p->H; ++h) {
    dA_log[h] = 0.0;
    ddt_bias[h] = 0.0;
  }
  for (int64_t bb = 0; bb < p->B; ++bb) {
    const int64_t L = valid_length(p, valid_len, bb);
    for (int64_t t = 0; t < p->T; ++t) {
      for (int64_t h = 0; h < p->H; ++h) {
        const int64_t gi = G_IDX(p, bb, t, h);
        if (t >= L) {
          da[gi] = 0.0;
          db[gi] = 0.0;
          continue;
        }
        const double x = a[gi] + dt_bias[h];
        const double dsp = x > 20.0 ? 1.0 : sigmoid(x);
        const double g = -exp(A_log[h]) * softplus(x);
        const double be = sigmoid(b[gi]);
        da[gi] = dg[gi] * (-exp(A_log[h])) * dsp;
        db[gi] = dbeta[gi] * be * (1.0 - be);
        ddt_bias[h] += da[gi];
        dA_log[h] += dg[gi] * g;
      }
    }
  }
  return 0;
}

int oracle_abi_version(void) { return 1; }
