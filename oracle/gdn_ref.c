/*
 * Oracle: token-by-token fp64 gated delta rule (TEST INFRASTRUCTURE ONLY).
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
 * reference legs may load this file's library. The CUDA path never links,
 * includes or calls it, and it shares no code with the CUDA path.
 *
 * What it computes, per sequence n and value head hv (key head h = hv / HG,
 * HG = Hv / H, the grouping of "Optimizing GDN Chunk Prefill on Intel AMX
 * CPU", section 4):
 *
 *   S (dk x dv, one row per key dimension, fp64) = initial_state[n,hv]^T or 0
 *   for each token t of sequence n:
 *       alpha = exp(g[t,hv])                              decay
 *       pred  = alpha * S^T k_t                           what S predicts for k_t
 *       S     = alpha * S + beta[t,hv] * k_t (v_t - pred)^T   write the correction
 *       o_t   = scale * S^T q_t                           read with the updated S
 *   final_state[n,hv] = S^T
 *
 * With per-channel gates (g_per_channel != 0; g is then [T, Hv, dk]) the
 * decay is a diagonal matrix over the key dimension, one factor per row of S:
 *       pred  = (diag(alpha_t) S)^T k_t
 *       S     = diag(alpha_t) S + beta[t,hv] * k_t (v_t - pred)^T
 * which is the scalar case when all dk factors are equal. This is the reading
 * of the per-channel ("KDA") gate the graph-capture RFC for the GDN/KDA chunk
 * paths lists beside GDN (section "What needs to change", the KDA forward
 * kernels): the same delta-rule write, with a gate per key channel.
 *
 * This is the per-token update described in "Chunking Qwen3.5's gated
 * DeltaNet for 1.5x faster prefill on Apple Silicon" (section "What is the
 * gated delta rule in Qwen3.5?": decay, correction from the state's
 * prediction for the key, write-back, read), with the state held as
 * [dv, dk] at the boundary exactly as the AMX note's section 9 describes
 * ("CPU / Triton-facing state: [N, Hv, V, K]"); the transpose here is the
 * same layout bridge its tests use.
 *
 * Optional q/k L2 normalisation (AMX note, section 7): x / sqrt(sum x^2 + eps),
 * done in fp64 before the recurrence. scale <= 0 or NaN means 1/sqrt(dk).
 * cu_seqlens == NULL means one sequence covering all T rows. Rows outside
 * [cu_seqlens[0], cu_seqlens[N]) are left untouched in out.
 *
 * Plain C11, no SIMD intrinsics, no fast-math. OpenMP is used only across
 * independent (sequence, value head) lanes; each lane's arithmetic is serial
 * and in a fixed order, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GDN_REF_OK 0
#define GDN_REF_BAD_ARG (-1)
#define GDN_REF_NO_MEMORY (-2)

static void l2_normalise(const double* x, double* y, int64_t d, double eps) {
  double ss = 0.0;
  for (int64_t i = 0; i < d; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss + eps);
  for (int64_t i = 0; i < d; ++i) y[i] = x[i] * r;
}

/* One (sequence, value-head) lane. S is dk x dv, row-major (S[i*dv + j]). */
static void run_lane(int64_t t0, int64_t t1, int64_t H, int64_t Hv, int64_t dk,
                     int64_t dv, int64_t h, int64_t hv, const double* q,
                     const double* k, const double* v, const double* g,
                     const double* beta, double scale, int qk_l2norm,
                     double eps, int g_per_channel, double* S, double* pred,
                     double* kt, double* qt, double* out) {
  for (int64_t t = t0; t < t1; ++t) {
    const double* kraw = k + (t * H + h) * dk;
    const double* qraw = q + (t * H + h) * dk;
    if (qk_l2norm) {
      l2_normalise(kraw, kt, dk, eps);
      l2_normalise(qraw, qt, dk, eps);
    } else {
      memcpy(kt, kraw, (size_t)dk * sizeof(double));
      memcpy(qt, qraw, (size_t)dk * sizeof(double));
    }
    /* per-channel gates: alpha is folded into each row below and is 1 here */
    const double* gk = g_per_channel ? g + (t * Hv + hv) * dk : NULL;
    const double alpha = gk ? 1.0 : exp(g[t * Hv + hv]);
    const double b = beta[t * Hv + hv];
    const double* vt = v + (t * Hv + hv) * dv;

    /* pred = alpha * S^T k, or (diag(alpha_i) S)^T k with per-channel gates */
    for (int64_t j = 0; j < dv; ++j) pred[j] = 0.0;
    for (int64_t i = 0; i < dk; ++i) {
      const double ki = gk ? exp(gk[i]) * kt[i] : kt[i];
      const double* Si = S + i * dv;
      for (int64_t j = 0; j < dv; ++j) pred[j] += Si[j] * ki;
    }
    for (int64_t j = 0; j < dv; ++j) pred[j] *= alpha;

    /* S = alpha * S + beta * k (v - pred)^T, alpha per row with per-channel gates */
    for (int64_t i = 0; i < dk; ++i) {
      const double bki = b * kt[i];
      const double ai = gk ? exp(gk[i]) : alpha;
      double* Si = S + i * dv;
      for (int64_t j = 0; j < dv; ++j) Si[j] = ai * Si[j] + bki * (vt[j] - pred[j]);
    }

    /* o = scale * S^T q (after the update) */
    double* ot = out + (t * Hv + hv) * dv;
    for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
    for (int64_t i = 0; i < dk; ++i) {
      const double qi = qt[i];
      const double* Si = S + i * dv;
      for (int64_t j = 0; j < dv; ++j) ot[j] += Si[j] * qi;
    }
    for (int64_t j = 0; j < dv; ++j) ot[j] *= scale;
  }
}

int gdn_ref_forward(int64_t T, int64_t N, int64_t H, int64_t Hv, int64_t dk,
                    int64_t dv, const double* q, const double* k,
                    const double* v, const double* g, const double* beta,
                    double scale, const double* initial_state,
                    const int64_t* cu_seqlens, int qk_l2norm, double eps,
                    double* out, double* final_state, int nthreads, int g_per_channel) {
  if (T < 0 || N < 1 || H < 1 || Hv < 1 || dk < 1 || dv < 1) return GDN_REF_BAD_ARG;
  if (Hv % H != 0) return GDN_REF_BAD_ARG;
  if (!q || !k || !v || !g || !beta || !out) return GDN_REF_BAD_ARG;
  if (!cu_seqlens && N != 1) return GDN_REF_BAD_ARG;
  if (cu_seqlens) {
    for (int64_t n = 0; n < N; ++n)
      if (cu_seqlens[n] < 0 || cu_seqlens[n + 1] < cu_seqlens[n] || cu_seqlens[n + 1] > T)
        return GDN_REF_BAD_ARG;
  }
  if (!(scale > 0.0)) scale = 1.0 / sqrt((double)dk); /* also catches NaN */
  const int64_t HG = Hv / H;
  const int64_t lanes = N * Hv;
  int rc = GDN_REF_OK;

#ifdef _OPENMP
  if (nthreads < 1) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double* S = (double*)malloc((size_t)(dk * dv) * sizeof(double));
    double* pred = (double*)malloc((size_t)dv * sizeof(double));
    double* kt = (double*)malloc((size_t)dk * sizeof(double));
    double* qt = (double*)malloc((size_t)dk * sizeof(double));
    int ok = S && pred && kt && qt;
    if (!ok) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      rc = GDN_REF_NO_MEMORY;
    }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t lane = 0; lane < lanes; ++lane) {
      if (!ok) continue;
      const int64_t n = lane / Hv, hv = lane % Hv, h = hv / HG;
      const int64_t t0 = cu_seqlens ? cu_seqlens[n] : 0;
      const int64_t t1 = cu_seqlens ? cu_seqlens[n + 1] : T;
      /* boundary layout [dv, dk] -> working layout [dk, dv] */
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j)
          S[i * dv + j] = initial_state ? initial_state[((n * Hv + hv) * dv + j) * dk + i] : 0.0;
      run_lane(t0, t1, H, Hv, dk, dv, h, hv, q, k, v, g, beta, scale, qk_l2norm, eps,
               g_per_channel, S, pred, kt, qt, out);
      if (final_state)
        for (int64_t i = 0; i < dk; ++i)
          for (int64_t j = 0; j < dv; ++j)
            final_state[((n * Hv + hv) * dv + j) * dk + i] = S[i * dv + j];
    }
    free(S);
    free(pred);
    free(kt);
    free(qt);
  }
  return rc;
}

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int gdn_ref_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Backward of the token recurrence above (scalar gates): the exact adjoint of
 * each step, applied from the last token to the first. Given d_out [T,Hv,dv]
 * (the gradient of a loss with respect to out) and d_final [N,Hv,dv,dk] (with
 * respect to final_state, NULL for none), it writes the gradients with respect
 * to every input: dq, dk [T,H,dk] (summed over the value heads that share a key
 * head), dv [T,Hv,dv], dg, dbeta [T,Hv] and d_initial [N,Hv,dv,dk] (NULL: not
 * written). q/k L2 normalisation is not part of this function.
 *
 * One forward step, with alpha = exp(g_t), b = beta_t:
 *     D = alpha S_prev;  pred = D^T k;  delta = v - pred;
 *     S = D + b k delta^T;  o = scale S^T q
 * and its adjoint, with dS the gradient flowing into S:
 *     dS += scale q do^T;            dq  = scale S do
 *     dD  = dS;  db = k^T dS delta;  dk  = b dS delta;  ddelta = b dS^T k
 *     dv  = ddelta;  dpred = -ddelta
 *     dD += k dpred^T;               dk += D dpred
 *     dS_prev = alpha dD;            dg  = alpha <S_prev, dD>
 * The states the adjoint needs are recomputed: S is stored every 64 tokens on
 * the way forward and each 64-token segment is replayed before its adjoint.
 */
static void lane_backward(int64_t t0, int64_t t1, int64_t H, int64_t Hv, int64_t dk,
                          int64_t dv, int64_t h, int64_t hv, const double* q,
                          const double* k, const double* v, const double* g,
                          const double* beta, double scale, const double* dout,
                          double* S, double* ckpt, double* seg, double* dS, double* dD,
                          double* tmp_v, double* tmp_k, double* dq, double* dk_out,
                          double* dv_out, double* dg, double* dbeta) {
  const int64_t n = t1 - t0, KV = dk * dv;
  const int64_t nseg = (n + 63) / 64;
  /* forward, keeping the state at the start of each 64-token segment */
  for (int64_t s = 0; s < nseg; ++s) {
    memcpy(ckpt + s * KV, S, (size_t)KV * sizeof(double));
    const int64_t a = t0 + 64 * s, e = a + 64 < t1 ? a + 64 : t1;
    for (int64_t t = a; t < e; ++t) {
      const double alpha = exp(g[t * Hv + hv]), b = beta[t * Hv + hv];
      const double* kt = k + (t * H + h) * dk;
      const double* vt = v + (t * Hv + hv) * dv;
      for (int64_t j = 0; j < dv; ++j) tmp_v[j] = 0.0;
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j) tmp_v[j] += alpha * S[i * dv + j] * kt[i];
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j)
          S[i * dv + j] = alpha * S[i * dv + j] + b * kt[i] * (vt[j] - tmp_v[j]);
    }
  }
  /* adjoint, segment by segment from the end; dS holds the incoming gradient */
  for (int64_t s = nseg - 1; s >= 0; --s) {
    const int64_t a = t0 + 64 * s, e = a + 64 < t1 ? a + 64 : t1;
    /* replay: seg[m] = state after token a + m - 1 (seg[0] = segment start) */
    memcpy(seg, ckpt + s * KV, (size_t)KV * sizeof(double));
    for (int64_t t = a; t < e; ++t) {
      const double* Sp = seg + (t - a) * KV;
      double* Sn = seg + (t - a + 1) * KV;
      const double alpha = exp(g[t * Hv + hv]), b = beta[t * Hv + hv];
      const double* kt = k + (t * H + h) * dk;
      const double* vt = v + (t * Hv + hv) * dv;
      for (int64_t j = 0; j < dv; ++j) tmp_v[j] = 0.0;
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j) tmp_v[j] += alpha * Sp[i * dv + j] * kt[i];
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j)
          Sn[i * dv + j] = alpha * Sp[i * dv + j] + b * kt[i] * (vt[j] - tmp_v[j]);
    }
    for (int64_t t = e - 1; t >= a; --t) {
      const double* Sp = seg + (t - a) * KV;      /* S_prev */
      const double* St = seg + (t - a + 1) * KV;  /* S after token t */
      const double alpha = exp(g[t * Hv + hv]), b = beta[t * Hv + hv];
      const double* kt = k + (t * H + h) * dk;
      const double* qt = q + (t * H + h) * dk;
      const double* vt = v + (t * Hv + hv) * dv;
      const double* dot = dout + (t * Hv + hv) * dv;
      double* dqt = dq + (t * H + h) * dk;
      double* dkt = dk_out + (t * H + h) * dk;
      double* dvt = dv_out + (t * Hv + hv) * dv;
      /* read: dS += scale q do^T; dq += scale S do */
      for (int64_t i = 0; i < dk; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < dv; ++j) {
          dS[i * dv + j] += scale * qt[i] * dot[j];
          acc += St[i * dv + j] * dot[j];
        }
        dqt[i] += scale * acc;
      }
      /* delta = v - (alpha S_prev)^T k, recomputed */
      for (int64_t j = 0; j < dv; ++j) tmp_v[j] = 0.0;
      for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j) tmp_v[j] += alpha * Sp[i * dv + j] * kt[i];
      for (int64_t j = 0; j < dv; ++j) tmp_v[j] = vt[j] - tmp_v[j];  /* delta */
      /* write: db = k^T dS delta; dk = b dS delta; ddelta = b dS^T k */
      double db = 0.0;
      for (int64_t i = 0; i < dk; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < dv; ++j) acc += dS[i * dv + j] * tmp_v[j];
        tmp_k[i] = acc;                       /* (dS delta)_i */
        db += kt[i] * acc;
      }
      dbeta[t * Hv + hv] = db;
      for (int64_t i = 0; i < dk; ++i) dkt[i] += b * tmp_k[i];
      for (int64_t j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < dk; ++i) acc += dS[i * dv + j] * kt[i];
        dvt[j] = b * acc;                     /* dv = ddelta; dpred = -ddelta */
      }
      /* dD = dS + k dpred^T; dk += D dpred with D = alpha S_prev */
      for (int64_t i = 0; i < dk; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < dv; ++j) {
          dD[i * dv + j] = dS[i * dv + j] - kt[i] * dvt[j];
          acc += alpha * Sp[i * dv + j] * dvt[j];
        }
        dkt[i] -= acc;
      }
      /* decay: dg = alpha <S_prev, dD>; dS_prev = alpha dD */
      double da = 0.0;
      for (int64_t i = 0; i < KV; ++i) {
        da += Sp[i] * dD[i];
        dS[i] = alpha * dD[i];
      }
      dg[t * Hv + hv] = alpha * da;
    }
  }
}

int gdn_ref_backward(int64_t T, int64_t N, int64_t H, int64_t Hv, int64_t dk, int64_t dv,
                     const double* q, const double* k, const double* v, const double* g,
                     const double* beta, double scale, const double* initial_state,
                     const int64_t* cu_seqlens, const double* d_out, const double* d_final,
                     double* dq, double* dk_out, double* dv_out, double* dg, double* dbeta,
                     double* d_initial, int nthreads) {
  if (T < 0 || N < 1 || H < 1 || Hv < 1 || dk < 1 || dv < 1) return GDN_REF_BAD_ARG;
  if (Hv % H != 0) return GDN_REF_BAD_ARG;
  if (!q || !k || !v || !g || !beta || !d_out || !dq || !dk_out || !dv_out || !dg || !dbeta)
    return GDN_REF_BAD_ARG;
  if (!cu_seqlens && N != 1) return GDN_REF_BAD_ARG;
  if (cu_seqlens)
    for (int64_t n = 0; n < N; ++n)
      if (cu_seqlens[n] < 0 || cu_seqlens[n + 1] < cu_seqlens[n] || cu_seqlens[n + 1] > T)
        return GDN_REF_BAD_ARG;
  if (!(scale > 0.0)) scale = 1.0 / sqrt((double)dk);
  const int64_t HG = Hv / H, KV = dk * dv;
  int64_t max_len = 0;
  for (int64_t n = 0; n < N; ++n) {
    const int64_t len = cu_seqlens ? cu_seqlens[n + 1] - cu_seqlens[n] : T;
    if (len > max_len) max_len = len;
  }
  const int64_t max_seg = (max_len + 63) / 64 + 1;
  memset(dq, 0, (size_t)(T * H * dk) * sizeof(double));
  memset(dk_out, 0, (size_t)(T * H * dk) * sizeof(double));
  memset(dv_out, 0, (size_t)(T * Hv * dv) * sizeof(double));
  memset(dg, 0, (size_t)(T * Hv) * sizeof(double));
  memset(dbeta, 0, (size_t)(T * Hv) * sizeof(double));
  int rc = GDN_REF_OK;
  /* value heads of one key head write the same dq/dk rows: one task per
     (sequence, key head), its value heads in order */
  const int64_t tasks = N * H;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double* S = (double*)malloc((size_t)KV * sizeof(double));
    double* ckpt = (double*)malloc((size_t)(max_seg * KV) * sizeof(double));
    double* seg = (double*)malloc((size_t)(65 * KV) * sizeof(double));
    double* dS = (double*)malloc((size_t)KV * sizeof(double));
    double* dD = (double*)malloc((size_t)KV * sizeof(double));
    double* tv = (double*)malloc((size_t)dv * sizeof(double));
    double* tk = (double*)malloc((size_t)dk * sizeof(double));
    int ok = S && ckpt && seg && dS && dD && tv && tk;
    if (!ok) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      rc = GDN_REF_NO_MEMORY;
    }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t task = 0; task < tasks; ++task) {
      if (!ok) continue;
      const int64_t n = task / H, h = task % H;
      const int64_t first = cu_seqlens ? cu_seqlens[n] : 0;
      const int64_t end = cu_seqlens ? cu_seqlens[n + 1] : T;
      for (int64_t hv = h * HG; hv < (h + 1) * HG; ++hv) {
        for (int64_t i = 0; i < dk; ++i)
          for (int64_t j = 0; j < dv; ++j) {
            const size_t at = (size_t)(((n * Hv + hv) * dv + j) * dk + i);
            S[i * dv + j] = initial_state ? initial_state[at] : 0.0;
            dS[i * dv + j] = d_final ? d_final[at] : 0.0;
          }
        lane_backward(first, end, H, Hv, dk, dv, h, hv, q, k, v, g, beta, scale, d_out, S, ckpt,
                      seg, dS, dD, tv, tk, dq, dk_out, dv_out, dg, dbeta);
        if (d_initial)
          for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j)
              d_initial[((n * Hv + hv) * dv + j) * dk + i] = dS[i * dv + j];
      }
    }
    free(S); free(ckpt); free(seg); free(dS); free(dD); free(tv); free(tk);
  }
  return rc;
}
