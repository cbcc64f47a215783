/*
 * oracle_bwd.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct fp64 gradients of softmax attention, used to
 * check the CUDA backward kernels.  Shares nothing with the CUDA library.
 *
 * Definition ("GPU Engineering: Correctness, Throughput, and Attention",
 * sections 22.5 and 22.7): with S = scale * Q K^T (causal rule j > i +
 * query_offset -> -inf), P = softmax(S) row by row, O = P V and a loss
 * gradient G = dO on O:
 *   dV = P^T dO,   dP = dO V^T,
 *   dS = P * (dP - rowsum(P * dP))      (vector-Jacobian product of softmax)
 *   dQ = scale * dS K,   dK = scale * dS^T Q.
 * A row with no admissible key has P = 0 and contributes nothing (the lab's
 * zero-gradient policy).  The row correction rowsum(P * dP) is taken from its
 * definition here; the page's identity rowsum(P * dP) = rowsum(dO * O) is
 * pinned by the tests instead.
 *
 * Grouped K/V heads: query head h of batch b uses K/V head b*Hkv + h/(H/Hkv),
 * so dK/dV of a K/V head sum the contributions of its whole group.  Work is
 * split over K/V heads, so no two threads write the same dK/dV row.
 *
 * The value width dv may differ from the key width d (V enters only through
 * O = P V, so the formulas above hold unchanged): V, dO and dV have dv
 * columns, Q, K, dQ and dK have d.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

enum { BWD_F64 = 0, BWD_BF16 = 1 };

typedef struct {
  const void *q, *k, *v, *dout;
  int elem;
  int64_t B, H, Hkv, Nq, Nk, d, dv_dim;
  int causal;
  int64_t query_offset;
  double scale;
  double *dq, *dk, *dv;
  int64_t kv_begin, kv_end; /* this worker's K/V heads (flattened b*Hkv + hk) */
} bwd_job_t;

static double ld(const void *base, int elem, int64_t idx) {
  if (elem == BWD_F64) return ((const double *)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static void *bwd_worker(void *arg) {
  const bwd_job_t *J = (const bwd_job_t *)arg;
  const int64_t Nk = J->Nk, d = J->d, e = J->dv_dim, G = J->H / J->Hkv;
  double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
  double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
  double *dp = (double *)malloc(sizeof(double) * (size_t)Nk);
  if (!s || !p || !dp) {
    free(s); free(p); free(dp);
    return (void *)1;
  }
  for (int64_t kvh = J->kv_begin; kvh < J->kv_end; ++kvh) {
    const int64_t b = kvh / J->Hkv, hk = kvh % J->Hkv;
    const int64_t kv_row0 = kvh * Nk; /* first K/V row of this head */
    for (int64_t g = 0; g < G; ++g) {
      const int64_t h = hk * G + g;
      for (int64_t i = 0; i < J->Nq; ++i) {
        const int64_t qrow = (b * J->H + h) * J->Nq + i;
        double M = -INFINITY;
        for (int64_t j = 0; j < Nk; ++j) {
          double dot = 0.0;
          for (int64_t c = 0; c < d; ++c)
            dot += ld(J->q, J->elem, qrow * d + c) * ld(J->k, J->elem, (kv_row0 + j) * d + c);
          s[j] = dot * J->scale;
          if (J->causal && j > i + J->query_offset) s[j] = -INFINITY;
          if (s[j] > M) M = s[j];
        }
        for (int64_t c = 0; c < d; ++c) J->dq[qrow * d + c] = 0.0;
        if (M == -INFINITY) continue; /* no admissible key: no gradient */
        double Z = 0.0;
        for (int64_t j = 0; j < Nk; ++j) {
          p[j] = exp(s[j] - M);
          Z += p[j];
        }
        double corr = 0.0;
        for (int64_t j = 0; j < Nk; ++j) {
          p[j] /= Z;
          double acc = 0.0;
          for (int64_t c = 0; c < e; ++c)
            acc += ld(J->dout, J->elem, qrow * e + c) * ld(J->v, J->elem, (kv_row0 + j) * e + c);
          dp[j] = acc;
          corr += p[j] * dp[j];
        }
        for (int64_t j = 0; j < Nk; ++j) {
#if ORACLE_PLANT == 8 /* softmax row correction dropped */
          const double ds = p[j] * dp[j];
#else
          const double ds = p[j] * (dp[j] - corr);
#endif
          for (int64_t c = 0; c < d; ++c) {
            const double kc = ld(J->k, J->elem, (kv_row0 + j) * d + c);
            const double qc = ld(J->q, J->elem, qrow * d + c);
            J->dq[qrow * d + c] += J->scale * ds * kc;
#if ORACLE_PLANT == 9 /* score scale missing from dK */
            J->dk[(kv_row0 + j) * d + c] += ds * qc;
#else
            J->dk[(kv_row0 + j) * d + c] += J->scale * ds * qc;
#endif
          }
          for (int64_t c = 0; c < e; ++c)
            J->dv[(kv_row0 + j) * e + c] += p[j] * ld(J->dout, J->elem, qrow * e + c);
        }
      }
    }
  }
  free(s); free(p); free(dp);
  return NULL;
}

/*
 * q: [B][H][Nq][d]; k: [B][Hkv][Nk][d]; v: [B][Hkv][Nk][dv_dim]; dout:
 * [B][H][Nq][dv_dim] (contiguous, same element type).  Writes dq
 * [B][H][Nq][d], dk [B][Hkv][Nk][d] and dv [B][Hkv][Nk][dv_dim] (double).
 * Returns 0, -1 on invalid arguments, -2 on allocation failure.
 */
int oracle_attention_bwd(const void *q, const void *k, const void *v, const void *dout,
                         int elem, int64_t B, int64_t H, int64_t Hkv, int64_t Nq, int64_t Nk,
                         int64_t d, int64_t dv_dim, int causal, int64_t query_offset,
                         double scale, double *dq, double *dk, double *dv, int n_threads) {
  if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
  if (elem != BWD_F64 && elem != BWD_BF16) return -1;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1 || dv_dim < 1) return -1;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0 || !isfinite(scale)) return -1;
  const int64_t n_kv = B * Hkv;
  memset(dk, 0, sizeof(double) * (size_t)(n_kv * Nk * d));
  memset(dv, 0, sizeof(double) * (size_t)(n_kv * Nk * dv_dim));
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (n_kv < n_threads) n_threads = (int)n_kv;
  bwd_job_t jobs[256];
  pthread_t tids[256];
  int started[256] = {0};
  int status = 0;
  for (int t = 0; t < n_threads; ++t) {
    bwd_job_t J = {q, k, v, dout, elem, B, H, Hkv, Nq, Nk, d, dv_dim, causal, query_offset,
                   scale, dq, dk, dv, n_kv * t / n_threads, n_kv * (t + 1) / n_threads};
    jobs[t] = J;
    if (n_threads > 1 && pthread_create(&tids[t], NULL, bwd_worker, &jobs[t]) == 0)
      started[t] = 1;
  }
  for (int t = 0; t < n_threads; ++t) {
    if (started[t]) {
      void *ret = NULL;
      pthread_join(tids[t], &ret);
      if (ret != NULL) status = -2;
    } else if (bwd_worker(&jobs[t]) != NULL) {
      status = -2;
    }
  }
  return status;
}
