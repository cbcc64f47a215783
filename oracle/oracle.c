/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU definition of softmax attention in
 * IEEE double precision.  It exists to check the CUDA path; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no source, header, table or helper with the CUDA library.
 *
 * What it computes (per head (b,h) and query row i), following
 * "GPU Engineering: Correctness, Throughput, and Attention":
 *   - section 22.7 (worked lab): scores S = Q K^T * scale, with the causal
 *     rule that key position j is excluded when j > i + query_offset, and the
 *     explicit policy that a row with no admissible key has output 0 and
 *     log-normaliser -infinity;
 *   - section 22.5: the online-softmax recurrence reaches, in real
 *     arithmetic, exactly the stable full softmax; so the oracle is that full
 *     softmax written out densely (max, then exponentials, then one sum),
 *     not the tiled recurrence.
 *
 *   s_j   = scale * sum_c q[i][c] * k[j][c]           j in [key_lo, key_hi)
 *   s_j   = -inf   if causal and j > i + query_offset
 *   M     = max_j s_j
 *   if M == -inf:  o[i][:] = 0,  lse[i] = -inf
 *   else:          w_j = exp(s_j - M),  Z = sum_j w_j
 *                  o[i][c] = sum_j w_j * v[j][c] / Z
 *                  lse[i]  = M + log(Z)              (natural logarithm)
 *
 * Grouped K/V heads (GQA/MQA, named among FlashAttention's production
 * features in "GPU Kernels: CUDA, HIP & Triton", section 7.6): K and V have
 * Hkv heads; query head h of batch b reads K/V head b*Hkv + h / (H / Hkv).
 * Hkv = H is ordinary multi-head attention.
 *
 * Inputs are either IEEE doubles or bfloat16 bit patterns; a bfloat16 value
 * is widened exactly (its 16 bits are the top half of an IEEE single).
 * The key range [key_lo, key_hi) defaults to every key; a narrower range is
 * attention over a contiguous subset of keys, used to pin the split-key
 * merge.  Rows may be restricted to a caller-given list (a deterministic
 * sample), in which case outputs are packed in list order.
 *
 * Planted mistakes (ORACLE_PLANT=n at compile time) exist only so the test
 * suite can show that its pins catch each of them; the default build has
 * ORACLE_PLANT undefined.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

enum { ORACLE_F64 = 0, ORACLE_BF16 = 1 };

typedef struct {
  const void *q, *k, *v;
  int elem;
  int64_t B, H, Hkv, Nq, Nk, d, dv;
  int causal;
  int64_t query_offset;
  double scale;
  int64_t key_lo, key_hi;
  const int64_t *rows; /* flattened (b*H + h)*Nq + i, or NULL for all rows */
  int64_t n_rows;
  double *o, *lse;
  int64_t row_begin, row_end; /* this worker's slice of the row list */
} job_t;

static double load(const void *base, int elem, int64_t idx) {
  if (elem == ORACLE_F64) return ((const double *)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* One query row of one head, by the dense definition above. */
static void one_row(const job_t *J, int64_t flat_row, double *s, double *o_out,
                    double *lse_out) {
  const int64_t bh = flat_row / J->Nq;
  const int64_t i = flat_row % J->Nq;
  const int64_t q_base = flat_row * J->d;
  const int64_t b = bh / J->H, h = bh % J->H;
#if ORACLE_PLANT == 7 /* grouped heads mapped round-robin instead of in blocks */
  const int64_t kv_head = (b * J->Hkv + h % J->Hkv) * J->Nk;
#else
  const int64_t kv_head = (b * J->Hkv + h / (J->H / J->Hkv)) * J->Nk;
#endif

  double M = -INFINITY;
  for (int64_t j = J->key_lo; j < J->key_hi; ++j) {
    double dot = 0.0;
    for (int64_t c = 0; c < J->d; ++c) {
#if ORACLE_PLANT == 5 /* transposed operand: reads K column-major */
      double kv = load(J->k, J->elem, kv_head * J->d + c * J->Nk + j);
#else
      double kv = load(J->k, J->elem, (kv_head + j) * J->d + c);
#endif
      dot += load(J->q, J->elem, q_base + c) * kv;
    }
    double sj = dot * J->scale;
#if ORACLE_PLANT == 1 /* causal mask dropped */
    (void)0;
#elif ORACLE_PLANT == 2 /* causal mask off by one: excludes the diagonal */
    if (J->causal && j >= i + J->query_offset) sj = -INFINITY;
#else
    if (J->causal && j > i + J->query_offset) sj = -INFINITY;
#endif
    s[j - J->key_lo] = sj;
    if (sj > M) M = sj;
  }

  if (M == -INFINITY) { /* no admissible key: explicit policy */
    for (int64_t c = 0; c < J->dv; ++c) o_out[c] = 0.0;
    *lse_out = -INFINITY;
    return;
  }

  double Z = 0.0;
  for (int64_t c = 0; c < J->dv; ++c) o_out[c] = 0.0;
  for (int64_t j = J->key_lo; j < J->key_hi; ++j) {
#if ORACLE_PLANT == 3 /* wrong sign in the exponent */
    double w = exp(M - s[j - J->key_lo]);
    if (s[j - J->key_lo] == -INFINITY) w = 0.0;
#else
    double w = exp(s[j - J->key_lo] - M);
#endif
    Z += w;
    for (int64_t c = 0; c < J->dv; ++c)
      o_out[c] += w * load(J->v, J->elem, (kv_head + j) * J->dv + c);
  }
#if ORACLE_PLANT == 4 /* forgot to normalise the output */
  (void)0;
#else
  for (int64_t c = 0; c < J->dv; ++c) o_out[c] /= Z;
#endif
#if ORACLE_PLANT == 6 /* log-normaliser without the row maximum */
  *lse_out = log(Z);
#else
  *lse_out = M + log(Z);
#endif
}

static void *worker(void *arg) {
  const job_t *J = (const job_t *)arg;
  double *s = (double *)malloc(sizeof(double) * (size_t)(J->key_hi - J->key_lo + 1));
  if (!s) return (void *)1;
  for (int64_t r = J->row_begin; r < J->row_end; ++r) {
    int64_t flat = J->rows ? J->rows[r] : r;
    one_row(J, flat, s, J->o + r * J->dv, J->lse + r);
  }
  free(s);
  return NULL;
}

/*
 * Returns 0 on success, -1 on invalid arguments, -2 on allocation failure.
 * q: [B][H][Nq][d], k: [B][Hkv][Nk][d], v: [B][Hkv][Nk][dv] (contiguous);
 * H must be a multiple of Hkv.
 * o: [n_out][dv], lse: [n_out] where n_out = n_rows if rows != NULL else B*H*Nq.
 */
int oracle_attention(const void *q, const void *k, const void *v, int elem,
                     int64_t B, int64_t H, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                     int64_t dv, int causal, int64_t query_offset, double scale,
                     int64_t key_lo, int64_t key_hi, const int64_t *rows,
                     int64_t n_rows, double *o, double *lse, int n_threads) {
  if (!q || !k || !v || !o || !lse) return -1;
  if (elem != ORACLE_F64 && elem != ORACLE_BF16) return -1;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1 || dv < 1) return -1;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return -1;
  if (key_lo < 0 || key_hi > Nk || key_lo > key_hi) return -1;
  if (!isfinite(scale)) return -1;
  const int64_t total_rows = B * H * Nq;
  const int64_t n_out = rows ? n_rows : total_rows;
  if (rows) {
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= total_rows) return -1;
  }
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (n_out < n_threads) n_threads = n_out > 0 ? (int)n_out : 1;

  job_t base = {q, k, v, elem, B, H, Hkv, Nq, Nk, d, dv, causal, query_offset,
                scale, key_lo, key_hi, rows, n_rows, o, lse, 0, 0};
  job_t jobs[256];
  pthread_t tids[256];
  int started[256] = {0};
  int status = 0;
  for (int t = 0; t < n_threads; ++t) {
    jobs[t] = base;
    jobs[t].row_begin = n_out * t / n_threads;
    jobs[t].row_end = n_out * (t + 1) / n_threads;
    if (n_threads == 1) break;
    if (pthread_create(&tids[t], NULL, worker, &jobs[t]) == 0) started[t] = 1;
  }
  if (n_threads == 1) {
    if (worker(&jobs[0]) != NULL) status = -2;
    return status;
  }
  for (int t = 0; t < n_threads; ++t) {
    if (started[t]) {
      void *ret = NULL;
      pthread_join(tids[t], &ret);
      if (ret != NULL) status = -2;
    } else if (worker(&jobs[t]) != NULL) {
      status = -2;
    }
  }
  return status;
}

int oracle_plant(void) { return ORACLE_PLANT; }
