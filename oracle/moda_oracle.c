/*
 * MoDA forward oracle: plain, slow, fp64, one query row at a time.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do. It shares no code, header or helper with the CUDA
 * library.
 *
 * What it computes (Mixture-of-Depths Attention, arXiv 2603.15619):
 *   For query row (t, h) with hk = floor(h / G), G = Hq / Hk (contiguous
 *   groups of G query heads share one KV head; the paper's 1-based
 *   phi(h) = ceil(h/G), Sec. 2.1 Eq. (2)):
 *     z_j       = scale * <q[t,h,:], k[j,hk,:]>          for j = 0..t
 *                 (causal, self included: M_ij = 0 iff j <= i, Eq. (2))
 *     z_{t+1+l} = scale * <q[t,h,:], kd[l,t,hk,:]>      for l = 0..L-1
 *                 (the L depth slots written for the SAME position t,
 *                  Sec. 2.2 "MoDA" and Fig. 1)
 *     p = softmax(z) over the joint row (ONE shared denominator, the
 *         expanded form of Sec. 2.2 in the reading notes, Sec. 二.2)
 *     o[t,h,:]  = sum_j p_j v[j,hk,:] + sum_l p_{t+1+l} vd[l,t,hk,:]
 *     lse[t,h]  = max(z) + ln(sum exp(z - max(z)))   (natural log, in the
 *                 scaled-score domain; the pages define no lse, this is the
 *                 FlashAttention convention)
 *
 * The depth stream is read in its UNPACKED layout [L, T, Hk, d], the order
 * in which layers append slots, so that a bug in the relayout kernel cannot
 * cancel against a matching bug here.
 *
 * Inputs are bf16 bit patterns (uint16). They are widened exactly to double
 * (bf16 -> fp32 is a 16-bit shift, fp32 -> fp64 is exact). All arithmetic is
 * double precision; the joint score row is materialised explicitly.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double dot_bf16(const uint16_t* a, const uint16_t* b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += bf16_to_double(a[c]) * bf16_to_double(b[c]);
  return s;
}

/* Returns 0 on success, -1 on a bad argument, -2 on allocation failure. */
int moda_oracle_row(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const uint16_t* kd, const uint16_t* vd, int T, int Hq,
                    int Hk, int d, int L, double scale, int t, int h,
                    double* o, double* lse, double* p_out) {
  if (T < 1 || Hq < 1 || Hk < 1 || d < 1 || L < 0) return -1;
  if (Hq % Hk != 0) return -1;
  if (t < 0 || t >= T || h < 0 || h >= Hq) return -1;
  if (L > 0 && (kd == NULL || vd == NULL)) return -1;
  const int G = Hq / Hk;
  const int hk = h / G;
  const int64_t n = (int64_t)t + 1 + L; /* joint row length */
  double* z = (double*)malloc((size_t)n * sizeof(double));
  if (!z) return -2;

  const uint16_t* qrow = q + ((int64_t)t * Hq + h) * d;
  /* sequence logits, causal: keys 0..t */
  for (int64_t j = 0; j <= t; ++j) {
    const uint16_t* krow = k + (j * Hk + hk) * d;
    z[j] = scale * dot_bf16(qrow, krow, d);
  }
  /* depth logits: slot l of the same position t */
  for (int l = 0; l < L; ++l) {
    const uint16_t* kdrow = kd + (((int64_t)l * T + t) * Hk + hk) * d;
    z[t + 1 + l] = scale * dot_bf16(qrow, kdrow, d);
  }
  /* one softmax over the joint row */
  double m = z[0];
  for (int64_t j = 1; j < n; ++j)
    if (z[j] > m) m = z[j];
  double Z = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    z[j] = exp(z[j] - m); /* z now holds unnormalised weights */
    Z += z[j];
  }
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (int64_t j = 0; j <= t; ++j) {
    const double pj = z[j] / Z;
    const uint16_t* vrow = v + (j * Hk + hk) * d;
    for (int c = 0; c < d; ++c) o[c] += pj * bf16_to_double(vrow[c]);
  }
  for (int l = 0; l < L; ++l) {
    const double pl = z[t + 1 + l] / Z;
    const uint16_t* vdrow = vd + (((int64_t)l * T + t) * Hk + hk) * d;
    for (int c = 0; c < d; ++c) o[c] += pl * bf16_to_double(vdrow[c]);
  }
  *lse = m + log(Z);
  if (p_out)
    for (int64_t j = 0; j < n; ++j) p_out[j] = z[j] / Z;
  free(z);
  return 0;
}

/* ---- many rows, optionally split over threads (outer loop only) ---- */

typedef struct {
  const uint16_t *q, *k, *v, *kd, *vd;
  int T, Hq, Hk, d, L;
  double scale;
  const int64_t *ts, *hs;
  int64_t begin, end;
  double *o, *lse;
  int status;
} rows_job;

static void* rows_worker(void* arg) {
  rows_job* jb = (rows_job*)arg;
  jb->status = 0;
  for (int64_t i = jb->begin; i < jb->end; ++i) {
    int rc = moda_oracle_row(jb->q, jb->k, jb->v, jb->kd, jb->vd, jb->T, jb->Hq,
                             jb->Hk, jb->d, jb->L, jb->scale, (int)jb->ts[i],
                             (int)jb->hs[i], jb->o + i * jb->d, jb->lse + i, NULL);
    if (rc != 0) {
      jb->status = rc;
      break;
    }
  }
  return NULL;
}

/* Computes rows (ts[i], hs[i]) for i < n into o[i*d .. i*d+d) and lse[i].
 * nthreads <= 1 runs on the calling thread. Returns 0 or the first error. */
int moda_oracle_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const uint16_t* kd, const uint16_t* vd, int T, int Hq,
                     int Hk, int d, int L, double scale, const int64_t* ts,
                     const int64_t* hs, int64_t n, double* o, double* lse,
                     int nthreads) {
  if (n < 0) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  rows_job* jobs = (rows_job*)calloc((size_t)nthreads, sizeof(rows_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -2;
  }
  /* interleave-free contiguous split: rows are passed in caller order */
  for (int i = 0; i < nthreads; ++i) {
    rows_job* jb = &jobs[i];
    jb->q = q; jb->k = k; jb->v = v; jb->kd = kd; jb->vd = vd;
    jb->T = T; jb->Hq = Hq; jb->Hk = Hk; jb->d = d; jb->L = L;
    jb->scale = scale; jb->ts = ts; jb->hs = hs;
    jb->begin = n * i / nthreads;
    jb->end = n * (i + 1) / nthreads;
    jb->o = o; jb->lse = lse;
  }
  int status = 0;
  if (nthreads == 1) {
    rows_worker(&jobs[0]);
    status = jobs[0].status;
  } else {
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
      if (pthread_create(&th[i], NULL, rows_worker, &jobs[i]) != 0) break;
      ++started;
    }
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    if (started < nthreads) {
      /* finish the remainder on this thread */
      for (int i = started; i < nthreads; ++i) rows_worker(&jobs[i]);
    }
    for (int i = 0; i < nthreads && status == 0; ++i) status = jobs[i].status;
  }
  free(jobs);
  free(th);
  return status;
}
