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

/* ------------------------------------------------------------------------
 * Backward of the joint-softmax forward above, fp64, one query row at a time
 * (the gradient of the MoDA forward of Sec. 2.2 with respect to every input;
 * the pages time forward + backward in Table 2 and Table 7 but do not spell
 * the backward out, so this is the chain rule through the definition):
 *
 *   for row (t, h) with joint row z, p = softmax(z), o = sum_c p_c val_c:
 *     D      = <dO[t,h,:], o>
 *     dp_c   = <dO[t,h,:], val_c>
 *     ds_c   = p_c (dp_c - D)              (gradient w.r.t. z_c)
 *     dq[t,h]        += scale * sum_c ds_c key_c
 *     dk[j,hk]       += scale * ds_j q[t,h]        j <= t
 *     dv[j,hk]       += p_j dO[t,h]
 *     dkd[l,t,hk]    += scale * ds_{t+1+l} q[t,h]  (same position only)
 *     dvd[l,t,hk]    += p_{t+1+l} dO[t,h]
 *
 * dO is bf16 bits like the other inputs; every gradient is double. The depth
 * gradients use the UNPACKED layout [L, T, Hk, d]. Rows are split over
 * threads; each thread accumulates dk/dv/dkd/dvd privately and the copies are
 * summed in thread order, so results do not depend on scheduling.
 * ------------------------------------------------------------------------ */
/* Where one row's gradient contributions go. Sequence key j >= k_lo lands at
 * dk + ((j - k_lo)*Hk + hk)*d (keys below k_lo are not accumulated); depth
 * slot l lands at dkd_row + l*dkd_stride. */
typedef struct {
  double *dq_row, *dk, *dv, *dkd_row, *dvd_row;
  int k_lo;
  int64_t dkd_stride;
} bwd_dst;

/* Gradient contributions of query row (t, h); work buffers z[T+L], o, g, qr[d]. */
static void bwd_row(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const uint16_t* kd, const uint16_t* vd, const uint16_t* dO, int T, int Hq,
                    int Hk, int d, int L, double scale, int t, int h, const bwd_dst* dst,
                    double* z, double* o, double* g, double* qr) {
  const int G = Hq / Hk, hk = h / G;
  const int64_t row = (int64_t)t * Hq + h;
  const uint16_t* qrow = q + row * d;
  const uint16_t* dorow = dO + row * d;
  for (int c = 0; c < d; ++c) {
    qr[c] = bf16_to_double(qrow[c]);
    g[c] = bf16_to_double(dorow[c]);
  }
  const int64_t n = (int64_t)t + 1 + L;
  for (int64_t j = 0; j <= t; ++j) z[j] = scale * dot_bf16(qrow, k + (j * Hk + hk) * d, d);
  for (int l = 0; l < L; ++l)
    z[t + 1 + l] = scale * dot_bf16(qrow, kd + (((int64_t)l * T + t) * Hk + hk) * d, d);
  double m = z[0];
  for (int64_t j = 1; j < n; ++j)
    if (z[j] > m) m = z[j];
  double Z = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    z[j] = exp(z[j] - m);
    Z += z[j];
  }
  for (int64_t j = 0; j < n; ++j) z[j] /= Z; /* z now holds p */
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    const uint16_t* val = j <= t ? v + (j * Hk + hk) * d
                                 : vd + (((int64_t)(j - t - 1) * T + t) * Hk + hk) * d;
    for (int c = 0; c < d; ++c) o[c] += z[j] * bf16_to_double(val[c]);
  }
  double D = 0.0;
  for (int c = 0; c < d; ++c) D += g[c] * o[c];
  for (int64_t j = 0; j < n; ++j) {
    const int is_seq = j <= t;
    const int64_t kv_off = is_seq ? (j * Hk + hk) * d
                                  : (((int64_t)(j - t - 1) * T + t) * Hk + hk) * d;
    const uint16_t* key = (is_seq ? k : kd) + kv_off;
    const uint16_t* val = (is_seq ? v : vd) + kv_off;
    double dp = 0.0;
    for (int c = 0; c < d; ++c) dp += g[c] * bf16_to_double(val[c]);
    const double p = z[j];
    const double ds = p * (dp - D);
    double *dkey = NULL, *dval = NULL;
    if (is_seq) {
      if (j >= dst->k_lo) {
        dkey = dst->dk + ((j - dst->k_lo) * Hk + hk) * d;
        dval = dst->dv + ((j - dst->k_lo) * Hk + hk) * d;
      }
    } else if (dst->dkd_row) {
      dkey = dst->dkd_row + (j - t - 1) * dst->dkd_stride;
      dval = dst->dvd_row + (j - t - 1) * dst->dkd_stride;
    }
    for (int c = 0; c < d; ++c) {
      dst->dq_row[c] += scale * ds * bf16_to_double(key[c]);
      if (dkey) {
        dkey[c] += scale * ds * qr[c];
        dval[c] += p * g[c];
      }
    }
  }
}

typedef struct {
  const uint16_t *q, *k, *v, *kd, *vd, *dO;
  int T, Hq, Hk, d, L;
  double scale;
  const int64_t* rows; /* row = t*Hq + h; NULL means rows begin..end-1 */
  int64_t begin, end;
  int k_lo;
  int rows_mode;       /* 0: full layouts; 1: per-row depth outputs, dk/dv tail */
  double *dq, *dk, *dv, *dkd, *dvd; /* dq (and per-row depth) disjoint; dk/dv private */
  int status;
} bwd_job;

static void* bwd_worker(void* arg) {
  bwd_job* jb = (bwd_job*)arg;
  const int T = jb->T, Hq = jb->Hq, Hk = jb->Hk, d = jb->d, L = jb->L;
  const int G = Hq / Hk;
  double* z = (double*)malloc(((size_t)T + L) * sizeof(double));
  double* o = (double*)malloc((size_t)d * sizeof(double));
  double* g = (double*)malloc((size_t)d * sizeof(double));
  double* qr = (double*)malloc((size_t)d * sizeof(double));
  jb->status = 0;
  if (!z || !o || !g || !qr) {
    jb->status = -2;
    free(z); free(o); free(g); free(qr);
    return NULL;
  }
  for (int64_t i = jb->begin; i < jb->end; ++i) {
    const int64_t row = jb->rows ? jb->rows[i] : i;
    const int t = (int)(row / Hq), h = (int)(row % Hq), hk = h / G;
    bwd_dst dst;
    dst.k_lo = jb->k_lo;
    dst.dk = jb->dk;
    dst.dv = jb->dv;
    if (jb->rows_mode) {
      dst.dq_row = jb->dq + i * d;
      dst.dkd_row = L ? jb->dkd + i * (int64_t)L * d : NULL;
      dst.dvd_row = L ? jb->dvd + i * (int64_t)L * d : NULL;
      dst.dkd_stride = d;
    } else {
      dst.dq_row = jb->dq + row * d;
      dst.dkd_row = L ? jb->dkd + ((int64_t)t * Hk + hk) * d : NULL;
      dst.dvd_row = L ? jb->dvd + ((int64_t)t * Hk + hk) * d : NULL;
      dst.dkd_stride = (int64_t)T * Hk * d;
    }
    bwd_row(jb->q, jb->k, jb->v, jb->kd, jb->vd, jb->dO, T, Hq, Hk, d, L, jb->scale, t, h, &dst,
            z, o, g, qr);
  }
  free(z); free(o); free(g); free(qr);
  return NULL;
}

/* Runs jobs[0..nthreads) (job 0 on the calling thread); returns the first error. */
static int run_bwd_jobs(bwd_job* jobs, int nthreads) {
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!th) return -2;
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, bwd_worker, &jobs[i]) != 0) break;
    ++started;
  }
  bwd_worker(&jobs[0]);
  for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
  for (int i = started + 1; i < nthreads; ++i) bwd_worker(&jobs[i]);
  free(th);
  int status = 0;
  for (int i = 0; i < nthreads && status == 0; ++i) status = jobs[i].status;
  return status;
}

/* All gradients of the forward: dq[T,Hq,d], dk/dv[T,Hk,d], dkd/dvd[L,T,Hk,d]
 * (double, overwritten). kd/vd/dkd/dvd may be NULL when L == 0. Every thread
 * accumulates dk/dv/dkd/dvd privately; the copies are summed in thread order. */
int moda_oracle_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const uint16_t* kd, const uint16_t* vd, const uint16_t* dO, int T, int Hq,
                    int Hk, int d, int L, double scale, double* dq, double* dk, double* dv,
                    double* dkd, double* dvd, int nthreads) {
  if (T < 1 || Hq < 1 || Hk < 1 || d < 1 || L < 0 || Hq % Hk != 0) return -1;
  if (L > 0 && (!kd || !vd || !dkd || !dvd)) return -1;
  const int64_t rows = (int64_t)T * Hq;
  const size_t nq = (size_t)rows * d, nk = (size_t)T * Hk * d, nd = (size_t)L * T * Hk * d;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > rows) nthreads = (int)rows;
  bwd_job* jobs = (bwd_job*)calloc((size_t)nthreads, sizeof(bwd_job));
  double* priv = (double*)calloc((size_t)nthreads * (2 * nk + 2 * nd), sizeof(double));
  if (!jobs || !priv) {
    free(jobs); free(priv);
    return -2;
  }
  memset(dq, 0, nq * sizeof(double));
  for (int i = 0; i < nthreads; ++i) {
    bwd_job* jb = &jobs[i];
    double* base = priv + (size_t)i * (2 * nk + 2 * nd);
    jb->q = q; jb->k = k; jb->v = v; jb->kd = kd; jb->vd = vd; jb->dO = dO;
    jb->T = T; jb->Hq = Hq; jb->Hk = Hk; jb->d = d; jb->L = L; jb->scale = scale;
    jb->rows = NULL;
    jb->begin = rows * i / nthreads;
    jb->end = rows * (i + 1) / nthreads;
    jb->k_lo = 0;
    jb->rows_mode = 0;
    jb->dq = dq;
    jb->dk = base; jb->dv = base + nk; jb->dkd = base + 2 * nk; jb->dvd = base + 2 * nk + nd;
  }
  const int status = run_bwd_jobs(jobs, nthreads);
  memset(dk, 0, nk * sizeof(double));
  memset(dv, 0, nk * sizeof(double));
  if (L > 0) {
    memset(dkd, 0, nd * sizeof(double));
    memset(dvd, 0, nd * sizeof(double));
  }
  for (int i = 0; i < nthreads; ++i) {
    const bwd_job* jb = &jobs[i];
    for (size_t e = 0; e < nk; ++e) {
      dk[e] += jb->dk[e];
      dv[e] += jb->dv[e];
    }
    for (size_t e = 0; e < nd; ++e) {
      dkd[e] += jb->dkd[e];
      dvd[e] += jb->dvd[e];
    }
  }
  free(jobs); free(priv);
  return status;
}

/* Gradient contributions of the listed rows only (row = t*Hq + h):
 *   dq_rows[i][:]                 dq of row i (complete)
 *   dkd_rows[i][l][:], dvd_rows   row i's share of the depth gradients of its
 *                                 position (the sum over the G heads of a
 *                                 position is the full depth gradient there)
 *   dk_tail[j-k_lo][hk][:], dv_tail  the listed rows' share of the gradients
 *                                 of keys k_lo <= j < T (complete when every
 *                                 row of positions >= k_lo is listed)
 * Used to check large workloads without an O(T^2) full backward. */
int moda_oracle_bwd_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const uint16_t* kd, const uint16_t* vd, const uint16_t* dO, int T,
                         int Hq, int Hk, int d, int L, double scale, const int64_t* rows,
                         int64_t n, int k_lo, double* dq_rows, double* dk_tail, double* dv_tail,
                         double* dkd_rows, double* dvd_rows, int nthreads) {
  if (T < 1 || Hq < 1 || Hk < 1 || d < 1 || L < 0 || Hq % Hk != 0 || n < 0) return -1;
  if (k_lo < 0 || k_lo > T) return -1;
  if (L > 0 && (!kd || !vd || !dkd_rows || !dvd_rows)) return -1;
  for (int64_t i = 0; i < n; ++i)
    if (rows[i] < 0 || rows[i] >= (int64_t)T * Hq) return -1;
  const size_t nk = (size_t)(T - k_lo) * Hk * d;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  bwd_job* jobs = (bwd_job*)calloc((size_t)nthreads, sizeof(bwd_job));
  double* priv = (double*)calloc((size_t)nthreads * 2 * (nk ? nk : 1), sizeof(double));
  if (!jobs || !priv) {
    free(jobs); free(priv);
    return -2;
  }
  memset(dq_rows, 0, (size_t)n * d * sizeof(double));
  if (L > 0) {
    memset(dkd_rows, 0, (size_t)n * L * d * sizeof(double));
    memset(dvd_rows, 0, (size_t)n * L * d * sizeof(double));
  }
  for (int i = 0; i < nthreads; ++i) {
    bwd_job* jb = &jobs[i];
    jb->q = q; jb->k = k; jb->v = v; jb->kd = kd; jb->vd = vd; jb->dO = dO;
    jb->T = T; jb->Hq = Hq; jb->Hk = Hk; jb->d = d; jb->L = L; jb->scale = scale;
    jb->rows = rows;
    jb->begin = n * i / nthreads;
    jb->end = n * (i + 1) / nthreads;
    jb->k_lo = k_lo;
    jb->rows_mode = 1;
    jb->dq = dq_rows; jb->dkd = dkd_rows; jb->dvd = dvd_rows;
    jb->dk = priv + (size_t)i * 2 * (nk ? nk : 1);
    jb->dv = jb->dk + nk;
  }
  const int status = run_bwd_jobs(jobs, nthreads);
  memset(dk_tail, 0, nk * sizeof(double));
  memset(dv_tail, 0, nk * sizeof(double));
  for (int i = 0; i < nthreads; ++i)
    for (size_t e = 0; e < nk; ++e) {
      dk_tail[e] += jobs[i].dk[e];
      dv_tail[e] += jobs[i].dv[e];
    }
  free(jobs); free(priv);
  return status;
}

/*
 * Depth key or value of an FFN layer.
 *
 * Where the depth KV comes from (reading notes, Sec. 二.3; summary, Sec. 2.2,
 * the MoDA "write" step): attention layers append the K, V they already
 * computed, while an FFN layer obtains its pair through a light KV projection
 * of the FFN's INPUT X. MoDA keeps only the grouped depth key/value
 * projections (no depth query). Plain reading: a linear map without bias,
 *   out[r, n] = sum_{c < Dm} x[t_r, c] * w[n, c]     for n < N,
 * with x [T, Dm], the weight one row per output feature, w [N, Dm], N = Hk*d
 * (feature n = hk*d + j is element j of KV head hk), and t_r = rows[r].
 * The sum is taken in double precision in the order of c and returned
 * unrounded in out [n_rows, N]. The caller calls it once with W_K and once
 * with W_V.
 *
 * Returns 0, or -1 on a bad argument.
 */
int moda_oracle_kv_proj(const uint16_t* x, const uint16_t* w, int T, int Dm, int N,
                        const int64_t* rows, int64_t n_rows, double* out) {
  if (!x || !w || !out || T < 1 || Dm < 1 || N < 1 || n_rows < 0) return -1;
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t t = rows ? rows[r] : r;
    if (t < 0 || t >= T) return -1;
    const uint16_t* xrow = x + t * (int64_t)Dm;
    for (int n = 0; n < N; ++n) {
      const uint16_t* wrow = w + (int64_t)n * Dm;
      double s = 0.0;
      for (int c = 0; c < Dm; ++c) s += bf16_to_double(xrow[c]) * bf16_to_double(wrow[c]);
      out[r * (int64_t)N + n] = s;
    }
  }
  return 0;
}

/*
 * Depth probability mass: how much the queries of one layer read each depth
 * slot.
 *
 * The bounded depth cache (summary, Sec. 6.2 "bounded depth KV slot cache")
 * keeps a fixed budget of S slots and, in its dynamic-selection form, scores
 * the cached entries by utility and keeps the top S. The pages give no
 * formula for the utility. Reading: the probability mass that the joint
 * softmax of Sec. 2.2 gives the slot, summed over the rows that read it,
 *   mass[hk*L + l] = sum over listed rows (t, h) with floor(h/G) = hk of
 *                    p_{t,h}(depth slot l),
 * p_{t,h} being the joint row of moda_oracle_row (its entry t + 1 + l).
 * Rows are (ts[i], hs[i]) for i < n; threads accumulate privately and the
 * copies are summed in thread order. Returns 0, -1 on a bad argument, -2 on
 * allocation failure.
 */
typedef struct {
  const uint16_t *q, *k, *v, *kd, *vd;
  int T, Hq, Hk, d, L;
  double scale;
  const int64_t *ts, *hs;
  int64_t begin, end;
  double* mass; /* private [Hk*L] */
  int status;
} mass_job;

static void* mass_worker(void* arg) {
  mass_job* jb = (mass_job*)arg;
  jb->status = 0;
  const int G = jb->Hq / jb->Hk;
  double* o = (double*)malloc((size_t)jb->d * sizeof(double));
  double* p = (double*)malloc(((size_t)jb->T + (size_t)jb->L) * sizeof(double));
  if (!o || !p) {
    jb->status = -2;
    free(o);
    free(p);
    return NULL;
  }
  for (int64_t i = jb->begin; i < jb->end; ++i) {
    const int t = (int)jb->ts[i], h = (int)jb->hs[i];
    double lse;
    int rc = moda_oracle_row(jb->q, jb->k, jb->v, jb->kd, jb->vd, jb->T, jb->Hq, jb->Hk, jb->d,
                             jb->L, jb->scale, t, h, o, &lse, p);
    if (rc != 0) {
      jb->status = rc;
      break;
    }
    double* m = jb->mass + (int64_t)(h / G) * jb->L;
    for (int l = 0; l < jb->L; ++l) m[l] += p[t + 1 + l];
  }
  free(o);
  free(p);
  return NULL;
}

int moda_oracle_depth_mass(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const uint16_t* kd, const uint16_t* vd, int T, int Hq, int Hk, int d,
                           int L, double scale, const int64_t* ts, const int64_t* hs, int64_t n,
                           double* mass, int nthreads) {
  if (n < 0 || L < 1 || Hk < 1 || Hq % Hk != 0 || !mass) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  const size_t nm = (size_t)Hk * L;
  mass_job* jobs = (mass_job*)calloc((size_t)nthreads, sizeof(mass_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  double* priv = (double*)calloc((size_t)nthreads * nm, sizeof(double));
  if (!jobs || !th || !priv) {
    free(jobs); free(th); free(priv);
    return -2;
  }
  for (int i = 0; i < nthreads; ++i) {
    mass_job* jb = &jobs[i];
    jb->q = q; jb->k = k; jb->v = v; jb->kd = kd; jb->vd = vd;
    jb->T = T; jb->Hq = Hq; jb->Hk = Hk; jb->d = d; jb->L = L; jb->scale = scale;
    jb->ts = ts; jb->hs = hs;
    jb->begin = n * i / nthreads;
    jb->end = n * (i + 1) / nthreads;
    jb->mass = priv + (size_t)i * nm;
  }
  int started = 0;
  if (nthreads > 1)
    for (int i = 0; i < nthreads; ++i) {
      if (pthread_create(&th[i], NULL, mass_worker, &jobs[i]) != 0) break;
      ++started;
    }
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  for (int i = started; i < nthreads; ++i) mass_worker(&jobs[i]);
  int status = 0;
  for (int i = 0; i < nthreads && status == 0; ++i) status = jobs[i].status;
  memset(mass, 0, nm * sizeof(double));
  for (int i = 0; i < nthreads; ++i)
    for (size_t e = 0; e < nm; ++e) mass[e] += jobs[i].mass[e];
  free(jobs); free(th); free(priv);
  return status;
}
