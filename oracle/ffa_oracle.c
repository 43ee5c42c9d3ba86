/*
 * Flexible-mask attention oracle: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load this library.  It shares
 * no code, header or constant with the CUDA path.
 *
 * What it computes (MagiAttention pages, quickstart card "Single-GPU
 * Flex-Flash-Attention"; FlagAttention user guide, "Dense attention"):
 *   - tokens are packed: q[Tq][Hq][D], k/v[Tk][Hkv][D], bf16, converted to
 *     double exactly;
 *   - the mask is a list of slices (q_range, k_range, mask_type), ranges
 *     half-open [start, end);
 *   - inside a slice, query row i sees keys [lo_s(i), hi_s(i)) where the
 *     start moves with the row when bit 1 (value 2) of the type is set and
 *     the end moves with the row when bit 0 (value 1) is set, so that causal
 *     is bottom-right aligned (card "Calculate KV Interval Boundaries for Mask
 *     Types"; FlagAttention "Rectangular causal attention is bottom-right
 *     aligned");
 *   - a row sees the union of its intervals over the slices that contain it;
 *   - x_j = scale * <q_i, k_j>, lse_i = log sum_j exp(x_j) (natural log, the
 *     row log-normalizer), out_i = sum_j exp(x_j - lse_i) v_j;
 *     scale defaults to 1/sqrt(D);
 *   - a row that sees no key gives out = 0 and lse = -inf;
 *   - query head h reads key/value head h / (Hq / Hkv) (grouped-query heads).
 * Backward (standard softmax-attention gradient of the same function, fed
 * dOut):  P = exp(x - lse), dV_j = sum_i P_ij dO_i, dP_ij = <dO_i, v_j>,
 * delta_i = <dO_i, O_i>, dS = P (dP - delta), dQ_i = scale sum_j dS_ij k_j,
 * dK_j = scale sum_i dS_ij q_i, summed over the query heads of a kv head.
 *
 * Attention sink (quickstart card "Single-GPU Flex-Flash-Attention", the
 * `sink` argument, and the FlashAttention-with-sink cards, layouts "sh"
 * [n_sink][Hq] and "ssh" [Tq][n_sink][Hq], fp32).  The pages show the
 * argument but not its formula; the reading used here: each sink value
 * sigma_s is a logit, not multiplied by the softmax scale, that joins the
 * row's normaliser only,
 *     lse_i = log( sum_j exp(x_j) + sum_s exp(sigma_s) ),
 *     out_i = sum_j exp(x_j - lse_i) v_j,
 * so a row that sees no key gets out = 0 and lse = log sum_s exp(sigma_s).
 * Its gradient follows from that definition:
 *     dsink_s = - sum_i exp(sigma_s - lse_i) delta_i
 * (summed over the rows of the head for "sh", one value per row for "ssh").
 *
 * Softcap (quickstart card: the `softcap` argument, default 0; no formula on
 * the pages).  Reading: for c > 0 every score is capped smoothly,
 *     x_j = c * tanh(scale * <q_i, k_j> / c),
 * and the backward carries the chain-rule factor 1 - tanh^2 into dS:
 *     dS = P (dP - delta) (1 - (x / c)^2),  dQ = scale dS K,  dK = scale dS^T Q.
 * c <= 0 means no cap.
 *
 * Every loop below is the definition written out, with no blocking, fusion or
 * reordering.  OpenMP only splits independent (head, row) or (head, key)
 * pairs across threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int qs, qe, ks, ke, type;
} slice_t;

/* Exact bf16 -> double: a bf16 is the high half of an IEEE single. */
static double bf16_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double dot_bf16(const uint16_t* a, const uint16_t* b, int d) {
  double s = 0.0;
  for (int t = 0; t < d; ++t) s += bf16_to_double(a[t]) * bf16_to_double(b[t]);
  return s;
}

/* Interval of keys that row i sees inside slice s; empty when lo >= hi.
 * Returns 0 when the row is outside the slice's q range. */
static int slice_row_interval(const slice_t* s, long i, long* lo, long* hi) {
  if (i < s->qs || i >= s->qe) return 0;
  long start = s->ks, end = s->ke;
  if (s->type & 2) start += i - s->qs;       /* start shifts with the row */
  if (s->type & 1) end -= s->qe - 1 - i;     /* end clamps bottom-right   */
  *lo = start;
  *hi = end;
  return 1;
}

/* Does row i see key j under any slice? */
static int visible(const slice_t* sl, int ns, long i, long j) {
  for (int s = 0; s < ns; ++s) {
    long lo, hi;
    if (slice_row_interval(&sl[s], i, &lo, &hi) && lo <= j && j < hi) return 1;
  }
  return 0;
}

static slice_t* read_slices(const int* qr, const int* kr, const int* ty, int ns) {
  slice_t* sl = (slice_t*)malloc(sizeof(slice_t) * (ns > 0 ? ns : 1));
  for (int s = 0; s < ns; ++s) {
    sl[s].qs = qr[2 * s];
    sl[s].qe = qr[2 * s + 1];
    sl[s].ks = kr[2 * s];
    sl[s].ke = kr[2 * s + 1];
    sl[s].type = ty[s];
  }
  return sl;
}

typedef struct {
  const uint16_t *q, *k, *v;
  long Tq, Tk;
  int Hq, Hkv, D;
  const slice_t* sl;
  int ns;
  double scale;
  double softcap;     /* <= 0: no cap */
  const double* sink; /* NULL: no sink */
  int n_sink;
  int sink_layout;    /* 0: [n_sink][Hq], 1: [Tq][n_sink][Hq] */
} problem_t;

/* Score of a (row, key) pair from its dot product: scale * dot, capped. */
static double score(const problem_t* P, double dot) {
  const double x = P->scale * dot;
  return P->softcap > 0.0 ? P->softcap * tanh(x / P->softcap) : x;
}

/* d score / d(scale * dot) at score x: 1 - tanh^2 under a cap, else 1. */
static double score_grad(const problem_t* P, double x) {
  if (P->softcap <= 0.0) return 1.0;
  const double t = x / P->softcap;
  return 1.0 - t * t;
}

/* Sink logit s of (head h, row i). */
static double sink_value(const problem_t* P, int h, long i, int s) {
  if (P->sink_layout == 0) return P->sink[(size_t)s * P->Hq + h];
  return P->sink[((size_t)i * P->n_sink + s) * P->Hq + h];
}

/* Forward for one (head, row): fills out_row[D] and returns lse.
 * xbuf holds Tk doubles (scores of the visible keys), vis holds Tk flags. */
static double row_forward(const problem_t* P, int h, long i, double* out_row, double* xbuf,
                          unsigned char* vis) {
  const int D = P->D;
  const int hk = h / (P->Hq / P->Hkv);
  const uint16_t* qi = P->q + ((size_t)i * P->Hq + h) * D;
  memset(vis, 0, (size_t)P->Tk);
  /* V(i): union of the row's intervals over the slices that contain it */
  for (int s = 0; s < P->ns; ++s) {
    long lo, hi;
    if (!slice_row_interval(&P->sl[s], i, &lo, &hi)) continue;
    for (long j = lo; j < hi; ++j) vis[j] = 1;
  }
  double m = -INFINITY;
  long cnt = 0;
  for (long j = 0; j < P->Tk; ++j) {
    if (!vis[j]) continue;
    xbuf[j] = score(P, dot_bf16(qi, P->k + ((size_t)j * P->Hkv + hk) * D, D));
    if (xbuf[j] > m) m = xbuf[j];
    ++cnt;
  }
  /* sink logits join the normaliser (and its maximum, for a stable sum) */
  const int ns = P->sink ? P->n_sink : 0;
  for (int s = 0; s < ns; ++s) {
    const double sv = sink_value(P, h, i, s);
    if (sv > m) m = sv;
  }
  for (int t = 0; t < D; ++t) out_row[t] = 0.0;
  if (m == -INFINITY) return -INFINITY; /* no visible key and no (finite) sink */
  double sum = 0.0;
  for (long j = 0; j < P->Tk; ++j)
    if (vis[j]) sum += exp(xbuf[j] - m);
  for (int s = 0; s < ns; ++s) sum += exp(sink_value(P, h, i, s) - m);
  const double lse = m + log(sum);
  if (cnt == 0) return lse;
  for (long j = 0; j < P->Tk; ++j) {
    if (!vis[j]) continue;
    const double p = exp(xbuf[j] - lse);
    const uint16_t* vj = P->v + ((size_t)j * P->Hkv + hk) * D;
    for (int t = 0; t < D; ++t) out_row[t] += p * bf16_to_double(vj[t]);
  }
  return lse;
}

int ffa_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Forward on a subset of query rows (rows == NULL: all rows, n_rows = Tq).
 * out: [n_rows][Hq][D], lse: [Hq][n_rows]. */
int ffa_oracle_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, long Tq, long Tk,
                   int Hq, int Hkv, int D, const int* q_ranges, const int* k_ranges,
                   const int* mask_types, int num_slices, double scale, double softcap,
                   const double* sink, int n_sink, int sink_layout, const long* rows, long n_rows,
                   double* out, double* lse) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return 1;
  if (n_sink < 0 || (n_sink > 0 && !sink) || sink_layout < 0 || sink_layout > 1) return 1;
  slice_t* sl = read_slices(q_ranges, k_ranges, mask_types, num_slices);
  problem_t P = {q, k, v, Tq, Tk, Hq, Hkv, D, sl, num_slices, scale, softcap, sink, n_sink,
                 sink_layout};
  const long n = rows ? n_rows : Tq;
#pragma omp parallel
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
    unsigned char* vis = (unsigned char*)malloc((size_t)(Tk > 0 ? Tk : 1));
#pragma omp for schedule(dynamic, 4)
    for (long w = 0; w < n * Hq; ++w) {
      const long r = w / Hq;
      const int h = (int)(w % Hq);
      const long i = rows ? rows[r] : r;
      lse[(size_t)h * n + r] = row_forward(&P, h, i, out + ((size_t)r * Hq + h) * D, xbuf, vis);
    }
    free(xbuf);
    free(vis);
  }
  free(sl);
  return 0;
}

/* Backward.  dq for the rows in dq_rows (NULL: all rows) -> dq[n][Hq][D];
 * dk, dv for the keys in dkv_keys (NULL: all keys) -> dk/dv[n][Hkv][D].
 * lse and O are the oracle's own (recomputed per row in fp64). */
int ffa_oracle_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                   long Tq, long Tk, int Hq, int Hkv, int D, const int* q_ranges,
                   const int* k_ranges, const int* mask_types, int num_slices, double scale,
                   double softcap, const double* sink, int n_sink, int sink_layout,
                   const long* dq_rows,
                   long n_dq_rows, double* dq, const long* dkv_keys, long n_keys, double* dk,
                   double* dv) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return 1;
  if (n_sink < 0 || (n_sink > 0 && !sink) || sink_layout < 0 || sink_layout > 1) return 1;
  slice_t* sl = read_slices(q_ranges, k_ranges, mask_types, num_slices);
  problem_t P = {q, k, v, Tq, Tk, Hq, Hkv, D, sl, num_slices, scale, softcap, sink, n_sink,
                 sink_layout};
  const int g = Hq / Hkv;
  const long nq = dq_rows ? n_dq_rows : Tq;
  const long nk = dkv_keys ? n_keys : Tk;

  /* dQ rows */
#pragma omp parallel
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
    unsigned char* vis = (unsigned char*)malloc((size_t)(Tk > 0 ? Tk : 1));
    double* o = (double*)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 4)
    for (long w = 0; w < nq * Hq; ++w) {
      const long r = w / Hq;
      const int h = (int)(w % Hq);
      const int hk = h / g;
      const long i = dq_rows ? dq_rows[r] : r;
      double* dqi = dq + ((size_t)r * Hq + h) * D;
      for (int t = 0; t < D; ++t) dqi[t] = 0.0;
      const double lse = row_forward(&P, h, i, o, xbuf, vis);
      if (lse == -INFINITY) continue;
      const uint16_t* doi = dout + ((size_t)i * Hq + h) * D;
      double delta = 0.0;
      for (int t = 0; t < D; ++t) delta += bf16_to_double(doi[t]) * o[t];
      for (long j = 0; j < Tk; ++j) {
        if (!vis[j]) continue;
        const double p = exp(xbuf[j] - lse);
        const double dp = dot_bf16(doi, v + ((size_t)j * Hkv + hk) * D, D);
        const double ds = p * (dp - delta) * score_grad(&P, xbuf[j]);
        const uint16_t* kj = k + ((size_t)j * Hkv + hk) * D;
        for (int t = 0; t < D; ++t) dqi[t] += scale * ds * bf16_to_double(kj[t]);
      }
    }
    free(xbuf);
    free(vis);
    free(o);
  }

  if (nk > 0) {
    /* rows that see at least one requested key need their lse and delta */
    unsigned char* want = (unsigned char*)calloc((size_t)(Tk > 0 ? Tk : 1), 1);
    for (long r = 0; r < nk; ++r) want[dkv_keys ? dkv_keys[r] : r] = 1;
    unsigned char* need = (unsigned char*)calloc((size_t)(Tq > 0 ? Tq : 1), 1);
#pragma omp parallel for schedule(dynamic, 64)
    for (long i = 0; i < Tq; ++i) {
      for (int s = 0; s < num_slices && !need[i]; ++s) {
        long lo, hi;
        if (!slice_row_interval(&sl[s], i, &lo, &hi)) continue;
        for (long j = lo; j < hi; ++j)
          if (want[j]) { need[i] = 1; break; }
      }
    }
    double* lse_all = (double*)malloc(sizeof(double) * (size_t)Hq * (Tq > 0 ? Tq : 1));
    double* delta_all = (double*)malloc(sizeof(double) * (size_t)Hq * (Tq > 0 ? Tq : 1));
#pragma omp parallel
    {
      double* xbuf = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
      unsigned char* vis = (unsigned char*)malloc((size_t)(Tk > 0 ? Tk : 1));
      double* o = (double*)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 4)
      for (long w = 0; w < Tq * Hq; ++w) {
        const long i = w / Hq;
        const int h = (int)(w % Hq);
        if (!need[i]) continue;
        const double lse = row_forward(&P, h, i, o, xbuf, vis);
        const uint16_t* doi = dout + ((size_t)i * Hq + h) * D;
        double delta = 0.0;
        for (int t = 0; t < D; ++t) delta += bf16_to_double(doi[t]) * o[t];
        lse_all[(size_t)h * Tq + i] = lse;
        delta_all[(size_t)h * Tq + i] = delta;
      }
      free(xbuf);
      free(vis);
      free(o);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (long w = 0; w < nk * Hkv; ++w) {
      const long r = w / Hkv;
      const int hk = (int)(w % Hkv);
      const long j = dkv_keys ? dkv_keys[r] : r;
      double* dkj = dk + ((size_t)r * Hkv + hk) * D;
      double* dvj = dv + ((size_t)r * Hkv + hk) * D;
      for (int t = 0; t < D; ++t) dkj[t] = dvj[t] = 0.0;
      const uint16_t* kj = k + ((size_t)j * Hkv + hk) * D;
      const uint16_t* vj = v + ((size_t)j * Hkv + hk) * D;
      for (long i = 0; i < Tq; ++i) {
        if (!need[i] || !visible(sl, num_slices, i, j)) continue;
        for (int h = hk * g; h < (hk + 1) * g; ++h) {
          const uint16_t* qi = q + ((size_t)i * Hq + h) * D;
          const uint16_t* doi = dout + ((size_t)i * Hq + h) * D;
          const double x = score(&P, dot_bf16(qi, kj, D));
          const double p = exp(x - lse_all[(size_t)h * Tq + i]);
          const double dp = dot_bf16(doi, vj, D);
          const double ds = p * (dp - delta_all[(size_t)h * Tq + i]) * score_grad(&P, x);
          for (int t = 0; t < D; ++t) {
            dvj[t] += p * bf16_to_double(doi[t]);
            dkj[t] += scale * ds * bf16_to_double(qi[t]);
          }
        }
      }
    }
    free(want);
    free(need);
    free(lse_all);
    free(delta_all);
  }
  free(sl);
  return 0;
}

/* Gradient of the sink logits: dsink_s = - sum_i exp(sigma_s - lse_i) delta_i,
 * with the oracle's own lse and O.  Layout 0 ([n_sink][Hq]): summed over all
 * rows of the head, in row order; layout 1 ([Tq][n_sink][Hq]): one value per
 * row, for the rows in `rows` (NULL: all) -> dsink[n][n_sink][Hq]. */
int ffa_oracle_dsink(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const uint16_t* dout, long Tq, long Tk, int Hq, int Hkv, int D,
                     const int* q_ranges, const int* k_ranges, const int* mask_types,
                     int num_slices, double scale, double softcap, const double* sink,
                     int n_sink, int sink_layout, const long* rows, long n_rows, double* dsink) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return 1;
  if (n_sink <= 0 || !sink || sink_layout < 0 || sink_layout > 1) return 1;
  if (sink_layout == 0 && rows) return 1; /* a per-head sum needs every row */
  slice_t* sl = read_slices(q_ranges, k_ranges, mask_types, num_slices);
  problem_t P = {q, k, v, Tq, Tk, Hq, Hkv, D, sl, num_slices, scale, softcap, sink, n_sink,
                 sink_layout};
  const long n = rows ? n_rows : Tq;
  /* per (row, head, sink) term, then the sums in a fixed order */
  double* term = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * Hq * n_sink);
#pragma omp parallel
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
    unsigned char* vis = (unsigned char*)malloc((size_t)(Tk > 0 ? Tk : 1));
    double* o = (double*)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 4)
    for (long w = 0; w < n * Hq; ++w) {
      const long r = w / Hq;
      const int h = (int)(w % Hq);
      const long i = rows ? rows[r] : r;
      const double lse = row_forward(&P, h, i, o, xbuf, vis);
      const uint16_t* doi = dout + ((size_t)i * Hq + h) * D;
      double delta = 0.0;
      for (int t = 0; t < D; ++t) delta += bf16_to_double(doi[t]) * o[t];
      for (int s = 0; s < n_sink; ++s)
        term[((size_t)r * n_sink + s) * Hq + h] = -exp(sink_value(&P, h, i, s) - lse) * delta;
    }
    free(xbuf);
    free(vis);
    free(o);
  }
  if (sink_layout == 0) {
    for (int s = 0; s < n_sink; ++s)
      for (int h = 0; h < Hq; ++h) {
        double acc = 0.0;
        for (long r = 0; r < n; ++r) acc += term[((size_t)r * n_sink + s) * Hq + h];
        dsink[(size_t)s * Hq + h] = acc;
      }
  } else {
    memcpy(dsink, term, sizeof(double) * (size_t)n * Hq * n_sink);
  }
  free(term);
  free(sl);
  return 0;
}
