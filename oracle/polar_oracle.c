/*
 * Plain fp64 CPU oracle for causal Polar Attention (prefill and decode).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the tests, the smoke check and the bench's CPU-baseline leg load it.
 * It shares no code, header, constant or helper with the CUDA library.
 *
 * Source: "ATMA: Length-Invariant Language Modeling via Polar Attention and
 * Gated-Delta Compression Memory" (technical summaries, es/it/fr pages),
 *   §2.1  out = content + count + memory (three additive streams)
 *   §2.1 item 1 (direction / "what" channel): the sum of matched values is
 *         projected onto the unit sphere; a length temperature sharpens the
 *         distribution as context grows; an extreme-value-corrected null
 *         floor calibrates logits against random noise
 *   §2.1 item 2 (magnitude / "how much" channel): participation ratio
 *         (inverse Simpson index) n_eff of the attention distribution, gated
 *         by confidence in signal detection, through a bounded, monotone,
 *         saturating tanh-of-log map
 *   §2.1 item 3 (memory channel): an additive stream, taken here as input
 *   §2.2 fused kernel: participation ratios computed online with streaming
 *         accumulators and squared correction factors, O(block) memory
 *   §2 decoder-only stack => causal attention; §3 training length 2K.
 *
 * The pages give these ingredients in words only.  The functional forms are
 * this project's pinned reading (each one is stated where it is used):
 *   tau   = max(1, ln n / ln T0),   T0 = 2048 (training length 2K)
 *   s_j   = tau * (q . k_j) / sqrt(d),  j < n  (n = i+1 causal keys)
 *   m = max s,  e_j = exp(s_j - m),  l = sum e,  Q2 = sum e^2
 *   n_eff = l^2 / Q2 = 1 / sum p_j^2          (inverse Simpson index)
 *   sigma = tau * sigma_k * |q| / sqrt(d),  b = sigma * sqrt(2 ln n)
 *           (floor_order 2: b = sigma * [r - (ln ln n + ln 4 pi)/(2 r)
 *            + gamma / r], r = sqrt(2 ln n), the second-order expected
 *            maximum of n iid N(0,1) (Gumbel location plus the Euler-gamma
 *            mean shift); b = 0 at n = 1)
 *   conf  = sigmoid(m + ln l - b)   (mass on real keys next to a null slot
 *                                    of logit b and value zero)
 *   u     = a / max(|a|, eps),  a = sum p_j v_j       (unit sphere)
 *   count = conf * tanh(ln n_eff / kappa),  kappa = ln T0
 *   out   = u + count * w_count[h] + mem
 *
 * Three forms are provided:
 *   - the definition (two passes per row, the whole logit row held);
 *   - the streamed form (tiles of keys, running max with exp(dm) on l and
 *     acc and exp(2 dm) on Q2: the pages' "squared correction factors");
 *   - split partials merged afterwards (decode split-KV).
 * All are fp64.  Threads split rows; every row is computed independently.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  double log_t0;  /* ln T0 */
  double kappa;   /* tanh-log scale */
  double sigma_k; /* assumed std of a key component under the null */
  double eps;     /* norm guard of the unit-sphere projection */
  int floor_order; /* 1: leading-order null floor, 2: second order */
} oracle_consts;

#define EULER_GAMMA 0.57721566490153286061

/* Per-row streaming state: running reference max m, normaliser l, sum of
 * squares Q2, unnormalised value accumulator acc[d]. */
typedef struct {
  double m, l, q2;
  double* acc;
} row_state;

static double dot(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int x = 0; x < d; ++x) s += a[x] * b[x];
  return s;
}

/* Length temperature (§2.1 item 1): neutral up to T0 keys, log-length
 * sharpening beyond. */
static double temperature(long n, const oracle_consts* c) {
  double t = log((double)n) / c->log_t0;
  return t > 1.0 ? t : 1.0;
}

/* Epilogue shared by every form: given the state over all n keys of the row,
 * produce direction u, n_eff, confidence and count (§2.1 items 1-2). */
static void finish_row(const row_state* st, const double* q, long n, int d,
                       const oracle_consts* c, double* u, double* n_eff,
                       double* conf, double* count) {
  double tau = temperature(n, c);
  /* participation ratio of p_j = e_j / l: 1/sum p^2 = l^2 / Q2 */
  double ne = st->l * st->l / st->q2;
  /* null floor: expected maximum of n iid N(0, sigma^2) noise logits,
   * leading order sigma*sqrt(2 ln n); second order adds the Gumbel
   * location correction and the Euler-gamma mean shift */
  double qn = sqrt(dot(q, q, d));
  double sigma = tau * c->sigma_k * qn / sqrt((double)d);
  double r = sqrt(2.0 * log((double)n));
  double b = sigma * r;
  if (c->floor_order == 2) {
    b = 0.0;
    if (n >= 2)
      b = sigma * (r - (log(log((double)n)) + log(4.0 * M_PI)) / (2.0 * r) + EULER_GAMMA / r);
  }
  double lse = st->m + log(st->l);
  double cf = 1.0 / (1.0 + exp(-(lse - b)));
  /* direction: a = acc / l, projected on the unit sphere */
  double an = 0.0;
  for (int x = 0; x < d; ++x) {
    double a = st->acc[x] / st->l;
    an += a * a;
  }
  an = sqrt(an);
  double den = an > c->eps ? an : c->eps;
  for (int x = 0; x < d; ++x) u[x] = (st->acc[x] / st->l) / den;
  *n_eff = ne;
  *conf = cf;
  *count = cf * tanh(log(ne) / c->kappa);
}

/* Definition form: hold the whole logit row, take the exact max, sum. */
static void state_two_pass(const double* q, const double* K, const double* V,
                           long n, int d, double tau, row_state* st,
                           double* s /* scratch[n] */) {
  double scale = tau / sqrt((double)d);
  double m = -INFINITY;
  for (long j = 0; j < n; ++j) {
    s[j] = scale * dot(q, K + j * d, d);
    if (s[j] > m) m = s[j];
  }
  double l = 0.0, q2 = 0.0;
  memset(st->acc, 0, sizeof(double) * d);
  for (long j = 0; j < n; ++j) {
    double e = exp(s[j] - m);
    l += e;
    q2 += e * e;
    const double* vj = V + j * d;
    for (int x = 0; x < d; ++x) st->acc[x] += e * vj[x];
  }
  st->m = m;
  st->l = l;
  st->q2 = q2;
}

/* Streamed form over keys [j0, j1) in tiles of `tile` keys, continuing the
 * state st (§2.2: streaming accumulators, squared correction factors).
 * tau is the temperature of the full row (it depends on n, not on the tile). */
static void state_stream(const double* q, const double* K, const double* V,
                         long j0, long j1, int d, double tau, long tile,
                         row_state* st) {
  double scale = tau / sqrt((double)d);
  for (long t0 = j0; t0 < j1; t0 += tile) {
    long t1 = t0 + tile < j1 ? t0 + tile : j1;
    double mt = -INFINITY;
    for (long j = t0; j < t1; ++j) {
      double sj = scale * dot(q, K + j * d, d);
      if (sj > mt) mt = sj;
    }
    double mnew = st->m > mt ? st->m : mt;
    double alpha = (st->m == -INFINITY) ? 0.0 : exp(st->m - mnew);
    st->l *= alpha;
    st->q2 *= alpha * alpha; /* squared correction factor */
    for (int x = 0; x < d; ++x) st->acc[x] *= alpha;
    for (long j = t0; j < t1; ++j) {
      double sj = scale * dot(q, K + j * d, d);
      double e = exp(sj - mnew);
      st->l += e;
      st->q2 += e * e;
      const double* vj = V + j * d;
      for (int x = 0; x < d; ++x) st->acc[x] += e * vj[x];
    }
    st->m = mnew;
  }
}

static void state_init(row_state* st) {
  st->m = -INFINITY;
  st->l = 0.0;
  st->q2 = 0.0;
}

/* Merge partial states over disjoint key sets (decode split-KV combine):
 * rebase every partial on the common max M with weight w = exp(m_s - M),
 * w on l and acc, w^2 on Q2. */
static void state_merge(row_state* dst, const row_state* parts, int nparts,
                        int d) {
  double M = -INFINITY;
  for (int s = 0; s < nparts; ++s)
    if (parts[s].m > M) M = parts[s].m;
  dst->m = M;
  dst->l = 0.0;
  dst->q2 = 0.0;
  memset(dst->acc, 0, sizeof(double) * d);
  for (int s = 0; s < nparts; ++s) {
    if (parts[s].m == -INFINITY) continue; /* empty split */
    double w = exp(parts[s].m - M);
    dst->l += w * parts[s].l;
    dst->q2 += w * w * parts[s].q2;
    for (int x = 0; x < d; ++x) dst->acc[x] += w * parts[s].acc[x];
  }
}

/* ---------------------------------------------------------------- rows -- */

typedef struct {
  const double *q, *k, *v, *mem, *w; /* one head: q/k/v/mem [T][d], w [d] */
  int T, d;
  const long* rows; /* query row indices i (n = i + 1 keys) */
  long nrows;
  const oracle_consts* c;
  int mode;  /* 0 definition, 1 streamed */
  long tile; /* tile of the streamed form */
  double *out, *neff, *conf; /* out [nrows][d], neff/conf [nrows] */
  long r0, r1, stride;       /* this worker's rows[]: r0, r0 + stride, ... < r1 */
  int status;
} rows_job;

static void* rows_worker(void* arg) {
  rows_job* jb = (rows_job*)arg;
  int d = jb->d;
  double* s = (double*)malloc(sizeof(double) * (size_t)(jb->T > 0 ? jb->T : 1));
  double* acc = (double*)malloc(sizeof(double) * d);
  double* u = (double*)malloc(sizeof(double) * d);
  if (!s || !acc || !u) {
    jb->status = -2;
    free(s);
    free(acc);
    free(u);
    return NULL;
  }
  for (long r = jb->r0; r < jb->r1; r += jb->stride) {
    long i = jb->rows[r];
    long n = i + 1;
    const double* qi = jb->q + i * d;
    double tau = temperature(n, jb->c);
    row_state st;
    st.acc = acc;
    if (jb->mode == 0) {
      state_two_pass(qi, jb->k, jb->v, n, d, tau, &st, s);
    } else {
      state_init(&st);
      memset(acc, 0, sizeof(double) * d);
      state_stream(qi, jb->k, jb->v, 0, n, d, tau, jb->tile, &st);
    }
    double ne, cf, cnt;
    finish_row(&st, qi, n, d, jb->c, u, &ne, &cf, &cnt);
    double* o = jb->out + r * d;
    const double* mi = jb->mem + i * d;
    for (int x = 0; x < d; ++x) o[x] = u[x] + cnt * jb->w[x] + mi[x];
    jb->neff[r] = ne;
    jb->conf[r] = cf;
  }
  free(s);
  free(acc);
  free(u);
  jb->status = 0;
  return NULL;
}

static int run_rows(rows_job* proto, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (proto->nrows < nthreads) nthreads = proto->nrows > 0 ? (int)proto->nrows : 1;
  rows_job jobs[256];
  pthread_t th[256];
  /* rows are dealt out round-robin (worker t takes rows t, t + nthreads,
   * ...): a causal row's cost grows with its index, so contiguous slices
   * would leave the last worker with most of the work */
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *proto;
    jobs[t].r0 = t;
    jobs[t].r1 = proto->nrows;
    jobs[t].stride = nthreads;
    jobs[t].status = -1;
  }
  if (nthreads == 1) {
    rows_worker(&jobs[0]);
    return jobs[0].status;
  }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, rows_worker, &jobs[t]);
  int st = 0;
  for (int t = 0; t < nthreads; ++t) {
    pthread_join(th[t], NULL);
    if (jobs[t].status != 0) st = jobs[t].status;
  }
  return st;
}

/* Causal prefill rows of ONE head.  rows[r] = query index i; the row sees
 * keys 0..i.  mode 0 = definition, 1 = streamed in tiles of `tile` keys. */
int oracle_polar_rows(const double* q, const double* k, const double* v,
                      const double* mem, const double* w, int T, int d,
                      double log_t0, double kappa, double sigma_k, double eps,
                      int floor_order, const long* rows, long nrows, int mode, long tile,
                      double* out, double* neff, double* conf, int nthreads) {
  if (T < 1 || d < 1 || nrows < 0 || (mode == 1 && tile < 1)) return -1;
  if (floor_order != 1 && floor_order != 2) return -1;
  for (long r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= T) return -1;
  oracle_consts c = {log_t0, kappa, sigma_k, eps, floor_order};
  rows_job jb;
  memset(&jb, 0, sizeof(jb));
  jb.q = q; jb.k = k; jb.v = v; jb.mem = mem; jb.w = w;
  jb.T = T; jb.d = d; jb.rows = rows; jb.nrows = nrows; jb.c = &c;
  jb.mode = mode; jb.tile = tile;
  jb.out = out; jb.neff = neff; jb.conf = conf;
  return run_rows(&jb, nthreads);
}

/* Full causal prefill: q,k,v,mem [B][H][T][d], w [H][d];
 * out [B][H][T][d], neff/conf [B][H][T]. */
int oracle_polar_fwd(const double* q, const double* k, const double* v,
                     const double* mem, const double* w, int B, int H, int T,
                     int d, double log_t0, double kappa, double sigma_k,
                     double eps, int floor_order, int mode, long tile, double* out,
                     double* neff, double* conf, int nthreads) {
  if (B < 0 || H < 0 || T < 1 || d < 1) return -1;
  long* rows = (long*)malloc(sizeof(long) * T);
  if (!rows) return -2;
  for (long i = 0; i < T; ++i) rows[i] = i;
  int st = 0;
  for (long bh = 0; bh < (long)B * H && st == 0; ++bh) {
    long h = bh % H;
    size_t off = (size_t)bh * T * d;
    st = oracle_polar_rows(q + off, k + off, v + off, mem + off, w + h * d, T,
                           d, log_t0, kappa, sigma_k, eps, floor_order, rows, T,
                           mode, tile,
                           out + off, neff + (size_t)bh * T,
                           conf + (size_t)bh * T, nthreads);
  }
  free(rows);
  return st;
}

/* Decode: one query per (b, h) against a cache of Tkv keys, all visible
 * (n = Tkv).  nsplit = 0: definition form over the whole cache.
 * nsplit >= 1: the cache is cut into nsplit contiguous chunks of
 * ceil(Tkv / nsplit) keys, each chunk streamed in tiles of `tile` keys from
 * an empty state, and the partial states merged.
 * q, mem [B][H][d]; k, v [B][H][Tkv][d]; w [H][d]; out [B][H][d];
 * neff, conf [B][H].  Threads take (b, h) problems round-robin. */
typedef struct {
  const double *q, *k, *v, *mem, *w;
  int H, Tkv, d, nsplit;
  long tile;
  const oracle_consts* c;
  double *out, *neff, *conf;
  long bh0, bh1, stride;
  int status;
} decode_job;

static void* decode_worker(void* arg) {
  decode_job* jb = (decode_job*)arg;
  const int d = jb->d, Tkv = jb->Tkv, nsplit = jb->nsplit;
  const double *q = jb->q, *k = jb->k, *v = jb->v, *mem = jb->mem, *w = jb->w;
  const oracle_consts* c = jb->c;
  int ns = nsplit > 0 ? nsplit : 1;
  double* s = (double*)malloc(sizeof(double) * Tkv);
  double* accs = (double*)malloc(sizeof(double) * (size_t)d * (ns + 1));
  row_state* parts = (row_state*)malloc(sizeof(row_state) * ns);
  double* u = (double*)malloc(sizeof(double) * d);
  if (!s || !accs || !parts || !u) {
    free(s); free(accs); free(parts); free(u);
    jb->status = -2;
    return NULL;
  }
  for (long bh = jb->bh0; bh < jb->bh1; bh += jb->stride) {
    long h = bh % jb->H;
    const double* qi = q + bh * d;
    const double* K = k + (size_t)bh * Tkv * d;
    const double* V = v + (size_t)bh * Tkv * d;
    long n = Tkv;
    double tau = temperature(n, c);
    row_state st;
    st.acc = accs + (size_t)d * ns;
    if (nsplit == 0) {
      state_two_pass(qi, K, V, n, d, tau, &st, s);
    } else {
      long chunk = (n + ns - 1) / ns;
      for (int p = 0; p < ns; ++p) {
        parts[p].acc = accs + (size_t)d * p;
        state_init(&parts[p]);
        memset(parts[p].acc, 0, sizeof(double) * d);
        long j0 = (long)p * chunk, j1 = j0 + chunk < n ? j0 + chunk : n;
        if (j0 < j1) state_stream(qi, K, V, j0, j1, d, tau, jb->tile, &parts[p]);
      }
      state_merge(&st, parts, ns, d);
    }
    double ne, cf, cnt;
    finish_row(&st, qi, n, d, c, u, &ne, &cf, &cnt);
    for (int x = 0; x < d; ++x)
      jb->out[bh * d + x] = u[x] + cnt * w[h * d + x] + mem[bh * d + x];
    jb->neff[bh] = ne;
    jb->conf[bh] = cf;
  }
  free(s); free(accs); free(parts); free(u);
  jb->status = 0;
  return NULL;
}

int oracle_polar_decode(const double* q, const double* k, const double* v,
                        const double* mem, const double* w, int B, int H,
                        int Tkv, int d, double log_t0, double kappa,
                        double sigma_k, double eps, int floor_order, int nsplit,
                        long tile, double* out, double* neff, double* conf,
                        int nthreads) {
  if (B < 0 || H < 0 || Tkv < 1 || d < 1 || nsplit < 0 || tile < 1) return -1;
  if (floor_order != 1 && floor_order != 2) return -1;
  oracle_consts c = {log_t0, kappa, sigma_k, eps, floor_order};
  const long nbh = (long)B * H;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nbh < nthreads) nthreads = nbh > 0 ? (int)nbh : 1;
  decode_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    decode_job* jb = &jobs[t];
    jb->q = q; jb->k = k; jb->v = v; jb->mem = mem; jb->w = w;
    jb->H = H; jb->Tkv = Tkv; jb->d = d; jb->nsplit = nsplit; jb->tile = tile;
    jb->c = &c;
    jb->out = out; jb->neff = neff; jb->conf = conf;
    jb->bh0 = t; jb->bh1 = nbh; jb->stride = nthreads;
    jb->status = -1;
  }
  if (nthreads == 1) {
    decode_worker(&jobs[0]);
    return jobs[0].status;
  }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, decode_worker, &jobs[t]);
  int st = 0;
  for (int t = 0; t < nthreads; ++t) {
    pthread_join(th[t], NULL);
    if (jobs[t].status != 0) st = jobs[t].status;
  }
  return st;
}
