/*
 * gdn_oracle.c — fp64 reference of the Gated DeltaNet state path.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library.  It
 * shares no code, header, table or constant with the CUDA engine.
 *
 * Everything here is the plain token-by-token definition, in double precision,
 * in the order the definition states it:
 *
 *   conv  : y[t][c] = SiLU( sum_{i=0..3} w[c][i] * xh[t-3+i][c] ), where xh is
 *           the carried three-row window followed by the new rows (depthwise
 *           causal convolution with a rolling state; "Hybrid linear attention
 *           (gated DeltaNet)", section "Why this family is different", item 1)
 *   norm  : q <- q_scale * q / sqrt(sum q^2 + eps);  k <- k / sqrt(sum k^2 + eps)
 *   step  : S <- a*S - a*b*(S k) k^T + b*v k^T   (= a S (I - b k k^T) + b v k^T,
 *           the gated delta rule of Yang, Kautz and Hatamizadeh, "Gated Delta
 *           Networks", 2024) with a = exp(g)
 *   output: o = S q, taken after the update
 *
 * Checkpoints: after every token whose absolute 1-based position is a multiple
 * of the block size, the state and the conv window are recorded ("Prefix
 * caching on Gated DeltaNet hybrids", section "Why hits were wrong": a full
 * block keeps the state after its last token).
 *
 * Parity pins live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define CONV_K 4

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Pre-conv row tau of one sequence: tau < 0 reads the carried window
 * (win row 3+tau), tau >= 0 reads the new rows. */
static double hist(const double* x, const double* win, int64_t conv_dim, int64_t tau,
                   int64_t c) {
  if (tau < 0) return win[(CONV_K - 1 + tau) * conv_dim + c];
  return x[tau * conv_dim + c];
}

/* One channel of the causal conv followed by SiLU; tap 3 multiplies row t. */
static double conv_silu_channel(const double* x, const double* win, const double* w,
                                int64_t conv_dim, int64_t t, int64_t c) {
  double z = 0.0;
  for (int i = 0; i < CONV_K; ++i) z += w[c * CONV_K + i] * hist(x, win, conv_dim, t - 3 + i, c);
  return silu(z);
}

static void l2norm(double* v, int n, double scale, double eps) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += v[i] * v[i];
  double f = scale / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) v[i] *= f;
}

/* One step of the gated delta rule on S [dv][dk]; writes o [dv]. */
static void delta_step(int dk, int dv, double* S, const double* q, const double* k,
                       const double* v, double a, double b, double* u, double* o) {
  for (int r = 0; r < dv; ++r) {
    double acc = 0.0;
    for (int c = 0; c < dk; ++c) acc += S[r * dk + c] * k[c];
    u[r] = acc;
  }
  for (int r = 0; r < dv; ++r)
    for (int c = 0; c < dk; ++c)
      S[r * dk + c] = a * S[r * dk + c] - a * b * u[r] * k[c] + b * v[r] * k[c];
  for (int r = 0; r < dv; ++r) {
    double acc = 0.0;
    for (int c = 0; c < dk; ++c) acc += S[r * dk + c] * q[c];
    o[r] = acc;
  }
}

/* The bare recurrence over T steps for one head with given (already
 * normalised) q, k [T][dk], v [T][dv] and per-step a, b.  S [dv][dk] is
 * updated in place; o [T][dv]. */
int gdn_oracle_recurrence(int dk, int dv, int64_t T, const double* q, const double* k,
                          const double* v, const double* a, const double* b, double* S,
                          double* o) {
  double* u = (double*)malloc(sizeof(double) * (size_t)dv);
  if (!u) return 1;
  for (int64_t t = 0; t < T; ++t)
    delta_step(dk, dv, S, q + t * dk, k + t * dk, v + t * dv, a[t], b[t], u, o + t * dv);
  free(u);
  return 0;
}

/* Conv + SiLU over all channels: y [T][conv_dim] from x [T][conv_dim], the
 * window [3][conv_dim] and w [conv_dim][4]. */
int gdn_oracle_conv_silu(int64_t conv_dim, int64_t T, const double* x, const double* win,
                         const double* w, double* y) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t c = 0; c < conv_dim; ++c)
      y[t * conv_dim + c] = conv_silu_channel(x, win, w, conv_dim, t, c);
  return 0;
}

int gdn_oracle_l2norm(int n, double* v, double scale, double eps) {
  l2norm(v, n, scale, eps);
  return 0;
}

/* ------------------------------------------------------------------------- */

typedef struct {
  int Hqk, Hv, dk, dv;
  double q_scale, eps;
  int64_t conv_dim, B;
  int32_t N;
  const int64_t *cu, *start;
  const double *x, *g, *beta, *w;
  double *S, *win, *o;
  const int64_t* ck_off;
  double* ck_S;
  int64_t next;  /* work counter */
} job_t;

/* Work item (sequence s, value head h): the whole token loop of one head. */
static void run_item(job_t* J, int64_t item) {
  const int s = (int)(item / J->Hv), h = (int)(item % J->Hv);
  const int dk = J->dk, dv = J->dv, grp = J->Hv / J->Hqk, j = h / grp;
  const int64_t cd = J->conv_dim, t0 = J->cu[s], T = J->cu[s + 1] - t0;
  const double* x = J->x + t0 * cd;
  const double* win = J->win + (int64_t)s * (CONV_K - 1) * cd;
  double* S = J->S + ((int64_t)s * J->Hv + h) * dv * dk;
  const int64_t cq = (int64_t)j * dk, ck = (int64_t)J->Hqk * dk + (int64_t)j * dk,
                cv = 2 * (int64_t)J->Hqk * dk + (int64_t)h * dv;
  double* q = (double*)malloc(sizeof(double) * (size_t)(2 * dk + 2 * dv));
  double* k = q + dk;
  double* v = k + dk;
  double* u = v + dv;
  int64_t nck = 0;
  for (int64_t t = 0; t < T; ++t) {
    for (int c = 0; c < dk; ++c) q[c] = conv_silu_channel(x, win, J->w, cd, t, cq + c);
    for (int c = 0; c < dk; ++c) k[c] = conv_silu_channel(x, win, J->w, cd, t, ck + c);
    for (int c = 0; c < dv; ++c) v[c] = conv_silu_channel(x, win, J->w, cd, t, cv + c);
    l2norm(q, dk, J->q_scale, J->eps);
    l2norm(k, dk, 1.0, J->eps);
    const double a = exp(J->g[(t0 + t) * J->Hv + h]);
    const double b = J->beta[(t0 + t) * J->Hv + h];
    double* o = J->o + ((t0 + t) * J->Hv + h) * dv;
    delta_step(dk, dv, S, q, k, v, a, b, u, o);
    if ((J->start[s] + t + 1) % J->B == 0) {
      double* dst = J->ck_S + ((J->ck_off[s] + nck) * J->Hv + h) * (int64_t)dv * dk;
      memcpy(dst, S, sizeof(double) * (size_t)dv * dk);
      ++nck;
    }
  }
  free(q);
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  const int64_t total = (int64_t)J->N * J->Hv;
  for (;;) {
    int64_t item = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (item >= total) break;
    run_item(J, item);
  }
  return NULL;
}

/* Window after the last token of a sequence prefix: the last three pre-conv
 * rows of [carried window ; x[0..t_end)]. */
static void window_after(const double* x, const double* win0, int64_t cd, int64_t t_end,
                         double* out) {
  for (int r = 0; r < CONV_K - 1; ++r) {
    int64_t tau = t_end - (CONV_K - 1) + r;
    for (int64_t c = 0; c < cd; ++c) out[r * cd + c] = hist(x, win0, cd, tau, c);
  }
}

int gdn_oracle_num_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/* Prefill of N sequences packed along the token axis.
 *   x [T][conv_dim], g/beta [T][Hv], conv_w [conv_dim][4]
 *   S   [N][Hv][dv][dk]  in: initial state, out: final state
 *   win [N][3][conv_dim] in: initial window, out: final window
 *   o   [T][Hv][dv]
 *   ck_off [N+1] prefix sums of the boundaries each sequence crosses;
 *   ck_S [ck_off[N]][Hv][dv][dk] and ck_win [ck_off[N]][3][conv_dim] receive
 *   the checkpoint after every crossed boundary, in order.
 * nthreads <= 0 uses every online core.  Returns 0 on success. */
int gdn_oracle_prefill(int Hqk, int Hv, int dk, int dv, double q_scale, double eps,
                       int32_t N, const int64_t* cu_seqlens, const int64_t* start_pos,
                       int64_t block_size, const double* x, const double* g,
                       const double* beta, const double* conv_w, double* S, double* win,
                       double* o, const int64_t* ck_off, double* ck_S, double* ck_win,
                       int nthreads) {
  if (Hqk <= 0 || Hv % Hqk != 0 || dk <= 0 || dv <= 0 || block_size <= 0 || N < 0) return 1;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.Hqk = Hqk; J.Hv = Hv; J.dk = dk; J.dv = dv; J.q_scale = q_scale; J.eps = eps;
  J.conv_dim = 2 * (int64_t)Hqk * dk + (int64_t)Hv * dv;
  J.B = block_size; J.N = N; J.cu = cu_seqlens; J.start = start_pos;
  J.x = x; J.g = g; J.beta = beta; J.w = conv_w; J.S = S; J.win = win; J.o = o;
  J.ck_off = ck_off; J.ck_S = ck_S; J.next = 0;

  if (nthreads <= 0) nthreads = gdn_oracle_num_threads();
  int64_t items = (int64_t)N * Hv;
  if (nthreads > items) nthreads = (int)(items > 0 ? items : 1);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  int started = 0;
  for (int i = 1; i < nthreads; ++i)
    if (pthread_create(&th[i], NULL, worker, &J) == 0) ++started; else break;
  worker(&J);
  for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
  free(th);

  /* Conv windows: checkpoints first (they read the initial window), then the
   * final window replaces the carried one. */
  const int64_t cd = J.conv_dim, wsz = (CONV_K - 1) * cd;
  double* tmp = (double*)malloc(sizeof(double) * (size_t)wsz);
  for (int32_t s = 0; s < N; ++s) {
    const int64_t t0 = cu_seqlens[s], T = cu_seqlens[s + 1] - t0;
    const double* xs = x + t0 * cd;
    double* w0 = win + (int64_t)s * wsz;
    int64_t nck = 0;
    for (int64_t t = 0; t < T; ++t)
      if ((start_pos[s] + t + 1) % block_size == 0) {
        window_after(xs, w0, cd, t + 1, ck_win + (ck_off[s] + nck) * wsz);
        ++nck;
      }
    window_after(xs, w0, cd, T, tmp);
    memcpy(w0, tmp, sizeof(double) * (size_t)wsz);
  }
  free(tmp);
  return 0;
}
