/*
 * Plain, slow CPU oracle for partitioned attention with attention-state reuse.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's compute path may include, link or call
 * this file; only the test suite, the package's smoke check and the CPU-baseline leg of the
 * benchmark use it. It shares no code with the CUDA path.
 *
 * Source of the method: "DiTango: Cost-Effective Parallel Diffusion Generation with Selective
 * Attention State Reuse" (gist.science/paper/2607.15650), Technical Summary, Methodology:
 *   - 1. Anchor-Guided Selection Planner (compute-or-reuse per partition pair);
 *   - 2. State-Centric Parallel Runtime, "State Composition": an attention state is the pair
 *     (output, log-sum-exp); states combine associatively and commutatively.
 * and, for the optional rotary prologue, "Accelerating Video Generation Inference with
 * Sequential-Parallel 3D Positional Encoding Using a Global Time Index"
 * (gist.science/es/paper/2603.06664), section 2 (Causal-RoPE SP: t_global = t_local + s,
 * precomputed sin/cos), with the three channel groups t / x / y named in "Kaleido"
 * (gist.science/es/paper/2607.13770), Methodology 1.
 *
 * The pages print no formula. The readings used here (each the plainest one consistent with
 * the text) are:
 *   state of query row r against KV partition j:
 *     z_c = scale * <q_r, k_c>  (c in partition j)
 *     lse = m + ln sum_c exp(z_c - m),  m = max_c z_c
 *     O   = sum_c exp(z_c - lse) v_c    (normalised within partition j only)
 *   merge of states (O_s, lse_s):
 *     L = M + ln sum_s exp(lse_s - M), M = max_s lse_s;  O = sum_s exp(lse_s - L) O_s
 *   partitions: contiguous; the first N mod P partitions hold one extra row.
 *   3D RoPE: token n -> (t = n / (Hl*Wl) + s, h = (n / Wl) mod Hl, w = n mod Wl);
 *     channel pair m = (2m, 2m+1); the first dt/2 pairs rotate with t, the next dh/2 with h,
 *     the last dw/2 with w; pair k of an axis of width d_a turns by pos * theta^(-2k/d_a);
 *     (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a), in fp64; for a bf16 (fp32)
 *     configuration the attention reads the rotated q and k stored in that dtype, i.e. the
 *     fp64 rotation rounded once, nearest-even (a bf16 pipeline hands its attention kernel the
 *     output of the fused projection + RoPE step as bf16 tensors: Causal-RoPE SP page,
 *     section 2, operator fusion).
 * All arithmetic is fp64. Inputs arrive as fp64 copies of the values in the config dtype.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- partitioning ------------------------------------------------------------------- */

/* Contiguous partition offsets, offsets[0] = 0, offsets[P] = N. */
void oracle_partition_offsets(int64_t N, int32_t P, int64_t* offsets) {
  int64_t base = N / P, extra = N % P, acc = 0;
  offsets[0] = 0;
  for (int32_t p = 0; p < P; ++p) {
    acc += base + (p < extra ? 1 : 0);
    offsets[p + 1] = acc;
  }
}

/* ---- rounding to the storage dtypes --------------------------------------------------- */

/* Round a double to the nearest bfloat16 value (ties to even), returned as a double.
 * Written from the format's definition: 8 significant bits, exponent range of fp32. */
double oracle_round_bf16(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  double m = frexp(fabs(x), &e); /* |x| = m * 2^e, m in [0.5, 1) */
  int exp_unbiased = e - 1;      /* |x| = (2m) * 2^(e-1), 2m in [1,2) */
  int q;                          /* quantum exponent: spacing of bf16 values near x */
  if (exp_unbiased < -126) {
    q = -126 - 7; /* subnormal range: fixed spacing 2^-133 */
  } else {
    q = exp_unbiased - 7;
  }
  double scaled = ldexp(fabs(x), -q);
  double r = nearbyint(scaled); /* default rounding mode: to nearest, ties to even */
  double y = ldexp(r, q);
  if (y > 3.3895313892515355e38) y = INFINITY; /* above max bf16 (0x7F7F) rounds to inf */
  return x < 0 ? -y : y;
}

double oracle_round_f32(double x) { return (double)(float)x; }

static double round_to(double x, int mode) {
  if (mode == 1) return oracle_round_bf16(x);
  if (mode == 2) return oracle_round_f32(x);
  return x;
}

/* ---- 3D rotary embedding -------------------------------------------------------------- */

/* Rotate one d-vector x at position (t, h, w) into y. */
void oracle_rope_rotate(const double* x, double* y, int32_t d, int32_t dt, int32_t dh, int32_t dw,
                        int64_t t, int64_t h, int64_t w, double theta) {
  int32_t pairs = d / 2;
  for (int32_t m = 0; m < pairs; ++m) {
    int64_t pos;
    int32_t k, width;
    if (m < dt / 2) {
      pos = t; k = m; width = dt;
    } else if (m < dt / 2 + dh / 2) {
      pos = h; k = m - dt / 2; width = dh;
    } else {
      pos = w; k = m - dt / 2 - dh / 2; width = dw;
    }
    double ang = (double)pos * pow(theta, -2.0 * (double)k / (double)width);
    double c = cos(ang), s = sin(ang);
    double x0 = x[2 * m], x1 = x[2 * m + 1];
    y[2 * m] = x0 * c - x1 * s;
    y[2 * m + 1] = x0 * s + x1 * c;
  }
  (void)dw;
}

typedef struct {
  const double* x;
  double* y;
  int64_t B, N, H;
  int32_t d, dt, dh, dw;
  int64_t Hl, Wl, s;
  double theta;
  int round_mode;
  int64_t tok_begin, tok_end; /* over B*N tokens */
} rope_job;

static void* rope_worker(void* arg) {
  rope_job* jb = (rope_job*)arg;
  for (int64_t bn = jb->tok_begin; bn < jb->tok_end; ++bn) {
    int64_t n = bn % jb->N;
    int64_t t = n / (jb->Hl * jb->Wl) + jb->s;
    int64_t h = (n / jb->Wl) % jb->Hl;
    int64_t w = n % jb->Wl;
    for (int64_t hd = 0; hd < jb->H; ++hd) {
      const double* xv = jb->x + (bn * jb->H + hd) * jb->d;
      double* yv = jb->y + (bn * jb->H + hd) * jb->d;
      oracle_rope_rotate(xv, yv, jb->d, jb->dt, jb->dh, jb->dw, t, h, w, jb->theta);
      for (int32_t e = 0; e < jb->d; ++e) yv[e] = round_to(yv[e], jb->round_mode);
    }
  }
  return NULL;
}

/* Rotate a [B, N, H, d] tensor in fp64. round_mode: 0 keep fp64, 1 round to bf16, 2 round to
 * fp32 (the attention inputs are the rotated tensors stored in the config dtype: one rounding of
 * the fp64 rotation, nearest-even). */
void oracle_rope_apply(const double* x, double* y, int64_t B, int64_t N, int64_t H, int32_t d,
                       int32_t dt, int32_t dh, int32_t dw, int64_t Hl, int64_t Wl, int64_t s,
                       double theta, int32_t round_mode, int32_t nthreads) {
  if (nthreads < 1) nthreads = 1;
  int64_t total = B * N;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  rope_job* jobs = (rope_job*)malloc(sizeof(rope_job) * (size_t)nthreads);
  for (int32_t i = 0; i < nthreads; ++i) {
    rope_job jb = {x, y, B, N, H, d, dt, dh, dw, Hl, Wl, s, theta, round_mode,
                   total * i / nthreads, total * (i + 1) / nthreads};
    jobs[i] = jb;
    pthread_create(&th[i], NULL, rope_worker, &jobs[i]);
  }
  for (int32_t i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  free(th);
  free(jobs);
}

/* ---- attention state of one query row against one KV partition ------------------------- */

/* q: d values; k, v: rows [c0, c1) of a [N, H, d]-strided head slice, row stride `rs`.
 * Writes O (d values) and lse. `z` is scratch of at least (c1 - c0) doubles. */
void oracle_pair_state(const double* q, const double* k, const double* v, int64_t rs, int64_t c0,
                       int64_t c1, int32_t d, double scale, double* z, double* O, double* lse) {
  double m = -INFINITY;
  for (int64_t c = c0; c < c1; ++c) {
    const double* kc = k + c * rs;
    double acc = 0.0;
    for (int32_t e = 0; e < d; ++e) acc += q[e] * kc[e];
    z[c - c0] = scale * acc;
    if (z[c - c0] > m) m = z[c - c0];
  }
  double sum = 0.0;
  for (int64_t c = c0; c < c1; ++c) sum += exp(z[c - c0] - m);
  double L = m + log(sum);
  for (int32_t e = 0; e < d; ++e) O[e] = 0.0;
  for (int64_t c = c0; c < c1; ++c) {
    double p = exp(z[c - c0] - L);
    const double* vc = v + c * rs;
    for (int32_t e = 0; e < d; ++e) O[e] += p * vc[e];
  }
  *lse = L;
}

/* ---- merge of attention states ---------------------------------------------------------- */

/* Merge n states (O_s: n x d row-major, lse_s: n) into (O, lse). */
void oracle_merge(const double* O_s, const double* lse_s, int32_t n, int32_t d, double* O,
                  double* lse) {
  double M = -INFINITY;
  for (int32_t s = 0; s < n; ++s)
    if (lse_s[s] > M) M = lse_s[s];
  double sum = 0.0;
  for (int32_t s = 0; s < n; ++s) sum += exp(lse_s[s] - M);
  double L = M + log(sum);
  for (int32_t e = 0; e < d; ++e) O[e] = 0.0;
  for (int32_t s = 0; s < n; ++s) {
    double w = exp(lse_s[s] - L);
    for (int32_t e = 0; e < d; ++e) O[e] += w * O_s[(int64_t)s * d + e];
  }
  *lse = L;
}

/* ---- one step over a list of query rows ------------------------------------------------- */

typedef struct {
  /* inputs: fp64 [B, N, H, d] (q and k already rotated if the config rotates them) */
  const double *q, *k, *v;
  int64_t B, N, H;
  int32_t d, P;
  const int64_t* offsets; /* P + 1 */
  const uint8_t* reuse;   /* P x P, 1 = reuse the cached state */
  double scale;
  /* rows: nrows triples (b, h, r) */
  const int64_t* rows;
  int64_t nrows;
  /* per-row state cache: O [nrows, P, d], lse [nrows, P]; persists across steps */
  double *cache_O, *cache_lse;
  int32_t cache_round; /* rounding of a stored O: 0 none (lse kept too), 1 bf16, 2 fp32;
                        * with 1 or 2 the stored lse is rounded to fp32 */
  /* outputs: fresh states of this step [nrows, P, d] / [nrows, P] (NaN where reused),
   * merged out [nrows, d], out_lse [nrows] */
  double *fresh_O, *fresh_lse, *out, *out_lse;
  int64_t row_begin, row_end;
} step_job;

static int32_t partition_of(const int64_t* offsets, int32_t P, int64_t r) {
  int32_t lo = 0, hi = P - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) / 2;
    if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

static void* step_worker(void* arg) {
  step_job* jb = (step_job*)arg;
  const int32_t d = jb->d, P = jb->P;
  int64_t maxn = 0;
  for (int32_t p = 0; p < P; ++p) {
    int64_t n = jb->offsets[p + 1] - jb->offsets[p];
    if (n > maxn) maxn = n;
  }
  double* z = (double*)malloc(sizeof(double) * (size_t)(maxn > 0 ? maxn : 1));
  double* Ost = (double*)malloc(sizeof(double) * (size_t)P * (size_t)d);
  double* lst = (double*)malloc(sizeof(double) * (size_t)P);
  const int64_t rs = jb->H * d; /* row stride of one head inside [N, H, d] */
  for (int64_t ri = jb->row_begin; ri < jb->row_end; ++ri) {
    int64_t b = jb->rows[3 * ri], h = jb->rows[3 * ri + 1], r = jb->rows[3 * ri + 2];
    int32_t i = partition_of(jb->offsets, P, r);
    const double* qr = jb->q + ((b * jb->N + r) * jb->H + h) * d;
    const double* kb = jb->k + (b * jb->N * jb->H + h) * d;
    const double* vb = jb->v + (b * jb->N * jb->H + h) * d;
    double* cO = jb->cache_O + ri * P * d;
    double* cl = jb->cache_lse + ri * P;
    for (int32_t j = 0; j < P; ++j) {
      double* fO = jb->fresh_O + (ri * P + j) * d;
      if (jb->reuse[i * P + j]) {
        for (int32_t e = 0; e < d; ++e) fO[e] = NAN;
        jb->fresh_lse[ri * P + j] = NAN;
        continue; /* the cached state of an earlier step stands */
      }
      double lse;
      oracle_pair_state(qr, kb, vb, rs, jb->offsets[j], jb->offsets[j + 1], d, jb->scale, z, fO,
                        &lse);
      jb->fresh_lse[ri * P + j] = lse;
      for (int32_t e = 0; e < d; ++e) cO[j * d + e] = round_to(fO[e], jb->cache_round);
      cl[j] = jb->cache_round ? oracle_round_f32(lse) : lse; /* a stored lse is fp32 */
    }
    for (int32_t j = 0; j < P; ++j) {
      for (int32_t e = 0; e < d; ++e) Ost[j * d + e] = cO[j * d + e];
      lst[j] = cl[j];
    }
    oracle_merge(Ost, lst, P, d, jb->out + ri * d, jb->out_lse + ri);
  }
  free(z);
  free(Ost);
  free(lst);
  return NULL;
}

/* One step of partitioned attention with reuse for the listed rows. Every pair (i, j) with
 * reuse[i][j] == 0 is computed from this step's inputs and written to the row's cache; every
 * other pair keeps the cached state; then all P cached states of the row are merged. */
void oracle_rows_step(const double* q, const double* k, const double* v, int64_t B, int64_t N,
                      int64_t H, int32_t d, int32_t P, const int64_t* offsets,
                      const uint8_t* reuse, double scale, const int64_t* rows, int64_t nrows,
                      double* cache_O, double* cache_lse, int32_t cache_round, double* fresh_O,
                      double* fresh_lse, double* out, double* out_lse, int32_t nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nrows) nthreads = (int32_t)(nrows > 0 ? nrows : 1);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  step_job* jobs = (step_job*)malloc(sizeof(step_job) * (size_t)nthreads);
  for (int32_t t = 0; t < nthreads; ++t) {
    step_job jb = {q, k, v, B, N, H, d, P, offsets, reuse, scale, rows, nrows, cache_O,
                   cache_lse, cache_round, fresh_O, fresh_lse, out, out_lse,
                   nrows * t / nthreads, nrows * (t + 1) / nthreads};
    jobs[t] = jb;
    pthread_create(&th[t], NULL, step_worker, &jobs[t]);
  }
  for (int32_t t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
}

/* Elementwise rounding of an array (mode 1: bf16, 2: fp32), in place. */
void oracle_round_array(double* x, int64_t n, int32_t mode) {
  for (int64_t i = 0; i < n; ++i) x[i] = round_to(x[i], mode);
}
