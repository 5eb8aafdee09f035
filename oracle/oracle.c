/*
 * oracle.c -- plain, slow, float64 CPU reference for the DLR / S5 hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's product path links, calls or
 * includes this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header, table or constant with the CUDA path.
 *
 * Every routine is the plain definition, in the pages' order, with no blocking, fusion or
 * reordering. Float32 inputs are promoted to double on read; all arithmetic is double.
 *
 * Sources (cited by page title and section):
 *  - "Simplifying and Understanding State Space Models with Diagonal Linear RNNs"
 *    section 2 (DLR, Eq. 1 recurrence, Eq. 3/4 kernel K_j = sum_i w_i lambda_i^j and the
 *    Re cast y_k = sum_{j<=k} Re(K_j) u_{k-j}), section 2.1 (DLR-prod cast Re(K)*Im(K),
 *    bidirectional DLR as the sum of two independent DLRs), section 2.2 (lambda =
 *    exp(-(log Lambda)_re^2 + i (log Lambda)_im)).
 *  - "Simplified State Space Layers for Sequence Modeling" section 2.2 (the linear
 *    recurrence x_k = Abar x_{k-1} + Bbar u_k as a scan) and section 3 (diagonal MIMO
 *    system with B~, C~, diagonal D).
 *
 * Threads: independent (b, h) rows may run on separate pthreads; each row is computed by
 * exactly the same sequential loop whatever the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct { double re, im; } cplx;

static inline cplx c_mul(cplx a, cplx b) {
  cplx r = {a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
  return r;
}
static inline cplx c_add(cplx a, cplx b) {
  cplx r = {a.re + b.re, a.im + b.im};
  return r;
}

/* lambda = exp(-(log Lambda)_re^2 + i (log Lambda)_im)   [DLR paper, section 2.2] */
static inline cplx dlr_lambda(float a, float theta) {
  double ad = (double)a, td = (double)theta;
  double mag = exp(-ad * ad);
  cplx r = {mag * cos(td), mag * sin(td)};
  return r;
}

void orc_lambda(int64_t H, int64_t N, const float* log_re, const float* log_im,
                double* lam /* [H, N, 2] */) {
  for (int64_t i = 0; i < H * N; ++i) {
    cplx l = dlr_lambda(log_re[i], log_im[i]);
    lam[2 * i] = l.re;
    lam[2 * i + 1] = l.im;
  }
}

/*
 * Convolution kernel K_j = sum_n W_n lambda_n^j, j = 0..L-1, per channel h  [DLR paper,
 * section 2, Eq. 3/4]. The power lambda^j is formed by the recurrence p <- p * lambda.
 * cast: 0 -> Re K_j ; 1 -> Re K_j * Im K_j (DLR-prod) ; 2 -> complex K written as [H, L, 2].
 */
void orc_dlr_kernel(int64_t H, int64_t N, int64_t L, const float* log_re, const float* log_im,
                    const float* W, int cast, double* K) {
  cplx* acc = (cplx*)calloc((size_t)L, sizeof(cplx));
  for (int64_t h = 0; h < H; ++h) {
    memset(acc, 0, (size_t)L * sizeof(cplx));
    for (int64_t n = 0; n < N; ++n) {
      int64_t i = h * N + n;
      cplx lam = dlr_lambda(log_re[i], log_im[i]);
      cplx w = {(double)W[2 * i], (double)W[2 * i + 1]};
      cplx p = {1.0, 0.0};
      for (int64_t j = 0; j < L; ++j) {
        acc[j] = c_add(acc[j], c_mul(w, p));
        p = c_mul(p, lam);
      }
    }
    for (int64_t j = 0; j < L; ++j) {
      if (cast == 0) K[h * L + j] = acc[j].re;
      else if (cast == 1) K[h * L + j] = acc[j].re * acc[j].im;
      else { K[2 * (h * L + j)] = acc[j].re; K[2 * (h * L + j) + 1] = acc[j].im; }
    }
  }
  free(acc);
}

/* ---------------------------------------------------------------------------------------- */
/* Row-parallel driver                                                                         */

typedef void (*row_fn)(void* ctx, int64_t row);
typedef struct { row_fn fn; void* ctx; int64_t begin, end; } row_job;

static void* row_worker(void* arg) {
  row_job* j = (row_job*)arg;
  for (int64_t r = j->begin; r < j->end; ++r) j->fn(j->ctx, r);
  return NULL;
}

static void run_rows(row_fn fn, void* ctx, int64_t rows, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > rows) nthreads = (int)(rows > 0 ? rows : 1);
  if (nthreads == 1) {
    for (int64_t r = 0; r < rows; ++r) fn(ctx, r);
    return;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  row_job* jobs = (row_job*)malloc(sizeof(row_job) * (size_t)nthreads);
  int64_t per = (rows + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].begin = t * per < rows ? t * per : rows;
    jobs[t].end = (t + 1) * per < rows ? (t + 1) * per : rows;
    pthread_create(&th[t], NULL, row_worker, &jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
}

/* ---------------------------------------------------------------------------------------- */
/*
 * DLR recurrence with the Re cast [DLR paper, section 2, Eq. 1 and the Re cast]:
 *   x_{n,k} = lambda_n x_{n,k-1} + u_k        (input vector all ones, x_{-1} = x0 or 0)
 *   y_k     = sum_n Re(w_n x_{n,k})
 * u, y: [B, H, L] (y double). x0, xT: [B, H, N, 2] or NULL (initial / final state).
 */
typedef struct {
  int64_t B, H, N, L;
  const float *u, *log_re, *log_im, *W;
  const double* x0;
  double *y, *xT;
} rec_ctx;

static void rec_row(void* vctx, int64_t row) {
  rec_ctx* c = (rec_ctx*)vctx;
  int64_t h = row % c->H;
  const float* u = c->u + row * c->L;
  double* y = c->y + row * c->L;
  cplx* x = (cplx*)malloc(sizeof(cplx) * (size_t)c->N);
  cplx* lam = (cplx*)malloc(sizeof(cplx) * (size_t)c->N);
  cplx* w = (cplx*)malloc(sizeof(cplx) * (size_t)c->N);
  for (int64_t n = 0; n < c->N; ++n) {
    int64_t i = h * c->N + n;
    lam[n] = dlr_lambda(c->log_re[i], c->log_im[i]);
    w[n].re = c->W[2 * i];
    w[n].im = c->W[2 * i + 1];
    if (c->x0) {
      x[n].re = c->x0[2 * (row * c->N + n)];
      x[n].im = c->x0[2 * (row * c->N + n) + 1];
    } else {
      x[n].re = 0.0;
      x[n].im = 0.0;
    }
  }
  for (int64_t k = 0; k < c->L; ++k) {
    double uk = (double)u[k];
    double yk = 0.0;
    for (int64_t n = 0; n < c->N; ++n) {
      cplx xn = c_mul(lam[n], x[n]);
      xn.re += uk;
      x[n] = xn;
      yk += w[n].re * xn.re - w[n].im * xn.im;
    }
    y[k] = yk;
  }
  if (c->xT)
    for (int64_t n = 0; n < c->N; ++n) {
      c->xT[2 * (row * c->N + n)] = x[n].re;
      c->xT[2 * (row * c->N + n) + 1] = x[n].im;
    }
  free(x);
  free(lam);
  free(w);
}

void orc_dlr_recurrence(int64_t B, int64_t H, int64_t N, int64_t L, const float* u,
                        const float* log_re, const float* log_im, const float* W,
                        const double* x0, double* y, double* xT, int nthreads) {
  rec_ctx c = {B, H, N, L, u, log_re, log_im, W, x0, y, xT};
  run_rows(rec_row, &c, B * H, nthreads);
}

/*
 * Direct causal Toeplitz product y_k = sum_{j=0}^{k} kappa_{h,j} u_{k-j}  [DLR paper,
 * section 2: y_k = sum_{j<=k} Re(K_j) u_{k-j}; with kappa = Re K * Im K for DLR-prod].
 * u: [B, H, L] float; kappa: [H, L] double; y: [B, H, L] double (overwritten).
 */
typedef struct {
  int64_t H, L;
  const float* u;
  const double* kappa;
  double* y;
} toe_ctx;

static void toe_row(void* vctx, int64_t row) {
  toe_ctx* c = (toe_ctx*)vctx;
  int64_t h = row % c->H;
  const float* u = c->u + row * c->L;
  const double* kap = c->kappa + h * c->L;
  double* y = c->y + row * c->L;
  for (int64_t k = 0; k < c->L; ++k) {
    double s = 0.0;
    for (int64_t j = 0; j <= k; ++j) s += kap[j] * (double)u[k - j];
    y[k] = s;
  }
}

void orc_toeplitz_causal(int64_t B, int64_t H, int64_t L, const float* u, const double* kappa,
                         double* y, int nthreads) {
  toe_ctx c = {H, L, u, kappa, y};
  run_rows(toe_row, &c, B * H, nthreads);
}

/*
 * Diagonal complex recurrence over a precomputed drive v [S5 paper, section 2.2]:
 *   x_k = abar (.) x_{k-1} + v_k,  x_{-1} = 0;  k = 0..T-1, P states.
 * abar: [P, 2]; v, x: [T, P, 2] (double).
 */
void orc_diag_scan(int64_t T, int64_t P, const double* abar, const double* v, double* x) {
  for (int64_t p = 0; p < P; ++p) {
    cplx a = {abar[2 * p], abar[2 * p + 1]};
    cplx s = {0.0, 0.0};
    for (int64_t k = 0; k < T; ++k) {
      cplx vk = {v[2 * (k * P + p)], v[2 * (k * P + p) + 1]};
      s = c_add(c_mul(a, s), vk);
      x[2 * (k * P + p)] = s.re;
      x[2 * (k * P + p) + 1] = s.im;
    }
  }
}

/* The same scan with a multiplier that changes from step to step: x_k = abar_k x_{k-1} + v_k,
 * abar and v [T, P, 2]. */
void orc_diag_scan_tv(int64_t T, int64_t P, const double* abar, const double* v, double* x) {
  for (int64_t p = 0; p < P; ++p) {
    cplx s = {0.0, 0.0};
    for (int64_t k = 0; k < T; ++k) {
      cplx a = {abar[2 * (k * P + p)], abar[2 * (k * P + p) + 1]};
      cplx vk = {v[2 * (k * P + p)], v[2 * (k * P + p) + 1]};
      s = c_add(c_mul(a, s), vk);
      x[2 * (k * P + p)] = s.re;
      x[2 * (k * P + p) + 1] = s.im;
    }
  }
}

int orc_version(void) { return 1; }
