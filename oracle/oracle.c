/*
 * oracle.c -- plain float64 CPU oracle for the forward selective scan of a diagonal,
 * complex-valued, input-dependent linear recurrence.
 *
 * TEST INFRASTRUCTURE ONLY. This is the slow, obviously-correct definition that the CUDA
 * path is checked against. Only the tests, the smoke check and the bench's CPU-baseline leg
 * load it. It shares no code, header, table or helper with the CUDA library, and the CUDA
 * library never calls it: there is no CPU fallback built from this file.
 *
 * Sources (pages of the reference material, by title and section):
 *  - "Complex parallel scan" (fengwang.github.io, 2026-06-14), section 并行扫描的数学本质
 *    ("the mathematical essence of parallel scan"): the one-step operator O_t = (A_t, B_t x_t)
 *    acting as h -> A_t h + B_t x_t, the combine O_{t+1} (x) O_t, its associativity, and the
 *    remark that nothing in the derivation needs real numbers.
 *  - "Mamba-3 paper story" (ai.tomabc.com), the discretisation table (rows Exp-Euler and
 *    Exp-Trapezoidal: alpha_t, beta_t, gamma_t) and the section on the complex state space
 *    (real decay A times an input-dependent phase e^{i theta}).
 *  - "状态空间模型的对偶谱理论 2026" (blog.lonae.com), section 3.2, the sequential pseudocode listing
 *    (update h first, then read y from the updated h, summing over the state index).
 *  - "Mamba-3: 选择性状态空间模型的下一代架构" (metaphor-xennon), sections 2.1-2.2:
 *    y = C h + D x.
 *
 * Readings taken where the pages are silent or garbled (the full list is kept with the
 * design notes):
 *  - a_t = exp(dt[b,t,d] * A[d,n] + i * theta[b,t,n]); theta is not scaled by dt.
 *  - exp-Euler:      h_t = a_t h_{t-1} + dt_t Bc_t x_t                              (gamma = dt)
 *  - exp-trapezoid:  h_t = a_t h_{t-1} + (1-lam_t) dt_t a_t Bc_{t-1} x_{t-1}
 *                                      + lam_t dt_t Bc_t x_t,  Bc_{-1} x_{-1} = 0
 *    (beta_t = (1-lam_t) dt_t exp(dt_t A_t), where the exponential is the full complex
 *     a_t, rotation included, and dt is the current step's).
 *  - y[b,t,d] = Re(sum_n Cc[b,t,n] h_t[n]) + Dskip[d] x[b,t,d], from the updated h_t,
 *    with no conjugation.
 *  - the state before t = 0 is zero unless an initial state is passed in.
 *
 * Layouts (all row-major, float64; complex values interleaved re, im):
 *   x, dt, y : (B, L, D)        Bc, Cc : (B, L, N) complex      theta : (B, L, N)
 *   lam      : (B, L)           A      : (D, N) real            Dskip : (D)
 *   h0, h_last : (B, D, N) complex     x_prev : (B, D)     Bc_prev : (B, N) complex
 *   h_traj   : (B, L, D, N) complex
 */
#include <complex.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

typedef double complex cplx;

static cplx load_c(const double* p, int64_t i) { return p[2 * i] + I * p[2 * i + 1]; }
static void store_c(double* p, int64_t i, cplx v) { p[2 * i] = creal(v); p[2 * i + 1] = cimag(v); }

/* The transition factor a_t = exp(dt A + i theta): a real decay times a phase rotation
 * ("Mamba-3 paper story", complex state space section; alpha_t = exp(dt_t A_t) in its
 * discretisation table). */
static cplx transition(double dt, double A, double theta) { return cexp(dt * A + I * theta); }

/* The one-step operator O_t = (a_t, u_t) with h_t = a_t h_{t-1} + u_t ("Complex parallel
 * scan", section 并行扫描的数学本质). u_t is the input injected at step t:
 *   mode 0 (exp-Euler, gamma_t = dt_t):  u_t = dt_t x_t Bc_t
 *   mode 1 (exp-trapezoidal): u_t = beta_t Bc_{t-1} x_{t-1} + gamma_t Bc_t x_t with
 *          beta_t = (1 - lam_t) dt_t a_t and gamma_t = lam_t dt_t
 * ("Mamba-3 paper story", discretisation table). x_prev and B_prev are step t-1's input;
 * callers pass zero for them at the start of the sequence.
 * out = {Re a, Im a, Re u, Im u}. */
void oracle_operator(int mode, double dt, double A, double theta, double lam, double x, double x_prev,
                     const double* B, const double* B_prev, double* out) {
  cplx a = transition(dt, A, theta);         /* alpha_t */
  cplx v = (B[0] + I * B[1]) * x;            /* Bc_t x_t */
  cplx u;
  if (mode == 0) {
    double gamma = dt;
    u = gamma * v;
  } else {
    cplx v_prev = (B_prev[0] + I * B_prev[1]) * x_prev;   /* Bc_{t-1} x_{t-1} */
    cplx beta = (1.0 - lam) * dt * a;
    double gamma = lam * dt;
    u = beta * v_prev + gamma * v;
  }
  out[0] = creal(a); out[1] = cimag(a); out[2] = creal(u); out[3] = cimag(u);
}

/* The combine O2 (x) O1 = (a2 a1, a2 u1 + u2): applying O1 and then O2 equals applying the
 * combined operator once ("Complex parallel scan", section 并行扫描的数学本质). The diagonal
 * case, so a is a complex scalar per state. op = {Re a, Im a, Re u, Im u}. */
void oracle_combine(const double* op2, const double* op1, double* out) {
  cplx a2 = op2[0] + I * op2[1], u2 = op2[2] + I * op2[3];
  cplx a1 = op1[0] + I * op1[1], u1 = op1[2] + I * op1[3];
  cplx a = a2 * a1, u = a2 * u1 + u2;
  out[0] = creal(a); out[1] = cimag(a); out[2] = creal(u); out[3] = cimag(u);
}

/* O(h) = a h + u. */
void oracle_apply(const double* op, const double* h, double* out) {
  cplx a = op[0] + I * op[1], u = op[2] + I * op[3], hh = h[0] + I * h[1];
  cplx r = a * hh + u;
  out[0] = creal(r); out[1] = cimag(r);
}

typedef struct {
  const double *x, *dt, *A, *Bc, *Cc, *theta, *lam, *Dskip, *h0, *x_prev, *Bc_prev;
  double *y, *h_last, *h_traj;
  int64_t B, L, D, N;
  int mode;
  int64_t row_begin, row_step;
} job_t;

/* One (b, d) row: the sequential recurrence over t for every state n, then the output.
 * Loop form as in the sequential pseudocode listing of "状态空间模型的对偶谱理论 2026", section 3.2:
 * h is updated first and y_t is read from the updated h_t, summed over n; the D-skip term
 * follows "Mamba-3: 选择性状态空间模型的下一代架构", section 2.2 (y = C h + D x). */
static void run_row(const job_t* j, int64_t b, int64_t d, cplx* h) {
  const int64_t L = j->L, D = j->D, N = j->N;
  for (int64_t n = 0; n < N; ++n) h[n] = j->h0 ? load_c(j->h0, (b * D + d) * N + n) : 0.0;
  for (int64_t t = 0; t < L; ++t) {
    const int64_t td = (b * L + t) * D + d;
    const double xt = j->x[td], dtt = j->dt[td];
    double x_prev = 0.0;
    if (t > 0) x_prev = j->x[td - D];
    else if (j->x_prev) x_prev = j->x_prev[b * D + d];
    const double lam = j->mode == 1 ? j->lam[b * L + t] : 0.0;
    double acc = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const int64_t tn = (b * L + t) * N + n;
      double B_prev[2] = {0.0, 0.0};
      if (t > 0) { B_prev[0] = j->Bc[2 * (tn - N)]; B_prev[1] = j->Bc[2 * (tn - N) + 1]; }
      else if (j->Bc_prev) { B_prev[0] = j->Bc_prev[2 * (b * N + n)]; B_prev[1] = j->Bc_prev[2 * (b * N + n) + 1]; }
      double op[4];
      oracle_operator(j->mode, dtt, j->A[d * N + n], j->theta[tn], lam, xt, x_prev, &j->Bc[2 * tn], B_prev, op);
      h[n] = (op[0] + I * op[1]) * h[n] + (op[2] + I * op[3]);
      acc += creal(load_c(j->Cc, tn) * h[n]);
      if (j->h_traj) store_c(j->h_traj, td * N + n, h[n]);
    }
    j->y[td] = acc + j->Dskip[d] * xt;
  }
  if (j->h_last)
    for (int64_t n = 0; n < N; ++n) store_c(j->h_last, (b * j->D + d) * N + n, h[n]);
}

static void* worker(void* arg) {
  const job_t* j = (const job_t*)arg;
  cplx* h = (cplx*)malloc(sizeof(cplx) * (size_t)(j->N > 0 ? j->N : 1));
  if (!h) return (void*)1;
  for (int64_t r = j->row_begin; r < j->B * j->D; r += j->row_step) run_row(j, r / j->D, r % j->D, h);
  free(h);
  return NULL;
}

int oracle_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/* Forward scan over all (b, d) rows, rows split across `nthreads` POSIX threads (<= 0: all
 * online cores). The split is over independent rows only; each row is computed exactly as
 * run_row states. h0, x_prev, Bc_prev, h_last and h_traj may be NULL (zero initial state and
 * halo; outputs not wanted). lam may be NULL in mode 0.
 * Returns the number of threads used (> 0), or a negative value on bad arguments. */
int oracle_forward(const double* x, const double* dt, const double* A, const double* Bc, const double* Cc,
                   const double* theta, const double* lam, const double* Dskip, const double* h0,
                   const double* x_prev, const double* Bc_prev, double* y, double* h_last, double* h_traj,
                   int64_t B, int64_t L, int64_t D, int64_t N, int mode, int nthreads) {
  if (B < 0 || L < 0 || D < 0 || N < 0) return -1;
  if (mode != 0 && mode != 1) return -2;
  if (mode == 1 && !lam && B * L > 0) return -3;
  if (nthreads <= 0) nthreads = oracle_default_threads();
  if ((int64_t)nthreads > B * D) nthreads = (int)(B * D > 0 ? B * D : 1);
  job_t base = {x, dt, A, Bc, Cc, theta, lam, Dskip, h0, x_prev, Bc_prev, y, h_last, h_traj, B, L, D, N, mode, 0, 1};
  if (nthreads == 1) {
    if (worker(&base)) return -4;
    return 1;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nthreads);
  if (!th || !jobs) { free(th); free(jobs); return -4; }
  int rc = 0, started = 0;
  for (int i = 0; i < nthreads; ++i) {
    jobs[i] = base;
    jobs[i].row_begin = i;
    jobs[i].row_step = nthreads;
    if (pthread_create(&th[i], NULL, worker, &jobs[i]) != 0) { rc = -5; break; }
    ++started;
  }
  for (int i = 0; i < started; ++i) {
    void* ret = NULL;
    pthread_join(th[i], &ret);
    if (ret) rc = -4;
  }
  free(th);
  free(jobs);
  return rc < 0 ? rc : nthreads;
}
