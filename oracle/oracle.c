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
 *  - zero-order hold (mode 2): h_t = a_t h_{t-1} + dt_t (e^{z_t} - 1)/z_t Bc_t x_t, z_t the
 *    exponent of a_t (the rotation included, as for beta_t)
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
 *   mode 2 (zero-order hold): u_t = gamma_t Bc_t x_t, gamma_t = dt_t (e^{z_t} - 1) / z_t,
 *          z_t = dt_t A + i theta_t
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
  } else if (mode == 1) {
    cplx v_prev = (B_prev[0] + I * B_prev[1]) * x_prev;   /* Bc_{t-1} x_{t-1} */
    cplx beta = (1.0 - lam) * dt * a;
    double gamma = lam * dt;
    u = beta * v_prev + gamma * v;
  } else {
    /* mode 2, zero-order hold: gamma = A^{-1}(exp(dt A) - I) ("Mamba-3 paper story",
     * discretisation table, row ZOH; the same B-bar in "Complex parallel scan", section
     * 硬件落地的挑战), with the complex exponent z = dt A + i theta in place of dt A as for
     * alpha_t: gamma = dt (e^z - 1) / z, which tends to dt as z -> 0 */
    cplx z = dt * A + I * theta;
    cplx phi = cabs(z) < 1e-6 ? 1.0 + z / 2.0 + z * z / 6.0 : (cexp(z) - 1.0) / z;
    cplx gamma = dt * phi;
    u = gamma * v;
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
  if (mode != 0 && mode != 1 && mode != 2) return -2;
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

/* ===================================================================================== *
 * Backward (reverse mode) of the scan above, for a sequence that starts from the zero
 * state with no step -1 halo.
 *
 * The pages name the backward pass and its recompute strategy without formulas ("Complex
 * parallel scan", sections 一个问题，两种命运 and 硬件落地的挑战: one reverse sweep after
 * the forward, states regenerated instead of stored, a backward kernel beside the forward
 * one). What follows is reverse-mode differentiation of the recurrence written out step by
 * step. For a complex quantity z the gradient is G(z) = dl/dRe z + i dl/dIm z, where
 * l = sum_{b,t,d} dy[b,t,d] y[b,t,d]. Two rules give every line below:
 *   w = p z (p fixed)          =>  G(z) += conj(p) G(w)
 *   w = exp(z)                 =>  G(z)  = conj(exp(z)) G(w)
 * and for y = Re(C h): G(h) += dy conj(C), G(C) += dy conj(h).
 * The adjoint of the state obeys the reversed recurrence
 *   ghat_t = dy_t conj(Cc_t) + conj(a_{t+1}) ghat_{t+1},  ghat_L = 0,
 * and ghat_t is the gradient of the step-t injection u_t; the transition a_t = exp(z_t),
 * z_t = dt_t A + i theta_t, receives G(a_t) = ghat_t conj(h_{t-1}) (plus, in the trapezoid
 * mode, ghat_t conj((1 - lam_t) dt_t x_{t-1} Bc_{t-1}) from beta_t), so that
 * d l / d(dt_t A) = Re G(z_t) and d l / d theta_t = Im G(z_t). In the zero-order hold the
 * injection's gamma_t = dt_t phi(z_t) depends on z_t too: G(z_t) gains conj(phi'(z_t)) dt_t
 * x_t conj(Bc_t) ghat_t, and dt_t's own factor gives Re(conj(phi) x_t conj(Bc_t) ghat_t).
 *
 * Outputs are fully written (zeroed first); complex gradients are (d/dRe, d/dIm) pairs in the
 * layouts of their inputs: dx, ddt (B,L,D); dA (D,N); dBc, dCc (B,L,N) complex;
 * dtheta (B,L,N); dlam (B,L) (mode 1; may be NULL in mode 0); dDskip (D).
 * ===================================================================================== */
typedef struct {
  const double *x, *dt, *A, *Bc, *Cc, *theta, *lam, *Dskip, *dy;
  double *dx, *ddt;                          /* per row, written by the row's owner only */
  double *dA, *dBc, *dCc, *dtheta, *dlam, *dD; /* shared: private copies per worker */
  int64_t B, L, D, N;
  int mode;
  int64_t row_begin, row_step;
} bjob_t;

/* Zero-order hold: phi(z) = (e^z - 1) / z, as in oracle_operator, and its derivative
 * phi'(z) = (e^z (z - 1) + 1) / z^2, from its power series sum_{k>=1} k z^{k-1} / (k+1)! where
 * the closed form would cancel (|z| < 1e-2: the first omitted term is below 1e-13 of 1/2). */
static cplx zoh_phi(cplx z) { return cabs(z) < 1e-6 ? 1.0 + z / 2.0 + z * z / 6.0 : (cexp(z) - 1.0) / z; }
static cplx zoh_dphi(cplx z) {
  if (cabs(z) < 1e-2)
    return 0.5 + z * (1.0 / 3.0 + z * (1.0 / 8.0 + z * (1.0 / 30.0 + z * (1.0 / 144.0 + z / 840.0))));
  return (cexp(z) * (z - 1.0) + 1.0) / (z * z);
}

static void backward_row(const bjob_t* j, int64_t b, int64_t d, cplx* hs, cplx* as, cplx* carry) {
  const int64_t L = j->L, D = j->D, N = j->N;
  /* forward sweep: keep every state h_t and transition a_t of this row */
  for (int64_t n = 0; n < N; ++n) carry[n] = 0.0;   /* used as h here */
  for (int64_t t = 0; t < L; ++t) {
    const int64_t td = (b * L + t) * D + d;
    const double xt = j->x[td], dtt = j->dt[td];
    const double x_prev = t > 0 ? j->x[td - D] : 0.0;
    const double lam = j->mode == 1 ? j->lam[b * L + t] : 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const int64_t tn = (b * L + t) * N + n;
      double B_prev[2] = {0.0, 0.0};
      if (t > 0) { B_prev[0] = j->Bc[2 * (tn - N)]; B_prev[1] = j->Bc[2 * (tn - N) + 1]; }
      double op[4];
      oracle_operator(j->mode, dtt, j->A[d * N + n], j->theta[tn], lam, xt, x_prev, &j->Bc[2 * tn], B_prev, op);
      carry[n] = (op[0] + I * op[1]) * carry[n] + (op[2] + I * op[3]);
      hs[t * N + n] = carry[n];
      as[t * N + n] = op[0] + I * op[1];
    }
  }
  /* reverse sweep */
  for (int64_t n = 0; n < N; ++n) carry[n] = 0.0;   /* conj(a_{t+1}) ghat_{t+1} */
  for (int64_t t = L - 1; t >= 0; --t) {
    const int64_t td = (b * L + t) * D + d;
    const double xt = j->x[td], dtt = j->dt[td], dyt = j->dy[td];
    const double x_prev = t > 0 ? j->x[td - D] : 0.0;
    const double lam = j->mode == 1 ? j->lam[b * L + t] : 0.0;
    double P = 0.0;   /* sum_n Re(conj(Bc_t) ghat_t): d l / d(coefficient of Bc_t) */
    double R = 0.0;   /* sum_n Re(conj(a_t Bc_{t-1}) ghat_t): the same for beta_t's term */
    double dz_re = 0.0;
    double Q = 0.0;   /* zero-order hold: d l / d dt_t through gamma's factor dt_t */
    for (int64_t n = 0; n < N; ++n) {
      const int64_t tn = (b * L + t) * N + n;
      const cplx a = as[t * N + n];
      const cplx h = hs[t * N + n];
      const cplx h_prev = t > 0 ? hs[(t - 1) * N + n] : 0.0;
      const cplx ghat = dyt * conj(load_c(j->Cc, tn)) + carry[n];
      /* output y_t = Re(Cc_t h_t) */
      store_c(j->dCc, tn, load_c(j->dCc, tn) + dyt * conj(h));
      /* injection */
      const cplx Bt = load_c(j->Bc, tn);
      cplx Ga = ghat * conj(h_prev);
      cplx Gz_phi = 0.0;   /* zero-order hold: G(z) through gamma = dt phi(z) */
      if (j->mode == 0) {
        store_c(j->dBc, tn, load_c(j->dBc, tn) + (dtt * xt) * ghat);
        P += creal(conj(Bt) * ghat);
      } else if (j->mode == 2) {
        /* u_t = gamma_t x_t Bc_t: G(gamma) = x conj(Bc) ghat, G(phi) = dt G(gamma),
         * G(z) += conj(phi'(z)) G(phi); the factor dt in gamma gives Re(conj(phi) G(gamma)) */
        const cplx z = dtt * j->A[d * N + n] + I * j->theta[tn];
        const cplx phi = zoh_phi(z), gam = dtt * phi;
        const cplx Ggam = xt * conj(Bt) * ghat;
        store_c(j->dBc, tn, load_c(j->dBc, tn) + (xt * conj(gam)) * ghat);
        P += creal(conj(gam * Bt) * ghat);
        Q += creal(conj(phi) * Ggam);
        Gz_phi = conj(zoh_dphi(z)) * (dtt * Ggam);
      } else {
        store_c(j->dBc, tn, load_c(j->dBc, tn) + (lam * dtt * xt) * ghat);
        P += creal(conj(Bt) * ghat);
        if (t > 0) {
          const cplx Bp = load_c(j->Bc, tn - N);
          const double c2 = (1.0 - lam) * dtt * x_prev;     /* beta_t's term is c2 a_t Bc_{t-1} */
          R += creal(conj(a * Bp) * ghat);
          store_c(j->dBc, tn - N, load_c(j->dBc, tn - N) + c2 * conj(a) * ghat);
          Ga += ghat * conj(c2 * Bp);
        }
      }
      /* transition a_t = exp(dt_t A + i theta_t) (and, in mode 2, gamma's phi(z)) */
      const cplx Gz = conj(a) * Ga + Gz_phi;
      j->dA[d * N + n] += dtt * creal(Gz);
      dz_re += j->A[d * N + n] * creal(Gz);
      j->dtheta[tn] += cimag(Gz);
      carry[n] = conj(a) * ghat;
    }
    double gx, gdt;
    if (j->mode == 0) {
      gx = dtt * P;
      gdt = xt * P;
    } else if (j->mode == 2) {
      gx = P;
      gdt = Q;
    } else {
      gx = lam * dtt * P;
      gdt = lam * xt * P + (1.0 - lam) * x_prev * R;
      j->dlam[b * L + t] += dtt * xt * P - dtt * x_prev * R;
      if (t > 0) j->dx[td - D] += (1.0 - lam) * dtt * R;
    }
    j->dx[td] += gx + j->Dskip[d] * dyt;
    j->ddt[td] += gdt + dz_re;
    j->dD[d] += dyt * xt;
  }
}

static void* bworker(void* arg) {
  const bjob_t* j = (const bjob_t*)arg;
  const size_t LN = (size_t)(j->L > 0 ? j->L : 1) * (size_t)(j->N > 0 ? j->N : 1);
  cplx* hs = (cplx*)malloc(sizeof(cplx) * LN);
  cplx* as = (cplx*)malloc(sizeof(cplx) * LN);
  cplx* carry = (cplx*)malloc(sizeof(cplx) * (size_t)(j->N > 0 ? j->N : 1));
  if (!hs || !as || !carry) { free(hs); free(as); free(carry); return (void*)1; }
  for (int64_t r = j->row_begin; r < j->B * j->D; r += j->row_step) backward_row(j, r / j->D, r % j->D, hs, as, carry);
  free(hs); free(as); free(carry);
  return NULL;
}

/* Reverse-mode gradients of l = sum dy * y for oracle_forward with h0 = 0 and no halo, rows
 * split across `nthreads` POSIX threads (<= 0: all online cores); the shared gradients are
 * summed from private per-thread copies. Returns the number of threads used (> 0), or a
 * negative value on bad arguments or allocation failure. */
int oracle_backward(const double* x, const double* dt, const double* A, const double* Bc, const double* Cc,
                    const double* theta, const double* lam, const double* Dskip, const double* dy,
                    double* dx, double* ddt, double* dA, double* dBc, double* dCc, double* dtheta, double* dlam,
                    double* dDskip, int64_t B, int64_t L, int64_t D, int64_t N, int mode, int nthreads) {
  if (B < 0 || L < 0 || D < 0 || N < 0) return -1;
  if (mode != 0 && mode != 1 && mode != 2) return -2;
  if (mode == 1 && (!lam || !dlam) && B * L > 0) return -3;
  const size_t nBLD = (size_t)(B * L * D), nDN = (size_t)(D * N), nBLN = (size_t)(B * L * N), nBL = (size_t)(B * L);
  for (size_t i = 0; i < nBLD; ++i) { dx[i] = 0.0; ddt[i] = 0.0; }
  for (size_t i = 0; i < nDN; ++i) dA[i] = 0.0;
  for (size_t i = 0; i < 2 * nBLN; ++i) { dBc[i] = 0.0; dCc[i] = 0.0; }
  for (size_t i = 0; i < nBLN; ++i) dtheta[i] = 0.0;
  if (dlam) for (size_t i = 0; i < nBL; ++i) dlam[i] = 0.0;
  for (int64_t i = 0; i < D; ++i) dDskip[i] = 0.0;
  if (nthreads <= 0) nthreads = oracle_default_threads();
  if ((int64_t)nthreads > B * D) nthreads = (int)(B * D > 0 ? B * D : 1);
  /* per-thread private copies of the shared gradients: dA, dBc, dCc, dtheta, dlam, dD */
  const size_t priv = nDN + 4 * nBLN + nBLN + nBL + (size_t)D;
  double* buf = (double*)calloc(priv * (size_t)nthreads + 1, sizeof(double));
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  bjob_t* jobs = (bjob_t*)malloc(sizeof(bjob_t) * (size_t)nthreads);
  if (!buf || !th || !jobs) { free(buf); free(th); free(jobs); return -4; }
  int rc = 0, started = 0;
  for (int i = 0; i < nthreads; ++i) {
    double* p = buf + priv * (size_t)i;
    bjob_t jb = {x, dt, A, Bc, Cc, theta, lam, Dskip, dy, dx, ddt,
                 p, p + nDN, p + nDN + 2 * nBLN, p + nDN + 4 * nBLN, p + nDN + 5 * nBLN, p + nDN + 5 * nBLN + nBL,
                 B, L, D, N, mode, i, nthreads};
    jobs[i] = jb;
    if (nthreads == 1) {
      if (bworker(&jobs[i])) rc = -4;
      started = 0;
      break;
    }
    if (pthread_create(&th[i], NULL, bworker, &jobs[i]) != 0) { rc = -5; break; }
    ++started;
  }
  for (int i = 0; i < started; ++i) {
    void* ret = NULL;
    pthread_join(th[i], &ret);
    if (ret) rc = -4;
  }
  if (rc == 0) {
    for (int i = 0; i < nthreads; ++i) {
      const bjob_t* jb = &jobs[i];
      for (size_t k = 0; k < nDN; ++k) dA[k] += jb->dA[k];
      for (size_t k = 0; k < 2 * nBLN; ++k) { dBc[k] += jb->dBc[k]; dCc[k] += jb->dCc[k]; }
      for (size_t k = 0; k < nBLN; ++k) dtheta[k] += jb->dtheta[k];
      if (dlam) for (size_t k = 0; k < nBL; ++k) dlam[k] += jb->dlam[k];
      for (int64_t k = 0; k < D; ++k) dDskip[k] += jb->dD[k];
    }
  }
  free(buf); free(th); free(jobs);
  return rc < 0 ? rc : nthreads;
}

/* ===================================================================================== *
 * MIMO scan: P input/output channels of a head share one complex state per (b, head, n).
 * "Mamba-3 paper story" (MIMO section and its SISO/MIMO table) widens B and C from vectors to
 * N x P matrices so that one state serves P channels, raising the work per byte; its
 * formulas were lost from the page. Reading taken (the SISO sharing carried over):
 *   a_t = exp(dt[b,t,h] A[h,n] + i theta[b,t,n])
 *   v_t[n] = sum_p Bm[b,t,n,p] x[b,t,h,p]                       (the rank-P injection)
 *   exp-Euler:  h_t = a_t h_{t-1} + dt_t v_t
 *   trapezoid:  h_t = a_t h_{t-1} + (1 - lam_t) dt_t a_t v_{t-1} + lam_t dt_t v_t,  v_{-1} = 0
 *   y[b,t,h,p] = Re(sum_n Cm[b,t,n,p] h_t[n]) + Dskip[h,p] x[b,t,h,p]
 * Layouts (float64; complex interleaved): x, y (B,L,H,P); dt (B,L,H); A (H,N);
 * Bm, Cm (B,L,N,P) complex; theta (B,L,N); lam (B,L); Dskip (H,P).
 * With P = 1 this is the scan above with one channel per head.
 * ===================================================================================== */
typedef struct {
  const double *x, *dt, *A, *Bm, *Cm, *theta, *lam, *Dskip;
  double* y;
  int64_t B, L, H, P, N;
  int mode;
  int64_t row_begin, row_step;
} mjob_t;

static void mimo_row(const mjob_t* j, int64_t b, int64_t hd, cplx* h, cplx* v_prev) {
  const int64_t L = j->L, H = j->H, P = j->P, N = j->N;
  for (int64_t n = 0; n < N; ++n) { h[n] = 0.0; v_prev[n] = 0.0; }
  for (int64_t t = 0; t < L; ++t) {
    const double dtt = j->dt[(b * L + t) * H + hd];
    const double lam = j->mode == 1 ? j->lam[b * L + t] : 0.0;
    const double* xt = &j->x[((b * L + t) * H + hd) * P];
    for (int64_t n = 0; n < N; ++n) {
      const int64_t tn = (b * L + t) * N + n;
      cplx v = 0.0;
      for (int64_t p = 0; p < P; ++p) v += load_c(j->Bm, tn * P + p) * xt[p];
      const cplx a = transition(dtt, j->A[hd * N + n], j->theta[tn]);
      cplx u;
      if (j->mode == 0) u = dtt * v;
      else u = (1.0 - lam) * dtt * a * v_prev[n] + lam * dtt * v;
      h[n] = a * h[n] + u;
      v_prev[n] = v;
    }
    for (int64_t p = 0; p < P; ++p) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) acc += creal(load_c(j->Cm, ((b * L + t) * N + n) * P + p) * h[n]);
      j->y[((b * L + t) * H + hd) * P + p] = acc + j->Dskip[hd * P + p] * xt[p];
    }
  }
}

static void* mworker(void* arg) {
  const mjob_t* j = (const mjob_t*)arg;
  cplx* h = (cplx*)malloc(sizeof(cplx) * (size_t)(j->N > 0 ? 2 * j->N : 2));
  if (!h) return (void*)1;
  for (int64_t r = j->row_begin; r < j->B * j->H; r += j->row_step) mimo_row(j, r / j->H, r % j->H, h, h + j->N);
  free(h);
  return NULL;
}

/* MIMO forward over all (b, head) rows, split across `nthreads` POSIX threads (<= 0: all
 * online cores). Returns the number of threads used (> 0) or a negative value on bad
 * arguments. */
int oracle_forward_mimo(const double* x, const double* dt, const double* A, const double* Bm, const double* Cm,
                        const double* theta, const double* lam, const double* Dskip, double* y, int64_t B, int64_t L,
                        int64_t H, int64_t P, int64_t N, int mode, int nthreads) {
  if (B < 0 || L < 0 || H < 0 || P < 0 || N < 0) return -1;
  if (mode != 0 && mode != 1) return -2;
  if (mode == 1 && !lam && B * L > 0) return -3;
  if (nthreads <= 0) nthreads = oracle_default_threads();
  if ((int64_t)nthreads > B * H) nthreads = (int)(B * H > 0 ? B * H : 1);
  mjob_t base = {x, dt, A, Bm, Cm, theta, lam, Dskip, y, B, L, H, P, N, mode, 0, 1};
  if (nthreads == 1) return mworker(&base) ? -4 : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  mjob_t* jobs = (mjob_t*)malloc(sizeof(mjob_t) * (size_t)nthreads);
  if (!th || !jobs) { free(th); free(jobs); return -4; }
  int rc = 0, started = 0;
  for (int i = 0; i < nthreads; ++i) {
    jobs[i] = base;
    jobs[i].row_begin = i;
    jobs[i].row_step = nthreads;
    if (pthread_create(&th[i], NULL, mworker, &jobs[i]) != 0) { rc = -5; break; }
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

/* ===================================================================================== *
 * Backward (reverse mode) of the MIMO scan, from the zero state: the gradients of
 * l = sum dy[b,t,h,p] y[b,t,h,p], written out with the rules of the single-input backward
 * above. Per (b, head) and state n the adjoint is
 *   ghat_t = sum_p dy_t[p] conj(Cm_t[n,p]) + conj(a_{t+1}) ghat_{t+1},
 * the gradient of the step-t injection u_t. exp-Euler u_t = dt_t v_t gives
 * G(v_t) = dt_t ghat_t; the trapezoid u_t = c1 v_t + c2 a_t v_{t-1} (c1 = lam_t dt_t,
 * c2 = (1 - lam_t) dt_t) gives G(v_t) = c1 ghat_t + c2' conj(a_{t+1}) ghat_{t+1} (c2' of step
 * t + 1) and G(a_t) gains ghat_t conj(c2 v_{t-1}). v_t[n] = sum_p Bm_t[n,p] x_t[p] then gives
 * G(Bm_t[n,p]) = x_t[p] G(v_t[n]) and dx_t[p] += Re(conj(Bm_t[n,p]) G(v_t[n])).
 * Outputs are zeroed first and fully written: dx (B,L,H,P), ddt (B,L,H), dA (H,N),
 * dBm, dCm (B,L,N,P) complex, dtheta (B,L,N), dlam (B,L) (trapezoid; may be NULL otherwise),
 * dDskip (H,P). Single-threaded (a test reference for small sizes). Returns 0, or a negative
 * value on bad arguments or allocation failure.
 * ===================================================================================== */
int oracle_backward_mimo(const double* x, const double* dt, const double* A, const double* Bm, const double* Cm,
                         const double* theta, const double* lam, const double* Dskip, const double* dy,
                         double* dx, double* ddt, double* dA, double* dBm, double* dCm, double* dtheta,
                         double* dlam, double* dDskip, int64_t B, int64_t L, int64_t H, int64_t P, int64_t N,
                         int mode) {
  if (B < 0 || L < 0 || H < 0 || P < 0 || N < 0) return -1;
  if (mode != 0 && mode != 1) return -2;
  if (mode == 1 && (!lam || !dlam) && B * L > 0) return -3;
  for (int64_t i = 0; i < B * L * H * P; ++i) dx[i] = 0.0;
  for (int64_t i = 0; i < B * L * H; ++i) ddt[i] = 0.0;
  for (int64_t i = 0; i < H * N; ++i) dA[i] = 0.0;
  for (int64_t i = 0; i < 2 * B * L * N * P; ++i) { dBm[i] = 0.0; dCm[i] = 0.0; }
  for (int64_t i = 0; i < B * L * N; ++i) dtheta[i] = 0.0;
  if (dlam) for (int64_t i = 0; i < B * L; ++i) dlam[i] = 0.0;
  for (int64_t i = 0; i < H * P; ++i) dDskip[i] = 0.0;
  const size_t LN = (size_t)(L > 0 ? L : 1) * (size_t)(N > 0 ? N : 1);
  cplx* hs = (cplx*)malloc(sizeof(cplx) * LN);
  cplx* as = (cplx*)malloc(sizeof(cplx) * LN);
  cplx* vs = (cplx*)malloc(sizeof(cplx) * LN);
  cplx* cg = (cplx*)malloc(sizeof(cplx) * (size_t)(N > 0 ? 2 * N : 2));
  if (!hs || !as || !vs || !cg) { free(hs); free(as); free(vs); free(cg); return -4; }
  cplx* cv = cg + N;   /* G(v_t) carried from step t + 1 (trapezoid) */
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t hd = 0; hd < H; ++hd) {
      /* forward sweep: keep h_t, a_t and v_t of this row */
      for (int64_t n = 0; n < N; ++n) cg[n] = 0.0;   /* used as h here */
      for (int64_t t = 0; t < L; ++t) {
        const double dtt = dt[(b * L + t) * H + hd];
        const double lm = mode == 1 ? lam[b * L + t] : 0.0;
        const double* xt = &x[((b * L + t) * H + hd) * P];
        for (int64_t n = 0; n < N; ++n) {
          const int64_t tn = (b * L + t) * N + n;
          cplx v = 0.0;
          for (int64_t p = 0; p < P; ++p) v += load_c(Bm, tn * P + p) * xt[p];
          const cplx a = transition(dtt, A[hd * N + n], theta[tn]);
          const cplx vp = t > 0 ? vs[(t - 1) * N + n] : 0.0;
          const cplx u = mode == 0 ? dtt * v : (1.0 - lm) * dtt * a * vp + lm * dtt * v;
          cg[n] = a * cg[n] + u;
          hs[t * N + n] = cg[n];
          as[t * N + n] = a;
          vs[t * N + n] = v;
        }
      }
      /* reverse sweep */
      for (int64_t n = 0; n < N; ++n) { cg[n] = 0.0; cv[n] = 0.0; }
      for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t th = (b * L + t) * H + hd;
        const double dtt = dt[th];
        const double lm = mode == 1 ? lam[b * L + t] : 0.0;
        const double c1 = mode == 0 ? dtt : lm * dtt, c2 = (1.0 - lm) * dtt;
        const double* xt = &x[th * P];
        const double* dyt = &dy[th * P];
        double dc1 = 0.0, dc2 = 0.0, dz_re = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          const int64_t tn = (b * L + t) * N + n;
          const cplx a = as[t * N + n], h = hs[t * N + n];
          const cplx h_prev = t > 0 ? hs[(t - 1) * N + n] : 0.0;
          const cplx v = vs[t * N + n];
          cplx ghat = cg[n];
          for (int64_t p = 0; p < P; ++p) {
            ghat += dyt[p] * conj(load_c(Cm, tn * P + p));
            store_c(dCm, tn * P + p, load_c(dCm, tn * P + p) + dyt[p] * conj(h));
          }
          const cplx Gv = c1 * ghat + cv[n];
          dc1 += creal(conj(v) * ghat);
          cplx Ga = ghat * conj(h_prev);
          cplx next_cv = 0.0;
          if (mode == 1 && t > 0) {
            const cplx vp = vs[(t - 1) * N + n];
            Ga += ghat * conj(c2 * vp);
            dc2 += creal(conj(a * vp) * ghat);
            next_cv = c2 * conj(a) * ghat;   /* G(v_{t-1}) from this step's beta term */
          }
          for (int64_t p = 0; p < P; ++p) {
            store_c(dBm, tn * P + p, load_c(dBm, tn * P + p) + xt[p] * Gv);
            dx[th * P + p] += creal(conj(load_c(Bm, tn * P + p)) * Gv);
          }
          const cplx Gz = conj(a) * Ga;
          dA[hd * N + n] += dtt * creal(Gz);
          dz_re += A[hd * N + n] * creal(Gz);
          dtheta[tn] += cimag(Gz);
          cg[n] = conj(a) * ghat;
          cv[n] = next_cv;
        }
        if (mode == 0) {
          ddt[th] += dc1 + dz_re;
        } else {
          ddt[th] += lm * dc1 + (1.0 - lm) * dc2 + dz_re;
          dlam[b * L + t] += dtt * dc1 - dtt * dc2;
        }
        for (int64_t p = 0; p < P; ++p) {
          dDskip[hd * P + p] += dyt[p] * xt[p];
          dx[th * P + p] += Dskip[hd * P + p] * dyt[p];
        }
      }
    }
  }
  free(hs); free(as); free(vs); free(cg);
  return 0;
}
