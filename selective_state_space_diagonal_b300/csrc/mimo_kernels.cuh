// mimo_kernels.cuh -- the MIMO scan: the P channels of a head share one complex state.
//
//   a_t     = exp(dt[b,t,h] A[h,n] + i theta[b,t,n])
//   v_t[n]  = sum_p Bm[b,t,n,p] x[b,t,h,p]
//   exp-Euler   h_t = a_t h_{t-1} + dt_t v_t
//   trapezoid   h_t = a_t h_{t-1} + (1 - lam_t) dt_t a_t v_{t-1} + lam_t dt_t v_t
//   y[b,t,h,p] = Re(sum_n Cm[b,t,n,p] h_t[n]) + Dskip[h,p] x[b,t,h,p]
//
// "Mamba-3 paper story" (MIMO section) widens B and C to N x P so that one state serves P
// channels: per state and step the work grows with P while the state's traffic does not. The
// kernels mirror the zero-order-hold ones:
//   mimo_rot_kernel     e^{i theta} per (b, t, n)
//   mimo_chunk_kernel   per (b, c, h, n): the chunk's end state from a zero entry state and
//                       the product of a over the chunk                     (chunks > 1 only)
//   mimo_combine_kernel per (b, h, n): each chunk's entry state
//   mimo_out_kernel     blocks of OUT_THREADS / N heads of one (b, c), a thread per (head, n): the
//                       recurrence over the chunk with y, each 8-step group's shared inputs
//                       staged in shared memory first; each lane keeps its P partial outputs
//                       for the group and a reduce-scatter over the head's N lanes leaves
//                       every (step, channel) sum in one lane
#pragma once

#include "device_util.cuh"

namespace csscan {
namespace mimo {

constexpr int GROUP = 8;
// Threads per block of mimo_out_kernel. Blocks of 128 threads compiled for 9 resident
// blocks per SM (56 registers) hold 1152 threads per SM, so 16 x 640 x 16 (b, head, n) rows
// run in one wave; 256-thread blocks at 64 registers held 1024 and needed a second, 8 %
// full wave (11.5 -> 8.4 ms). With P = 8 the 56-register cap spills the 64 partial outputs,
// so those kernels keep 128 registers (4 blocks).
constexpr int OUT_THREADS = 128;
template <int P> struct OutOcc {
  static constexpr int MIN_BLOCKS = P <= 4 ? 9 : 4;
};
constexpr float LOG2E = 1.4426950408889634f;

struct Params {
  const void* x;       // (B, L, H, P)
  const void* dt;      // (B, L, H)
  const void* Bm;      // (B, L, N, P, 2)
  const void* Cm;      // (B, L, N, P, 2)
  const void* lam;     // (B, L) trapezoid only
  const float* A;      // (H, N)
  const float* Dskip;  // (H, P)
  float* y;            // (B, L, H, P)
  const float2* rot;   // (B, L, N)
  float2* chunk;       // (B, C, H, N, 2): end state | entry state, product of a
  int B, L, H, N, P;
  int TC, C;
};

template <typename Tin>
__global__ void __launch_bounds__(256) mimo_rot_kernel(const void* theta, float2* rot, long long total) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= total) return;
  float s, c;
  sincosf(load_in<Tin>(static_cast<const Tin*>(theta), i), &s, &c);
  rot[i] = make_float2(c, s);
}

struct Thread {
  long long b;
  int c, h, n;
  bool ok;
};
__device__ __forceinline__ Thread thread_of(const Params& p) {
  const long long gid = (long long)blockIdx.x * 256 + threadIdx.x;
  Thread r;
  r.ok = gid < (long long)p.B * p.C * p.H * p.N;
  const long long g = r.ok ? gid : 0;
  r.n = int(g % p.N);
  long long q = g / p.N;
  r.h = int(q % p.H);
  q /= p.H;
  r.c = int(q % p.C);
  r.b = q / p.C;
  return r;
}
__device__ __forceinline__ float2* rec_of(const Params& p, long long b, int c, int h, int n) {
  return p.chunk + ((((b * p.C + c) * p.H + h) * p.N) + n) * 2;
}

// The step's rank-P injection v = sum_p Bm[n, p] x[p] and x itself (for the D-skip).
template <typename Tin, int P>
__device__ __forceinline__ float2 inject(const Params& p, long long b, int t, int h, int n, float (&xs)[P]) {
  const Tin* X = static_cast<const Tin*>(p.x);
  const Tin* BM = static_cast<const Tin*>(p.Bm);
  const long long th = ((b * p.L + t) * p.H + h) * P;
  const long long tn = ((b * p.L + t) * p.N + n) * P;
  float vr = 0.f, vi = 0.f;
#pragma unroll
  for (int q = 0; q < P; ++q) {
    xs[q] = load_in<Tin>(X, th + q);
    const float2 bb = load_pair<Tin>(BM, tn + q);
    vr = fmaf(bb.x, xs[q], vr);
    vi = fmaf(bb.y, xs[q], vi);
  }
  return make_float2(vr, vi);
}

// One step: h <- a h + u. vp carries v_{t-1} (trapezoid). ar, ai return a.
template <typename Tin, int MODE>
__device__ __forceinline__ void mimo_step(const Params& p, long long b, int t, int h, int n, float a2, float2 v,
                                          float2& vp, float& hr, float& hi, float& ar, float& ai) {
  const Tin* DT = static_cast<const Tin*>(p.dt);
  const float dtt = load_in<Tin>(DT, (b * p.L + t) * p.H + h);
  const float2 ro = p.rot[(b * p.L + t) * p.N + n];
  const float r = ex2_approx(dtt * a2);
  ar = r * ro.x;
  ai = r * ro.y;
  float ur, ui;
  if (MODE == 0) {
    ur = dtt * v.x;
    ui = dtt * v.y;
  } else {
    const float lm = load_in<Tin>(static_cast<const Tin*>(p.lam), b * p.L + t);
    const float c1 = lm * dtt, c2 = (1.f - lm) * dtt;
    ur = c1 * v.x + c2 * (ar * vp.x - ai * vp.y);
    ui = c1 * v.y + c2 * (ar * vp.y + ai * vp.x);
    vp = v;
  }
  const float nr = fmaf(ar, hr, fmaf(-ai, hi, ur));
  const float ni = fmaf(ar, hi, fmaf(ai, hr, ui));
  hr = nr;
  hi = ni;
}

template <typename Tin, int MODE, int P>
__device__ __forceinline__ float2 v_before(const Params& p, long long b, int tc, int h, int n) {
  if (MODE == 0 || tc == 0) return make_float2(0.f, 0.f);
  float xs[P];
  return inject<Tin, P>(p, b, tc - 1, h, n, xs);
}

template <typename Tin, int MODE, int P>
__global__ void __launch_bounds__(256) mimo_chunk_kernel(const Params p) {
  const Thread th = thread_of(p);
  if (!th.ok) return;
  const float a2 = p.A[(long long)th.h * p.N + th.n] * LOG2E;
  const int tc = th.c * p.TC, te = min(p.L, tc + p.TC);
  float hr = 0.f, hi = 0.f, Pr = 1.f, Pi = 0.f;
  float2 vp = v_before<Tin, MODE, P>(p, th.b, tc, th.h, th.n);
  for (int t = tc; t < te; ++t) {
    float xs[P];
    const float2 v = inject<Tin, P>(p, th.b, t, th.h, th.n, xs);
    float ar, ai;
    mimo_step<Tin, MODE>(p, th.b, t, th.h, th.n, a2, v, vp, hr, hi, ar, ai);
    const float qr = ar * Pr - ai * Pi, qi = ar * Pi + ai * Pr;
    Pr = qr;
    Pi = qi;
  }
  float2* rec = rec_of(p, th.b, th.c, th.h, th.n);
  rec[0] = make_float2(hr, hi);
  rec[1] = make_float2(Pr, Pi);
}

__global__ void __launch_bounds__(256) mimo_combine_kernel(const Params p) {
  const long long gid = (long long)blockIdx.x * 256 + threadIdx.x;
  if (gid >= (long long)p.B * p.H * p.N) return;
  const int n = int(gid % p.N);
  const long long bh = gid / p.N;
  const int h = int(bh % p.H);
  const long long b = bh / p.H;
  float hr = 0.f, hi = 0.f;
  for (int c = 0; c < p.C; ++c) {
    float2* rec = rec_of(p, b, c, h, n);
    const float2 U = rec[0], Pm = rec[1];
    rec[0] = make_float2(hr, hi);
    const float nr = Pm.x * hr - Pm.y * hi + U.x, ni = Pm.x * hi + Pm.y * hr + U.y;
    hr = nr;
    hi = ni;
  }
}

// The recurrence over chunk c with y. A block owns HB = OUT_THREADS / N heads of one (b, c): thread
// (head hl, state n), the N lanes of a head neighbours in a warp (N <= 32). For each group of
// GROUP steps the block first stages, coalesced, what its lanes share -- e^{i theta}, Bm and Cm
// per (t, n), x and dt per (t, head), lam per t -- in shared memory. Each lane then keeps its P
// partial outputs for the group and a reduce-scatter over the head's N lanes leaves every
// (step, channel) sum in one lane. Grid: (ceil(H / HB), C, B).
template <int N, int P> struct MimoStage {
  static constexpr int HB = OUT_THREADS / N;               // heads per block
  static constexpr int TN = GROUP * N;                     // (t, n) entries of a group
  static constexpr int TH = GROUP * HB;                    // (t, head) entries of a group
  static constexpr int OFF_ROT = 0;                        // float2 [GROUP][N]
  static constexpr int OFF_BM = OFF_ROT + TN * 8;          // float2 [GROUP][N][P]
  static constexpr int OFF_CM = OFF_BM + TN * P * 8;       // float2 [GROUP][N][P]
  static constexpr int OFF_X = OFF_CM + TN * P * 8;        // float [GROUP][HB][P]
  static constexpr int OFF_DT = OFF_X + TH * P * 4;        // float [GROUP][HB]
  static constexpr int OFF_LAM = OFF_DT + TH * 4;          // float [GROUP]
  static constexpr int BYTES = OFF_LAM + GROUP * 4;
};

template <typename Tin, int MODE, int N, int P>
__global__ void __launch_bounds__(OUT_THREADS, OutOcc<P>::MIN_BLOCKS) mimo_out_kernel(const Params p) {
  using MS = MimoStage<N, P>;
  constexpr int HB = MS::HB;
  constexpr int E = GROUP * P;                   // (step, channel) entries of one group
  constexpr int HOLD = E >= N ? E / N : 1;
  constexpr int DUP = N > E ? N / E : 1;
  __shared__ __align__(16) unsigned char sm[MS::BYTES];
  float2 (*s_rot)[N] = reinterpret_cast<float2 (*)[N]>(sm + MS::OFF_ROT);
  float2 (*s_bm)[N][P] = reinterpret_cast<float2 (*)[N][P]>(sm + MS::OFF_BM);
  float2 (*s_cm)[N][P] = reinterpret_cast<float2 (*)[N][P]>(sm + MS::OFF_CM);
  float (*s_x)[HB][P] = reinterpret_cast<float (*)[HB][P]>(sm + MS::OFF_X);
  float (*s_dt)[HB] = reinterpret_cast<float (*)[HB]>(sm + MS::OFF_DT);
  float* s_lam = reinterpret_cast<float*>(sm + MS::OFF_LAM);

  const int tid = threadIdx.x;
  const int n = tid % N, hl = tid / N;
  const int h0 = blockIdx.x * HB;
  const int h = h0 + hl;
  const bool valid = h < p.H;
  const int hc = valid ? h : 0;
  const int c = blockIdx.y;
  const long long b = blockIdx.z;
  const Tin* X = static_cast<const Tin*>(p.x);
  const Tin* DT = static_cast<const Tin*>(p.dt);
  const Tin* BM = static_cast<const Tin*>(p.Bm);
  const Tin* CM = static_cast<const Tin*>(p.Cm);
  const Tin* LAM = static_cast<const Tin*>(p.lam);
  const float a2 = p.A[(long long)hc * N + n] * LOG2E;
  float Ds[P];
#pragma unroll
  for (int q = 0; q < P; ++q) Ds[q] = p.Dskip[(long long)hc * P + q];
  const int tc = c * p.TC, te = min(p.L, tc + p.TC);
  float hr = 0.f, hi = 0.f;
  if (p.C > 1 && valid) {
    const float2 hin = rec_of(p, b, c, h, n)[0];
    hr = hin.x;
    hi = hin.y;
  }
  float2 vp = valid ? v_before<Tin, MODE, P>(p, b, tc, hc, n) : make_float2(0.f, 0.f);
  for (int t0 = tc; t0 < te; t0 += GROUP) {
    const int ng = min(GROUP, te - t0);
    // ---- stage the group (steps past te or heads past H as zeros)
    for (int k = tid; k < GROUP * N * P; k += OUT_THREADS) {
      const int i = k / (N * P), r = k % (N * P);
      float2 bb = make_float2(0.f, 0.f), cc = make_float2(0.f, 0.f);
      if (i < ng) {
        const long long e = ((b * p.L + t0 + i) * N) * P + r;   // entry (t, n, q), n * P + q = r
        bb = load_pair<Tin>(BM, e);
        cc = load_pair<Tin>(CM, e);
      }
      (&s_bm[0][0][0])[k] = bb;
      (&s_cm[0][0][0])[k] = cc;
    }
    for (int k = tid; k < GROUP * N; k += OUT_THREADS) {
      const int i = k / N, nn = k % N;
      s_rot[i][nn] = i < ng ? p.rot[(b * p.L + t0 + i) * N + nn] : make_float2(0.f, 0.f);
    }
    for (int k = tid; k < GROUP * HB * P; k += OUT_THREADS) {
      const int i = k / (HB * P), r = k % (HB * P), hh = h0 + r / P;
      (&s_x[0][0][0])[k] = (i < ng && hh < p.H) ? load_in<Tin>(X, ((b * p.L + t0 + i) * p.H + h0) * P + r) : 0.f;
    }
    for (int k = tid; k < GROUP * HB; k += OUT_THREADS) {
      const int i = k / HB, r = k % HB;
      s_dt[i][r] = (i < ng && h0 + r < p.H) ? load_in<Tin>(DT, (b * p.L + t0 + i) * p.H + h0 + r) : 0.f;
    }
    if (MODE == 1 && tid < GROUP) s_lam[tid] = tid < ng ? load_in<Tin>(LAM, b * p.L + t0 + tid) : 0.f;
    __syncthreads();

    float part[1][E];
#pragma unroll
    for (int i = 0; i < GROUP; ++i) {
#pragma unroll
      for (int q = 0; q < P; ++q) part[0][i * P + q] = 0.f;
      if (i < ng) {
        float vr = 0.f, vi = 0.f;
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const float2 bb = s_bm[i][n][q];
          vr = fmaf(bb.x, s_x[i][hl][q], vr);
          vi = fmaf(bb.y, s_x[i][hl][q], vi);
        }
        const float dtt = s_dt[i][hl];
        const float2 ro = s_rot[i][n];
        const float r = ex2_approx(dtt * a2);
        const float ar = r * ro.x, ai = r * ro.y;
        float ur, ui;
        if (MODE == 0) {
          ur = dtt * vr;
          ui = dtt * vi;
        } else {
          const float lm = s_lam[i];
          const float c1 = lm * dtt, c2 = (1.f - lm) * dtt;
          ur = c1 * vr + c2 * (ar * vp.x - ai * vp.y);
          ui = c1 * vi + c2 * (ar * vp.y + ai * vp.x);
          vp = make_float2(vr, vi);
        }
        const float nr = fmaf(ar, hr, fmaf(-ai, hi, ur));
        const float ni = fmaf(ar, hi, fmaf(ai, hr, ui));
        hr = nr;
        hi = ni;
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const float2 cc = s_cm[i][n][q];
          float o = cc.x * hr - cc.y * hi;
          if (n == 0) o = fmaf(Ds[q], s_x[i][hl][q], o);
          part[0][i * P + q] = o;
        }
      }
    }
    const int base = butterfly<N, 1, E>(part, n);
    if ((n % DUP) == 0 && valid) {
#pragma unroll
      for (int k = 0; k < HOLD; ++k) {
        const int e = base + k, i = e / P, q = e % P;
        if (i < ng) p.y[((b * p.L + t0 + i) * p.H + h) * P + q] = part[0][k];
      }
    }
    __syncthreads();
  }
}

}  // namespace mimo
}  // namespace csscan
