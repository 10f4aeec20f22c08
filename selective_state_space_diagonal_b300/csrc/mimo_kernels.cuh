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
//   mimo_out_kernel     per (b, c, h, n): the recurrence over the chunk with y; each lane keeps
//                       its P partial outputs for 8 steps and a reduce-scatter over the
//                       head's N lanes leaves every (step, channel) sum in one lane
#pragma once

#include "device_util.cuh"

namespace csscan {
namespace mimo {

constexpr int GROUP = 8;
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

// The recurrence over chunk c with y. Lanes n = 0 .. N-1 of one (b, c, h) are neighbours in a
// warp (N <= 32); every lane of a warp runs the same number of groups (the shuffles span the
// warp) and a lane past its chunk's end (or past the problem) adds zeros and stores nothing.
template <typename Tin, int MODE, int N, int P>
__global__ void __launch_bounds__(256) mimo_out_kernel(const Params p) {
  constexpr int E = GROUP * P;                   // (step, channel) entries of one group
  constexpr int HOLD = E >= N ? E / N : 1;
  constexpr int DUP = N > E ? N / E : 1;
  const Thread th = thread_of(p);
  const long long b = th.b;
  const int h = th.h, n = th.n;
  const float a2 = p.A[(long long)h * N + n] * LOG2E;
  float Ds[P];
#pragma unroll
  for (int q = 0; q < P; ++q) Ds[q] = p.Dskip[(long long)h * P + q];
  const Tin* CM = static_cast<const Tin*>(p.Cm);
  const int tc = th.c * p.TC;
  const int te = th.ok ? min(p.L, tc + p.TC) : tc;
  const int ngroups = (p.TC + GROUP - 1) / GROUP;
  float hr = 0.f, hi = 0.f;
  if (p.C > 1 && th.ok) {
    const float2 h0 = rec_of(p, b, th.c, h, n)[0];
    hr = h0.x;
    hi = h0.y;
  }
  float2 vp = th.ok ? v_before<Tin, MODE, P>(p, b, tc, h, n) : make_float2(0.f, 0.f);
  for (int gi = 0; gi < ngroups; ++gi) {
    const int t0 = tc + gi * GROUP;
    float part[1][E];
#pragma unroll
    for (int i = 0; i < GROUP; ++i) {
      const int t = t0 + i;
#pragma unroll
      for (int q = 0; q < P; ++q) part[0][i * P + q] = 0.f;
      if (t < te) {
        float xs[P];
        const float2 v = inject<Tin, P>(p, b, t, h, n, xs);
        float ar, ai;
        mimo_step<Tin, MODE>(p, b, t, h, n, a2, v, vp, hr, hi, ar, ai);
        const long long tn = ((b * p.L + t) * p.N + n) * P;
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const float2 cc = load_pair<Tin>(CM, tn + q);
          float o = cc.x * hr - cc.y * hi;
          if (n == 0) o = fmaf(Ds[q], xs[q], o);
          part[0][i * P + q] = o;
        }
      }
    }
    const int base = butterfly<N, 1, E>(part, n);
    if ((n % DUP) == 0) {
#pragma unroll
      for (int k = 0; k < HOLD; ++k) {
        const int e = base + k, t = t0 + e / P, q = e % P;
        if (t < te) p.y[((b * p.L + t) * p.H + h) * P + q] = part[0][k];
      }
    }
  }
}

}  // namespace mimo
}  // namespace csscan
