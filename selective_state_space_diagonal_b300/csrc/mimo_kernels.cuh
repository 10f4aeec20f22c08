// mimo_kernels.cuh -- the MIMO scan: the P channels of a head share one complex state.
//
//   a_t     = exp(dt[b,t,h] A[h,n] + i theta[b,t,n])
//   v_t[n]  = sum_p Bm[b,t,n,p] x[b,t,h,p]
//   exp-Euler   h_t = a_t h_{t-1} + dt_t v_t
//   trapezoid   h_t = a_t h_{t-1} + (1 - lam_t) dt_t a_t v_{t-1} + lam_t dt_t v_t
//   y[b,t,h,p] = Re(sum_n Cm[b,t,n,p] h_t[n]) + Dskip[h,p] x[b,t,h,p]
//
// "Mamba-3 paper story" (MIMO section) widens B and C to N x P so that one state serves P
// channels: per state and step the work grows with P while the state's traffic does not.
//   mimo_rot_kernel     e^{i theta} per (b, t, n)                          (chunks > 1 only)
//   mimo_chunk_kernel   per (b, c, h, n): the chunk's end state from a zero entry state and
//                       the product of a over the chunk                     (chunks > 1 only)
//   mimo_combine_kernel per (b, h, n): each chunk's entry state
//   mimo_out_kernel     blocks of heads of one (b, c), a thread per (head, state pair): the
//                       recurrence over the chunk with y in a rotating frame (real decay),
//                       each 8-step group's rotated Bm, Cm and its x, dt staged in shared
//                       memory first; each lane keeps its P partial outputs for the group and
//                       a reduce-scatter over the head's lanes leaves every (step, channel)
//                       sum in one lane
#pragma once

#include "device_util.cuh"

namespace csscan {
namespace mimo {

constexpr int GROUP = 8;
// Threads per block of mimo_out_kernel and the resident blocks per SM it is compiled for:
// 128-thread blocks at 5 per SM (96 registers, room for the next group's loads in flight
// without spills; 80 registers spilled and ran 6 % slower) hold 640 threads per SM, so the
// 16 x 640 x 16 / 2 (b, head, state pair) threads of the large-batch MIMO workload run in one
// wave; with P = 8 the 64 partial outputs per lane need 128 registers (4 blocks).
constexpr int OUT_THREADS = 128;
template <int P> struct OutOcc {
  static constexpr int MIN_BLOCKS = P <= 4 ? 5 : 4;
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
  const float2* phase; // (B, L, N): e^{i Phi_t}, Phi from the step's group start (mimo_phase_kernel)
  const float2* rot;   // (B, L, N): e^{i theta} (time-chunk pass only)
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

// e^{i Phi_t} per (b, t, n), Phi_t the sum of theta from the first step of t's GROUP-step
// group (groups aligned to multiples of GROUP) through t: the rotating frame of mimo_out_kernel.
template <typename Tin>
__global__ void __launch_bounds__(256) mimo_phase_kernel(const void* theta, float2* ph, int L, int N, long long total) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;   // (b, group, n)
  if (i >= total) return;
  const int n = int(i % N);
  const long long bg = i / N;
  const int G = (L + GROUP - 1) / GROUP;
  const long long b = bg / G;
  const int t0 = int(bg % G) * GROUP;
  const Tin* th = static_cast<const Tin*>(theta);
  float phi = 0.f;
  for (int t = t0; t < min(t0 + GROUP, L); ++t) {
    const long long e = (b * L + t) * N + n;
    phi += load_in<Tin>(th, e);
    float s, c;
    sincosf(phi, &s, &c);
    ph[e] = make_float2(c, s);
  }
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

static __global__ void __launch_bounds__(256) mimo_combine_kernel(const Params p) {
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

// The recurrence over chunk c with y, in a rotating frame. A block owns HB = OUT_THREADS / NPT
// heads of one (b, c), NPT = N / 2 threads per head; thread (head hl, state pair g) holds the
// states 2g, 2g + 1 as packed float32x2. Within each group of GROUP steps, Phi_t is the sum of
// theta from the group's first step, and with g_t = e^{-i Phi_t} h_t the decay is real. For
// each group the block first stages what its lanes share: per (t, channel, state pair)
// Bt = e^{-i Phi_t} Bm and Ct = e^{+i Phi_t} Cm, e^{i Phi} after the group's last step (the
// frame reset), per (t, head) x and dt (one step more for the trapezoid's look-ahead) and
// per t lam. The trapezoid carries k_t = g_{t-1} + mu_t V_{t-1} with
// mu_t = (1 - lam_t) dt_t, q_t = lam_t dt_t and V_t = sum_p x_t[p] Bt_t[p]:
//     g_t = r_t k_t + q_t V_t,   k_{t+1} = g_t + mu_{t+1} V_t,   y_t[p] = Re(sum_n Ct_t[n,p] g_t) + Dskip x_t[p],
// with mu_{t+1} = 0 at the chunk's last step (exp-Euler: q = dt, mu = 0, k = g), so that per
// state and step the work is the rank-P injection and the P outputs on state pairs. Each lane keeps
// its P partial outputs of the group's steps; a reduce-scatter over the head's NPT lanes then
// leaves every (step, channel) sum in one lane. Grid: (ceil(H / HB), C, B).
template <int N, int P> struct MimoStage {
  static_assert(N >= 2 && N <= 32, "mimo_out_kernel handles N = 2 .. 32");
  static constexpr int NPT = N / 2;                        // threads (state pairs) per head
  static constexpr int HB = OUT_THREADS / NPT;             // heads per block
};

template <typename Tin, int MODE, int N, int P>
__global__ void __launch_bounds__(OUT_THREADS, OutOcc<P>::MIN_BLOCKS) mimo_out_kernel(const Params p) {
  using MS = MimoStage<N, P>;
  constexpr int NPT = MS::NPT, HB = MS::HB;
  constexpr int E = GROUP * P;                   // (step, channel) entries of one group
  constexpr int HOLD = E >= NPT ? E / NPT : 1;
  constexpr int DUP = NPT > E ? NPT / E : 1;
  __shared__ float4 s_bt[GROUP][P][N / 2];       // (Btr_n, Btr_n+1, Bti_n, Bti_n+1)
  __shared__ float4 s_ct[GROUP][P][N / 2];       // (Ctr_n, Ctr_n+1, -Cti_n, -Cti_n+1)
  __shared__ float2 s_rs[N];                     // e^{i Phi} after the group's last step
  __shared__ __align__(16) float s_x[GROUP][HB][P];
  __shared__ float s_dt[GROUP + 1][HB];
  __shared__ float s_lam[GROUP + 1];

  const int tid = threadIdx.x;
  const int g = tid % NPT, hl = tid / NPT;
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
  const float2 A2 = f2(p.A[(long long)hc * N + 2 * g] * LOG2E, p.A[(long long)hc * N + 2 * g + 1] * LOG2E);
  const int tc = c * p.TC, te = min(p.L, tc + p.TC);

  // k at the chunk's first step, in the standard frame: h_in + mu_tc v_{tc-1}
  float2 kr = f2(0.f, 0.f), ki = f2(0.f, 0.f);
  if (p.C > 1 && valid) {
    const float2 e0 = rec_of(p, b, c, h, 2 * g)[0], e1 = rec_of(p, b, c, h, 2 * g + 1)[0];
    kr = f2(e0.x, e1.x);
    ki = f2(e0.y, e1.y);
  }
  if (MODE == 1 && tc > 0 && valid) {
    const float mu = (1.f - load_in<Tin>(LAM, b * p.L + tc)) * load_in<Tin>(DT, (b * p.L + tc) * p.H + h);
    const float2 v0 = v_before<Tin, MODE, P>(p, b, tc, h, 2 * g), v1 = v_before<Tin, MODE, P>(p, b, tc, h, 2 * g + 1);
    kr = fma2(f2(mu, mu), f2(v0.x, v1.x), kr);
    ki = fma2(f2(mu, mu), f2(v0.y, v1.y), ki);
  }

  // Staging, split so that a group's global loads are in flight while the previous group is
  // computed: `fetch` loads this thread's share of a group into registers (steps past te and
  // heads past H as zeros, so that those steps leave k unchanged and add nothing), `commit`
  // rotates Bm and Cm into the group's frame and stores everything in shared memory.
  constexpr int RIT = (GROUP * N + OUT_THREADS - 1) / OUT_THREADS;
  constexpr int XIT = (GROUP * HB * P + OUT_THREADS - 1) / OUT_THREADS;
  constexpr int DIT = ((GROUP + 1) * HB + OUT_THREADS - 1) / OUT_THREADS;
  float2 f_ph[RIT], f_bm[RIT][P], f_cm[RIT][P];
  float f_x[XIT], f_dt[DIT], f_lam = 0.f;
  auto fetch = [&](int t0) {
    const int ng = min(GROUP, te - t0);
#pragma unroll
    for (int it = 0; it < RIT; ++it) {
      const int k = tid + it * OUT_THREADS, i = k / N, n = k % N;
      const bool ok = k < GROUP * N && i < ng;
      f_ph[it] = ok ? p.phase[(b * p.L + t0 + i) * N + n] : f2(1.f, 0.f);
#pragma unroll
      for (int pp = 0; pp < P; ++pp) {
        const long long e = ((b * p.L + t0 + i) * N + n) * P + pp;
        f_bm[it][pp] = ok ? load_pair<Tin>(BM, e) : f2(0.f, 0.f);
        f_cm[it][pp] = ok ? load_pair<Tin>(CM, e) : f2(0.f, 0.f);
      }
    }
#pragma unroll
    for (int it = 0; it < XIT; ++it) {
      const int k = tid + it * OUT_THREADS, i = k / (HB * P), r = k % (HB * P), hh = h0 + r / P;
      f_x[it] = (k < GROUP * HB * P && i < ng && hh < p.H) ? load_in<Tin>(X, ((b * p.L + t0 + i) * p.H + h0) * P + r) : 0.f;
    }
#pragma unroll
    for (int it = 0; it < DIT; ++it) {
      const int k = tid + it * OUT_THREADS, i = k / HB, r = k % HB;
      f_dt[it] = (k < (GROUP + 1) * HB && t0 + i < te && h0 + r < p.H)
                     ? load_in<Tin>(DT, (b * p.L + t0 + i) * p.H + h0 + r) : 0.f;
    }
    if (MODE == 1 && tid <= GROUP) f_lam = t0 + tid < te ? load_in<Tin>(LAM, b * p.L + t0 + tid) : 0.f;
  };
  auto commit = [&](int t0) {
    const int ng = min(GROUP, te - t0);
#pragma unroll
    for (int it = 0; it < RIT; ++it) {
      const int k = tid + it * OUT_THREADS, i = k / N, n = k % N;
      if (k < GROUP * N) {
        const float cs = f_ph[it].x, sn = f_ph[it].y;
        if (i == ng - 1) s_rs[n] = f_ph[it];
        const int q = n >> 1, odd = n & 1;
#pragma unroll
        for (int pp = 0; pp < P; ++pp) {
          const float2 bb = f_bm[it][pp], cc = f_cm[it][pp];
          float* bt = reinterpret_cast<float*>(&s_bt[i][pp][q]);
          bt[odd] = cs * bb.x + sn * bb.y;
          bt[2 + odd] = cs * bb.y - sn * bb.x;
          float* ct = reinterpret_cast<float*>(&s_ct[i][pp][q]);
          ct[odd] = cs * cc.x - sn * cc.y;
          ct[2 + odd] = -(cs * cc.y + sn * cc.x);
        }
      }
    }
#pragma unroll
    for (int it = 0; it < XIT; ++it) {
      const int k = tid + it * OUT_THREADS;
      if (k < GROUP * HB * P) (&s_x[0][0][0])[k] = f_x[it];
    }
#pragma unroll
    for (int it = 0; it < DIT; ++it) {
      const int k = tid + it * OUT_THREADS;
      if (k < (GROUP + 1) * HB) (&s_dt[0][0])[k] = f_dt[it];
    }
    if (MODE == 1 && tid <= GROUP) s_lam[tid] = f_lam;
  };

  fetch(tc);
  commit(tc);
  __syncthreads();
  for (int t0 = tc; t0 < te; t0 += GROUP) {
    const int ng = min(GROUP, te - t0);
    const bool more = t0 + GROUP < te;
    if (more) fetch(t0 + GROUP);

    float part[1][E];
#pragma unroll
    for (int i = 0; i < GROUP; ++i) {
      const float dtt = s_dt[i][hl];
      const float2 r = ex2_pair(mul2(f2(dtt, dtt), A2));
      // exp-Euler: w = dt x, g = k; trapezoid: V = sum_p x Bt, g = r k + q V, k = g + mu V
      const float wq = MODE == 1 ? 1.f : dtt;
      float2 sr = f2(0.f, 0.f), si = f2(0.f, 0.f);
#pragma unroll
      for (int pp = 0; pp < P; ++pp) {
        const float w = wq * s_x[i][hl][pp];
        const float4 bt = s_bt[i][pp][g];
        sr = fma2(f2(w, w), f2(bt.x, bt.y), sr);
        si = fma2(f2(w, w), f2(bt.z, bt.w), si);
      }
      float2 gr, gi;
      if (MODE == 1) {
        const float q = s_lam[i] * dtt, mu1 = (1.f - s_lam[i + 1]) * s_dt[i + 1][hl];
        gr = fma2(r, kr, mul2(f2(q, q), sr));
        gi = fma2(r, ki, mul2(f2(q, q), si));
        kr = fma2(f2(mu1, mu1), sr, gr);
        ki = fma2(f2(mu1, mu1), si, gi);
      } else {
        kr = fma2(r, kr, sr);
        ki = fma2(r, ki, si);
        gr = kr;
        gi = ki;
      }
#pragma unroll
      for (int pp = 0; pp < P; ++pp) {
        const float4 ct = s_ct[i][pp][g];
        const float2 o = fma2(f2(ct.x, ct.y), gr, mul2(f2(ct.z, ct.w), gi));
        part[0][i * P + pp] = o.x + o.y;
      }
    }
    {  // frame reset: back to the standard frame after the group's last step
      const float2 e0 = s_rs[2 * g], e1 = s_rs[2 * g + 1];
      const float2 cc = f2(e0.x, e1.x), ss = f2(e0.y, e1.y), nss = f2(-e0.y, -e1.y);
      const float2 nr = fma2(cc, kr, mul2(nss, ki)), ni = fma2(cc, ki, mul2(ss, kr));
      kr = nr;
      ki = ni;
    }
    const int base = butterfly<NPT, 1, E>(part, g);
    if ((g % DUP) == 0 && valid) {
#pragma unroll
      for (int k = 0; k < HOLD; ++k) {
        const int e = base + k, i = e / P, pp = e % P;
        if (i < ng) p.y[((b * p.L + t0 + i) * p.H + h) * P + pp] = fmaf(p.Dskip[(long long)h * P + pp], s_x[i][hl][pp], part[0][k]);
      }
    }
    __syncthreads();
    if (more) {
      commit(t0 + GROUP);
      __syncthreads();
    }
  }
}

}  // namespace mimo
}  // namespace csscan
