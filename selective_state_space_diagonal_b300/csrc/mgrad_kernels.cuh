// mgrad_kernels.cuh -- reverse-mode gradients of the MIMO scan (csscan_forward_mimo, from the
// zero state), with the states regenerated from checkpoints instead of stored.
//
// The forward ("Mamba-3 paper story", MIMO section, read as in csscan.h): per (b, head h,
// state n), a_t = exp(dt_t A[h,n] + i theta_t[n]), v_t = sum_p Bm_t[n,p] x_t[h,p],
//   h_t = a_t h_{t-1} + c1_t v_t + c2_t a_t v_{t-1},  y_t[h,p] = Re(sum_n Cm_t[n,p] h_t) + Dskip[h,p] x_t[h,p]
// with c1 = dt, c2 = 0 (exp-Euler) or c1 = lam dt, c2 = (1 - lam) dt (trapezoid). With
// G(z) = dl/dRe z + i dl/dIm z for l = sum dy y, walking t from the end:
//   ghat_t   = sum_p dy_t[p] conj(Cm_t[n,p]) + conj(a_{t+1}) ghat_{t+1}
//   G(v_t)   = c1_t ghat_t + c2_{t+1} conj(a_{t+1}) ghat_{t+1}
//   G(a_t)   = ghat_t conj(h_{t-1}) + c2_t ghat_t conj(v_{t-1}),   G(z_t) = conj(a_t) G(a_t)
//   dCm_t[n,p] += dy_t[p] conj(h_t),  dBm_t[n,p] += x_t[p] G(v_t),  dx_t[p] = sum_n Re(conj(Bm_t[n,p]) G(v_t)) + Dskip dy_t[p]
//   dA += dt Re G(z), ddt_t = lam Re(conj(v_t) ghat_t) + (1 - lam) Re(conj(a_t v_{t-1}) ghat_t) + sum_n A Re G(z)
//   (exp-Euler: ddt_t = sum_n Re(conj(v_t) ghat_t) + sum_n A Re G(z)), dtheta_t += Im G(z),
//   dlam_t += dt (Re(conj(v_t) ghat_t) - Re(conj(a_t v_{t-1}) ghat_t)), dDskip += dy x.
//
// Kernels (a thread per (b, h, n), the N lanes of a head contiguous, 128 / N heads per block; no
// time chunks: a thread walks the whole sequence, so the parallelism is B H N threads):
//   mckpt_kernel  the forward recurrence, storing the state before every 8-step segment;
//   mgrad_kernel  per segment, last to first: regenerate the segment's states from its
//                 checkpoint, walk it backwards; sums over n of a (t, h) by shuffles across the
//                 head's lanes; sums over h of a (t, n) by shuffles across the warp's heads, then
//                 over the block's warps through shared memory once per segment, then one atomic
//                 add per value and block.
// e^{i theta} comes from bwd::rot_kernel's table (B, L, N), shared by every head.
#pragma once

#include "backward_kernels.cuh"

namespace csscan {
namespace mgrad {

constexpr int SEG = 8;
constexpr int THREADS = 128;
constexpr float LOG2E = 1.4426950408889634f;

struct Params {
  const void* x;        // (B, L, H, P) input dtype
  const void* dt;       // (B, L, H)
  const void* Bm;       // (B, L, N, P, 2)
  const void* Cm;       // (B, L, N, P, 2)
  const void* lam;      // (B, L) trapezoid only
  const float* A;       // (H, N)
  const float* Dskip;   // (H, P)
  const float* dy;      // (B, L, H, P)
  const float2* rot;    // (B, L, N) e^{i theta}
  float2* ckpt;         // (B, S, H, N) state before segment s >= 1
  float* dx;            // (B, L, H, P)   written
  float* ddt;           // (B, L, H)      written
  float* dA;            // (H, N)         accumulated
  float* dBm;           // (B, L, N, P, 2) accumulated
  float* dCm;           // (B, L, N, P, 2) accumulated
  float* dtheta;        // (B, L, N)      accumulated
  float* dlam;          // (B, L)         accumulated (trapezoid)
  float* dD;            // (H, P)         accumulated
  int B, L, H, N, S;
};

// v_t[n] = sum_p Bm_t[n, p] x_t[h, p] of this thread's (b, t, h, n); zero outside the sequence
template <typename Tin, int P>
__device__ __forceinline__ float2 mimo_v(const Params& p, long long b, int t, int h, int n) {
  if (t < 0 || t >= p.L) return make_float2(0.f, 0.f);
  const Tin* X = static_cast<const Tin*>(p.x) + ((b * p.L + t) * p.H + h) * P;
  const Tin* BM = static_cast<const Tin*>(p.Bm) + ((b * p.L + t) * p.N + n) * P * 2;
  float vr = 0.f, vi = 0.f;
#pragma unroll
  for (int q = 0; q < P; ++q) {
    const float xv = load_in<Tin>(X, q);
    vr = fmaf(load_in<Tin>(BM, 2 * q), xv, vr);
    vi = fmaf(load_in<Tin>(BM, 2 * q + 1), xv, vi);
  }
  return make_float2(vr, vi);
}

// a_t and the injection weights (c1, c2) of step t for head h, state n
template <typename Tin, int MODE>
__device__ __forceinline__ void mimo_step_coef(const Params& p, long long b, int t, int h, int n, float a2,
                                               float2& a, float& c1, float& c2, float& dtt, float& lm) {
  dtt = load_in<Tin>(static_cast<const Tin*>(p.dt), (b * p.L + t) * p.H + h);
  lm = MODE == 1 ? load_in<Tin>(static_cast<const Tin*>(p.lam), b * p.L + t) : 0.f;
  const float r = ex2_approx(dtt * a2);
  const float2 ro = p.rot[(b * p.L + t) * p.N + n];
  a = make_float2(r * ro.x, r * ro.y);
  c1 = MODE == 1 ? lm * dtt : dtt;
  c2 = MODE == 1 ? (1.f - lm) * dtt : 0.f;
}

// Forward recurrence per (b, h, n), storing the state before every segment s >= 1.
template <typename Tin, int MODE, int P>
__global__ void __launch_bounds__(THREADS) mckpt_kernel(const Params p) {
  const int hpb = THREADS / p.N;
  const int n = threadIdx.x % p.N;
  const int h = blockIdx.x * hpb + threadIdx.x / p.N;
  const long long b = blockIdx.y;
  if (h >= p.H) return;
  const float a2 = p.A[(long long)h * p.N + n] * LOG2E;
  float hr = 0.f, hi = 0.f;
  float2 vp = make_float2(0.f, 0.f);
  for (int t = 0; t < p.L; ++t) {
    if (t > 0 && t % SEG == 0) p.ckpt[((b * p.S + t / SEG) * p.H + h) * p.N + n] = make_float2(hr, hi);
    float2 a;
    float c1, c2, dtt, lm;
    mimo_step_coef<Tin, MODE>(p, b, t, h, n, a2, a, c1, c2, dtt, lm);
    const float2 v = mimo_v<Tin, P>(p, b, t, h, n);
    // u = c1 v + c2 a v_{t-1}
    const float ur = fmaf(c1, v.x, c2 * (a.x * vp.x - a.y * vp.y));
    const float ui = fmaf(c1, v.y, c2 * (a.x * vp.y + a.y * vp.x));
    const float nr = fmaf(a.x, hr, fmaf(-a.y, hi, ur));
    const float ni = fmaf(a.x, hi, fmaf(a.y, hr, ui));
    hr = nr;
    hi = ni;
    vp = v;
  }
}

// Shared memory of mgrad_kernel: per segment step, the block's partial sums over its heads of
// dBm, dCm (re, im) per (n, p), dtheta per n and dlam.
template <int P>
struct MGradSmem {
  static constexpr int bytes(int N) { return SEG * N * P * 4 * 4 + SEG * N * 4 + SEG * 4; }
};

template <typename Tin, int MODE, int P>
__global__ void __launch_bounds__(THREADS) mgrad_kernel(const Params p) {
  extern __shared__ __align__(16) float s_mem[];
  const int N = p.N;
  float* s_bc = s_mem;                              // [SEG][N][P][4]: dBm re, im, dCm re, im
  float* s_th = s_mem + SEG * N * P * 4;            // [SEG][N]
  float* s_lm = s_th + SEG * N;                     // [SEG]
  const int hpb = THREADS / N;
  const int tid = threadIdx.x;
  const int n = tid % N;
  const int h = blockIdx.x * hpb + tid / N;
  const bool valid = h < p.H;
  const int hh = valid ? h : 0;
  const long long b = blockIdx.y;
  const unsigned lane = tid & 31u;
  // the N lanes of this head within the warp (N <= 32 divides 32)
  const unsigned gmask = N >= 32 ? 0xffffffffu : (((1u << N) - 1u) << (lane & ~unsigned(N - 1)));
  const float Ad = valid ? p.A[(long long)hh * N + n] : 0.f;
  // sum over the 32 / N heads of this warp (lanes n of every head), at every lane
  auto head_sum = [&](float v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
      if (o >= N) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  };
  const float a2 = Ad * LOG2E;
  for (int k = tid; k < SEG * N * P * 4 + SEG * N + SEG; k += THREADS) s_mem[k] = 0.f;

  float cgr = 0.f, cgi = 0.f;   // conj(a_{t+1}) ghat_{t+1}
  float cvr = 0.f, cvi = 0.f;   // c2_{t+1} conj(a_{t+1}) ghat_{t+1} (the trapezoid's term of G(v_t))
  float dA_acc = 0.f;
  float dD_acc[P];   // lane n = 0: dDskip[h, :]
#pragma unroll
  for (int q = 0; q < P; ++q) dD_acc[q] = 0.f;
  __syncthreads();

#pragma unroll 1
  for (int s = p.S - 1; s >= 0; --s) {
    const int t0 = s * SEG;
    const int nt = min(SEG, p.L - t0);
    // ---- regenerate the segment's states (and v) from its checkpoint
    float hsr[SEG], hsi[SEG], vsr[SEG], vsi[SEG];
    float h0r = 0.f, h0i = 0.f;
    if (valid && s > 0) {
      const float2 c = p.ckpt[((b * p.S + s) * p.H + hh) * N + n];
      h0r = c.x;
      h0i = c.y;
    }
    const float2 vprev0 = MODE == 1 ? mimo_v<Tin, P>(p, b, t0 - 1, hh, n) : make_float2(0.f, 0.f);
    {
      float hr = h0r, hi = h0i;
      float2 vp = vprev0;
#pragma unroll
      for (int i = 0; i < SEG; ++i) {
        float2 v = make_float2(0.f, 0.f);
        if (i < nt && valid) {
          float2 a;
          float c1, c2, dtt, lm;
          mimo_step_coef<Tin, MODE>(p, b, t0 + i, hh, n, a2, a, c1, c2, dtt, lm);
          v = mimo_v<Tin, P>(p, b, t0 + i, hh, n);
          const float ur = fmaf(c1, v.x, c2 * (a.x * vp.x - a.y * vp.y));
          const float ui = fmaf(c1, v.y, c2 * (a.x * vp.y + a.y * vp.x));
          const float nr = fmaf(a.x, hr, fmaf(-a.y, hi, ur));
          const float ni = fmaf(a.x, hi, fmaf(a.y, hr, ui));
          hr = nr;
          hi = ni;
        }
        hsr[i] = hr;
        hsi[i] = hi;
        vsr[i] = v.x;
        vsi[i] = v.y;
        vp = v;
      }
    }
    // ---- backwards through the segment
#pragma unroll
    for (int i = SEG - 1; i >= 0; --i) {
      if (i >= nt) continue;
      const int t = t0 + i;
      float2 a = make_float2(0.f, 0.f);
      float c1 = 0.f, c2 = 0.f, dtt = 0.f, lm = 0.f;
      if (valid) mimo_step_coef<Tin, MODE>(p, b, t, hh, n, a2, a, c1, c2, dtt, lm);
      const long long th = (b * p.L + t) * p.H + hh;
      const long long tn = (b * p.L + t) * N + n;
      const Tin* X = static_cast<const Tin*>(p.x) + th * P;
      const Tin* BM = static_cast<const Tin*>(p.Bm) + tn * P * 2;
      const Tin* CM = static_cast<const Tin*>(p.Cm) + tn * P * 2;
      const float* DY = p.dy + th * P;
      const float hr = hsr[i], hi = hsi[i];
      const float hpr = i > 0 ? hsr[i > 0 ? i - 1 : 0] : h0r;
      const float hpi = i > 0 ? hsi[i > 0 ? i - 1 : 0] : h0i;
      const float vr = vsr[i], vi = vsi[i];
      const float vpr = i > 0 ? vsr[i > 0 ? i - 1 : 0] : vprev0.x;
      const float vpi = i > 0 ? vsi[i > 0 ? i - 1 : 0] : vprev0.y;
      float dys[P], xs[P];
      float gr = cgr, gi = cgi;
#pragma unroll
      for (int q = 0; q < P; ++q) {
        dys[q] = valid ? DY[q] : 0.f;
        xs[q] = valid ? load_in<Tin>(X, q) : 0.f;
        const float cr = load_in<Tin>(CM, 2 * q), ci = load_in<Tin>(CM, 2 * q + 1);
        gr = fmaf(dys[q], cr, gr);     // + dy conj(Cm)
        gi = fmaf(-dys[q], ci, gi);
      }
      // G(v_t) = c1 ghat + c2_{t+1} conj(a_{t+1}) ghat_{t+1}
      const float Gvr = fmaf(c1, gr, cvr), Gvi = fmaf(c1, gi, cvi);
      float dc1 = vr * gr + vi * gi;   // Re(conj(v_t) ghat_t)
      float Gar = gr * hpr + gi * hpi, Gai = gi * hpr - gr * hpi;   // ghat conj(h_{t-1})
      float dc2 = 0.f;
      float ncvr = 0.f, ncvi = 0.f;
      if (MODE == 1) {
        Gar = fmaf(c2, gr * vpr + gi * vpi, Gar);   // + c2 ghat conj(v_{t-1})
        Gai = fmaf(c2, gi * vpr - gr * vpi, Gai);
        const float wr = a.x * vpr - a.y * vpi, wi = a.x * vpi + a.y * vpr;   // a_t v_{t-1}
        dc2 = wr * gr + wi * gi;
        ncvr = c2 * (a.x * gr + a.y * gi);   // c2 conj(a) ghat
        ncvi = c2 * (a.x * gi - a.y * gr);
      }
      float dxs[P];
#pragma unroll
      for (int q = 0; q < P; ++q) {
        const float br = load_in<Tin>(BM, 2 * q), bi = load_in<Tin>(BM, 2 * q + 1);
        dxs[q] = br * Gvr + bi * Gvi;   // Re(conj(Bm) G(v))
        // dBm (x G(v)) and dCm (dy conj(h)) summed over the warp's heads first (an absent
        // head contributes zeros), then one shared-memory add per warp
        const float bmr = head_sum(xs[q] * Gvr), bmi = head_sum(xs[q] * Gvi);
        const float cmr = head_sum(dys[q] * hr), cmi = head_sum(-dys[q] * hi);
        if (lane < unsigned(N)) {
          float* sb = s_bc + ((i * N + n) * P + q) * 4;
          atomicAdd(sb + 0, bmr);
          atomicAdd(sb + 1, bmi);
          atomicAdd(sb + 2, cmr);
          atomicAdd(sb + 3, cmi);
        }
      }
      const float Gzr = a.x * Gar + a.y * Gai;   // conj(a) G(a)
      const float Gzi = a.x * Gai - a.y * Gar;
      dA_acc = fmaf(dtt, Gzr, dA_acc);
      float dz = Ad * Gzr;
      const float gth = head_sum(Gzi);
      if (lane < unsigned(N)) atomicAdd(&s_th[i * N + n], gth);
      // sums over the head's N lanes: dc1, dc2, dz and dx[p]
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        if (o < N) {
          dc1 += __shfl_xor_sync(gmask, dc1, o);
          dc2 += __shfl_xor_sync(gmask, dc2, o);
          dz += __shfl_xor_sync(gmask, dz, o);
#pragma unroll
          for (int q = 0; q < P; ++q) dxs[q] += __shfl_xor_sync(gmask, dxs[q], o);
        }
      }
      if (valid && n == 0) {
        const float* Dk = p.Dskip + (long long)hh * P;
        float* dxo = p.dx + th * P;
#pragma unroll
        for (int q = 0; q < P; ++q) dxo[q] = fmaf(Dk[q], dys[q], dxs[q]);
        p.ddt[th] = MODE == 1 ? fmaf(lm, dc1, fmaf(1.f - lm, dc2, dz)) : dc1 + dz;
        if (MODE == 1) atomicAdd(&s_lm[i], dtt * (dc1 - dc2));
#pragma unroll
        for (int q = 0; q < P; ++q) dD_acc[q] = fmaf(dys[q], xs[q], dD_acc[q]);
      }
      // carries to step t - 1
      cgr = a.x * gr + a.y * gi;   // conj(a) ghat
      cgi = a.x * gi - a.y * gr;
      cvr = ncvr;
      cvi = ncvi;
    }
    // ---- the segment's sums over the block's heads: one atomic add per value
    __syncthreads();
    for (int k = tid; k < nt * N * P * 4; k += THREADS) {
      const int i = k / (N * P * 4), rem = k % (N * P * 4);
      const int nn = rem / (P * 4), q = (rem / 4) % P, c = rem % 4;
      const long long e = (((b * p.L + t0 + i) * N + nn) * P + q) * 2 + (c & 1);
      atomicAdd((c < 2 ? p.dBm : p.dCm) + e, s_bc[k]);
      s_bc[k] = 0.f;
    }
    for (int k = tid; k < nt * N; k += THREADS) {
      const int i = k / N, nn = k % N;
      atomicAdd(&p.dtheta[(b * p.L + t0 + i) * N + nn], s_th[k]);
      s_th[k] = 0.f;
    }
    if (MODE == 1 && tid < nt) {
      atomicAdd(&p.dlam[b * p.L + t0 + tid], s_lm[tid]);
      s_lm[tid] = 0.f;
    }
    __syncthreads();
  }
  if (valid) {
    atomicAdd(&p.dA[(long long)hh * N + n], dA_acc);
    if (n == 0) {
#pragma unroll
      for (int q = 0; q < P; ++q) atomicAdd(&p.dD[(long long)hh * P + q], dD_acc[q]);
    }
  }
}

}  // namespace mgrad
}  // namespace csscan
