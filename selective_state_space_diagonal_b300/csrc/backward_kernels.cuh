// backward_kernels.cuh -- reverse-mode gradients of the forward scan (zero initial state, no
// step -1 halo), with the states regenerated from checkpoints instead of stored.
//
// "Complex parallel scan" (sections 一个问题，两种命运 and 硬件落地的挑战) describes the training
// pattern this serves: one forward over the whole sequence, one backward sweep, states
// recomputed on the fly rather than written out, and a backward kernel beside the fused
// forward one. The formulas are reverse-mode differentiation of the recurrence of
// scan_kernels.cuh. With G(z) = dl/dRe z + i dl/dIm z for l = sum dy * y:
//   adjoint        ghat_t = dy_t conj(Cc_t) + conj(a_{t+1}) ghat_{t+1},   ghat_L = 0
//   transition     G(a_t) = ghat_t conj(h_{t-1})  (+ ghat_t (1-lam_t) dt_t x_{t-1} conj(Bc_{t-1}))
//                  G(z_t) = conj(a_t) G(a_t),  z_t = dt_t A + i theta_t
//                  dA += dt_t Re G(z_t),  ddt_t += A Re G(z_t),  dtheta_t += Im G(z_t)
//   injection      exp-Euler:  u_t = dt_t x_t Bc_t
//                  trapezoid:  u_t = lam_t dt_t x_t Bc_t + (1-lam_t) dt_t x_{t-1} a_t Bc_{t-1}
//                  with P_t = Re(conj(Bc_t) ghat_t) and R_t = Re(conj(a_t Bc_{t-1}) ghat_t)
//   output         dCc_t += dy_t conj(h_t),  dx_t += Dskip dy_t,  dDskip += dy_t x_t
//
// Three kernels:
//   rot_kernel    e^{i theta} per (b, t, n), shared by every channel;
//   ckpt_kernel   one thread per (b, d, n) runs the forward recurrence and stores the state
//                 before every segment of SEG steps;
//   grad_kernel   a thread owns one state n of K channels of one batch row. For each segment,
//                 last to first, and each of its channels it recomputes the segment's SEG states
//                 from the checkpoint into registers, then walks the segment backwards. Sums over
//                 n (dx, ddt, dlam) use a butterfly over the N lanes of a channel; sums over d
//                 (dBc, dCc, dtheta, dlam) accumulate in registers across the thread's channels,
//                 then across lanes and warps, and leave the block as one atomic add per value.
#pragma once

#include "device_util.cuh"

namespace csscan {
namespace bwd {

constexpr int SEG = 8;          // steps per recomputed segment = checkpoint spacing
constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr float LOG2E = 1.4426950408889634f;

struct Params {
  const void* x;       // (B, L, D) input dtype
  const void* dt;      // (B, L, D)
  const void* Bc;      // (B, L, N, 2)
  const void* Cc;      // (B, L, N, 2)
  const void* lam;     // (B, L) trapezoid only
  const float* A;      // (D, N)
  const float* Dskip;  // (D)
  const float* dy;     // (B, L, D)
  float* dx;           // (B, L, D)      written
  float* ddt;          // (B, L, D)      written
  float* dA;           // (D, N)         accumulated (zeroed by the host)
  float* dBc;          // (B, L, N, 2)   accumulated
  float* dCc;          // (B, L, N, 2)   accumulated
  float* dtheta;       // (B, L, N)      accumulated
  float* dlam;         // (B, L)         accumulated (trapezoid only)
  float* dD;           // (D)            accumulated
  const float2* rot;   // (B, L, N)      e^{i theta}
  float2* ckpt;        // (B, S, D, N)   state before segment s (s >= 1)
  int B, L, D, N, S;
};

// Channels per block of grad_kernel: K slots per thread x (32 / N) channels per warp x WARPS.
template <int N> struct GradTile {
  static_assert(N >= 2 && N <= 32 && (N & (N - 1)) == 0, "grad_kernel handles N = 2 .. 32");
  static constexpr int CPW = 32 / N;
  static constexpr int K = N < 16 ? N : 16;
  static constexpr int CB = K * CPW * WARPS;
};

template <typename Tin>
__global__ void __launch_bounds__(256) rot_kernel(const void* theta, float2* rot, long long total) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= total) return;
  float s, c;
  sincosf(load_in<Tin>(static_cast<const Tin*>(theta), i), &s, &c);
  rot[i] = make_float2(c, s);
}

// Forward recurrence per (b, d, n), storing h_{s SEG - 1} for s = 1 .. S-1.
template <typename Tin, int MODE>
__global__ void __launch_bounds__(256) ckpt_kernel(const Params p) {
  const long long gid = (long long)blockIdx.x * 256 + threadIdx.x;
  if (gid >= (long long)p.B * p.D * p.N) return;
  const int n = int(gid % p.N);
  const long long bd = gid / p.N;
  const int d = int(bd % p.D);
  const long long b = bd / p.D;
  const Tin* X = static_cast<const Tin*>(p.x);
  const Tin* DT = static_cast<const Tin*>(p.dt);
  const Tin* BC = static_cast<const Tin*>(p.Bc);
  const Tin* LAM = static_cast<const Tin*>(p.lam);
  const float a2 = p.A[(long long)d * p.N + n] * LOG2E;
  float hr = 0.f, hi = 0.f, xp = 0.f, bpr = 0.f, bpi = 0.f;
  for (int t = 0; t < p.L; ++t) {
    if (t > 0 && t % SEG == 0) p.ckpt[((b * p.S + t / SEG) * p.D + d) * p.N + n] = make_float2(hr, hi);
    const long long td = (b * p.L + t) * p.D + d;
    const long long tn = (b * p.L + t) * p.N + n;
    const float xt = load_in<Tin>(X, td), dtt = load_in<Tin>(DT, td);
    const float2 ro = p.rot[tn];
    const float r = ex2_approx(dtt * a2);
    const float ar = r * ro.x, ai = r * ro.y;
    const float br = load_in<Tin>(BC, 2 * tn), bi = load_in<Tin>(BC, 2 * tn + 1);
    float ur, ui;
    if (MODE == 0) {
      const float w = dtt * xt;
      ur = w * br;
      ui = w * bi;
    } else {
      const float lm = load_in<Tin>(LAM, b * p.L + t);
      const float w = lm * dtt * xt, c2 = (1.f - lm) * dtt * xp;
      ur = w * br + c2 * (ar * bpr - ai * bpi);
      ui = w * bi + c2 * (ar * bpi + ai * bpr);
      xp = xt;
      bpr = br;
      bpi = bi;
    }
    const float nr = fmaf(ar, hr, fmaf(-ai, hi, ur));
    const float ni = fmaf(ar, hi, fmaf(ai, hr, ui));
    hr = nr;
    hi = ni;
  }
}

// Reduce-scatter of V[SEG] over the N lanes of a channel group (lane bits below N): rounds
// with the high masks halve the array (each lane keeps one half and adds its partner's copy of
// it), rounds with the remaining masks add whole values. Afterwards a lane holds the group sum
// for t offsets base .. base + HOLD - 1.
template <int N, int NARR>
__device__ __forceinline__ int butterfly(float (&v)[NARR][SEG], int lane) {
  int base = 0;
  int len = SEG;
#pragma unroll
  for (int m = N / 2; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
    if (len > 1) {
      const int half = len / 2;
#pragma unroll
      for (int k = 0; k < NARR; ++k)
#pragma unroll
        for (int i = 0; i < SEG / 2; ++i)
          if (i < half) {
            const float send = upper ? v[k][i] : v[k][i + half];
            const float keep = upper ? v[k][i + half] : v[k][i];
            v[k][i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
      if (upper) base += half;
      len = half;
    } else {
#pragma unroll
      for (int k = 0; k < NARR; ++k) v[k][0] += __shfl_xor_sync(0xffffffffu, v[k][0], m);
    }
  }
  return base;
}

template <typename Tin, int MODE, int N>
__global__ void __launch_bounds__(THREADS) grad_kernel(const Params p) {
  using GT = GradTile<N>;
  constexpr int CPW = GT::CPW, K = GT::K, CB = GT::CB;
  constexpr int HOLD = SEG >= N ? SEG / N : 1;     // t values a lane holds after the butterfly
  constexpr int DUP = N > SEG ? N / SEG : 1;        // lanes holding the same t values
  // per (thread, slot) state carried from segment to segment: conj(a_{t+1}) ghat_{t+1} (re, im),
  // R_{t+1}, the dA partial sum; and the dDskip partial sum
  __shared__ float4 s_state[K][THREADS];
  __shared__ float s_dD[K][THREADS];
  __shared__ float s_acc[SEG][N][5];   // per (t, n): dBc re, im, dCc re, im, dtheta
  __shared__ float s_lam[SEG];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = lane % N, cl = lane / N;
  const long long b = blockIdx.y;
  const int dbase = blockIdx.x * CB;
  const Tin* X = static_cast<const Tin*>(p.x);
  const Tin* DT = static_cast<const Tin*>(p.dt);
  const Tin* BC = static_cast<const Tin*>(p.Bc);
  const Tin* CC = static_cast<const Tin*>(p.Cc);
  const Tin* LAM = static_cast<const Tin*>(p.lam);
  const long long L = p.L, D = p.D;

#pragma unroll 1
  for (int j = 0; j < K; ++j) {
    s_state[j][tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    s_dD[j][tid] = 0.f;
  }
  for (int k = tid; k < SEG * N * 5; k += THREADS) (&s_acc[0][0][0])[k] = 0.f;
  if (tid < SEG) s_lam[tid] = 0.f;
  __syncthreads();

#pragma unroll 1
  for (int s = p.S - 1; s >= 0; --s) {
    const int ts = s * SEG;
    const int nt = min(SEG, p.L - ts);
    float acc[SEG][5];
#pragma unroll
    for (int i = 0; i < SEG; ++i)
#pragma unroll
      for (int c = 0; c < 5; ++c) acc[i][c] = 0.f;
    float lam_acc[HOLD];
#pragma unroll
    for (int h = 0; h < HOLD; ++h) lam_acc[h] = 0.f;
    int hold_base = 0;

#pragma unroll 1
    for (int j = 0; j < K; ++j) {
      const int d = dbase + (j * WARPS + warp) * CPW + cl;
      const bool valid = d < p.D;
      const long long dd = valid ? d : 0;
      // an absent channel runs with x = dy = 0, which makes every contribution exactly zero
      const float vmask = valid ? 1.f : 0.f;
      const float a2 = p.A[dd * N + n] * LOG2E;
      const float Ad = p.A[dd * N + n];
      const float Ds = p.Dskip[dd];
      float4 st = s_state[j][tid];
      float cgr = st.x, cgi = st.y, Rn = st.z, dA_acc = st.w;
      float dD_acc = s_dD[j][tid];

      // ---- forward: the segment's states from the checkpoint
      float h0r = 0.f, h0i = 0.f;
      if (s > 0 && valid) {
        const float2 c = p.ckpt[((b * p.S + s) * D + dd) * N + n];
        h0r = c.x;
        h0i = c.y;
      }
      float hsr[SEG], hsi[SEG];
      {
        float hr = h0r, hi = h0i;
        float xp = 0.f, bpr = 0.f, bpi = 0.f;
        if (MODE == 1 && ts > 0) {
          const long long tn = (b * L + ts - 1) * N + n;
          xp = vmask * load_in<Tin>(X, (b * L + ts - 1) * D + dd);
          bpr = load_in<Tin>(BC, 2 * tn);
          bpi = load_in<Tin>(BC, 2 * tn + 1);
        }
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
          if (i < nt) {
            const long long t = ts + i;
            const long long td = (b * L + t) * D + dd;
            const long long tn = (b * L + t) * N + n;
            const float xt = vmask * load_in<Tin>(X, td), dtt = load_in<Tin>(DT, td);
            const float2 ro = p.rot[tn];
            const float r = ex2_approx(dtt * a2);
            const float ar = r * ro.x, ai = r * ro.y;
            const float br = load_in<Tin>(BC, 2 * tn), bi = load_in<Tin>(BC, 2 * tn + 1);
            float ur, ui;
            if (MODE == 0) {
              const float w = dtt * xt;
              ur = w * br;
              ui = w * bi;
            } else {
              const float lm = load_in<Tin>(LAM, b * L + t);
              const float w = lm * dtt * xt, c2 = (1.f - lm) * dtt * xp;
              ur = w * br + c2 * (ar * bpr - ai * bpi);
              ui = w * bi + c2 * (ar * bpi + ai * bpr);
              xp = xt;
              bpr = br;
              bpi = bi;
            }
            const float nr = fmaf(ar, hr, fmaf(-ai, hi, ur));
            const float ni = fmaf(ar, hi, fmaf(ai, hr, ui));
            hr = nr;
            hi = ni;
          }
          hsr[i] = hr;
          hsi[i] = hi;
        }
      }

      // ---- backward through the segment
      float g3[3][SEG];   // per t: dx, ddt, dlam partial sums over this lane's state
      // (1 - lam_{t+1}) dt_{t+1}: the next step's beta weight (zero past the end)
      float mnext = 0.f;
      if (MODE == 1 && ts + nt < p.L) {
        const long long t1 = ts + nt;
        mnext = (1.f - load_in<Tin>(LAM, b * L + t1)) * load_in<Tin>(DT, (b * L + t1) * D + dd);
      }
#pragma unroll
      for (int i = SEG - 1; i >= 0; --i) {
        g3[0][i] = 0.f;
        g3[1][i] = 0.f;
        g3[2][i] = 0.f;
        if (i < nt) {
          const long long t = ts + i;
          const long long td = (b * L + t) * D + dd;
          const long long tn = (b * L + t) * N + n;
          const float xt = vmask * load_in<Tin>(X, td), dtt = load_in<Tin>(DT, td);
          const float dyt = vmask * p.dy[td];
          const float2 ro = p.rot[tn];
          const float r = ex2_approx(dtt * a2);
          const float ar = r * ro.x, ai = r * ro.y;
          const float hr = hsr[i], hi = hsi[i];
          const float hpr = i > 0 ? hsr[i > 0 ? i - 1 : 0] : h0r;
          const float hpi = i > 0 ? hsi[i > 0 ? i - 1 : 0] : h0i;
          const float ccr = load_in<Tin>(CC, 2 * tn), cci = load_in<Tin>(CC, 2 * tn + 1);
          const float br = load_in<Tin>(BC, 2 * tn), bi = load_in<Tin>(BC, 2 * tn + 1);
          // adjoint of h_t
          const float gr = fmaf(dyt, ccr, cgr);
          const float gi = fmaf(-dyt, cci, cgi);
          // output: dCc_t += dy conj(h_t)
          acc[i][2] = fmaf(dyt, hr, acc[i][2]);
          acc[i][3] = fmaf(-dyt, hi, acc[i][3]);
          // transition through h_t = a_t h_{t-1}
          float Gar = gr * hpr + gi * hpi;
          float Gai = gi * hpr - gr * hpi;
          const float P = br * gr + bi * gi;
          float R = 0.f, gx, gdt, glam = 0.f;
          if (MODE == 0) {
            const float coef = dtt * xt;
            acc[i][0] = fmaf(coef, gr, acc[i][0]);
            acc[i][1] = fmaf(coef, gi, acc[i][1]);
            gx = dtt * P;
            gdt = xt * P;
          } else {
            const float lm = load_in<Tin>(LAM, b * L + t);
            const float coef = lm * dtt * xt;
            const float cn = mnext * xt;   // beta_{t+1} reaches Bc_t through conj(a_{t+1}) ghat_{t+1}
            acc[i][0] += coef * gr + cn * cgr;
            acc[i][1] += coef * gi + cn * cgi;
            float xp = 0.f;
            if (t > 0) {
              const long long tp = tn - N;
              xp = vmask * load_in<Tin>(X, td - D);
              const float bpr = load_in<Tin>(BC, 2 * tp), bpi = load_in<Tin>(BC, 2 * tp + 1);
              const float c2 = (1.f - lm) * dtt * xp;
              const float vr = ar * bpr - ai * bpi, vi = ar * bpi + ai * bpr;   // a_t Bc_{t-1}
              R = vr * gr + vi * gi;
              Gar += c2 * (gr * bpr + gi * bpi);
              Gai += c2 * (gi * bpr - gr * bpi);
            }
            gx = lm * dtt * P + mnext * Rn;
            gdt = lm * xt * P + (1.f - lm) * xp * R;
            glam = dtt * (xt * P - xp * R);
            mnext = (1.f - lm) * dtt;
          }
          // exponential: G(z) = conj(a) G(a)
          const float Gzr = ar * Gar + ai * Gai;
          const float Gzi = ar * Gai - ai * Gar;
          dA_acc = fmaf(dtt, Gzr, dA_acc);
          gdt = fmaf(Ad, Gzr, gdt);
          acc[i][4] += Gzi;
          if (n == 0) {
            gx = fmaf(Ds, dyt, gx);
            dD_acc = fmaf(dyt, xt, dD_acc);
          }
          g3[0][i] = gx;
          g3[1][i] = gdt;
          g3[2][i] = glam;
          // carry conj(a_t) ghat_t and R_t to step t - 1
          cgr = ar * gr + ai * gi;
          cgi = ar * gi - ai * gr;
          Rn = R;
        }
      }
      s_state[j][tid] = make_float4(cgr, cgi, Rn, dA_acc);
      s_dD[j][tid] = dD_acc;

      // ---- sums over n: dx and ddt of (t, d) are final; dlam goes on to the sum over d
      hold_base = butterfly<N, 3>(g3, n);
      const bool owner = (n % DUP) == 0;
#pragma unroll
      for (int h = 0; h < HOLD; ++h) {
        const int i = hold_base + h;
        if (owner && valid && i < nt) {
          const long long td = (b * L + ts + i) * D + dd;
          p.dx[td] = g3[0][h];
          p.ddt[td] = g3[1][h];
          lam_acc[h] += g3[2][h];
        }
      }
    }

    // ---- sums over d of this segment: lanes of one n, then warps, then one atomic per value
#pragma unroll
    for (int m = N; m < 32; m <<= 1)
#pragma unroll
      for (int i = 0; i < SEG; ++i)
#pragma unroll
        for (int c = 0; c < 5; ++c) acc[i][c] += __shfl_xor_sync(0xffffffffu, acc[i][c], m);
    if (cl == 0) {
#pragma unroll
      for (int i = 0; i < SEG; ++i)
        if (i < nt)
#pragma unroll
          for (int c = 0; c < 5; ++c) atomicAdd(&s_acc[i][n][c], acc[i][c]);
    }
    if (MODE == 1) {
#pragma unroll
      for (int h = 0; h < HOLD; ++h)
        if ((n % DUP) == 0 && hold_base + h < nt) atomicAdd(&s_lam[hold_base + h], lam_acc[h]);
    }
    __syncthreads();
    for (int k = tid; k < nt * N * 5; k += THREADS) {
      const int i = k / (N * 5), rem = k % (N * 5), nn = rem / 5, c = rem % 5;
      float* v = &s_acc[i][nn][c];
      const long long tn = (b * L + ts + i) * N + nn;
      if (c < 2) atomicAdd(&p.dBc[2 * tn + c], *v);
      else if (c < 4) atomicAdd(&p.dCc[2 * tn + c - 2], *v);
      else atomicAdd(&p.dtheta[tn], *v);
      *v = 0.f;
    }
    if (MODE == 1 && tid < nt) {
      atomicAdd(&p.dlam[b * L + ts + tid], s_lam[tid]);
      s_lam[tid] = 0.f;
    }
    __syncthreads();
  }

  // ---- per-(d, n) and per-d sums over this batch row
#pragma unroll 1
  for (int j = 0; j < K; ++j) {
    const int d = dbase + (j * WARPS + warp) * CPW + cl;
    if (d < p.D) {
      atomicAdd(&p.dA[(long long)d * N + n], s_state[j][tid].w);
      if (n == 0) atomicAdd(&p.dD[d], s_dD[j][tid]);
    }
  }
}

}  // namespace bwd
}  // namespace csscan
