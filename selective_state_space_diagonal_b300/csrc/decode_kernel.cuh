// decode_kernel.cuh -- one step of the recurrence for a batch of sequences whose state lives in
// device memory: the recurrent (decode) regime, O(1) state per token.
//
// What it computes is one step of the scan of scan_kernels.cuh (the step operator of "Complex
// parallel scan", section 并行扫描的数学本质; alpha, beta, gamma of the discretisation table of
// "Mamba-3 paper story"; the output of "Mamba-3: 选择性状态空间模型的下一代架构", section 2.2):
//
//   a        = exp(dt[b,d] A[d,n]) e^{i theta[b,n]}
//   exp-Euler        h[b,d,n] <- a h + dt x[b,d] Bc[b,n]
//   exp-trapezoidal  h[b,d,n] <- a h + (1 - lam[b]) dt a x_prev[b,d] Bc_prev[b,n] + lam[b] dt x Bc
//   zero-order hold  h[b,d,n] <- a h + dt (a - 1) / z x Bc,   z = dt A + i theta
//   y[b,d]   = Re(sum_n Cc[b,n] h[b,d,n]) + Dskip[d] x[b,d]
//
// One thread updates two consecutive states of one (b, d) row; the N / 2 threads of a row are
// neighbouring lanes and sum their parts of y with shuffles. The state is read and written once
// (16 bytes per state), so the step is bound by memory bandwidth, not arithmetic.
#pragma once

#include "device_util.cuh"

namespace csscan {

struct DecodeParams {
  const void* x;        // (B, D)
  const void* dt;       // (B, D)
  const float* A;       // (D, N)
  const void* Bc;       // (B, N, 2)
  const void* Cc;       // (B, N, 2)
  const void* theta;    // (B, N)
  const void* lam;      // (B) trapezoid only
  const float* Dskip;   // (D)
  float* y;             // (B, D)
  float4* h;            // (B, D, N/2) pairs of states: (re_n, im_n, re_{n+1}, im_{n+1}), in place
  const void* x_prev;   // (B, D) trapezoid only, or null (zero)
  const void* Bc_prev;  // (B, N, 2) trapezoid only, or null (zero)
  long long rows;       // B * D
  int D, N;
};

template <typename Tin, int MODE, int NP>
__global__ void __launch_bounds__(256) decode_kernel(DecodeParams p) {
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gid / NP;                 // (b, d)
  const int q = int(gid % NP);                    // state pair
  const bool valid = row < p.rows;
  const long long r = valid ? row : 0;
  const int d = int(r % p.D);
  const long long b = r / p.D;
  const int n = 2 * q;
  const Tin* X = static_cast<const Tin*>(p.x);
  const Tin* DTp = static_cast<const Tin*>(p.dt);
  const Tin* BC = static_cast<const Tin*>(p.Bc);
  const Tin* CC = static_cast<const Tin*>(p.Cc);
  const Tin* TH = static_cast<const Tin*>(p.theta);

  const float xv = load_in<Tin>(X, r), dv = load_in<Tin>(DTp, r);
  const long long bn = b * p.N + n;
  float4 hv = valid ? __ldcs(p.h + r * NP + q) : make_float4(0.f, 0.f, 0.f, 0.f);
  float part = 0.f;
  float hn[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float rr = expf(dv * p.A[(long long)d * p.N + n + k]);
    float sn, cs;
    sincosf(load_in<Tin>(TH, bn + k), &sn, &cs);
    const float ar = rr * cs, ai = rr * sn;                       // a = r e^{i theta}
    const float br = load_in<Tin>(BC, 2 * (bn + k)), bi = load_in<Tin>(BC, 2 * (bn + k) + 1);
    float ur, ui;
    if (MODE == 0) {
      const float g = dv * xv;
      ur = g * br;
      ui = g * bi;
    } else if (MODE == 2) {
      // (e^z - 1) / z without cancellation: e^z - 1 = expm1(dt A) e^{i theta} + (e^{i theta} - 1),
      // cos theta - 1 = -2 sin^2(theta / 2); the limit 1 where |z|^2 underflows
      const float u = dv * p.A[(long long)d * p.N + n + k], th = load_in<Tin>(TH, bn + k);
      const float em = expm1f(u);
      float sh, chh;
      sincosf(0.5f * th, &sh, &chh);
      const float cm1 = -2.f * sh * sh, s1 = 2.f * sh * chh;
      const float er = fmaf(em, 1.f + cm1, cm1), ei = (1.f + em) * s1;
      const float z2 = fmaf(u, u, th * th);
      float gr = 1.f, gi = 0.f;
      if (z2 > 1e-30f) {
        gr = fmaf(er, u, ei * th) / z2;
        gi = fmaf(ei, u, -er * th) / z2;
      }
      const float g = dv * xv;
      ur = g * (gr * br - gi * bi);
      ui = g * (gr * bi + gi * br);
    } else {
      const float lam = load_in<Tin>(static_cast<const Tin*>(p.lam), b);
      const float g = lam * dv * xv;
      ur = g * br;
      ui = g * bi;
      if (p.x_prev != nullptr) {
        const float xp = load_in<Tin>(static_cast<const Tin*>(p.x_prev), r);
        const Tin* BP = static_cast<const Tin*>(p.Bc_prev);
        const float pr = load_in<Tin>(BP, 2 * (bn + k)), pi = load_in<Tin>(BP, 2 * (bn + k) + 1);
        const float gp = (1.f - lam) * dv * xp;                  // beta = (1 - lam) dt a
        const float vr = gp * pr, vi = gp * pi;
        ur = fmaf(ar, vr, fmaf(-ai, vi, ur));
        ui = fmaf(ar, vi, fmaf(ai, vr, ui));
      }
    }
    const float h_r = hn[2 * k], h_i = hn[2 * k + 1];
    const float nr = fmaf(ar, h_r, fmaf(-ai, h_i, ur));
    const float ni = fmaf(ar, h_i, fmaf(ai, h_r, ui));
    hn[2 * k] = nr;
    hn[2 * k + 1] = ni;
    const float cr = load_in<Tin>(CC, 2 * (bn + k)), ci = load_in<Tin>(CC, 2 * (bn + k) + 1);
    part = fmaf(cr, nr, fmaf(-ci, ni, part));
  }
  if (valid) __stcs(p.h + r * NP + q, make_float4(hn[0], hn[1], hn[2], hn[3]));
#pragma unroll
  for (int o = NP / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (valid && q == 0) p.y[r] = fmaf(p.Dskip[d], xv, part);
}

}  // namespace csscan
