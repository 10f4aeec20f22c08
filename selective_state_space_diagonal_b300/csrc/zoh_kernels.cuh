// zoh_kernels.cuh -- the forward scan with the zero-order-hold injection (mode 2):
//
//   h_t = a_t h_{t-1} + gamma_t Bc_t x_t,   a_t = e^{z_t},  z_t = dt_t A + i theta_t,
//   gamma_t = dt_t (e^{z_t} - 1) / z_t,     y_t = Re(sum_n Cc_t h_t) + Dskip x_t
//
// gamma is the ZOH row of the discretisation table of "Mamba-3 paper story"
// (A^{-1}(exp(dt A) - I)), with the complex exponent z in place of dt A as for alpha_t. Unlike
// the other two modes the injection weight is complex and differs per (t, d, n), so the
// rotating-frame scan kernel does not apply; these kernels run the recurrence directly:
//   zoh_table_kernel   per (b, t, n): cos theta, sin theta, theta, cos theta - 1
//   zoh_chunk_kernel   per (b, c, d, n): state at the chunk's end from a zero entry state and
//                      the product of a over the chunk  (only when the rows leave few threads)
//   zoh_combine_kernel per (b, d, n): walks the chunks for each chunk's entry state
//   zoh_out_kernel     blocks of OUT_THREADS / N channels of one (b, c), a thread per (channel, n): the
//                      recurrence over the chunk from its entry state, each 8-step group's
//                      shared inputs staged in shared memory first; the N lanes of a channel
//                      sum Re(Cc h) with a reduce-scatter and one stores y
// gamma is evaluated without cancellation: e^z - 1 = expm1(dt A) e^{i theta} + (e^{i theta} - 1)
// with cos theta - 1 = -2 sin^2(theta / 2), then divided by z.
#pragma once

#include "device_util.cuh"

namespace csscan {
namespace zoh {

constexpr int GROUP = 8;   // steps whose loads are issued together
constexpr int OUT_THREADS = 256;   // threads per block of zoh_out_kernel

struct Params {
  const void* x;       // (B, L, D)
  const void* dt;      // (B, L, D)
  const void* Bc;      // (B, L, N, 2)
  const void* Cc;      // (B, L, N, 2)
  const float* A;      // (D, N)
  const float* Dskip;  // (D)
  float* y;            // (B, L, D)
  const float4* tab;   // (B, L, N): cos theta, sin theta, theta, cos theta - 1
  float2* chunk;       // (B, C, D, N, 2): end state | entry state, product of a
  int B, L, D, N;
  int TC, C;
};

template <typename Tin>
__global__ void __launch_bounds__(256) zoh_table_kernel(const void* theta, float4* tab, long long total) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= total) return;
  const float th = load_in<Tin>(static_cast<const Tin*>(theta), i);
  float s, c, sh, ch;
  sincosf(th, &s, &c);
  sincosf(0.5f * th, &sh, &ch);
  tab[i] = make_float4(c, s, th, -2.f * sh * sh);
}

// One step of the recurrence: h <- a h + gamma Bc x. ar, ai return a.
__device__ __forceinline__ void zoh_step(float dtt, float xt, float Adn, float4 tb, float br, float bi, float& hr,
                                         float& hi, float& ar, float& ai) {
  const float zr = dtt * Adn, zi = tb.z;
  const float em = expm1f(zr);                       // e^{dt A} - 1
  const float r = 1.f + em;
  ar = r * tb.x;
  ai = r * tb.y;
  // e^z - 1 = em e^{i theta} + (e^{i theta} - 1)
  const float er = fmaf(em, tb.x, tb.w), ei = r * tb.y;
  const float zz = fmaf(zr, zr, zi * zi);
  float pr, pi;   // phi = (e^z - 1) / z
  if (zz > 1e-12f) {
    const float inv = __frcp_rn(zz);
    pr = (er * zr + ei * zi) * inv;
    pi = (ei * zr - er * zi) * inv;
  } else {        // |z| < 1e-6: 1 + z/2 + z^2/6
    pr = 1.f + 0.5f * zr + (zr * zr - zi * zi) * (1.f / 6.f);
    pi = 0.5f * zi + zr * zi * (1.f / 3.f);
  }
  const float w = dtt * xt;
  const float gr = w * pr, gi = w * pi;              // gamma x
  const float ur = gr * br - gi * bi, ui = gr * bi + gi * br;
  const float nr = fmaf(ar, hr, fmaf(-ai, hi, ur));
  const float ni = fmaf(ar, hi, fmaf(ai, hr, ui));
  hr = nr;
  hi = ni;
}

struct Thread {
  long long b;
  int c, d, n;
  bool ok;
};
__device__ __forceinline__ Thread thread_of(const Params& p) {
  const long long gid = (long long)blockIdx.x * 256 + threadIdx.x;
  Thread r;
  r.ok = gid < (long long)p.B * p.C * p.D * p.N;
  const long long g = r.ok ? gid : 0;
  r.n = int(g % p.N);
  long long q = g / p.N;
  r.d = int(q % p.D);
  q /= p.D;
  r.c = int(q % p.C);
  r.b = q / p.C;
  return r;
}
__device__ __forceinline__ float2* rec_of(const Params& p, long long b, int c, int d, int n) {
  return p.chunk + ((((b * p.C + c) * p.D + d) * p.N) + n) * 2;
}

// Inputs of GROUP steps t0 .. t0 + GROUP - 1 (clamped to te - 1), loaded before use.
template <typename Tin>
struct Group {
  float xs[GROUP], ds[GROUP], brs[GROUP], bis[GROUP], crs[GROUP], cis[GROUP];
  float4 tbs[GROUP];
  __device__ __forceinline__ void load(const Params& p, long long b, int d, int n, int t0, int te, bool with_c) {
    const Tin* X = static_cast<const Tin*>(p.x);
    const Tin* DT = static_cast<const Tin*>(p.dt);
    const Tin* BC = static_cast<const Tin*>(p.Bc);
    const Tin* CC = static_cast<const Tin*>(p.Cc);
#pragma unroll
    for (int i = 0; i < GROUP; ++i) {
      const int t = min(t0 + i, te - 1);
      const long long td = (b * p.L + t) * p.D + d;
      const long long tn = (b * p.L + t) * p.N + n;
      xs[i] = load_in<Tin>(X, td);
      ds[i] = load_in<Tin>(DT, td);
      tbs[i] = p.tab[tn];
      const float2 bb = load_pair<Tin>(BC, tn);
      brs[i] = bb.x;
      bis[i] = bb.y;
      if (with_c) {
        const float2 cc = load_pair<Tin>(CC, tn);
        crs[i] = cc.x;
        cis[i] = cc.y;
      }
    }
  }
};

template <typename Tin>
__global__ void __launch_bounds__(256) zoh_chunk_kernel(const Params p) {
  const Thread th = thread_of(p);
  if (!th.ok) return;
  const float Adn = p.A[(long long)th.d * p.N + th.n];
  const int tc = th.c * p.TC, te = min(p.L, tc + p.TC);
  float hr = 0.f, hi = 0.f, Pr = 1.f, Pi = 0.f;
  for (int t0 = tc; t0 < te; t0 += GROUP) {
    Group<Tin> g;
    g.load(p, th.b, th.d, th.n, t0, te, false);
#pragma unroll
    for (int i = 0; i < GROUP; ++i) {
      if (t0 + i < te) {
        float ar, ai;
        zoh_step(g.ds[i], g.xs[i], Adn, g.tbs[i], g.brs[i], g.bis[i], hr, hi, ar, ai);
        const float qr = ar * Pr - ai * Pi, qi = ar * Pi + ai * Pr;
        Pr = qr;
        Pi = qi;
      }
    }
  }
  float2* rec = rec_of(p, th.b, th.c, th.d, th.n);
  rec[0] = make_float2(hr, hi);
  rec[1] = make_float2(Pr, Pi);
}

__global__ void __launch_bounds__(256) zoh_combine_kernel(const Params p) {
  const long long gid = (long long)blockIdx.x * 256 + threadIdx.x;
  if (gid >= (long long)p.B * p.D * p.N) return;
  const int n = int(gid % p.N);
  const long long bd = gid / p.N;
  const int d = int(bd % p.D);
  const long long b = bd / p.D;
  float hr = 0.f, hi = 0.f;
  for (int c = 0; c < p.C; ++c) {
    float2* rec = rec_of(p, b, c, d, n);
    const float2 U = rec[0], P = rec[1];
    rec[0] = make_float2(hr, hi);
    const float nr = P.x * hr - P.y * hi + U.x, ni = P.x * hi + P.y * hr + U.y;
    hr = nr;
    hi = ni;
  }
}

// The recurrence over chunk c from its entry state, with y. A block owns CBZ = OUT_THREADS / N channels
// of one (b, c): thread (channel dl, state n), the N lanes of a channel neighbours in a warp
// (N <= 32). For each group of GROUP steps the block first stages, coalesced, what its lanes
// share -- the (cos, sin, theta, cos - 1) row, Bc and Cc per (t, n), x and dt per (t, channel)
// -- in shared memory. Each lane keeps its Re(Cc h) for the group (lane 0 adds Dskip x); a
// reduce-scatter over the N lanes then leaves each step's sum in one lane, which stores it.
// Grid: (ceil(D / CBZ), C, B).
template <typename Tin, int N>
__global__ void __launch_bounds__(OUT_THREADS) zoh_out_kernel(const Params p) {
  constexpr int CBZ = OUT_THREADS / N;
  constexpr int HOLD = GROUP >= N ? GROUP / N : 1;
  constexpr int DUP = N > GROUP ? N / GROUP : 1;
  __shared__ float4 s_tab[GROUP][N];
  __shared__ float4 s_bc[GROUP][N];      // Bc re, im, Cc re, im
  __shared__ float2 s_xd[GROUP][CBZ];    // x, dt
  const int tid = threadIdx.x;
  const int n = tid % N, dl = tid / N;
  const int d0 = blockIdx.x * CBZ;
  const int d = d0 + dl;
  const bool valid = d < p.D;
  const int dc = valid ? d : 0;
  const int c = blockIdx.y;
  const long long b = blockIdx.z;
  const Tin* X = static_cast<const Tin*>(p.x);
  const Tin* DT = static_cast<const Tin*>(p.dt);
  const Tin* BC = static_cast<const Tin*>(p.Bc);
  const Tin* CC = static_cast<const Tin*>(p.Cc);
  const float Adn = p.A[(long long)dc * N + n];
  const float Ds = p.Dskip[dc];
  const int tc = c * p.TC, te = min(p.L, tc + p.TC);
  float hr = 0.f, hi = 0.f;
  if (p.C > 1 && valid) {
    const float2 h0 = rec_of(p, b, c, d, n)[0];
    hr = h0.x;
    hi = h0.y;
  }
  for (int t0 = tc; t0 < te; t0 += GROUP) {
    const int ng = min(GROUP, te - t0);
    // ---- stage the group (steps past te and channels past D as zeros)
    for (int k = tid; k < GROUP * N; k += OUT_THREADS) {
      const int i = k / N, nn = k % N;
      float4 tb = make_float4(0.f, 0.f, 0.f, 0.f), bc = tb;
      if (i < ng) {
        const long long tn = (b * p.L + t0 + i) * N + nn;
        tb = p.tab[tn];
        const float2 bb = load_pair<Tin>(BC, tn), cc = load_pair<Tin>(CC, tn);
        bc = make_float4(bb.x, bb.y, cc.x, cc.y);
      }
      s_tab[i][nn] = tb;
      s_bc[i][nn] = bc;
    }
    for (int k = tid; k < GROUP * CBZ; k += OUT_THREADS) {
      const int i = k / CBZ, cd = k % CBZ;
      float2 v = make_float2(0.f, 0.f);
      if (i < ng && d0 + cd < p.D) {
        const long long td = (b * p.L + t0 + i) * p.D + d0 + cd;
        v = make_float2(load_in<Tin>(X, td), load_in<Tin>(DT, td));
      }
      s_xd[i][cd] = v;
    }
    __syncthreads();
    float part[1][GROUP];
#pragma unroll
    for (int i = 0; i < GROUP; ++i) {
      part[0][i] = 0.f;
      if (i < ng) {
        const float2 xd = s_xd[i][dl];
        const float4 bc = s_bc[i][n];
        float ar, ai;
        zoh_step(xd.y, xd.x, Adn, s_tab[i][n], bc.x, bc.y, hr, hi, ar, ai);
        part[0][i] = bc.z * hr - bc.w * hi;
        if (n == 0) part[0][i] = fmaf(Ds, xd.x, part[0][i]);
      }
    }
    const int base = butterfly<N, 1, GROUP>(part, n);
    if ((n % DUP) == 0 && valid) {
#pragma unroll
      for (int h = 0; h < HOLD; ++h) {
        const int i = base + h;
        if (i < ng) p.y[(b * p.L + t0 + i) * p.D + d] = part[0][h];
      }
    }
    __syncthreads();
  }
}

}  // namespace zoh
}  // namespace csscan
