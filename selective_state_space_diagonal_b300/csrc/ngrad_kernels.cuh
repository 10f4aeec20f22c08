// ngrad_kernels.cuh -- the gradient pass of csscan_backward in the rotating frame of the forward
// scan (nscan_kernels.cuh), for inputs that meet the tile-copy rules.
//
// Reverse-mode differentiation of the forward recurrence ("Complex parallel scan", sections
// 一个问题，两种命运 and 硬件落地的挑战: one forward over the sequence, one backward sweep,
// states recomputed rather than stored). Both modes are written as one recurrence over the
// look-ahead state s_t (the trapezoid's k_{t+1}; exp-Euler: s_t = h_t):
//   s_t = a_t s_{t-1} + w_t Bc_t,   a_t = exp(dt_t A + i theta_t)
//   y_t = Re(sum_n Cc_t s_t) - x_t m_t E_t + Dskip x_t
//   exp-Euler  w_t = dt_t x_t,                              m_t = 0
//   trapezoid  w_t = x_t (lam_t dt_t + mu_t dt_{t+1}),      m_t = mu_t dt_{t+1},  mu_t = 1 - lam_{t+1}
// (mu = 0 at the last step, E_t = sum_n Re(Cc_t Bc_t)). With G(z) = dl/dRe z + i dl/dIm z for
// l = sum dy y, the adjoint ghat_t = G(s_t) satisfies ghat_t = dy_t conj(Cc_t) + conj(a_{t+1})
// ghat_{t+1}. In the rotating frame of a 32-step sub-chunk (Phi the running sum of theta,
// g = e^{-i Phi} s, Bt = e^{-i Phi} Bc, Ct = e^{i Phi} Cc, r_t = exp(dt_t A)) the adjoint
// gamma = e^{-i Phi} ghat has a real decay,
//   gamma_t = dy_t conj(Ct_t) + r_{t+1} gamma_{t+1},
// and every gradient follows from gamma, g and the rotated tables:
//   G(z_t) = conj(a_t) G(a_t) = rho_t conj(g_{t-1}),  rho_t = r_t gamma_t   (z_t = dt_t A + i theta_t)
//     dA += dt_t Re G(z_t),  ddt_t += A Re G(z_t),  dtheta_t += Im G(z_t)
//   G(w_t)  = sum_n Re(conj(Bt_t) gamma_t)            (Gw)
//   dBc_t   = e^{+i Phi_t} sum_d w_t gamma_t  + G(E_t) conj(Cc_t)
//   dCc_t   = e^{-i Phi_t} sum_d dy_t conj(g_t) + G(E_t) conj(Bc_t),   G(E_t) = -sum_d dy_t x_t m_t
//   exp-Euler  dx_t = dt_t Gw_t + Dskip dy_t,  ddt_t = x_t Gw_t + sum_n A Re G(z_t)
//   trapezoid  dx_t = (lam_t dt_t + mu_t dt_{t+1}) Gw_t - dy_t m_t E_t + Dskip dy_t
//              ddt_t = x_t lam_t Gw_t + sum_n A Re G(z_t) + x_{t-1} mu_{t-1} (Gw_{t-1} - dy_{t-1} E_{t-1})
//              dlam_t = sum_d [x_t dt_t Gw_t - x_{t-1} dt_t (Gw_{t-1} - dy_{t-1} E_{t-1})]
//   dDskip += dy_t x_t.
//
// The work: a thread owns one state pair of K channels (one after the other); a block of 4
// warps owns BC channels of one batch row and one time chunk and walks its 8-step segments last to
// first. Per segment and channel the thread regenerates g over the segment from the checkpoint
// (the forward kernel's checkpoint variant stores the rotated state before every segment) into
// registers, then walks it backwards. Sums over n of a (t, d) (Gw, sum A Re G(z)) and sums over d
// of a (t, n) (dBc, dCc, dtheta) pass through shared memory once per segment: the first are
// written per step and summed per (t, d) by the block's threads, which then form dx, ddt, dlam;
// the second accumulate in registers over the thread's K channels and are summed per (t, n) over
// the block, leaving it as one vector atomic add per (t, state pair) and kind. dBc and dCc are
// accumulated in the rotated frame; ngrad_post_kernel rotates them back and adds the G(E) terms.
// The segments' inputs (x, dt, dy, the tables) arrive by tile copies into a 2-stage ring, the next
// segment's while the current one is worked.
#pragma once

#include "scan_kernels.cuh"

namespace csscan {
namespace ngrad {

constexpr int SEG = 8;   // checkpoint spacing and segment length
constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;

template <int N>
struct GTile {
  static_assert(N >= 2 && N <= 32 && (N & (N - 1)) == 0, "the gradient pass handles N = 2 .. 32");
  static constexpr int NG = N / 2;                    // lanes per channel (one state pair each)
  static constexpr int M = 32 / NG;                   // channel slots per warp
  static constexpr int K = M >= 16 ? 1 : 16 / M;      // channels per thread, one after the other
  static constexpr int BC = K * WARPS * M;            // channels per block
  static constexpr int SLOTS = WARPS * M;             // threads sharing a state pair
  static constexpr int NGR = NG > 8 ? 8 : NG;         // lanes per channel summed in shared memory
  static constexpr int ROWS = THREADS / BC;           // threads per channel in the per-(t, d) phase
  static constexpr int MIN_BLOCKS = 4;                // resident blocks per SM the kernel is compiled for
};

// One stage: x rows ts .. ts+7, dt rows ts .. ts+8, dy rows ts .. ts+7 of the block's channels,
// the trapezoid rows (lam_t, 1 - lam_{t+1}, E_t, 0), the two table planes (Bt, Ct) of rows ts ..
// ts+7 and e^{i Phi} after the last step of the sub-chunk holding ts. Rows past the sequence's end
// arrive as zeros. Then the scratch region: the segment's (dt, w) per (t, channel) [SEG][BC]
// float2, and the per-(t, d) partials of half a segment [SEG / 2][BC][TDW] float2, which the
// per-(t, n) partials of the half [SEG / 2][5][NG][SROW] floats overwrite once consumed (rows
// padded so that neither the writes nor the row sums meet bank conflicts).
template <int N, typename Tin, int MODE>
struct GStage {
  using GT = GTile<N>;
  static constexpr int SIN = int(sizeof(Tin));
  static constexpr int X_BYTES = SEG * GT::BC * SIN;
  static constexpr int DT_BYTES = (SEG + 1) * GT::BC * SIN;
  static constexpr int DY_BYTES = SEG * GT::BC * 4;
  static constexpr int AUX_BYTES = MODE == 1 ? SEG * 16 : 0;
  static constexpr int TAB_BYTES = SEG * 2 * 2 * N * 4;
  static constexpr int ROT_BYTES = 2 * N * 4;
  static constexpr int OFF_X = 0;
  static constexpr int OFF_DT = align128(OFF_X + X_BYTES);
  static constexpr int OFF_DY = align128(OFF_DT + DT_BYTES);
  static constexpr int OFF_AUX = align128(OFF_DY + DY_BYTES);
  static constexpr int OFF_TAB = align128(OFF_AUX + AUX_BYTES);
  static constexpr int OFF_ROT = align128(OFF_TAB + TAB_BYTES);
  static constexpr int BYTES = align128(OFF_ROT + ROT_BYTES);
  static constexpr int TX_BYTES = X_BYTES + DT_BYTES + DY_BYTES + AUX_BYTES + TAB_BYTES + ROT_BYTES;
  static constexpr int SROW = 2 * GT::SLOTS + 8;      // floats per (t, kind, pair) row
  static constexpr int TDW = GT::NGR + 2;             // float2 per (t, channel) row
  static constexpr int PRE_BYTES = SEG * GT::BC * 8;  // (dt, w) per (t, channel)
  static constexpr int TD_BYTES = (SEG / 2) * GT::BC * TDW * 8;
  static constexpr int TN_BYTES = (SEG / 2) * 5 * GT::NG * SROW * 4;
  static constexpr int SCR_BYTES = PRE_BYTES + (TD_BYTES > TN_BYTES ? TD_BYTES : TN_BYTES);
  static constexpr int SMEM = 2 * BYTES + SCR_BYTES + 128;
};

struct GradParams {
  CUtensorMap tm_x;     // (D, L, B) input dtype, box (BC, SEG, 1)
  CUtensorMap tm_dt;    // (D, L, B) input dtype, box (BC, SEG + 1, 1)
  CUtensorMap tm_dy;    // (D, L, B) f32, box (BC, SEG, 1)
  CUtensorMap tm_aux;   // (4, L, B) f32, box (4, SEG, 1)
  CUtensorMap tm_tab;   // (2N, 2, L, B) f32, box (2N, 2, SEG, 1)
  CUtensorMap tm_rot;   // (2N, 4 S32, B) f32, box (2N, 1, 1)
  const float* A;       // (D, N)
  const float* Dskip;   // (D)
  const float4* ckpt;   // (B, S8, D, N/2) state pairs (re, im, re', im') before segment s >= 1
  const float2* kap;    // (B, C, D, N) the true-frame adjoint carry entering chunk c's last step (C > 1)
  float* dx;            // (B, L, D) written
  float* ddt;           // (B, L, D) written (chunk starts completed by ngrad_fix_kernel)
  float* dA;            // (D, N) accumulated
  float* dBc;           // (B, L, N, 2) accumulated in the rotated frame (ngrad_post_kernel finishes)
  float* dCc;           // (B, L, N, 2) accumulated in the rotated frame
  float* dtheta;        // (B, L, N) accumulated
  float* dlam;          // (B, L) accumulated (trapezoid)
  float* dD;            // (D) accumulated
  float* ge;            // (B, L) G(E_t), accumulated (trapezoid)
  float* xb;            // (B, C, D) a chunk's last-step term of ddt at the next chunk's first step
  uint32_t* hdr;        // error word of the workspace header
  int B, L, D, S8, TC, C;
  int tab_ng;           // lane-group interleave of the table's state pairs
};

template <typename Tin, int MODE, int N>
__global__ void __launch_bounds__(THREADS, GTile<N>::MIN_BLOCKS) ngrad_kernel(const __grid_constant__ GradParams p) {
  using GT = GTile<N>;
  using SG = GStage<N, Tin, MODE>;
  constexpr int NG = GT::NG, M = GT::M, K = GT::K, BC = GT::BC, NGR = GT::NGR, ROWS = GT::ROWS;
  constexpr int SROW = SG::SROW, TDW = SG::TDW;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  float2* pre = reinterpret_cast<float2*>(smem + 2 * SG::BYTES);                  // (dt, w) per (t, channel)
  float* scr = reinterpret_cast<float*>(smem + 2 * SG::BYTES + SG::PRE_BYTES);   // per-(t, n) partials
  float2* tdp = reinterpret_cast<float2*>(scr);                                  // per-(t, d) partials
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ float4 s_carry[K][THREADS];   // per (channel, thread): the adjoint carry rho (re pair, im pair)
  __shared__ float2 s_dA[K][THREADS];      // per (channel, thread): dA of the pair
  __shared__ float s_pend[2][BC];          // ddt at a segment's first step without the previous step's term
  __shared__ float s_hpend[BC];            // the same at the segment's middle step
  __shared__ float s_lam[SEG + 1];         // per step of the segment (and the next segment's first)
  __shared__ float s_ge[SEG];

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane / M;     // state pair (states 2g, 2g + 1)
  const int c = lane % M;     // channel slot
  const int b = blockIdx.y, chunk = blockIdx.z;
  const int d0 = blockIdx.x * BC;
  const int64_t L = p.L, D = p.D;
  const int tc = chunk * p.TC, te = min(p.L, tc + p.TC);
  const int s_first = tc / SEG, s_last = (te - 1) / SEG;
  const int npair = N / (2 * p.tab_ng);
  const int pos = (g % npair) * p.tab_ng + g / npair;   // this pair's float4 within a table plane

  auto issue = [&](int s, int slot) {
    unsigned char* base = smem + slot * SG::BYTES;
    const int ts = s * SEG;
    mbar_arrive_expect_tx(&bar[slot], uint32_t(SG::TX_BYTES));
    tma_load_3d(base + SG::OFF_X, &p.tm_x, d0, ts, b, &bar[slot]);
    tma_load_3d(base + SG::OFF_DT, &p.tm_dt, d0, ts, b, &bar[slot]);
    tma_load_3d(base + SG::OFF_DY, &p.tm_dy, d0, ts, b, &bar[slot]);
    if (MODE == 1) tma_load_3d(base + SG::OFF_AUX, &p.tm_aux, 0, ts, b, &bar[slot]);
    tma_load_4d(base + SG::OFF_TAB, &p.tm_tab, 0, 0, ts, b, &bar[slot]);
    tma_load_3d(base + SG::OFF_ROT, &p.tm_rot, 0, 4 * (ts / T_SUB) + 3, b, &bar[slot]);
  };
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    prefetch_tmap(&p.tm_x);
    prefetch_tmap(&p.tm_dt);
    prefetch_tmap(&p.tm_dy);
    if (MODE == 1) prefetch_tmap(&p.tm_aux);
    prefetch_tmap(&p.tm_tab);
    prefetch_tmap(&p.tm_rot);
    issue(s_last, 0);
  }

  // ---- per (channel, thread): the true-frame carry entering the chunk's last step from the next
  // chunk (zero at the sequence's end), and the dA sums
#pragma unroll 1
  for (int k = 0; k < K; ++k) {
    const int d = d0 + (k * WARPS + w) * M + c;
    float4 cv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (chunk + 1 < p.C && d < p.D) {
      const float4 v = reinterpret_cast<const float4*>(p.kap + ((int64_t(b) * p.C + chunk) * D + d) * N)[g];
      cv = make_float4(v.x, v.z, v.y, v.w);
    }
    s_carry[k][tid] = cv;
    s_dA[k][tid] = f2(0.f, 0.f);
  }
  for (int i = tid; i < 2 * BC; i += THREADS) (&s_pend[0][0])[i] = 0.f;
  for (int i = tid; i < BC; i += THREADS) s_hpend[i] = 0.f;
  if (tid <= SEG) s_lam[tid] = 0.f;
  if (tid < SEG) s_ge[tid] = 0.f;

  // the channel and first step of this thread in the per-(t, d) phase
  const int cbA = tid % BC, rA = tid / BC;
  const int dA_ = d0 + cbA;
  const bool validA = dA_ < p.D;
  const float DsA = validA ? p.Dskip[dA_] : 0.f;
  float dD_acc = 0.f;
  __syncthreads();

  // checkpoint of (segment s, channel k of this thread): the rotated state before the segment;
  // and A of the channel's state pair
  auto ckpt_of = [&](int s, int k) {
    const int d = d0 + (k * WARPS + w) * M + c;
    return (s > 0 && d < p.D) ? __ldcg(p.ckpt + ((int64_t(b) * p.S8 + CSSCAN_BCK(p.hdr, s, p.S8, 31)) * D + d) * (N / 2) + g)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  auto a_of = [&](int k) {
    const int d = d0 + (k * WARPS + w) * M + c;
    return d < p.D ? __ldg(reinterpret_cast<const float2*>(p.A + int64_t(d) * N) + g) : f2(0.f, 0.f);
  };
  float4 ck_next = ckpt_of(s_last, 0);
  float2 A_next = a_of(0);

  bool aborted = false;
  int q = 0;
#pragma unroll 1
  for (int s = s_last; s >= s_first; --s, ++q) {
    const int slot = q & 1;
    // the other slot held segment s + 1, whose last reads ended before the barrier closing it
    if (tid == 0 && s > s_first) issue(s - 1, slot ^ 1);
    const bool ok = wait_bar_bounded(&bar[slot], uint32_t(q >> 1) & 1u);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const unsigned char* base = smem + slot * SG::BYTES;
    const Tin* sX = reinterpret_cast<const Tin*>(base + SG::OFF_X);
    const Tin* sDT = reinterpret_cast<const Tin*>(base + SG::OFF_DT);
    const float* sDY = reinterpret_cast<const float*>(base + SG::OFF_DY);
    const float4* sAUX = reinterpret_cast<const float4*>(base + SG::OFF_AUX);
    const float4* sTAB = reinterpret_cast<const float4*>(base + SG::OFF_TAB);   // [i][plane][N/2]
    const float4 rot = reinterpret_cast<const float4*>(base + SG::OFF_ROT)[g];   // (c, s) of states 2g, 2g+1
    const int ts = s * SEG;
    const int nt = min(SEG, p.L - ts);
    // (dt, w) once per (t, channel) for every lane of the channel
    for (int e = tid; e < SEG * BC; e += THREADS) {
      const float x = smem_in<Tin>(sX, e), dt = smem_in<Tin>(sDT, e);
      float wt;
      if constexpr (MODE == 1) {
        const float4 ax = sAUX[e / BC];
        wt = x * fmaf(ax.x, dt, ax.y * smem_in<Tin>(sDT, e + BC));
      } else {
        wt = x * dt;
      }
      pre[e] = f2(dt, wt);
    }
    __syncthreads();

    // Two halves, the later steps first: the per-(t, n) sums of a half live in registers only
    // while its four steps are worked, and its per-(t, d) partials share one scratch region with
    // them. Each half regenerates g from the segment's checkpoint (the later half through all
    // eight steps, keeping the last five states; the earlier half through its four).
    auto run_half = [&](auto half_tag) {
      constexpr int half = decltype(half_tag)::value;
      constexpr int H = SEG / 2;
      constexpr int i0 = half * H;
      // per-(t, n) sums over this thread's channels: Im G(z) as sum rho_i g_r - sum rho_r g_i (two
      // accumulators, subtracted once per half), dBc (re, im), dCc as (dy g_r, dy g_i) (negated once)
      float2 aT[H], aT2[H], aBr[H], aBi[H], aCr[H], aCi[H];
#pragma unroll
      for (int ii = 0; ii < H; ++ii) aT[ii] = aT2[ii] = aBr[ii] = aBi[ii] = aCr[ii] = aCi[ii] = f2(0.f, 0.f);

#pragma unroll 1
      for (int k = 0; k < K; ++k) {
        // this channel's checkpoint was loaded one channel earlier; load the next one now (the
        // first channel of the next half or segment after the last channel)
        const float4 ck = ck_next;
        const float2 A2 = A_next;
        if (k + 1 < K) ck_next = ckpt_of(s, k + 1);
        else if (half == 1) ck_next = ckpt_of(s, 0);
        else if (s > s_first) ck_next = ckpt_of(s - 1, 0);
        A_next = a_of(k + 1 < K ? k + 1 : 0);
        const int cb = (k * WARPS + w) * M + c;
        const float2 a2 = mul2(A2, f2(LOG2E_F, LOG2E_F));
        float4 cv = s_carry[k][tid];
        float2 cr = f2(cv.x, cv.y), ci = f2(cv.z, cv.w);
        // the carry arrives from the next sub-chunk's frame (or the next chunk at a sub-chunk
        // boundary): into this frame by e^{-i Phi_last}
        if (half == 1 && ((ts + SEG) % T_SUB) == 0) {
          const float2 cc = f2(rot.x, rot.z), ss = f2(rot.y, rot.w);
          const float2 nr = fma2(cc, cr, mul2(ss, ci));
          const float2 ni = fma2(cc, ci, mul2(f2(-ss.x, -ss.y), cr));
          cr = nr;
          ci = ni;
        }
        // ---- regenerate g (steps past the sequence's end have dt = 0 and a zero table row:
        // they leave g unchanged, and the adjoint below stays zero there)
        float2 gr0 = f2(ck.x, ck.z), gi0 = f2(ck.y, ck.w);
#pragma unroll
        for (int i = 0; i < i0; ++i) {
          const float2 pv = pre[i * BC + cb];
          const float2 r2 = ex2_pair(mul2(f2(pv.x, pv.x), a2));
          const float4 bt = sTAB[(i * 2) * (N / 2) + pos];
          const float2 w2 = f2(pv.y, pv.y);
          gr0 = fma2(r2, gr0, mul2(w2, f2(bt.x, bt.y)));
          gi0 = fma2(r2, gi0, mul2(w2, f2(bt.z, bt.w)));
        }
        float2 hr[H + 1], hi[H + 1], r2s[H];   // g_{i0-1} .. g_{i0+3}; decays of the half's steps
        hr[0] = gr0;
        hi[0] = gi0;
#pragma unroll
        for (int ii = 0; ii < H; ++ii) {
          const int i = i0 + ii;
          const float2 pv = pre[i * BC + cb];
          const float2 r2 = ex2_pair(mul2(f2(pv.x, pv.x), a2));
          r2s[ii] = r2;
          const float4 bt = sTAB[(i * 2) * (N / 2) + pos];
          const float2 w2 = f2(pv.y, pv.y);
          hr[ii + 1] = fma2(r2, hr[ii], mul2(w2, f2(bt.x, bt.y)));
          hi[ii + 1] = fma2(r2, hi[ii], mul2(w2, f2(bt.z, bt.w)));
        }
        // ---- backwards through the half
        float2 dA2 = s_dA[k][tid];
#pragma unroll
        for (int ii = H - 1; ii >= 0; --ii) {
          const int i = i0 + ii;
          const float2 pv = pre[i * BC + cb];   // dt, w
          const float dy = sDY[i * BC + cb];
          const float2 r2 = r2s[ii];
          const float4 bt = sTAB[(i * 2) * (N / 2) + pos];
          const float4 ct = sTAB[(i * 2 + 1) * (N / 2) + pos];   // (Re, Re', -Im, -Im')
          const float2 dy2 = f2(dy, dy);
          const float2 gr = fma2(dy2, f2(ct.x, ct.y), cr);   // gamma = carry + dy conj(Ct)
          const float2 gi = fma2(dy2, f2(ct.z, ct.w), ci);
          const float2 P2 = fma2(f2(bt.x, bt.y), gr, mul2(f2(bt.z, bt.w), gi));   // Re(conj(Bt) gamma)
          const float2 rr = mul2(r2, gr), ri = mul2(r2, gi);                      // rho = r gamma
          const float2 zr = fma2(rr, hr[ii], mul2(ri, hi[ii]));                   // Re G(z) = Re(rho conj(g_{t-1}))
          const float2 Q2 = mul2(A2, zr);
          dA2 = fma2(f2(pv.x, pv.x), zr, dA2);
          aT[ii] = fma2(ri, hr[ii], aT[ii]);                                      // Im G(z), in two parts
          aT2[ii] = fma2(rr, hi[ii], aT2[ii]);
          const float2 w2 = f2(pv.y, pv.y);
          aBr[ii] = fma2(w2, gr, aBr[ii]);
          aBi[ii] = fma2(w2, gi, aBi[ii]);
          aCr[ii] = fma2(dy2, hr[ii + 1], aCr[ii]);
          aCi[ii] = fma2(dy2, hi[ii + 1], aCi[ii]);
          float2 pq = f2(P2.x + P2.y, Q2.x + Q2.y);   // (Gw, sum A Re G(z)) partials of this pair
          cr = rr;
          ci = ri;
          if constexpr (NG > NGR) {   // N = 32: fold the upper half of the channel's lanes first
            pq.x += __shfl_xor_sync(0xffffffffu, pq.x, NGR * M);
            pq.y += __shfl_xor_sync(0xffffffffu, pq.y, NGR * M);
          }
          if (g < NGR) tdp[(ii * BC + cb) * TDW + g] = pq;
        }
        s_carry[k][tid] = make_float4(cr.x, cr.y, ci.x, ci.y);
        s_dA[k][tid] = dA2;
      }
      __syncthreads();

      // ---- per (t, d) of the half: dx, ddt, dlam, G(E), dDskip
      {
        auto sums = [&](int ii) {   // (Gw, sum A Re G(z)) of (half step ii, channel cbA)
          if constexpr (NGR == 1) {
            return tdp[(ii * BC + cbA) * TDW];
          } else {
            const float4* r4 = reinterpret_cast<const float4*>(tdp + (ii * BC + cbA) * TDW);
            float4 v = r4[0];
#pragma unroll
            for (int u = 1; u < NGR / 2; ++u) {
              const float4 a = r4[u];
              v.x += a.x;
              v.y += a.y;
              v.z += a.z;
              v.w += a.w;
            }
            return f2(v.x + v.z, v.y + v.w);
          }
        };
#pragma unroll
        for (int j0 = 0; j0 < H; j0 += ROWS) {
          const int ii = j0 + rA;
          const int i = i0 + ii;
          float lam_i = 0.f, ge_i = 0.f, lam_next = 0.f;   // trapezoid only
          (void)lam_i;
          (void)ge_i;
          (void)lam_next;
          if (i < nt && validA) {
            const float2 gq = sums(ii);
            const float x = smem_in<Tin>(sX, i * BC + cbA);
            const float dt = pre[i * BC + cbA].x;
            const float dy = sDY[i * BC + cbA];
            const int64_t row = CSSCAN_BCK(p.hdr, (int64_t(b) * L + ts + i) * D + dA_, int64_t(p.B) * L * D, 32);
            dD_acc = fmaf(dy, x, dD_acc);
            if constexpr (MODE == 0) {
              p.dx[row] = fmaf(dt, gq.x, DsA * dy);
              p.ddt[row] = fmaf(x, gq.x, gq.y);
            } else {
              const float4 ax = sAUX[i];   // lam_t, mu_t, E_t
              const float dtn = smem_in<Tin>(sDT, (i + 1) * BC + cbA);
              const float m = ax.y * dtn;
              p.dx[row] = fmaf(fmaf(ax.x, dt, m), gq.x, fmaf(-dy * m, ax.z, DsA * dy));
              const float own = fmaf(x * ax.x, gq.x, gq.y);
              lam_i = x * dt * gq.x;
              ge_i = -dy * x * m;
              if (ii > 0) {   // the previous step's terms of ddt_t and dlam_t
                const float2 gp = sums(ii - 1);
                const float xp = smem_in<Tin>(sX, (i - 1) * BC + cbA);
                const float4 ap = sAUX[i - 1];
                const float gwe = fmaf(-sDY[(i - 1) * BC + cbA], ap.z, gp.x);
                p.ddt[row] = fmaf(xp * ap.y, gwe, own);
                lam_i = fmaf(-xp * dt, gwe, lam_i);
              } else if (half == 1) {
                s_hpend[cbA] = own;          // completed by the earlier half's last step
              } else {
                s_pend[s & 1][cbA] = own;    // completed by the next segment's last step
              }
              if (ii == H - 1 && (half == 0 ? i + 1 < nt : ts + SEG < p.L)) {   // this step's terms at i + 1
                const float gwe = fmaf(-dy, ax.z, gq.x);
                const float crs = x * ax.y * gwe;
                lam_next = -x * dtn * gwe;
                const int64_t nxt = CSSCAN_BCK(p.hdr, row + D, int64_t(p.B) * L * D, 32);
                if (half == 0) {
                  p.ddt[nxt] = s_hpend[cbA] + crs;
                } else if (s < s_last) {
                  p.ddt[nxt] = s_pend[(s + 1) & 1][cbA] + crs;
                } else {
                  p.xb[CSSCAN_BCK(p.hdr, (int64_t(b) * p.C + chunk + 1) * D + dA_, int64_t(p.B) * p.C * D, 33)] = crs;
                }
              }
            }
          }
          if constexpr (MODE == 1) {
            // sums over the warp's channels (a warp's threads share the step), one shared add per warp
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
              lam_i += __shfl_xor_sync(0xffffffffu, lam_i, o);
              ge_i += __shfl_xor_sync(0xffffffffu, ge_i, o);
              lam_next += __shfl_xor_sync(0xffffffffu, lam_next, o);
            }
            if (lane == 0) {
              atomicAdd(&s_lam[i], lam_i);
              atomicAdd(&s_ge[i], ge_i);
              if (ii == H - 1) atomicAdd(&s_lam[i + 1], lam_next);
            }
          }
        }
      }
      __syncthreads();

      // ---- per (t, n) of the half: sums over the block's channels of dtheta, dBc, dCc (rotated
      // frame), written over the per-(t, d) partials
      {
        const int slot2 = w * M + c;
#pragma unroll
        for (int ii = 0; ii < H; ++ii) {
          float2* row = reinterpret_cast<float2*>(scr + ((ii * 5) * NG + g) * SROW) + slot2;
          row[0] = f2(aT[ii].x - aT2[ii].x, aT[ii].y - aT2[ii].y);
          row[(NG * SROW) / 2] = aBr[ii];
          row[2 * ((NG * SROW) / 2)] = aBi[ii];
          row[3 * ((NG * SROW) / 2)] = aCr[ii];
          row[4 * ((NG * SROW) / 2)] = f2(-aCi[ii].x, -aCi[ii].y);
        }
      }
      __syncthreads();
      {
        auto rsum = [&](int ii, int kind, int gg) {
          const float4* r4 = reinterpret_cast<const float4*>(scr + ((ii * 5 + kind) * NG + gg) * SROW);
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
          for (int u = 0; u < GT::SLOTS / 2; ++u) {
            const float4 a = r4[u];
            v.x += a.x;
            v.y += a.y;
            v.z += a.z;
            v.w += a.w;
          }
          return f2(v.x + v.z, v.y + v.w);   // (state 2gg, state 2gg + 1)
        };
        const int nh = min(H, nt - i0);
        for (int o = tid; o < nh * 3 * NG; o += THREADS) {
          const int ii = o / (3 * NG), rem = o % (3 * NG), kind = rem / NG, gg = rem % NG;
          const int64_t tn = CSSCAN_BCK(p.hdr, (int64_t(b) * L + ts + i0 + ii) * N + 2 * gg, int64_t(p.B) * L * N, 34);
          if (kind == 0) {
            atomicAdd(reinterpret_cast<float2*>(p.dtheta + tn), rsum(ii, 0, gg));
          } else {
            const float2 re = rsum(ii, 2 * kind - 1, gg), im = rsum(ii, 2 * kind, gg);
            float* dst = kind == 1 ? p.dBc : p.dCc;
            atomicAdd(reinterpret_cast<float4*>(dst + 2 * tn), make_float4(re.x, im.x, re.y, im.y));
          }
        }
      }
      __syncthreads();
    };
    run_half(std::integral_constant<int, 1>{});
    run_half(std::integral_constant<int, 0>{});

    if constexpr (MODE == 1) {
      if (tid <= SEG) {
        const int t = ts + tid;
        if (t < p.L && (tid < nt || tid == SEG)) atomicAdd(&p.dlam[int64_t(b) * L + t], s_lam[tid]);
        s_lam[tid] = 0.f;
      }
      if (tid < SEG) {
        if (tid < nt) atomicAdd(&p.ge[int64_t(b) * L + ts + tid], s_ge[tid]);
        s_ge[tid] = 0.f;
      }
      // (the next segment's first use of s_lam / s_ge comes after at least two barriers)
    }
  }

  if (aborted) {
    if (tid == 0) {
      record_error(p.hdr, ERR_PIPELINE, int(blockIdx.x), -3);
      // drain the copies still in flight (bounded)
      for (int u = q; u <= q + 1 && u <= s_last - s_first; ++u) wait_bar_bounded(&bar[u & 1], uint32_t(u >> 1) & 1u);
    }
    return;
  }

  // ---- the chunk's first step: ddt without the previous chunk's term (ngrad_fix_kernel adds it)
  if (MODE == 1 && rA == 0 && validA) p.ddt[(int64_t(b) * L + tc) * D + dA_] = s_pend[s_first & 1][cbA];
  if (validA) atomicAdd(&p.dD[dA_], dD_acc);
#pragma unroll 1
  for (int k = 0; k < K; ++k) {
    const int d = d0 + (k * WARPS + w) * M + c;
    if (d < p.D) atomicAdd(reinterpret_cast<float2*>(p.dA + int64_t(d) * N + 2 * g), s_dA[k][tid]);
  }
}

// ---------------------------------------------------------------------------- chunk carries
// Where the sequence is cut into C time chunks (whole 32-step sub-chunks), the gradient block of
// chunk c needs the adjoint carry entering its last step from chunk c + 1. The adjoint recurrence
// is affine per chunk: with kappa_c that (true-frame) carry,
//   kappa_{c-1} = V_c + G_c kappa_c,   G_c = exp(A sum_{t in c} dt_t) e^{-i sum_{t in c} theta_t},
// V_c being the carry out of chunk c's first step from a zero carry (the sub-chunk frames make the
// decays real; crossing into an earlier sub-chunk multiplies by e^{-i Phi_last} of that sub-chunk).
struct AdjParams {
  CUtensorMap tm_dy;   // (D, L, B) f32, box (CH, T_SUB, 1)
  CUtensorMap tm_dt;   // (D, L, B) input dtype, box (CH, T_SUB, 1)
  CUtensorMap tm_ct;   // the forward table (2N, 2, L, B) f32, box (2N, 1, T_SUB, 1): the Ct plane
  uint32_t* hdr;       // error word of the workspace header
  const float2* rot;   // (B, S32, 4, N) e^{i Phi} rows; row 3: after the sub-chunk's last step
  const float* dy;     // (B, L, D)
  const void* dt;      // (B, L, D) input dtype
  const float* A;      // (D, N)
  float2* V;           // (B, C, D, N)
  float* Sdt;          // (B, C, D)
  float2* P;           // (B, C, N) e^{-i sum theta} per chunk
  float2* kap;         // (B, C, D, N) kappa_c: the carry entering chunk c's last step
  int B, L, D, S32, TC, C, tab_ng;
};

// V_c and the chunk's sum of dt, for c >= 1: a thread per (b, c, channel, state group), the states
// of the forward kernel's thread (16, or N below 16) in the forward table's pair order; a block
// of 128 threads owns 128 / NG channels of one (b, c). Each 32-step sub-chunk's dy and dt rows of
// the block's channels and its Ct rows arrive by tile copies into a 2-slot ring (the next
// sub-chunk's while the current one is worked); rows past the sequence's end arrive as zeros and
// leave the carry unchanged.
template <int N, typename Tin>
struct AdjStage {
  static constexpr int NS = N >= 16 ? 16 : N;
  static constexpr int NG = N / NS;
  static constexpr int CH = 128 / NG;   // channels per block
  static constexpr int DY_BYTES = T_SUB * CH * 4;
  static constexpr int DT_BYTES = T_SUB * CH * int(sizeof(Tin));
  static constexpr int CT_BYTES = T_SUB * 2 * N * 4;
  static constexpr int OFF_DY = 0;
  static constexpr int OFF_DT = align128(OFF_DY + DY_BYTES);
  static constexpr int OFF_CT = align128(OFF_DT + DT_BYTES);
  static constexpr int BYTES = align128(OFF_CT + CT_BYTES);
  static constexpr int TX_BYTES = DY_BYTES + DT_BYTES + CT_BYTES;
  static constexpr int SMEM = 2 * BYTES + 128;
};

template <typename Tin, int N>
__global__ void __launch_bounds__(128) nadj_kernel(const __grid_constant__ AdjParams p) {
  using AS = AdjStage<N, Tin>;
  constexpr int NS = AS::NS, NG = AS::NG, CH = AS::CH, NPAIR = NS / 2;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  __shared__ __align__(8) uint64_t bar[2];
  const int tid = threadIdx.x;
  const int cl = tid / NG, g = tid % NG;
  const int d0 = blockIdx.x * CH;
  const int d = d0 + cl;
  const int c = blockIdx.y + 1;
  const int b = blockIdx.z;
  const int tc = c * p.TC, te = min(p.L, tc + p.TC);
  const int f_first = tc / T_SUB, f_last = (te - 1) / T_SUB;
  auto issue = [&](int f, int slot) {
    unsigned char* base = smem + slot * AS::BYTES;
    mbar_arrive_expect_tx(&bar[slot], uint32_t(AS::TX_BYTES));
    tma_load_3d(base + AS::OFF_DY, &p.tm_dy, d0, f * T_SUB, b, &bar[slot]);
    tma_load_3d(base + AS::OFF_DT, &p.tm_dt, d0, f * T_SUB, b, &bar[slot]);
    tma_load_4d(base + AS::OFF_CT, &p.tm_ct, 0, 1, f * T_SUB, b, &bar[slot]);
  };
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    prefetch_tmap(&p.tm_dy);
    prefetch_tmap(&p.tm_dt);
    prefetch_tmap(&p.tm_ct);
    issue(f_last, 0);
  }
  __syncthreads();
  const bool valid = d < p.D;
  float2 a2[NPAIR], cr[NPAIR], ci[NPAIR];
#pragma unroll
  for (int q = 0; q < NPAIR; ++q) {
    const int n = g * NS + 2 * q;
    a2[q] = valid ? f2(p.A[int64_t(d) * N + n] * LOG2E_F, p.A[int64_t(d) * N + n + 1] * LOG2E_F) : f2(0.f, 0.f);
    cr[q] = ci[q] = f2(0.f, 0.f);
  }
  float sdt = 0.f;
  bool aborted = false;
  int k = 0;
  for (int f = f_last; f >= f_first; --f, ++k) {
    const int slot = k & 1;
    // the other slot held sub-chunk f + 1, consumed before the barrier that closed it
    if (tid == 0 && f > f_first) issue(f - 1, slot ^ 1);
    if (f < f_last) {   // into sub-chunk f from f + 1: e^{-i Phi_last(f)}
      const float2* rr = p.rot + ((int64_t(b) * p.S32 + f) * 4 + 3) * N + g * NS;
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) {
        const float2 r0 = rr[2 * q], r1 = rr[2 * q + 1];
        const float2 cc = f2(r0.x, r1.x), ss = f2(r0.y, r1.y);
        const float2 nr = fma2(cc, cr[q], mul2(ss, ci[q]));
        const float2 ni = fma2(cc, ci[q], mul2(f2(-ss.x, -ss.y), cr[q]));
        cr[q] = nr;
        ci[q] = ni;
      }
    }
    const bool ok = wait_bar_bounded(&bar[slot], uint32_t(k >> 1) & 1u);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const unsigned char* base = smem + slot * AS::BYTES;
    const float* sdy = reinterpret_cast<const float*>(base + AS::OFF_DY) + cl;
    const Tin* sdtp = reinterpret_cast<const Tin*>(base + AS::OFF_DT) + cl;
    const float4* sct = reinterpret_cast<const float4*>(base + AS::OFF_CT) + g;
#pragma unroll 4
    for (int r = T_SUB - 1; r >= 0; --r) {
      const float dy = sdy[r * CH];
      const float dt = smem_in<Tin>(sdtp, r * CH);
      sdt += dt;
      const float2 dy2 = f2(dy, dy), dt2 = f2(dt, dt);
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) {
        const float4 cv = sct[r * (N / 2) + q * p.tab_ng];   // Ct: (Re, Re', -Im, -Im')
        const float2 r2 = ex2_pair(mul2(dt2, a2[q]));
        const float2 gr = fma2(dy2, f2(cv.x, cv.y), cr[q]);
        const float2 gi = fma2(dy2, f2(cv.z, cv.w), ci[q]);
        cr[q] = mul2(r2, gr);
        ci[q] = mul2(r2, gi);
      }
    }
    __syncthreads();
  }
  if (aborted) {
    if (tid == 0) {
      record_error(p.hdr, ERR_PIPELINE, int(blockIdx.x), -4);
      for (int u = k; u <= k + 1 && u <= f_last - f_first; ++u) wait_bar_bounded(&bar[u & 1], uint32_t(u >> 1) & 1u);
    }
    return;
  }
  if (!valid) return;
  float4* v4 = reinterpret_cast<float4*>(p.V + ((int64_t(b) * p.C + c) * p.D + d) * N + g * NS);
#pragma unroll
  for (int q = 0; q < NPAIR; ++q) v4[q] = make_float4(cr[q].x, ci[q].x, cr[q].y, ci[q].y);
  if (g == 0) p.Sdt[(int64_t(b) * p.C + c) * p.D + d] = sdt;
}

// P_c = e^{-i sum theta over chunk c} as the product of its sub-chunks' e^{-i Phi_last}.
static __global__ void __launch_bounds__(256) nphase_kernel(const AdjParams p, int N) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= int64_t(p.B) * p.C * N) return;
  const int n = int(gid % N);
  const int64_t bc = gid / N;
  const int c = int(bc % p.C);
  const int b = int(bc / p.C);
  const int tc = c * p.TC, te = min(p.L, tc + p.TC);
  float pr = 1.f, pi = 0.f;
  for (int f = tc / T_SUB; f <= (te - 1) / T_SUB; ++f) {
    const float2 r = p.rot[((int64_t(b) * p.S32 + f) * 4 + 3) * N + n];
    const float nr = pr * r.x + pi * r.y, ni = pi * r.x - pr * r.y;   // times conj(r)
    pr = nr;
    pi = ni;
  }
  p.P[gid] = make_float2(pr, pi);
}

// kappa_c for every chunk, walking from the last: a thread per (b, d, n).
static __global__ void __launch_bounds__(256) ncombine_kernel(const AdjParams p, int N) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= int64_t(p.B) * p.D * N) return;
  const int n = int(gid % N);
  const int64_t bd = gid / N;
  const int d = int(bd % p.D);
  const int b = int(bd / p.D);
  const float a2 = p.A[int64_t(d) * N + n] * LOG2E_F;
  float kr = 0.f, ki = 0.f;
  for (int c = p.C - 1; c >= 1; --c) {
    const int64_t bcd = (int64_t(b) * p.C + c) * p.D + d;
    p.kap[bcd * N + n] = make_float2(kr, ki);
    const float e = ex2_approx(a2 * p.Sdt[bcd]);
    const float2 P = p.P[(int64_t(b) * p.C + c) * N + n];
    const float gr = e * P.x, gi = e * P.y;
    const float2 V = p.V[bcd * N + n];
    const float nr = V.x + gr * kr - gi * ki, ni = V.y + gr * ki + gi * kr;
    kr = nr;
    ki = ni;
  }
  p.kap[(int64_t(b) * p.C * p.D + d) * N + n] = make_float2(kr, ki);
}

// dBc, dCc from the rotated-frame sums: thread per (b, sub-chunk, n), the sub-chunk's running phase
// recomputed exactly as the table kernel forms it, plus the trapezoid's G(E) terms.
template <typename Tin, int MODE>
__global__ void __launch_bounds__(256) ngrad_post_kernel(const void* theta, const void* Bc, const void* Cc,
                                                         const float* ge, float* dBc, float* dCc, int B, int L, int N,
                                                         int S32) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= int64_t(B) * S32 * N) return;
  const int n = int(gid % N);
  const int64_t bs = gid / N;
  const int s = int(bs % S32);
  const int b = int(bs / S32);
  const Tin* th = static_cast<const Tin*>(theta);
  const int t0 = s * T_SUB, t1 = min(t0 + T_SUB, L);
  float phi = 0.f, cs, sn;
  for (int t = t0; t < t1; ++t) {
    const int64_t tn = (int64_t(b) * L + t) * N + n;
    phi += load_in<Tin>(th, tn);
    sincosf(phi, &sn, &cs);
    const float2 bv = reinterpret_cast<const float2*>(dBc)[tn];
    const float2 cv = reinterpret_cast<const float2*>(dCc)[tn];
    float br = cs * bv.x - sn * bv.y, bi = cs * bv.y + sn * bv.x;   // e^{+i Phi} sum w gamma
    float cr = cs * cv.x + sn * cv.y, ci = cs * cv.y - sn * cv.x;   // e^{-i Phi} sum dy conj(g)
    if (MODE == 1) {
      const float e = ge[int64_t(b) * L + t];
      const float2 cc = load_pair<Tin>(static_cast<const Tin*>(Cc), tn);
      const float2 bc = load_pair<Tin>(static_cast<const Tin*>(Bc), tn);
      br = fmaf(e, cc.x, br);
      bi = fmaf(-e, cc.y, bi);
      cr = fmaf(e, bc.x, cr);
      ci = fmaf(-e, bc.y, ci);
    }
    reinterpret_cast<float2*>(dBc)[tn] = make_float2(br, bi);
    reinterpret_cast<float2*>(dCc)[tn] = make_float2(cr, ci);
  }
}

// ddt at the first step of chunks 1 .. C-1: add the previous chunk's last-step term.
static __global__ void __launch_bounds__(256) ngrad_fix_kernel(const float* xb, float* ddt, int B, int L, int D, int C,
                                                        int TC) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= int64_t(B) * (C - 1) * D) return;
  const int d = int(gid % D);
  const int64_t bc = gid / D;
  const int c = int(bc % (C - 1)) + 1;
  const int b = int(bc / (C - 1));
  ddt[(int64_t(b) * L + int64_t(c) * TC) * D + d] += xb[(int64_t(b) * C + c) * D + d];
}

}  // namespace ngrad
}  // namespace csscan
