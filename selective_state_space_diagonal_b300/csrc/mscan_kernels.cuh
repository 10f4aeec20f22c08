// mscan_kernels.cuh -- the MIMO scan on the staged, rotating-frame design of nscan_kernels.cuh:
// the P channels of a head share one complex state ("Mamba-3 paper story", MIMO section).
//
//   a_t     = exp(dt[b,t,h] A[h,n] + i theta[b,t,n])
//   v_t[n]  = sum_p Bm[b,t,n,p] x[b,t,h,p]
//   exp-Euler   h_t = a_t h_{t-1} + dt_t v_t
//   trapezoid   h_t = a_t h_{t-1} + (1 - lam_t) dt_t a_t v_{t-1} + lam_t dt_t v_t
//   y[b,t,h,p] = Re(sum_n Cm[b,t,n,p] h_t[n]) + Dskip[h,p] x[b,t,h,p]
//
// How:
// 1. Rotating frame over sub-chunks of M_SUB steps: with Phi the running sum of theta,
//    Bt = e^{-i Phi} Bm and Ct = e^{+i Phi} Cm (per (b, t, n, p), written once by
//    mtable_kernel for all heads) make the decay real, r = 2^{dt A log2 e}.
// 2. Trapezoid look-ahead as in nscan_kernels.cuh: with c_t = lam_t dt_t + (1 - lam_{t+1})
//    dt_{t+1} and m_t = (1 - lam_{t+1}) dt_{t+1}, the carried k_{t+1} = r_t k_t + c_t V_t
//    (V_t = sum_p x_t[p] Bt_t[., p]) and
//        y_t[p] = Re(sum_n Ct_t[n, p] k_{t+1}[n]) - m_t sum_q x_t[q] E_t[p, q] + Dskip x_t[p],
//    E_t[p, q] = sum_n Re(Cm_t[n, p] Bm_t[n, q]) (frame-invariant, one P x P matrix per (b, t),
//    written by mtable_kernel): the same per-element work as exp-Euler (c = dt, m = 0).
// 3. Thread tile: one head and NS consecutive states of it for all P channels (NG = N / NS
//    lanes per head), NS chosen so that a thread handles about 16 channel-state elements per
//    step. Per step and state pair: the decay (shared by the P channels), the rank-P
//    injection (P packed FMAs per component), the update, and per channel the packed FMAs of
//    Re(Ct k). The partial outputs of G steps are reduce-scattered over the head's NG lanes at
//    once (independent shuffles rather than a dependent chain per step), which leaves each lane
//    the channels of one step to finish and store.
// 4. Staging, chunks and carries exactly as in nscan_kernels.cuh (3-stage TMA ring released per
//    warp, serial or decoupled carries with bounded waits); the state is not normalised (the
//    injection is not a per-channel scalar times a table entry).
#pragma once

#include "scan_kernels.cuh"

namespace csscan {

constexpr int M_SUB = 16;                 // sub-chunk (frame and stage) length
constexpr int MRING_BYTES = 96 * 1024;    // shared memory for the ring of one block

// Trapezoid aux row of P channels: E[p][q] (row-major), then lam_t and 1 - lam_{t+1} as one
// 8-byte aligned pair at this offset.
__host__ __device__ constexpr int mimo_lam_offset(int P) { return (P * P + 1) / 2 * 2; }

template <int N, int NS, int P>
struct MTile {
  static constexpr int NG = N / NS;       // lanes per head
  static constexpr int NPAIR = NS / 2;
  static constexpr int HPW = 32 / NG;     // heads per warp
  static constexpr int DH = WARPS * HPW;  // heads per block
  static constexpr int W4 = N / 2;        // float4 per (plane, channel) row of the table
  static constexpr int LAMW = mimo_lam_offset(P);       // offset of lam_t in the trapezoid row
  static constexpr int AUXW = (LAMW + 2 + 3) / 4 * 4;   // floats per trapezoid row
  static_assert(NS >= 2 && NS % 2 == 0 && N % NS == 0 && NG <= 16 && (NG & (NG - 1)) == 0, "unsupported tile");
  static_assert(DH * P <= 256 && DH <= 256, "tile wider than one tile copy");
};

template <int N, int NS, int P, typename Tin, int MODE>
struct MStage {
  using TL = MTile<N, NS, P>;
  static constexpr int SIN = int(sizeof(Tin));
  static constexpr int X_ROWS = M_SUB + 1, DT_ROWS = MODE == 1 ? M_SUB + 2 : M_SUB + 1, TAB_ROWS = M_SUB;
  static constexpr int AUX_ROWS = M_SUB + 1;
  static constexpr int X_BYTES = X_ROWS * TL::DH * P * SIN;
  static constexpr int DT_BYTES = DT_ROWS * TL::DH * SIN;
  static constexpr int TAB_BYTES = TAB_ROWS * 2 * P * 2 * N * 4;
  static constexpr int AUX_BYTES = MODE == 1 ? AUX_ROWS * TL::AUXW * 4 : 0;
  static constexpr int ROT_BYTES = 2 * N * 4;
  static constexpr int OFF_X = 0;
  static constexpr int OFF_DT = align128(OFF_X + X_BYTES);
  static constexpr int OFF_TAB = align128(OFF_DT + DT_BYTES);
  static constexpr int OFF_AUX = align128(OFF_TAB + TAB_BYTES);
  static constexpr int OFF_ROT = align128(OFF_AUX + AUX_BYTES);
  static constexpr int BYTES = align128(OFF_ROT + ROT_BYTES);
  static constexpr int TX_BYTES = X_BYTES + DT_BYTES + TAB_BYTES + AUX_BYTES + ROT_BYTES;
  static constexpr int FIT = MRING_BYTES / BYTES;
  static constexpr int NST = FIT >= 3 ? 3 : 2;
  static constexpr int SMEM = NST * BYTES + 128;
};

struct MTableParams {
  const void* Bm;      // (B, L, N, P, 2)
  const void* Cm;      // (B, L, N, P, 2)
  const void* theta;   // (B, L, N)
  const void* lam;     // (B, L), trapezoid only
  float* tab;          // (B, L, 2, P, 2N): Bt and Ct planes, per channel the state pairs as
                       // (Re, Re', Im, Im') (Ct's imaginary parts negated), interleaved by lane group
  float* aux;          // (B, L, auxw): E_t[p][q] (row-major), then at mimo_lam_offset(P) lam_t and
                       // 1 - lam_{t+1} (0 at t = L-1) (trapezoid)
  float* rot;          // (B, S, N, 2): e^{i Phi} after the sub-chunk's last step
  int B, L, N, P, S, ng, auxw;
  uint32_t* hdr;       // workspace header (error word of bounds-checked builds)
};

// One thread per (b, sub-chunk, n): the running phase, the rotated Bm and Cm of every channel,
// e^{i Phi} at the sub-chunk's end, and (trapezoid) E_t by shuffle sums over the N lanes of the
// sub-chunk, which are neighbours in a warp.
template <typename Tin, int MODE, int P>
__global__ void __launch_bounds__(256) mtable_kernel(MTableParams p) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = int64_t(p.B) * p.S * p.N;
  if (gid >= total) return;
  const int n = int(gid % p.N);
  const int64_t bs = gid / p.N;
  const int s = int(bs % p.S);
  const int b = int(bs / p.S);
  const Tin* th = static_cast<const Tin*>(p.theta);
  const Tin* Bm = static_cast<const Tin*>(p.Bm);
  const Tin* Cm = static_cast<const Tin*>(p.Cm);
  const Tin* lam = static_cast<const Tin*>(p.lam);
  const int t0 = s * M_SUB, t1 = min(t0 + M_SUB, p.L);
  const int npair = p.N / (2 * p.ng);
  const int idx = (((n >> 1) % npair) * p.ng + (n >> 1) / npair) * 4 + (n & 1);
  const int W = 2 * p.N;
  const unsigned gmask = p.N >= 32 ? 0xffffffffu : (((1u << p.N) - 1u) << ((threadIdx.x & 31) & ~(p.N - 1)));
  float phi = 0.f, cs = 1.f, sn = 0.f;
  for (int t = t0; t < t1; ++t) {
    const int64_t tn = (int64_t(b) * p.L + t) * p.N + n;
    phi += load_in<Tin>(th, tn);
    sincosf(phi, &sn, &cs);
    float* row = p.tab + CSSCAN_BCK(p.hdr, int64_t(b) * p.L + t, int64_t(p.B) * p.L, 21) * (2 * P * W);
    float br[P], bi[P], cr[P], ci[P];
#pragma unroll
    for (int q = 0; q < P; ++q) {
      const int64_t e = (tn * P + q) * 2;
      br[q] = load_in<Tin>(Bm, e);
      bi[q] = load_in<Tin>(Bm, e + 1);
      cr[q] = load_in<Tin>(Cm, e);
      ci[q] = load_in<Tin>(Cm, e + 1);
      float* bt = row + q * W;
      float* ct = row + (P + q) * W;
      bt[idx] = cs * br[q] + sn * bi[q];        // Re(e^{-i Phi} Bm)
      bt[idx + 2] = cs * bi[q] - sn * br[q];    // Im(e^{-i Phi} Bm)
      ct[idx] = cs * cr[q] - sn * ci[q];        // Re(e^{+i Phi} Cm)
      ct[idx + 2] = -(cs * ci[q] + sn * cr[q]); // -Im(e^{+i Phi} Cm)
    }
    if (MODE == 1) {
      float* a = p.aux + (int64_t(b) * p.L + t) * p.auxw;
#pragma unroll
      for (int pp = 0; pp < P; ++pp)
#pragma unroll
        for (int q = 0; q < P; ++q) {
          float E = cr[pp] * br[q] - ci[pp] * bi[q];
          for (int o = p.N / 2; o >= 1; o >>= 1) E += __shfl_xor_sync(gmask, E, o);
          if (n == 0) a[pp * P + q] = E;
        }
      if (n == 0) {
        const int64_t tb = int64_t(b) * p.L + t;
        a[mimo_lam_offset(P)] = load_in<Tin>(lam, tb);
        a[mimo_lam_offset(P) + 1] = (t + 1 < p.L) ? 1.f - load_in<Tin>(lam, tb + 1) : 0.f;
      }
    }
  }
  float* rr = p.rot + ((int64_t(b) * p.S + s) * p.N + n) * 2;
  rr[0] = cs;
  rr[1] = sn;
}

// Parameters of mscan_kernel: the carry workspace as in ScanParams.
struct MScanParams {
  CUtensorMap tm_x;    // (H P, L, B) input dtype, box (DH P, X_ROWS, 1)
  CUtensorMap tm_dt;   // (H, L, B) input dtype, box (DH, DT_ROWS, 1)
  CUtensorMap tm_tab;  // (2N, 2P, L, B) f32, box (2N, 2P, M_SUB, 1)
  CUtensorMap tm_aux;  // (AUXW, L, B) f32, box (AUXW, AUX_ROWS, 1)
  CUtensorMap tm_rot;  // (2N, S, B) f32, box (2N, 1, 1)
  const float* A;      // (H, N)
  const float* Dskip;  // (H, P)
  float* y;            // (B, L, H, P)
  Workspace ws;
  int B, L, H, N;
  int n_htiles, n_tiles, TC, n_chunks, n_units;
  int silent_chunk;
  long long poll_limit;
};

// Streaming store of K consecutive floats (p aligned to 4 K bytes; K = 1, 2, 4 or 8).
template <int K>
__device__ __forceinline__ void store_row(float* p, const float (&v)[K]) {
  if constexpr (K % 4 == 0) {
#pragma unroll
    for (int i = 0; i < K / 4; ++i)
      __stcs(reinterpret_cast<float4*>(p) + i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
  } else if constexpr (K == 2) {
    __stcs(reinterpret_cast<float2*>(p), make_float2(v[0], v[1]));
  } else {
    __stcs(p, v[0]);
  }
}

template <int N, int NS, int P, typename Tin, int MODE, int CARRY>
__global__ void __launch_bounds__(THREADS, 2) mscan_kernel(const __grid_constant__ MScanParams p) {
  using TL = MTile<N, NS, P>;
  using SG = MStage<N, NS, P, Tin, MODE>;
  constexpr int NG = TL::NG, NPAIR = TL::NPAIR, HPW = TL::HPW, DH = TL::DH, W4 = TL::W4;
  constexpr int NST = SG::NST;
  // steps per reduce-scatter of the partial outputs over the NG lanes of a head, the entries
  // reduced at once, and the entries (channels of one step) a lane holds afterwards
  constexpr int G = NG * P <= 32 ? NG : 32 / P;
  constexpr int LEN = G * P;
  constexpr int HOLDN = LEN / NG;
  static_assert(LEN >= NG && P % HOLDN == 0 && M_SUB % G == 0, "unsupported output split");

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
  __shared__ int s_ctl[8];
  __shared__ int s_done[MAX_STAGES];
  __shared__ int s_issued;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  // Lanes of one state group are consecutive (a warp holds HPW heads for each of the NG groups):
  // a table load then has one address per quarter-warp, which the shared-memory pipe serves in
  // two wavefronts per 128-bit load; with the groups interleaved lane by lane it takes four.
  const int g = lane / HPW;                        // state group of this thread
  const int hl = (tid >> 5) * HPW + lane % HPW;    // head of this thread within the block's tile
  const int n0 = g * NS;
  uint32_t* hdr = p.ws.hdr;

  if (tid == 0) {
    s_ctl[0] = int(atomicAdd(&hdr[H_TICKET], 1u));
    s_ctl[1] = int(ld_relaxed_gpu(&hdr[H_EPOCH]) & 0x3FFFFFFFu);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full_bar[i], 1);
      s_done[i] = 0;
    }
    fence_mbar_init();
    prefetch_tmap(&p.tm_x);
    prefetch_tmap(&p.tm_dt);
    prefetch_tmap(&p.tm_tab);
    if (MODE == 1) prefetch_tmap(&p.tm_aux);
    prefetch_tmap(&p.tm_rot);
  }
  __syncthreads();
  const int unit = s_ctl[0];
  const uint32_t epoch = uint32_t(s_ctl[1]);
  if (unit >= p.n_units) {
    if (tid == 0) {
      record_error(hdr, ERR_PIPELINE, unit, -2);
      const uint32_t prev = atomicAdd(&hdr[H_DONE], 1u);
      if (prev == uint32_t(p.n_units) - 1u) {
        atomicExch(&hdr[H_TICKET], 0u);
        atomicExch(&hdr[H_DONE], 0u);
        __threadfence();
        atomicAdd(&hdr[H_EPOCH], 1u);
      }
    }
    return;
  }
  const int c = unit / p.n_tiles;
  const int j = unit % p.n_tiles;
  const int b = j / p.n_htiles;
  const int h0 = (j % p.n_htiles) * DH;
  const int h = h0 + hl;
  const bool hvalid = h < p.H;
  const int tc = c * p.TC;
  const int te = min(tc + p.TC, p.L);
  const int s_begin = tc / M_SUB;
  const int n_sub = (te - tc + M_SUB - 1) / M_SUB;
  const bool silent = (c == p.silent_chunk);
  const int64_t L = p.L, H = p.H;

  bool pass1 = false;
  if (CARRY == CARRY_DECOUPLED) {
    if (c == 0) {
      pass1 = true;
    } else {
      if (tid == 0) s_ctl[2] = flag_ready(ld_acquire_gpu(&p.ws.flags[CSSCAN_BCK(hdr, (c - 1) * p.n_tiles + j, p.n_units, 18)]), epoch, ST_INCL);
      __syncthreads();
      pass1 = !s_ctl[2];
    }
  }
  const int total_stages = n_sub * (pass1 ? 2 : 1);

  auto issue = [&](int gs) {
    const int slot = gs % NST;
    s_issued = gs + 1;
    const int sub = s_begin + (gs % n_sub);
    unsigned char* base = smem + slot * SG::BYTES;
    mbar_arrive_expect_tx(&full_bar[slot], uint32_t(SG::TX_BYTES));
    tma_load_3d(base + SG::OFF_X, &p.tm_x, h0 * P, sub * M_SUB, b, &full_bar[slot]);
    tma_load_3d(base + SG::OFF_DT, &p.tm_dt, h0, sub * M_SUB, b, &full_bar[slot]);
    tma_load_4d(base + SG::OFF_TAB, &p.tm_tab, 0, 0, sub * M_SUB, b, &full_bar[slot]);
    if (MODE == 1) tma_load_3d(base + SG::OFF_AUX, &p.tm_aux, 0, sub * M_SUB, b, &full_bar[slot]);
    tma_load_3d(base + SG::OFF_ROT, &p.tm_rot, 0, sub, b, &full_bar[slot]);
  };
  if (tid == 0) {
    for (int gs = 0; gs < min(NST, total_stages); ++gs) issue(gs);
  }

  float2 Ap[NPAIR];
#pragma unroll
  for (int q = 0; q < NPAIR; ++q)
    Ap[q] = hvalid ? f2(p.A[int64_t(h) * N + n0 + 2 * q] * LOG2E_F, p.A[int64_t(h) * N + n0 + 2 * q + 1] * LOG2E_F)
                   : f2(0.f, 0.f);

  // the step within a group and the channels p0 .. p0 + HOLDN - 1 this lane writes, and their
  // Dskip
  const int hold_base = butterfly_base<NG, LEN>(g);
  const int s_hold = hold_base / P, p0 = hold_base % P;
  float Dsk[HOLDN];
#pragma unroll
  for (int v = 0; v < HOLDN; ++v) Dsk[v] = hvalid ? p.Dskip[int64_t(h) * P + p0 + v] : 0.f;

  float2 sr[NPAIR], si[NPAIR];   // state pairs (re), (im) in the current frame
  float2 Rr[NPAIR], Ri[NPAIR];   // chunk rotation product (aggregate pass)
  float sdt_acc = 0.f;
  int gstage = 0;
  bool aborted = false;

  // per-step scalars of the software pipeline: the head's P inputs scaled by the injection
  // weight, the raw inputs (D-skip, trapezoid correction), dt (and dt_{t+1}), the correction
  // weight m, and the step's decays beside them
  struct Scal {
    float x[P], cx[P];
    float dt, dtn, m;
  };

  auto run_pass = [&](auto with_y_tag) {
    constexpr bool WITH_Y = decltype(with_y_tag)::value;
    Scal cur;
    float2 ec[NPAIR];
    for (int i = 0; i < n_sub; ++i, ++gstage) {
      const int slot = gstage % NST;
      if (!wait_bar_bounded(&full_bar[slot], uint32_t(gstage / NST) & 1u)) {
        aborted = true;
        return;
      }
      const unsigned char* base = smem + slot * SG::BYTES;
      const Tin* sx = reinterpret_cast<const Tin*>(base + SG::OFF_X) + hl * P;
      const Tin* sdt = reinterpret_cast<const Tin*>(base + SG::OFF_DT) + hl;
      const float4* stab = reinterpret_cast<const float4*>(base + SG::OFF_TAB) + g;   // pair q at q * NG
      const float* saux = reinterpret_cast<const float*>(base + SG::OFF_AUX);
      const float4* srot = reinterpret_cast<const float4*>(base + SG::OFF_ROT) + g * NPAIR;
      const int t_sub0 = (s_begin + i) * M_SUB;
      const int nt = min(M_SUB, te - t_sub0);
      float* yrow = p.y + ((b * L + t_sub0) * H + h) * P;   // used only by the lanes of valid heads

      auto prep = [&](int tt, const Scal& pv, Scal& sc, float2 (&e)[NPAIR]) {
        smem_row<Tin, P>(sx + CSSCAN_BCKO(hdr, tt * (DH * P), hl * P, SG::X_ROWS * DH * P, 11), sc.x);
        float cw;
        if constexpr (MODE == 1) {
          sc.dt = pv.dtn;
          sc.dtn = smem_in<Tin>(sdt, CSSCAN_BCKO(hdr, (tt + 1) * DH, hl, SG::DT_ROWS * DH, 12));
          const float2 lm =
              *reinterpret_cast<const float2*>(saux + CSSCAN_BCK(hdr, tt, SG::AUX_ROWS, 13) * TL::AUXW + TL::LAMW);
          sc.m = lm.y * sc.dtn;
          cw = fmaf(lm.x, sc.dt, sc.m);
        } else {
          sc.dt = smem_in<Tin>(sdt, CSSCAN_BCKO(hdr, tt * DH, hl, SG::DT_ROWS * DH, 12));
          sc.dtn = 0.f;
          sc.m = 0.f;
          cw = sc.dt;
        }
#pragma unroll
        for (int q = 0; q < P; ++q) sc.cx[q] = cw * sc.x[q];
        const float2 dt2 = f2(sc.dt, sc.dt);
#pragma unroll
        for (int k = 0; k < NPAIR; ++k) e[k] = ex2_pair(mul2(dt2, Ap[k]));
      };
      if (i == 0) {
        Scal z;
        z.dtn = smem_in<Tin>(sdt, 0);
        prep(0, z, cur, ec);
      }

      // One step: the decays and scalars of step tt+1 (software pipeline), the rank-P injection
      // and the update of every state pair, and (WITH_Y) this lane's P partial outputs into
      // part[u * P ..].
      auto step = [&](int tt, int u, float (&part)[1][LEN]) {
        const float4* row = stab + CSSCAN_BCK(hdr, tt, SG::TAB_ROWS, 14) * (2 * P * W4);
        Scal nxt;
        float2 en[NPAIR];
        prep(tt + 1, cur, nxt, en);
        float2 acc[P];
#pragma unroll
        for (int q = 0; q < P; ++q) acc[q] = f2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NPAIR; ++k) {
          float2 vr = f2(0.f, 0.f), vi = f2(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < P; ++q) {
            const float4 bb = row[q * W4 + k * NG];
            const float2 w2 = f2(cur.cx[q], cur.cx[q]);
            vr = fma2(w2, f2(bb.x, bb.y), vr);
            vi = fma2(w2, f2(bb.z, bb.w), vi);
          }
          sr[k] = fma2(ec[k], sr[k], vr);
          si[k] = fma2(ec[k], si[k], vi);
          if (WITH_Y) {
#pragma unroll
            for (int q = 0; q < P; ++q) {
              const float4 cc = row[(P + q) * W4 + k * NG];
              acc[q] = fma2(f2(cc.z, cc.w), si[k], fma2(f2(cc.x, cc.y), sr[k], acc[q]));
            }
          }
        }
        if (WITH_Y) {
#pragma unroll
          for (int q = 0; q < P; ++q) part[0][u * P + q] = acc[q].x + acc[q].y;
        } else {
          sdt_acc += cur.dt;
        }
        cur = nxt;
#pragma unroll
        for (int k = 0; k < NPAIR; ++k) ec[k] = en[k];
      };

      // Groups of G steps; the partial outputs of a group are reduce-scattered over the head's
      // lanes at once (independent shuffles), after which each lane holds channels p0 .. of one
      // step, adds Dskip x and the trapezoid correction and stores them. Rows past the sequence's
      // end (a ragged last sub-chunk) arrive as zeros: dt = 0 and a zero table leave the state
      // unchanged, and their outputs are not stored.
#pragma unroll(G >= 8 ? 1 : 8 / G)
      for (int tt = 0; tt < nt; tt += G) {
        float part[1][LEN];
#pragma unroll
        for (int u = 0; u < G; ++u) step(tt + u, u, part);
        if (WITH_Y) {
          butterfly<NG, 1, LEN, HPW>(part, g);
          const int t = tt + s_hold;
          if (hvalid && t < nt) {
            float xa[P];   // the step's inputs: the held channels' Dskip term and the correction
            smem_row<Tin, P>(sx + CSSCAN_BCKO(hdr, t * (DH * P), hl * P, SG::X_ROWS * DH * P, 11), xa);
            float out[HOLDN];
            float m = 0.f;
            if constexpr (MODE == 1) m = saux[t * TL::AUXW + TL::LAMW + 1] * smem_in<Tin>(sdt, (t + 1) * DH);
#pragma unroll
            for (int v = 0; v < HOLDN; ++v) {
              // x of channel p0 + v (p0 is 0 unless a step's channels are split over lanes)
              float xv = xa[v];
              if constexpr (HOLDN < P) {
#pragma unroll
                for (int q = HOLDN; q < P; q += HOLDN) xv = (p0 == q) ? xa[q + v] : xv;
              }
              float corr = 0.f;
              if constexpr (MODE == 1) {
                float er[P];
                smem_row<float, P>(saux + t * TL::AUXW + (p0 + v) * P, er);
#pragma unroll
                for (int q = 0; q < P; ++q) corr = fmaf(xa[q], er[q], corr);
              }
              out[v] = fmaf(Dsk[v], xv, fmaf(-m, corr, part[0][v]));
            }
            store_row<HOLDN>(yrow + CSSCAN_BCKO(hdr, int64_t(t) * H * P + p0, ((b * L + t_sub0) * H + h) * P,
                                                int64_t(p.B) * L * H * P, 16),
                             out);
          }
        }
      }

      // frame reset: rotate the state by e^{i Phi_last} of this sub-chunk
#pragma unroll
      for (int k = 0; k < NPAIR; ++k) {
        const float4 rr = srot[k];
        const float2 cc = f2(rr.x, rr.z), ss = f2(rr.y, rr.w), nss = f2(-rr.y, -rr.w);
        const float2 nr = fma2(cc, sr[k], mul2(nss, si[k]));
        const float2 ni = fma2(cc, si[k], mul2(ss, sr[k]));
        sr[k] = nr;
        si[k] = ni;
        if (!WITH_Y) {
          const float2 r2 = fma2(cc, Rr[k], mul2(nss, Ri[k]));
          const float2 i2 = fma2(cc, Ri[k], mul2(ss, Rr[k]));
          Rr[k] = r2;
          Ri[k] = i2;
        }
      }
      // release the stage (as in nscan_kernel: the last warp to finish refills the slot)
      asm volatile("" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        if (atomicAdd(&s_done[slot], 1) == WARPS - 1) {
          s_done[slot] = 0;
          if (gstage + NST < total_stages) issue(gstage + NST);
        }
      }
    }
  };
  auto run_pass_sync = [&](auto with_y_tag) {
    run_pass(with_y_tag);
    aborted = __syncthreads_or(aborted) != 0;
  };

  auto rec_of = [&](float2* base, int u) {
    return base + (int64_t(CSSCAN_BCK(hdr, u, p.n_units, 17)) * DH + hl) * N + n0;
  };
  auto load_states = [&](const float2* rec, float2* re, float2* im) {
    const float4* r4 = reinterpret_cast<const float4*>(rec);
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
      const float4 v = __ldcg(r4 + q);
      re[q] = f2(v.x, v.z);
      im[q] = f2(v.y, v.w);
    }
  };
  auto store_states = [&](float2* rec, const float2* re, const float2* im) {
    float4* r4 = reinterpret_cast<float4*>(rec);
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) __stcg(r4 + q, make_float4(re[q].x, im[q].x, re[q].y, im[q].y));
  };
  auto unit_of = [&](int chunk) { return chunk * p.n_tiles + j; };
  auto publish = [&](uint32_t status) {
    __threadfence();
    __syncthreads();
    if (tid == 0 && !silent) st_release_gpu(&p.ws.flags[CSSCAN_BCK(hdr, unit, p.n_units, 18)], (epoch << 2) | status);
  };

  float2 hr[NPAIR], hi[NPAIR];
#pragma unroll
  for (int q = 0; q < NPAIR; ++q) { hr[q] = f2(0.f, 0.f); hi[q] = f2(0.f, 0.f); }
  bool incl_published = false;

  if (CARRY == CARRY_DECOUPLED && pass1) {
    // ---- pass 1: aggregate from a zero carry-in
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
      sr[q] = f2(0.f, 0.f);
      si[q] = f2(0.f, 0.f);
      Rr[q] = f2(1.f, 1.f);
      Ri[q] = f2(0.f, 0.f);
    }
    run_pass_sync(std::false_type{});
    if (!aborted) {
      if (!silent) {
        store_states(rec_of(p.ws.agg, unit), sr, si);
        if (g == 0) __stcg(p.ws.sdt + int64_t(unit) * DH + hl, sdt_acc);
        if (hl == 0) {
          float4* r4 = reinterpret_cast<float4*>(p.ws.crot + int64_t(unit) * N + n0);
#pragma unroll
          for (int q = 0; q < NPAIR; ++q) __stcg(r4 + q, make_float4(Rr[q].x, Ri[q].x, Rr[q].y, Ri[q].y));
        }
      }
      publish(ST_AGG);

      // ---- decoupled look-back over windows of 32 predecessors
      float Sd = 0.f;
      float2 Qr[NPAIR], Qi[NPAIR];
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) { Qr[q] = f2(1.f, 1.f); Qi[q] = f2(0.f, 0.f); }
      auto accumulate = [&](const float2* rec) {
        const float2 sd2 = f2(Sd, Sd);
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(rec) + q);
          const float2 ur = f2(v.x, v.z), ui = f2(v.y, v.w);
          const float2 e = ex2_pair(mul2(sd2, Ap[q]));
          const float2 mr = mul2(e, Qr[q]), mi = mul2(e, Qi[q]);
          hr[q] = fma2(mr, ur, fma2(f2(-mi.x, -mi.y), ui, hr[q]));
          hi[q] = fma2(mr, ui, fma2(mi, ur, hi[q]));
        }
      };
      int pred = c - 1;
      while (true) {
        if (tid < 32) {
          const int cp = pred - tid;
          int count = 0, found = 0, tout = 0;
          long long polls = 0;
          while (true) {
            uint32_t st = ST_INCL;   // before the sequence: the zero initial state acts as a final state
            if (cp >= 0) {
              const uint32_t f = ld_acquire_gpu(&p.ws.flags[CSSCAN_BCK(hdr, unit_of(cp), p.n_units, 18)]);
              st = ((f >> 2) == epoch) ? (f & 3u) : ST_NONE;
            }
            const unsigned incl = __ballot_sync(0xffffffffu, st == ST_INCL);
            const unsigned ready = __ballot_sync(0xffffffffu, st != ST_NONE);
            const int first = incl ? __ffs(incl) - 1 : 32;
            const unsigned need = first >= 31 ? 0xffffffffu : ((2u << first) - 1u);
            if ((need & ~ready) == 0u) { count = first; found = first < 32; break; }
            if (++polls > p.poll_limit) {
              count = (~ready == 0u) ? 32 : __ffs(~ready) - 1;
              tout = 1;
              break;
            }
            __nanosleep(polls < 32 ? 64 : 512);
          }
          if (tid == 0) {
            s_ctl[3] = count;
            s_ctl[4] = found;
            s_ctl[5] = tout;
            if (tout) record_error(hdr, ERR_LOOKBACK, unit, pred - count);
          }
        }
        __syncthreads();
        const int count = s_ctl[3], found = s_ctl[4], tout = s_ctl[5];
        for (int i = 0; i < count; ++i) {
          const int u2 = unit_of(pred - i);
          accumulate(rec_of(p.ws.agg, u2));
          Sd += __ldcg(p.ws.sdt + int64_t(u2) * DH + hl);
          const float4* cr4 = reinterpret_cast<const float4*>(p.ws.crot + int64_t(u2) * N + n0);
#pragma unroll
          for (int q = 0; q < NPAIR; ++q) {
            const float4 v = __ldcg(cr4 + q);
            const float2 rr = f2(v.x, v.z), ri = f2(v.y, v.w);
            const float2 nr = fma2(Qr[q], rr, mul2(f2(-Qi[q].x, -Qi[q].y), ri));
            const float2 ni = fma2(Qr[q], ri, mul2(Qi[q], rr));
            Qr[q] = nr;
            Qi[q] = ni;
          }
        }
        __syncthreads();
        if (found) {
          const int cp = pred - count;
          if (cp >= 0) accumulate(rec_of(p.ws.inc, unit_of(cp)));
          break;
        }
        if (tout) break;
        pred -= 32;
      }
      // ---- publish this chunk's final state: h_end = P h_in + U, P = exp(A sum dt) R
      const float2 sd2 = f2(sdt_acc, sdt_acc);
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) {
        const float2 e = ex2_pair(mul2(sd2, Ap[q]));
        const float2 pr = mul2(e, Rr[q]), pi = mul2(e, Ri[q]);
        sr[q] = fma2(pr, hr[q], fma2(f2(-pi.x, -pi.y), hi[q], sr[q]));   // scratch for the store
        si[q] = fma2(pr, hi[q], fma2(pi, hr[q], si[q]));
      }
      if (!silent) store_states(rec_of(p.ws.inc, unit), sr, si);
      publish(ST_INCL);
      incl_published = true;
    }
  } else if (CARRY != CARRY_NONE && c > 0) {
    if (tid == 0) {
      const uint32_t* fp = &p.ws.flags[CSSCAN_BCK(hdr, unit_of(c - 1), p.n_units, 18)];
      long long polls = 0;
      int tout = 0;
      while (!flag_ready(ld_acquire_gpu(fp), epoch, ST_INCL)) {
        if (++polls > p.poll_limit) { tout = 1; break; }
        __nanosleep(polls < 32 ? 64 : 512);
      }
      s_ctl[5] = tout;
      if (tout) record_error(hdr, ERR_LOOKBACK, unit, c - 1);
    }
    __syncthreads();
    if (!s_ctl[5]) load_states(rec_of(p.ws.inc, unit_of(c - 1)), hr, hi);
  }

  if (!aborted) {
    // ---- pass 2: from the carry-in, writing y
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
      sr[q] = hr[q];
      si[q] = hi[q];
    }
    run_pass_sync(std::true_type{});
  }
  if (!aborted) {
    if (CARRY != CARRY_NONE && !incl_published) {
      if (!silent) store_states(rec_of(p.ws.inc, unit), sr, si);
      publish(ST_INCL);
    }
  } else {
    if (tid == 0) {
      record_error(hdr, ERR_PIPELINE, unit, -1);
      for (int gs = max(0, s_issued - NST); gs < s_issued; ++gs)
        wait_bar_bounded(&full_bar[gs % NST], uint32_t(gs / NST) & 1u);
    }
  }

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&hdr[H_DONE], 1u);
    if (prev == uint32_t(p.n_units) - 1u) {
      atomicExch(&hdr[H_TICKET], 0u);
      atomicExch(&hdr[H_DONE], 0u);
      __threadfence();
      atomicAdd(&hdr[H_EPOCH], 1u);
    }
  }
}

}  // namespace csscan
