// nscan_kernels.cuh -- forward scan kernels of the exp-Euler and exp-trapezoidal modes with the
// complex state normalised by the magnitude of its injection weight.
//
// What they compute is the recurrence of "Complex parallel scan" (section 并行扫描的数学本质)
// with the exp-Euler / exp-trapezoidal coefficients of the discretisation table and the complex
// phase of "Mamba-3 paper story", exactly as scan_kernels.cuh does; how they compute it:
//
// 1. Rotating frame (as in scan_kernels.cuh). Within a sub-chunk of T_SUB steps the state is
//    kept as g = e^{-i Phi} h, Phi the running sum of theta, so the decay is the real
//    r_t = 2^{dt_t A log2 e}; the rotated Bt = e^{-i Phi} Bc and Ct = e^{+i Phi} Cc come from
//    per-(b, t, n) tables shared by every channel, and the state is rotated back once per
//    sub-chunk.
// 2. Normalised state. Both modes inject a real per-(t, d) weight times Bt_t:
//        k_t = r_t k_{t-1} + w_t Bt_t,
//    exp-Euler w_t = dt_t x_t; trapezoid (look-ahead form of scan_kernels.cuh, k_{t+1} there)
//    w_t = x_t (lam_t dt_t + (1 - lam_{t+1}) dt_{t+1}). With sigma_t = w_t + sign(w_t) FLOOR and
//    s_t = k_t / sigma_t this is
//        s_t = rho_t s_{t-1} + Bt_t,   rho_t = 2^{dt_t A log2 e} (sigma_{t-1} / sigma_t),
//        y_t = sigma_t Re(sum_n Ct_t s_t) (+ the trapezoid correction and Dskip x_t):
//    the injection is the table entry itself, the per-(t, d) ratio costs one MUFU reciprocal per
//    channel and step, and the per-element product w_t Bt_t becomes one packed multiply of the
//    decay by the ratio: 6 FP32 lane-ops per element where the unnormalised update takes 7, and
//    every lane of a warp reads the same table row (broadcast shared-memory loads). FLOOR
//    (1e-20) changes an injection by at most 1e-20 |Bt| (a zero input gives an output of order
//    1e-20, not 0). The ratio's rounding is a relative error of a few ulps per step, the same
//    order as that of the hardware 2^x.
// 3. Thread tile. A thread owns one channel and NS consecutive states of it (NG = N / NS lanes
//    per channel, combined with shuffles); a block of 4 warps owns DT = 128 / NG channels.
//    The per-channel scalars (x, dt, the weight, its logarithm) are formed once per step for
//    NS elements and the output needs no shuffle when NG = 1.
// 4. Chunks, carries, bounded waits and the workspace records: as in scan_kernels.cuh, with
//    the chunk aggregate U = sigma_last s_last.
#pragma once

#include "scan_kernels.cuh"

namespace csscan {

constexpr float NSCAN_FLOOR = 1e-20f;
// Shared memory for the ring of one block (at least 2 stages): 80 KB holds three stages of the
// bf16 N = 16 tile, which leaves two blocks per SM; measured on B300, a third stage (the warps
// release stages independently and drift apart) with two resident blocks beats two stages with
// three resident blocks.
constexpr int NRING_BYTES = 80 * 1024;

template <int N, int NS>
struct NTile {
  static constexpr int NG = N / NS;
  static constexpr int NPAIR = NS / 2;
  static constexpr int CPW = 32 / NG;
  static constexpr int DT = WARPS * CPW;
  // table row: two planes (Bt, Ct) of W = 2N floats, state pairs interleaved by lane group
  static constexpr int PLANES = 2;
  static constexpr int W = 2 * N;
  static constexpr int W4 = W / 4;
  static_assert(NS >= 2 && NS % 2 == 0 && N % NS == 0 && NG <= 32 && (NG & (NG - 1)) == 0, "unsupported tile");
};

// One staged sub-chunk: x rows t0 .. t0+32 and dt rows t0 .. t0+32 (t0+33 in the trapezoid mode,
// its dt_{t+1}; the row past the sub-chunk feeds the software pipeline), table rows t0 .. t0+31
// (two planes of 2N floats: Bt and Ct, per state pair (re, re', im, im')), the trapezoid's
// (lam_t, 1 - lam_{t+1}, E_t, 0) rows t0 .. t0+32 and e^{i Phi} after the sub-chunk's last step.
template <int N, int NS, typename Tin, int MODE>
struct NStage {
  static constexpr int DT = NTile<N, NS>::DT;
  static constexpr int SIN = int(sizeof(Tin));
  static constexpr int X_ROWS = T_SUB + 1, DT_ROWS = MODE == 1 ? T_SUB + 2 : T_SUB + 1, TAB_ROWS = T_SUB;
  static constexpr int AUX_ROWS = T_SUB + 1;
  static constexpr int X_BYTES = X_ROWS * DT * SIN;
  static constexpr int DT_BYTES = DT_ROWS * DT * SIN;
  static constexpr int TAB_BYTES = TAB_ROWS * NTile<N, NS>::PLANES * NTile<N, NS>::W * 4;
  static constexpr int AUX_BYTES = MODE == 1 ? AUX_ROWS * 16 : 0;
  static constexpr int ROT_BYTES = 2 * N * 4;
  static constexpr int OFF_X = 0;
  static constexpr int OFF_DT = align128(OFF_X + X_BYTES);
  static constexpr int OFF_TAB = align128(OFF_DT + DT_BYTES);
  static constexpr int OFF_AUX = align128(OFF_TAB + TAB_BYTES);
  static constexpr int OFF_ROT = align128(OFF_AUX + AUX_BYTES);
  static constexpr int BYTES = align128(OFF_ROT + ROT_BYTES);
  static constexpr int TX_BYTES = X_BYTES + DT_BYTES + TAB_BYTES + AUX_BYTES + ROT_BYTES;
  static constexpr int FIT = NRING_BYTES / BYTES;
  static constexpr int NST = FIT >= 3 ? 3 : 2;
  static constexpr int SMEM = NST * BYTES + 128;
};

// ------------------------------------------------------------------------- table kernel
// One thread per (b, sub-chunk, n): the running phase Phi, the two table planes of every step,
// e^{i Phi} after local steps 7, 15, 23 and the last (the layout of scan_kernels.cuh's rot), and
// for the trapezoid the row (lam_t, 1 - lam_{t+1} (0 at t = L-1), E_t = sum_n Re(Cc_t Bc_t), 0).
template <typename Tin, int MODE>
__global__ void __launch_bounds__(256) ntable_kernel(TableParams p) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = int64_t(p.B) * p.S * p.N;
  if (gid >= total) return;
  const int n = int(gid % p.N);
  const int64_t bs = gid / p.N;
  const int s = int(bs % p.S);
  const int b = int(bs / p.S);
  const Tin* th = static_cast<const Tin*>(p.theta);
  const Tin* Bc = static_cast<const Tin*>(p.Bc);
  const Tin* Cc = static_cast<const Tin*>(p.Cc);
  const Tin* lam = static_cast<const Tin*>(p.lam);
  const int t0 = s * T_SUB, t1 = min(t0 + T_SUB, p.L);
  // position of state n's real part within a plane: pair j = n / 2 is pair q = j % npair of lane
  // group g = j / npair, stored at float4 q * ng + g (neighbouring groups read neighbouring banks)
  const int npair = p.N / (2 * p.ng);
  const int idx = (((n >> 1) % npair) * p.ng + (n >> 1) / npair) * 4 + (n & 1);
  const int W = p.plane_w;
  float phi = 0.f, cs = 1.f, sn = 0.f;
  float* rr = p.rot + ((int64_t(b) * p.S + s) * 4 * p.N + n) * 2;
  // E_t by a shuffle sum over the N lanes of (b, s), neighbours in a warp when N <= 32
  const bool lane_sum = MODE == 1 && p.N <= 32;
  const unsigned gmask = p.N >= 32 ? 0xffffffffu : (((1u << p.N) - 1u) << ((threadIdx.x & 31) & ~(p.N - 1)));
  // groups of 8 steps: every load of a group is issued before its arithmetic, so that the
  // group's memory latencies overlap (the phase itself is a running sum)
  for (int tg = t0; tg < t1; tg += 8) {
    float ths[8], brs[8], bis[8], crs[8], cis[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t tn = (int64_t(b) * p.L + min(tg + i, t1 - 1)) * p.N + n;
      ths[i] = load_in<Tin>(th, tn);
      brs[i] = load_in<Tin>(Bc, 2 * tn);
      bis[i] = load_in<Tin>(Bc, 2 * tn + 1);
      crs[i] = load_in<Tin>(Cc, 2 * tn);
      cis[i] = load_in<Tin>(Cc, 2 * tn + 1);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = tg + i;
      if (t >= t1) break;
      phi += ths[i];
      sincosf(phi, &sn, &cs);
      if (((t - t0) & 7) == 7) {
        rr[((t - t0) >> 3) * 2 * p.N] = cs;
        rr[((t - t0) >> 3) * 2 * p.N + 1] = sn;
      }
      const float br = brs[i], bi = bis[i];
      const float cr = crs[i], ci = cis[i];
      const float btr = cs * br + sn * bi;   // Re(e^{-i Phi} Bc)
      const float bti = cs * bi - sn * br;   // Im(e^{-i Phi} Bc)
      float* row = p.tab + CSSCAN_BCK(p.hdr, int64_t(b) * p.L + t, int64_t(p.B) * p.L, 20) * (p.planes * W);
      row[idx] = btr;
      row[idx + 2] = bti;
      row[W + idx] = cs * cr - sn * ci;        // Re(e^{+i Phi} Cc)
      row[W + idx + 2] = -(cs * ci + sn * cr); // -Im(e^{+i Phi} Cc)
      if (p.planes == 3) {
        row[2 * W + idx] = -btr;
        row[2 * W + idx + 2] = -bti;
      }
      if (lane_sum) {
        float E = cr * br - ci * bi;
        for (int o = p.N / 2; o >= 1; o >>= 1) E += __shfl_xor_sync(gmask, E, o);
        if (n == 0) {
          const int64_t tb = int64_t(b) * p.L + t;
          const float mu = (t + 1 < p.L) ? 1.f - load_in<Tin>(lam, tb + 1) : 0.f;
          reinterpret_cast<float4*>(p.aux)[tb] = make_float4(load_in<Tin>(lam, tb), mu, E, 0.f);
        }
      }
    }
  }
  for (int r = 0; r < 4; ++r) {   // rows past the sub-chunk's last step hold the last step's value
    if (8 * r + 7 > t1 - 1 - t0) {
      rr[r * 2 * p.N] = cs;
      rr[r * 2 * p.N + 1] = sn;
    }
  }
  if (MODE == 1 && n == 0 && !lane_sum) {   // N = 64: one lane sums the row
    for (int t = t0; t < t1; ++t) {
      const int64_t tb = int64_t(b) * p.L + t;
      float E = 0.f;
      for (int m = 0; m < p.N; ++m) {
        const int64_t tm = tb * p.N + m;
        E += load_in<Tin>(Cc, 2 * tm) * load_in<Tin>(Bc, 2 * tm) - load_in<Tin>(Cc, 2 * tm + 1) * load_in<Tin>(Bc, 2 * tm + 1);
      }
      const float mu = (t + 1 < p.L) ? 1.f - load_in<Tin>(lam, tb + 1) : 0.f;
      reinterpret_cast<float4*>(p.aux)[tb] = make_float4(load_in<Tin>(lam, tb), mu, E, 0.f);
    }
  }
}

// ------------------------------------------------------------------------- scan kernel
// Parameters: ScanParams of scan_kernels.cuh, with tm_tab a 4-D map (2N, 2, L, B) boxed
// (2N, 2, T_SUB, 1), tm_aux (4, L, B) boxed (4, AUX_ROWS, 1), tm_rot boxed (2N, 1, 1), tm_x boxed
// (DT, X_ROWS, 1) and tm_dt boxed (DT, DT_ROWS, 1).
// Two resident blocks per SM (the ring allows no more for the large tiles): up to 255 registers,
// which the decoupled variant needs to hold its look-back state without spilling.
constexpr int NSCAN_MIN_BLOCKS = 2;

// CKPT: the checkpoint variant the backward pass launches: no y; instead, before every 8-step
// segment s >= 1, the state after step 8 s - 1 in the rotating frame of the 32-step sub-chunk
// that holds step 8 s (the look-ahead state k in the trapezoid mode; the true state after the
// frame reset when 8 s starts a sub-chunk) into p.ckpt, (B, S8, D, N) complex.
template <int N, int NS, typename Tin, int MODE, int CARRY, bool CKPT = false>
__global__ void __launch_bounds__(THREADS, NSCAN_MIN_BLOCKS) nscan_kernel(const __grid_constant__ ScanParams p) {
  using TL = NTile<N, NS>;
  using SG = NStage<N, NS, Tin, MODE>;
  constexpr int NG = TL::NG, NPAIR = TL::NPAIR, CPW = TL::CPW, DT = TL::DT;
  constexpr int NST = SG::NST;
  constexpr int W4 = TL::W4;  // float4 per table plane (with padding)
  constexpr int PL = TL::PLANES;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
  __shared__ int s_ctl[8];
  __shared__ int s_done[MAX_STAGES];   // warps finished with the stage in each slot
  __shared__ int s_issued;             // stages issued so far

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  // The lanes of one state group are contiguous (a warp holds CPW channels for each of the NG
  // groups): a table load then has one address per quarter-warp (two shared-memory wavefronts per
  // 128-bit load; with the groups interleaved lane by lane it takes four).
  const int g = lane / CPW;                       // state group of this thread
  const int cl = (tid >> 5) * CPW + lane % CPW;   // channel of this thread within the block's tile
  const int n0 = g * NS;                          // first state of this thread
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
    // only possible if the ticket counter was not reset: touch no data, report, count out
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
  const int b = j / p.n_dtiles;
  const int d0 = (j % p.n_dtiles) * DT;
  const int d = d0 + cl;
  const bool dvalid = d < p.D;
  const int tc = c * p.TC;
  const int te = min(tc + p.TC, p.L);
  const int s_begin = tc / T_SUB;
  const int n_sub = (te - tc + T_SUB - 1) / T_SUB;
  const bool silent = (c == p.silent_chunk);
  const int64_t L = p.L, D = p.D;

  // ---- which passes: decoupled chunks first compute their aggregate, unless the
  // predecessor's final state is already visible.
  bool pass1 = false;
  if (CARRY == CARRY_DECOUPLED) {
    if (c == 0) {
      pass1 = true;
    } else {
      if (tid == 0) s_ctl[2] = flag_ready(ld_acquire_gpu(&p.ws.flags[CSSCAN_BCK(hdr, (c - 1) * p.n_tiles + j, p.n_units, 8)]), epoch, ST_INCL);
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
    tma_load_3d(base + SG::OFF_X, &p.tm_x, d0, sub * T_SUB, b, &full_bar[slot]);
    tma_load_3d(base + SG::OFF_DT, &p.tm_dt, d0, sub * T_SUB, b, &full_bar[slot]);
    tma_load_4d(base + SG::OFF_TAB, &p.tm_tab, 0, 0, sub * T_SUB, b, &full_bar[slot]);
    if (MODE == 1) tma_load_3d(base + SG::OFF_AUX, &p.tm_aux, 0, sub * T_SUB, b, &full_bar[slot]);
    tma_load_3d(base + SG::OFF_ROT, &p.tm_rot, 0, 4 * sub + 3, b, &full_bar[slot]);
  };
  if (tid == 0) {
    for (int gs = 0; gs < min(NST, total_stages); ++gs) issue(gs);
  }

  // ---- per-thread constants: log2(e) A of this channel's states, Dskip
  float2 Ap[NPAIR];
#pragma unroll
  for (int q = 0; q < NPAIR; ++q)
    Ap[q] = dvalid ? f2(p.A[int64_t(d) * p.N + n0 + 2 * q] * LOG2E_F, p.A[int64_t(d) * p.N + n0 + 2 * q + 1] * LOG2E_F)
                   : f2(0.f, 0.f);
  const float Dsk = dvalid ? p.Dskip[d] : 0.f;

  // trapezoid: the carries are the look-ahead state k_t = h_{t-1} + p_t Bc_{t-1} (it enters the
  // recurrence exactly as h does, k_{t+1} = a_t k_t + w_t Bc_t, so chunks compose on it), and only
  // the sequence's first step needs the halo p_0 Bc_{-1}, p_0 = (1 - lam_0) dt_0 x_{-1}, from the
  // caller's step -1 (x_prev, Bc_prev); at t = L - 1, 1 - lam_L is 0 and k_L = h_{L-1}.
  const bool has_halo = MODE == 1 && tc == 0 && p.x_prev != nullptr;
  auto add_halo = [&](float2* re, float2* im) {
    if (!has_halo || !dvalid) return;
    const Tin* dtin = static_cast<const Tin*>(p.dt);
    const Tin* lamin = static_cast<const Tin*>(p.lam);
    const float xprev = load_in<Tin>(static_cast<const Tin*>(p.x_prev), int64_t(b) * D + d);
    const Tin* bsrc = static_cast<const Tin*>(p.Bc_prev) + int64_t(b) * p.N * 2;
    const float hp = (1.f - load_in<Tin>(lamin, b * L + tc)) * load_in<Tin>(dtin, (b * L + tc) * D + d) * xprev;
    const float2 hp2 = f2(hp, hp);
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
      const int n = n0 + 2 * q;
      re[q] = fma2(hp2, f2(load_in<Tin>(bsrc, 2 * n), load_in<Tin>(bsrc, 2 * n + 2)), re[q]);
      im[q] = fma2(hp2, f2(load_in<Tin>(bsrc, 2 * n + 1), load_in<Tin>(bsrc, 2 * n + 3)), im[q]);
    }
  };

  float2 sr[NPAIR], si[NPAIR];   // normalised state pairs (re), (im) in the current frame
  float2 Rr[NPAIR], Ri[NPAIR];   // chunk rotation product (aggregate pass)
  float sdt_acc = 0.f;           // sum of dt over the chunk (aggregate pass)
  float aw_last = 1.f;           // signed sigma of the last step taken: the true state is aw_last * s
  int gstage = 0;
  bool aborted = false;

  // Per-step scalars of the software pipeline: what the output of a step needs (x, the signed
  // weight scale sigma, the trapezoid's correction p_{t+1} E_t) and what the next step needs
  // (sigma, and the trapezoid's dt_{t+1}). The step's decays live beside it in a float2[NPAIR].
  struct Scal {
    float x, sig, pc, E, dt, dtn;
  };

  // One pass over the chunk's sub-chunks, starting from the true state in (sr, si). WITH_Y: write
  // y; otherwise accumulate the aggregate's sum of dt and rotation. Software pipeline: step t+1's
  // scalars, logarithm and decays are formed during step t (they do not depend on the state), so
  // the state update never waits for the MUFU; the stage holds row 32 of x, aux and dt (and 33 of
  // dt), i.e. the next sub-chunk's first step, so the pipeline runs on across sub-chunks.
  auto run_pass = [&](auto with_y_tag) {
    constexpr bool WITH_Y = decltype(with_y_tag)::value;   // the final pass (from the true carry-in)
    constexpr bool OUT = WITH_Y && !CKPT;                  // ... writing y
    constexpr bool CK = WITH_Y && CKPT;                    // ... writing checkpoints
    Scal cur;
    float2 ec[NPAIR];
    for (int i = 0; i < n_sub; ++i, ++gstage) {
      const int slot = gstage % NST;
      if (!wait_bar_bounded(&full_bar[slot], uint32_t(gstage / NST) & 1u)) {
        aborted = true;   // a tile copy never arrived: stop consuming (the block agrees below)
        return;
      }
      const unsigned char* base = smem + slot * SG::BYTES;
      const Tin* sx = reinterpret_cast<const Tin*>(base + SG::OFF_X) + cl;
      const Tin* sdt = reinterpret_cast<const Tin*>(base + SG::OFF_DT) + cl;
      const float4* stab = reinterpret_cast<const float4*>(base + SG::OFF_TAB) + g;   // pair q at q * NG
      const float4* saux = reinterpret_cast<const float4*>(base + SG::OFF_AUX);
      const float4* srot = reinterpret_cast<const float4*>(base + SG::OFF_ROT) + g * NPAIR;
      const int t_sub0 = (s_begin + i) * T_SUB;
      const int nt = min(T_SUB, te - t_sub0);
      float* yrow = p.y + (b * L + t_sub0) * D + d;

      // scalars and decays of local step tt (rows tt of x and aux, tt and tt + 1 of dt), given the
      // previous step's scalars
      auto prep = [&](int tt, const Scal& pv, Scal& sc, float2 (&e)[NPAIR]) {
        const float x = smem_in<Tin>(sx, CSSCAN_BCKO(hdr, tt * DT, cl, SG::X_ROWS * DT, 1));
        float w, dt;
        if constexpr (MODE == 1) {
          dt = pv.dtn;   // dt_t was the previous step's look-ahead
          const float dtn = smem_in<Tin>(sdt, CSSCAN_BCKO(hdr, (tt + 1) * DT, cl, SG::DT_ROWS * DT, 2));
          const float4 a = saux[CSSCAN_BCK(hdr, tt, SG::AUX_ROWS, 3)];   // (lam_t, 1 - lam_{t+1}, E_t, 0)
          const float m = a.y * dtn;
          w = x * fmaf(a.x, dt, m);
          sc.pc = m * x;
          sc.E = a.z;
          sc.dtn = dtn;
        } else {
          dt = smem_in<Tin>(sdt, CSSCAN_BCKO(hdr, tt * DT, cl, SG::DT_ROWS * DT, 2));
          w = x * dt;
          sc.pc = 0.f;
          sc.E = 0.f;
          sc.dtn = 0.f;
        }
        sc.x = x;
        sc.dt = dt;
        // sigma = w + sign(w) FLOOR
        sc.sig = __uint_as_float(__float_as_uint(fabsf(w) + NSCAN_FLOOR) | (__float_as_uint(w) & 0x80000000u));
        const float2 dt2 = f2(dt, dt);
        // decay times sigma_{t-1} / sigma_t as a packed multiply by the signed ratio
        const float q = pv.sig * rcp_approx(sc.sig);
        const float2 q2 = f2(q, q);
#pragma unroll
        for (int k = 0; k < NPAIR; ++k) e[k] = mul2(ex2_pair(mul2(dt2, Ap[k])), q2);
      };
      if (i == 0) {   // the pass starts from the unscaled state: sigma_{-1} = 1
        Scal one;
        one.sig = 1.f;
        one.dtn = smem_in<Tin>(sdt, 0);
        prep(0, one, cur, ec);
      }

      auto step = [&](int tt) {
        const float4* row = stab + CSSCAN_BCK(hdr, tt, SG::TAB_ROWS, 4) * (PL * W4);
        Scal nxt;
        float2 en[NPAIR];
        prep(tt + 1, cur, nxt, en);
        float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);   // Re(Ct s), even and odd pairs
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          const float4 bb = row[q * NG];
          sr[q] = fma2(ec[q], sr[q], f2(bb.x, bb.y));
          si[q] = fma2(ec[q], si[q], f2(bb.z, bb.w));
          if (OUT) {
            const float4 cc = row[W4 + q * NG];
            float2& acc = (q & 1) ? acc1 : acc0;
            acc = fma2(f2(cc.z, cc.w), si[q], fma2(f2(cc.x, cc.y), sr[q], acc));
          }
        }
        if (OUT) {
          float ys = (acc0.x + acc0.y) + (acc1.x + acc1.y);
#pragma unroll
          for (int o = 1; o < NG; o <<= 1) ys += __shfl_xor_sync(0xffffffffu, ys, o * CPW);
          const float yv = fmaf(cur.sig, ys, fmaf(-cur.pc, cur.E, Dsk * cur.x));
          if (g == 0 && dvalid)
            __stcs(yrow + CSSCAN_BCKO(hdr, tt * D, (b * L + t_sub0) * D + d, int64_t(p.B) * L * D, 6), yv);
        } else if (!WITH_Y) {
          sdt_acc += cur.dt;
        }
        aw_last = cur.sig;
        cur = nxt;
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) ec[q] = en[q];
      };

      // the true state (sigma of the last step times s) before segment s8, as (re, im) per state
      auto store_ckpt = [&](int s8) {
        if (!dvalid) return;
        float4* r4 = p.ckpt + ((int64_t(b) * p.S8 + CSSCAN_BCK(hdr, s8, p.S8, 9)) * D + d) * (N / 2) + n0 / 2;
#pragma unroll
        for (int q = 0; q < NPAIR; ++q)
          __stcg(r4 + q, make_float4(aw_last * sr[q].x, aw_last * si[q].x, aw_last * sr[q].y, aw_last * si[q].y));
      };
      int tt = 0;
      for (; tt + 8 <= nt; tt += 8) {
#pragma unroll
        for (int u = 0; u < 8; ++u) step(tt + u);
        if (CK && tt + 8 < T_SUB && t_sub0 + tt + 8 < p.L) store_ckpt((t_sub0 + tt + 8) / 8);
      }
      for (; tt < nt; ++tt) step(tt);

      // frame reset: rotate the state by e^{i Phi_last} of this sub-chunk
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) {
        const float4 rr = srot[q];
        const float2 cc = f2(rr.x, rr.z), ss = f2(rr.y, rr.w), nss = f2(-rr.y, -rr.w);
        const float2 nr = fma2(cc, sr[q], mul2(nss, si[q]));
        const float2 ni = fma2(cc, si[q], mul2(ss, sr[q]));
        sr[q] = nr;
        si[q] = ni;
        if (!WITH_Y) {
          const float2 r2 = fma2(cc, Rr[q], mul2(nss, Ri[q]));
          const float2 i2 = fma2(cc, Ri[q], mul2(ss, Rr[q]));
          Rr[q] = r2;
          Ri[q] = i2;
        }
      }
      if (CK && nt == T_SUB && t_sub0 + T_SUB < p.L) store_ckpt((t_sub0 + T_SUB) / 8);
      // release the stage: the last warp to finish with it refills the slot with stage
      // gstage + NST, so the warps of a block never wait for one another between stages
      // (every value the warp loaded from the stage has been consumed by arithmetic above, so
      // the loads are complete; the empty asm keeps the compiler from sinking any of them)
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
  // every thread of the block learns whether any of its warps stopped on a missing copy
  auto run_pass_sync = [&](auto with_y_tag) {
    run_pass(with_y_tag);
    aborted = __syncthreads_or(aborted) != 0;
  };

  // ---- per-state helpers on the workspace records (float2 per state, states contiguous)
  auto rec_of = [&](float2* base, int u) {
    return base + (int64_t(CSSCAN_BCK(hdr, u, p.n_units, 7)) * DT + cl) * p.N + n0;
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
  // stores the true state aw_last * (re, im)
  auto store_scaled = [&](float2* rec, const float2* re, const float2* im) {
    float4* r4 = reinterpret_cast<float4*>(rec);
#pragma unroll
    for (int q = 0; q < NPAIR; ++q)
      __stcg(r4 + q, make_float4(aw_last * re[q].x, aw_last * im[q].x, aw_last * re[q].y, aw_last * im[q].y));
  };
  auto unit_of = [&](int chunk) { return chunk * p.n_tiles + j; };
  auto publish = [&](uint32_t status) {
    __threadfence();
    __syncthreads();
    if (tid == 0 && !silent) st_release_gpu(&p.ws.flags[CSSCAN_BCK(hdr, unit, p.n_units, 8)], (epoch << 2) | status);
  };

  float2 hr[NPAIR], hi[NPAIR];   // carry-in h_{tc-1}
#pragma unroll
  for (int q = 0; q < NPAIR; ++q) { hr[q] = f2(0.f, 0.f); hi[q] = f2(0.f, 0.f); }
  bool incl_published = false;
  const bool has_h0 = (p.h0 != nullptr) && dvalid;
  auto h0rec = [&]() { return reinterpret_cast<const float2*>(p.h0) + (int64_t(b) * p.D + d) * p.N + n0; };

  if (CARRY == CARRY_DECOUPLED && pass1) {
    // ---- pass 1: aggregate from a zero carry-in
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
      sr[q] = f2(0.f, 0.f);
      si[q] = f2(0.f, 0.f);
      Rr[q] = f2(1.f, 1.f);
      Ri[q] = f2(0.f, 0.f);
    }
    add_halo(sr, si);
    run_pass_sync(std::false_type{});
    if (!aborted) {
      if (!silent) {
        store_scaled(rec_of(p.ws.agg, unit), sr, si);
        if (g == 0) __stcg(p.ws.sdt + int64_t(unit) * DT + cl, sdt_acc);
        if (cl == 0) {
          float4* r4 = reinterpret_cast<float4*>(p.ws.crot + int64_t(unit) * p.N + n0);
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
      // h_in += exp(A Sd) Q * rec   (the accumulated multiplier of the chunks seen so far)
      auto accumulate = [&](const float2* rec, bool plain) {
        const float2 sd2 = f2(Sd, Sd);
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          const float4 v = plain ? reinterpret_cast<const float4*>(rec)[q] : __ldcg(reinterpret_cast<const float4*>(rec) + q);
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
            uint32_t st = ST_INCL;   // before the sequence: the initial state acts as a final state
            if (cp >= 0) {
              const uint32_t f = ld_acquire_gpu(&p.ws.flags[CSSCAN_BCK(hdr, unit_of(cp), p.n_units, 8)]);
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
          accumulate(rec_of(p.ws.agg, u2), false);
          Sd += __ldcg(p.ws.sdt + int64_t(u2) * DT + cl);
          const float4* cr4 = reinterpret_cast<const float4*>(p.ws.crot + int64_t(u2) * p.N + n0);
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
          if (cp < 0) {
            if (has_h0) accumulate(h0rec(), true);
          } else {
            accumulate(rec_of(p.ws.inc, unit_of(cp)), false);
          }
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
        const float2 ur = mul2(f2(aw_last, aw_last), sr[q]), ui = mul2(f2(aw_last, aw_last), si[q]);
        sr[q] = fma2(pr, hr[q], fma2(f2(-pi.x, -pi.y), hi[q], ur));   // scratch for the store
        si[q] = fma2(pr, hi[q], fma2(pi, hr[q], ui));
      }
      aw_last = 1.f;
      if (!silent) store_scaled(rec_of(p.ws.inc, unit), sr, si);
      publish(ST_INCL);
      incl_published = true;
    }
  } else if (CARRY != CARRY_NONE && c > 0) {
    // ---- serial carry, or a decoupled chunk whose predecessor had already published its
    // final state when this block started: wait for (or take) that final state
    if (tid == 0) {
      const uint32_t* fp = &p.ws.flags[CSSCAN_BCK(hdr, unit_of(c - 1), p.n_units, 8)];
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
  } else if (has_h0) {
    const float4* r4 = reinterpret_cast<const float4*>(h0rec());
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
      const float4 v = r4[q];
      hr[q] = f2(v.x, v.z);
      hi[q] = f2(v.y, v.w);
    }
  }

  if (!aborted) {
    // ---- pass 2: from the carry-in, writing y
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
      sr[q] = hr[q];
      si[q] = hi[q];
    }
    add_halo(sr, si);
    run_pass_sync(std::true_type{});
  }
  if (!aborted) {
    if (CARRY != CARRY_NONE && !incl_published) {
      if (!silent) store_scaled(rec_of(p.ws.inc, unit), sr, si);
      publish(ST_INCL);
    }
    if (c == p.n_chunks - 1 && p.h_last != nullptr && dvalid)
      store_scaled(reinterpret_cast<float2*>(p.h_last) + (int64_t(b) * p.D + d) * p.N + n0, sr, si);
  } else {
    // a tile copy never arrived: report, drain what is still in flight (bounded), leave
    if (tid == 0) {
      record_error(hdr, ERR_PIPELINE, unit, -1);
      for (int gs = max(0, s_issued - NST); gs < s_issued; ++gs)
        wait_bar_bounded(&full_bar[gs % NST], uint32_t(gs / NST) & 1u);
    }
  }

  // ---- last block out resets the ticket and advances the epoch for the next launch
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
