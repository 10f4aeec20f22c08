// scan_kernels.cuh -- the two kernels of the forward selective scan.
//
// Method (what the kernels compute is the recurrence of "Complex parallel scan",
// section 并行扫描的数学本质, with the exp-Euler / exp-trapezoidal coefficients of the
// discretisation table and the complex phase of "Mamba-3 paper story"; how they compute
// it is specific to this library):
//
// 1. Rotating frame. Within a sub-chunk of T_SUB steps starting at t0 let
//    Phi_t = sum_{k=t0..t} theta_k (per b, n). With g_t = e^{-i Phi_t} h_t the recurrence
//    becomes real-decay only: g_t = r_t g_{t-1} + e^{-i Phi_t} u_t, r_t = exp(dt_t A).
//    The phase work moves to per-(b,t,n) tables shared by every channel d:
//    Bt_t = e^{-i Phi_t} Bc_t and Ct_t = e^{+i Phi_t} Cc_t, and Re(Cc h) = Re(Ct g).
//    At the end of a sub-chunk the state is rotated back by e^{i Phi_last} (frame reset),
//    which keeps Phi small and accurate in float32.
// 2. Trapezoid look-ahead. With p_t = (1-lam_t) dt_t x_{t-1}, q_t = lam_t dt_t x_t and
//    k_t = g_{t-1} + p_t Bt_{t-1}, the trapezoidal step becomes
//        k_{t+1} = r_t k_t + (q_t + p_{t+1}) Bt_t,
//        y_t = Re(sum_n Ct_t k_{t+1}) - p_{t+1} E_t + Dskip x_t,  E_t = sum_n Re(Cc_t Bc_t),
//    the same per-element cost as exp-Euler (which is the case p = 0, q = dt x).
// 3. Thread tile. A block has 4 warps (one per SM sub-partition). A thread owns CH = 2
//    adjacent channels and NS consecutive states of each; NG = N / NS neighbouring lanes
//    share one channel pair and sum their partial outputs with a shuffle. Every table value
//    a thread loads from shared memory serves both of its channels.
// 4. Chunks. A thread block owns DT channels of one batch row for one chunk of TC steps.
//    The chunk's map h_in -> h_end is affine: h_end = P h_in + U with
//    P = exp(A sum dt) e^{i sum theta} (the combine of the step operators), so a chunk can
//    publish U before it knows h_in, and successors combine predecessors' (P, U) pairs
//    (decoupled look-back) or wait for the predecessor's final state (serial carry).
//    Chunk order comes from an atomic ticket, so a block only ever waits on blocks that
//    started earlier; every wait is bounded and reports a status instead of hanging.
// 5. Zero-order hold (MODE 2). The injection is dt x Bc (e^z - 1) / z with z = dt A + i theta,
//    a complex weight per (t, d, n) (ZOH row of the discretisation table of "Mamba-3 paper
//    story", complex exponent as for alpha_t). With e^z - 1 = E e^{i theta} + (e^{i theta} - 1),
//    E = e^{dt A} - 1, the frame injection is dt x (E beta_t + delta_t) / z, where
//    beta_t = Bt_t e^{i theta_t} and delta_t = Bt_t (e^{i theta_t} - 1) are per-(b, t, n) table
//    entries. A thread forms per element only E (a Taylor polynomial where |dt A| is small,
//    else r - 1), one complex product with conj(z) and a hardware reciprocal of |z|^2. The
//    table holds beta, delta and theta in base-2 units (times log2 e), so that the decay's
//    own argument v = dt A log2 e is Re z; |z|^2 carries a floor tau whose numerator partner
//    tau beta makes the weight tend to Bt as z -> 0.
#pragma once

#include <type_traits>

#include "device_util.cuh"

namespace csscan {

constexpr int T_SUB = 32;       // sub-chunk: one rotation frame and one staged tile
constexpr int CH = 2;           // channels per thread
constexpr int WARPS = 4;        // warps per block
constexpr int THREADS = WARPS * 32;
constexpr int MAX_STAGES = 4;   // depth of the shared-memory ring
constexpr int RING_BYTES = 56 * 1024;   // shared memory for the ring of one block
constexpr float LOG2E_F = 1.4426950408889634f;
// Zero-order hold: Taylor coefficients (ln 2)^k / k! of 2^v - 1, the |v| below which that
// polynomial (truncation below 3e-8 relative) replaces r - 1, and the floor tau of |z|^2.
constexpr float ZOH_C1 = 0.6931471805599453f, ZOH_C2 = 0.2402265069591007f;
constexpr float ZOH_C3 = 0.05550410866482158f, ZOH_C4 = 0.009618129107628477f;
constexpr float ZOH_V_POLY = 0.0625f;
constexpr float ZOH_TAU = 1e-30f;
constexpr float ZOH_TAU_LN2 = ZOH_TAU * 0.6931471805599453f;   // tau times beta / beta'

// Thread tile for N states: NS states per thread, NG lanes per channel pair, CPW channels
// per warp, DT channels per block.
template <int N>
struct Tile {
  static constexpr int NS = N >= 8 ? 8 : N;
  static constexpr int NG = N / NS;
  static constexpr int NPAIR = NS / 2;
  static constexpr int CPW = 32 / NG * CH;
  static constexpr int DT = WARPS * CPW;
  static_assert(NS % 2 == 0 && NG >= 1 && NG <= 32 && (NG & (NG - 1)) == 0, "unsupported N");
};

// Shared-memory stage: one sub-chunk of one block. Rows past the sub-chunk (one of x, aux and
// the table, two of dt) feed the software pipeline's look-ahead and the trapezoid's dt_{t+1}.
constexpr int align128(int v) { return (v + 127) & ~127; }
template <int N, typename Tin, int MODE>
struct Stage {
  static constexpr int DT = Tile<N>::DT;
  static constexpr int SIN = int(sizeof(Tin));
  static constexpr int X_ROWS = T_SUB + 1, DT_ROWS = T_SUB + 2, AUX_ROWS = T_SUB + 1, TAB_ROWS = T_SUB + 1;
  static constexpr int AUX_W = 8;                       // floats per aux row
  static constexpr int X_BYTES = X_ROWS * DT * SIN;
  static constexpr int DT_BYTES = DT_ROWS * DT * SIN;
  static constexpr int TABW = MODE == 2 ? 8 : 4;         // table floats per state and step
  static constexpr int TAB_BYTES = TAB_ROWS * TABW * N * 4;
  static constexpr int AUX_BYTES = MODE == 1 ? AUX_ROWS * AUX_W * 4 : 0;
  static constexpr int ROT_BYTES = 4 * 2 * N * 4;       // e^{i Phi} after local steps 7, 15, 23, last
  static constexpr int OFF_X = 0;
  static constexpr int OFF_DT = align128(OFF_X + X_BYTES);
  static constexpr int OFF_TAB = align128(OFF_DT + DT_BYTES);
  static constexpr int OFF_AUX = align128(OFF_TAB + TAB_BYTES);
  static constexpr int OFF_ROT = align128(OFF_AUX + AUX_BYTES);
  static constexpr int BYTES = align128(OFF_ROT + ROT_BYTES);
  static constexpr int TX_BYTES = X_BYTES + DT_BYTES + TAB_BYTES + AUX_BYTES + ROT_BYTES;
  static constexpr int FIT = RING_BYTES / BYTES;
  static constexpr int NST = FIT >= MAX_STAGES ? MAX_STAGES : (FIT >= 2 ? FIT : 2);
  static constexpr int SMEM = NST * BYTES + 128;        // + alignment slack
};

enum : uint32_t { ST_NONE = 0, ST_AGG = 1, ST_INCL = 2 };
enum : int { CARRY_NONE = 0, CARRY_SERIAL = 1, CARRY_DECOUPLED = 2 };
enum : uint32_t { ERR_LOOKBACK = 1u, ERR_PIPELINE = 2u, ERR_BOUNDS = 4u };
enum { H_EPOCH = 0, H_TICKET = 1, H_DONE = 2, H_ERROR = 3, H_ERR_UNIT = 4, H_ERR_PRED = 5 };

constexpr long long MBAR_WAIT_LIMIT = 1ll << 22;   // about 0.5 s of polling

struct Workspace {
  uint32_t* hdr;     // epoch, ticket, done, error, error unit, error predecessor
  uint32_t* flags;   // [units] (epoch << 2) | status
  float2* inc;       // [units][DT][N] final state of the chunk
  float2* agg;       // [units][DT][N] chunk aggregate U (state reached from zero)
  float* sdt;        // [units][DT]    sum of dt over the chunk
  float2* crot;      // [units][N]     e^{i sum theta} over the chunk
};

// ------------------------------------------------------------------------- table kernel
struct TableParams {
  const void* Bc;
  const void* Cc;
  const void* theta;
  const void* lam;
  float* tab;  // (B, L, N/2, 8): per state pair (Btr, Btr', Bti, Bti', Ctr, Ctr', -Cti, -Cti');
               // zero-order hold (B, L, N/2, 16): (beta re x2, beta im x2, Ct as above,
               // delta re x2, delta im x2, theta x2, theta^2 + tau x2), beta, delta and theta
               // times log2 e
  float* aux;  // (B, L, 8): lam_t, lam_t, mu, mu, E_t, E_t, 0, 0 with mu = 1 - lam_{t+1}
               // (0 at t = L-1) (trapezoid only)
  float* rot;  // (B, S, 4, N, 2): e^{i Phi} of sub-chunk s after its local steps 7, 15, 23 and
               // after its last step (row r: local step min(8 r + 7, last))
  int B, L, N, S;
  int ng;      // nscan table only: lane groups per channel; state pairs are stored interleaved
               // by group (pair q of group g at position q * ng + g)
  int planes;  // nscan table only: planes per row (Bt, Ct, and -Bt when 3)
  int plane_w; // nscan table only: floats per plane (2N plus padding)
  uint32_t* hdr;   // workspace header (error word of bounds-checked builds)
  int n_full;  // scan table only: states per (b, t) row of Bc, Cc and theta (N of the whole problem)
  int n_off;   // scan table only: first state of this part (the tables hold states n_off .. n_off + N - 1)
};

template <typename Tin, int MODE>
__global__ void __launch_bounds__(256) table_kernel(TableParams p) {
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
  const int t0 = s * T_SUB, t1 = min(t0 + T_SUB, p.L);
  const int q = n >> 1, odd = n & 1;
  float phi = 0.f, cs = 1.f, sn = 0.f;
  float* rr = p.rot + ((int64_t(b) * p.S + s) * 4 * p.N + n) * 2;   // row r at rr + r * 2N
  // trapezoid: E_t = sum_n Re(Cc_t Bc_t) by a shuffle sum over the N lanes of (b, s), which are
  // neighbours in a warp when N <= 32 (whole groups: the thread count is a multiple of N)
  const bool lane_sum = MODE == 1 && p.N <= 32;
  const unsigned gmask = p.N >= 32 ? 0xffffffffu : (((1u << p.N) - 1u) << ((threadIdx.x & 31) & ~(p.N - 1)));
  const Tin* lam = static_cast<const Tin*>(p.lam);
  // groups of 8 steps: every load of a group is issued before its arithmetic, so that the
  // group's memory latencies overlap (the phase itself is a running sum)
  for (int tg = t0; tg < t1; tg += 8) {
    float ths[8], brs[8], bis[8], crs[8], cis[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t tn = (int64_t(b) * p.L + min(tg + i, t1 - 1)) * p.n_full + p.n_off + n;   // this state in the inputs
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
      const float th_t = ths[i];
      phi += th_t;
      sincosf(phi, &sn, &cs);
      if (((t - t0) & 7) == 7) {
        rr[((t - t0) >> 3) * 2 * p.N] = cs;
        rr[((t - t0) >> 3) * 2 * p.N + 1] = sn;
      }
      const float br = brs[i], bi = bis[i];
      const float cr = crs[i], ci = cis[i];
      constexpr int TW = MODE == 2 ? 8 : 4;
      float* row = p.tab + (int64_t(b) * p.L + t) * (TW * p.N) + q * 2 * TW;
      const float btr = cs * br + sn * bi;   // Re(e^{-i Phi} Bc)
      const float bti = cs * bi - sn * br;   // Im(e^{-i Phi} Bc)
      if (MODE == 2) {
        // e^{i theta} - 1 without cancellation: cos theta - 1 = -2 sin^2(theta / 2)
        float sh, chh;
        sincosf(0.5f * th_t, &sh, &chh);
        const float cm1 = -2.f * sh * sh, s1 = 2.f * sh * chh, c1 = 1.f + cm1;
        row[odd] = LOG2E_F * (btr * c1 - bti * s1);        // beta = Bt e^{i theta}
        row[2 + odd] = LOG2E_F * (btr * s1 + bti * c1);
        row[8 + odd] = LOG2E_F * (btr * cm1 - bti * s1);   // delta = Bt (e^{i theta} - 1)
        row[10 + odd] = LOG2E_F * (btr * s1 + bti * cm1);
        const float tq = LOG2E_F * th_t;
        row[12 + odd] = tq;
        row[14 + odd] = fmaf(tq, tq, ZOH_TAU);
      } else {
        row[odd] = btr;
        row[2 + odd] = bti;
      }
      row[4 + odd] = cs * cr - sn * ci;    // Re(e^{+i Phi} Cc)
      row[6 + odd] = -(cs * ci + sn * cr); // -Im(e^{+i Phi} Cc)
      if (lane_sum) {
        float E = cr * br - ci * bi;
        for (int o = p.N / 2; o >= 1; o >>= 1) E += __shfl_xor_sync(gmask, E, o);
        if (n == 0) {
          const int64_t tb = int64_t(b) * p.L + t;
          const float lt = load_in<Tin>(lam, tb);
          const float mu = (t + 1 < p.L) ? 1.f - load_in<Tin>(lam, tb + 1) : 0.f;
          float4* a = reinterpret_cast<float4*>(p.aux) + 2 * tb;
          a[0] = make_float4(lt, lt, mu, mu);
          a[1] = make_float4(E, E, 0.f, 0.f);
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
      const float lt = load_in<Tin>(lam, tb);
      const float mu = (t + 1 < p.L) ? 1.f - load_in<Tin>(lam, tb + 1) : 0.f;
      float4* a = reinterpret_cast<float4*>(p.aux) + 2 * tb;
      a[0] = make_float4(lt, lt, mu, mu);
      a[1] = make_float4(E, E, 0.f, 0.f);
    }
  }
}

// ------------------------------------------------------------------------- scan kernel
struct ScanParams {
  CUtensorMap tm_x;    // (D, L, B) input dtype, box (DT, T_SUB + 1, 1)
  CUtensorMap tm_dt;   // (D, L, B) input dtype, box (DT, T_SUB + 2, 1)
  CUtensorMap tm_tab;  // (TABW N, L, B) f32, box (TABW N, T_SUB + 1, 1)
  CUtensorMap tm_aux;  // (8, L, B) f32, box (8, T_SUB + 1, 1)
  CUtensorMap tm_rot;  // (2N, 4S, B) f32, box (2N, 4, 1)
  const float* A;
  const float* Dskip;
  float* y;
  const void* x;
  const void* dt;
  const void* Bc;
  const void* lam;
  const float* h0;      // (B, D, N, 2) initial state or null
  float* h_last;        // (B, D, N, 2) final state or null
  const void* x_prev;   // (B, D) step -1 input (trapezoid halo) or null
  const void* Bc_prev;  // (B, N, 2) step -1 Bc (trapezoid halo) or null
  Workspace ws;
  int B, L, D, N, S;
  int n_dtiles, n_tiles, TC, n_chunks, n_units;
  int carry;
  int y_vec2;           // y is 8-byte aligned: store channel pairs as float2
  int silent_chunk;
  long long poll_limit;
  float4* ckpt;         // checkpoint variant: (B, S8, D, N/2) state pairs before every 8-step segment
  int S8;               // ceil(L / 8)
  // scan_kernel, a part of the states of a larger problem: N states n_off .. n_off + N - 1 of
  // n_full (the row length of A, h0 and h_last)
  int n_full, n_off;
};

__device__ __forceinline__ bool flag_ready(uint32_t f, uint32_t epoch, uint32_t need) {
  return (f >> 2) == epoch && (f & 3u) >= need;
}

__device__ __forceinline__ void record_error(uint32_t* hdr, uint32_t code, int unit, int pred) {
  if (atomicOr(&hdr[H_ERROR], code) == 0u) {
    hdr[H_ERR_UNIT] = uint32_t(unit);
    hdr[H_ERR_PRED] = uint32_t(pred);
  }
}

// ------------------------------------------------------------------------- bounds checks
// Builds with CSSCAN_BOUNDS_CHECK defined range-check the kernels' shared-memory and global
// indices: CSSCAN_BCKO(hdr, i, off, n, site) checks off + i against [0, n); outside it, the first
// failure records ERR_BOUNDS with the site number and the offending index in the workspace header,
// and the index is replaced by -off so that the access lands on the array's first element. The
// kernel then runs on to its end (no trap, and no early exit that would leave a barrier or a
// successor waiting); the host reads the error as CSSCAN_ERR_BOUNDS. Other builds compile the
// index unchanged.
#ifdef CSSCAN_BOUNDS_CHECK
static __device__ __noinline__ void bounds_fail(uint32_t* hdr, int site, long long j) {
  record_error(hdr, ERR_BOUNDS, site, int(j < -2147483647LL ? -2147483647LL : (j > 2147483647LL ? 2147483647LL : j)));
}
template <typename I>
__device__ __forceinline__ I bck_off(uint32_t* hdr, I i, long long off, long long n, int site) {
  const long long j = (long long)i + off;
  if (j < 0 || j >= n) {
    bounds_fail(hdr, site, j);
    return I(-off);
  }
  return i;
}
#define CSSCAN_BCKO(hdr, i, off, n, site) ::csscan::bck_off((hdr), (i), (long long)(off), (long long)(n), (site))
#else
#define CSSCAN_BCKO(hdr, i, off, n, site) (i)
#endif
#define CSSCAN_BCK(hdr, i, n, site) CSSCAN_BCKO(hdr, i, 0, n, site)

__device__ __forceinline__ bool wait_bar_bounded(uint64_t* bar, uint32_t parity) {
  for (long long i = 0; i < MBAR_WAIT_LIMIT; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 16) __nanosleep(64);
  }
  return false;
}

// Two adjacent channels of one staged row, widened to float32 and broadcast to both halves of
// a pair: returns (kept, kept) and (other, other), where a lane with swap = 1 keeps the second
// channel. The bf16 case widens with byte permutes whose selectors the lane holds in registers
// (two equivalent selectors per half, so that the two copies are not merged into one value plus
// a register copy).
struct Selectors {
  uint32_t k1, k2, o1, o2;   // kept channel (twice), other channel (twice)
};
__device__ __forceinline__ Selectors make_selectors(int swap) {
  // 0x1044 / 0x1055: the low 16 bits moved to the top (bytes 4, 5 are the zero operand);
  // 0x3244 / 0x3255: the high 16 bits in place
  return swap ? Selectors{0x3244u, 0x3255u, 0x1044u, 0x1055u} : Selectors{0x1044u, 0x1055u, 0x3244u, 0x3255u};
}
__device__ __forceinline__ uint32_t prmt(uint32_t v, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(v), "r"(sel));
  return d;
}
template <typename Tin> struct PairLoad;
template <> struct PairLoad<float> {
  static __device__ __forceinline__ void bcast(const float* p, const Selectors& sl, int swap, float2& a, float2& b) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    const float k = swap ? v.y : v.x, o = swap ? v.x : v.y;
    a = f2(k, k);
    b = f2(o, o);
  }
};
template <> struct PairLoad<uint16_t> {
  static __device__ __forceinline__ void bcast(const uint16_t* p, const Selectors& sl, int, float2& a, float2& b) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    a = f2(__uint_as_float(prmt(v, sl.k1)), __uint_as_float(prmt(v, sl.k2)));
    b = f2(__uint_as_float(prmt(v, sl.o1)), __uint_as_float(prmt(v, sl.o2)));
  }
};

// CARRY (== p.carry) selects what is compiled in: CARRY_NONE (one chunk per row), CARRY_SERIAL
// (each chunk waits for its predecessor's final state) or CARRY_DECOUPLED (aggregate pass,
// then look-back); the lighter variants keep no registers for the heavier ones.
// CKPT = true is the checkpoint variant for the backward pass: no y, and the true state
// h_t = e^{i Phi_t} (k_{t+1} - p_{t+1} Bt_t) after every 8th step stored to p.ckpt.
// Zero-order-hold update of one state pair of one channel in the rotating frame:
// k <- r k + w (E beta + delta) conj(z) / |z|^2 (plus the tau terms), all in base-2 units.
// v = dt A log2 e (both states), r = 2^v, w = dt x broadcast; (dr, di) delta, tq theta,
// ntq -theta, t2 theta^2 + tau, (fr, fi) tau ln 2 beta'.
__device__ __forceinline__ void zoh_update(float2& kr, float2& ki, float2 r, float2 v, float2 w, float2 btr,
                                           float2 bti, float2 dr, float2 di, float2 tq, float2 ntq, float2 t2,
                                           float2 fr, float2 fi) {
  float2 pe = fma2(v, f2(ZOH_C4, ZOH_C4), f2(ZOH_C3, ZOH_C3));
  pe = fma2(v, pe, f2(ZOH_C2, ZOH_C2));
  pe = fma2(v, pe, f2(ZOH_C1, ZOH_C1));
  pe = mul2(v, pe);
  const float2 rm1 = fma2(r, f2(1.f, 1.f), f2(-1.f, -1.f));
  const float2 E = f2(fabsf(v.x) < ZOH_V_POLY ? pe.x : rm1.x, fabsf(v.y) < ZOH_V_POLY ? pe.y : rm1.y);
  const float2 nr = fma2(E, btr, dr), ni = fma2(E, bti, di);
  const float2 z2 = fma2(v, v, t2);
  const float2 sw = mul2(w, f2(rcp_approx(z2.x), rcp_approx(z2.y)));
  const float2 mr = fma2(ni, tq, fma2(nr, v, fr));
  const float2 mi = fma2(ni, v, fma2(nr, ntq, fi));
  kr = fma2(r, kr, mul2(sw, mr));
  ki = fma2(r, ki, mul2(sw, mi));
}

// ACC = true: a later part of a state split (see ScanParams::n_off): this part's Re(sum_n Cc h)
// is added to y, which an earlier part wrote together with the Dskip term.
template <int N, typename Tin, int MODE, int CARRY, bool CKPT = false, bool ACC = false>
__global__ void __launch_bounds__(THREADS, 2) scan_kernel(const __grid_constant__ ScanParams p) {
  using TL = Tile<N>;
  using SG = Stage<N, Tin, MODE>;
  constexpr int NS = TL::NS, NG = TL::NG, NPAIR = TL::NPAIR, CPW = TL::CPW, DT = TL::DT;
  constexpr int NST = SG::NST;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  // stage buffers start on a 128-byte boundary (the host requests 128 spare bytes)
  unsigned char* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
  __shared__ int s_ctl[8];
  __shared__ int s_abort;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int g = lane % NG;                              // state group of this thread
  const int cl = (tid >> 5) * CPW + (lane / NG) * CH;   // first of this thread's two channels
  const int n0 = g * NS;                                // first state of this thread
  // Lanes g and g^1 split a channel pair's states; the odd one keeps (outputs) the second
  // channel, and every per-channel pair of this thread is ordered (kept, other).
  const int swp = NG > 1 ? (g & 1) : 0;
  const Selectors sel = make_selectors(swp);
  uint32_t* hdr = p.ws.hdr;

  if (tid == 0) {
    s_ctl[0] = int(atomicAdd(&hdr[H_TICKET], 1u));
    s_ctl[1] = int(ld_relaxed_gpu(&hdr[H_EPOCH]) & 0x3FFFFFFFu);
    s_abort = 0;
    for (int i = 0; i < NST; ++i) mbar_init(&full_bar[i], 1);
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
  const int d = d0 + cl;                 // channels d and d + 1 (D is even, so both or neither exist)
  const bool dvalid = d < p.D;
  auto chan = [&](int ch) { return d + (ch ^ swp); };   // channel of this thread's pair slot ch
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
      if (tid == 0) s_ctl[2] = flag_ready(ld_acquire_gpu(&p.ws.flags[(c - 1) * p.n_tiles + j]), epoch, ST_INCL);
      __syncthreads();
      pass1 = !s_ctl[2];
    }
  }
  const int total_stages = n_sub * (pass1 ? 2 : 1);

  auto issue = [&](int gs) {
    const int slot = gs % NST;
    const int sub = s_begin + (gs % n_sub);
    unsigned char* base = smem + slot * SG::BYTES;
    mbar_arrive_expect_tx(&full_bar[slot], uint32_t(SG::TX_BYTES));
    tma_load_3d(base + SG::OFF_X, &p.tm_x, d0, sub * T_SUB, b, &full_bar[slot]);
    tma_load_3d(base + SG::OFF_DT, &p.tm_dt, d0, sub * T_SUB, b, &full_bar[slot]);
    tma_load_3d(base + SG::OFF_TAB, &p.tm_tab, 0, sub * T_SUB, b, &full_bar[slot]);
    if (MODE == 1) tma_load_3d(base + SG::OFF_AUX, &p.tm_aux, 0, sub * T_SUB, b, &full_bar[slot]);
    tma_load_3d(base + SG::OFF_ROT, &p.tm_rot, 0, 4 * sub, b, &full_bar[slot]);
  };
  if (tid == 0) {
    for (int gs = 0; gs < min(NST, total_stages); ++gs) issue(gs);
  }

  // ---- per-thread constants: log2(e) A for both channels, Dskip
  float2 Ap[CH][NPAIR];
#pragma unroll
  for (int ch = 0; ch < CH; ++ch)
#pragma unroll
    for (int q = 0; q < NPAIR; ++q)
      Ap[ch][q] = dvalid ? f2(p.A[int64_t(chan(ch)) * p.n_full + p.n_off + n0 + 2 * q] * LOG2E_F,
                              p.A[int64_t(chan(ch)) * p.n_full + p.n_off + n0 + 2 * q + 1] * LOG2E_F)
                         : f2(0.f, 0.f);
  const float2 Ds = (dvalid && !ACC) ? f2(p.Dskip[chan(0)], p.Dskip[chan(1)]) : f2(0.f, 0.f);

  // trapezoid halo: k at the chunk start is h_in + p_tc Bc_{tc-1}, p_tc = (1-lam_tc) dt_tc x_{tc-1}
  float2 halo_p = f2(0.f, 0.f);
  float2 hbr[NPAIR], hbi[NPAIR];
#pragma unroll
  for (int q = 0; q < NPAIR; ++q) { hbr[q] = f2(0.f, 0.f); hbi[q] = f2(0.f, 0.f); }
  if (MODE == 1 && (tc > 0 || p.x_prev != nullptr)) {
    const Tin* xin = static_cast<const Tin*>(p.x);
    const Tin* dtin = static_cast<const Tin*>(p.dt);
    const Tin* lamin = static_cast<const Tin*>(p.lam);
    const Tin* bsrc;
    float2 xprev = f2(0.f, 0.f);
    if (tc > 0) {
      if (dvalid) xprev = f2(load_in<Tin>(xin, (b * L + tc - 1) * D + chan(0)), load_in<Tin>(xin, (b * L + tc - 1) * D + chan(1)));
      bsrc = static_cast<const Tin*>(p.Bc) + (b * L + tc - 1) * p.N * 2;
    } else {
      const Tin* xp = static_cast<const Tin*>(p.x_prev);
      if (dvalid) xprev = f2(load_in<Tin>(xp, int64_t(b) * D + chan(0)), load_in<Tin>(xp, int64_t(b) * D + chan(1)));
      bsrc = static_cast<const Tin*>(p.Bc_prev) + int64_t(b) * p.N * 2;
    }
    const float2 dt_tc = dvalid ? f2(load_in<Tin>(dtin, (b * L + tc) * D + chan(0)), load_in<Tin>(dtin, (b * L + tc) * D + chan(1)))
                                : f2(0.f, 0.f);
    const float mu = 1.f - load_in<Tin>(lamin, b * L + tc);
    halo_p = f2(mu * dt_tc.x * xprev.x, mu * dt_tc.y * xprev.y);
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
      const int n = n0 + 2 * q;
      hbr[q] = f2(load_in<Tin>(bsrc, 2 * n), load_in<Tin>(bsrc, 2 * n + 2));
      hbi[q] = f2(load_in<Tin>(bsrc, 2 * n + 1), load_in<Tin>(bsrc, 2 * n + 3));
    }
  }

  float2 kr[CH][NPAIR], ki[CH][NPAIR];   // state pairs (re), (im) in the current frame
  float2 Rr[NPAIR], Ri[NPAIR];           // chunk rotation product (pass 1)
  float2 sdt_acc = f2(0.f, 0.f);         // sum of dt over the chunk, both channels (pass 1)
  int gstage = 0;
  bool aborted = false;

  // What a step needs from its scalars: the injection weight of each channel broadcast to a
  // pair (exp-Euler: dt x; trapezoid: lam dt x + pc), dt (aggregate pass), and for the output
  // x, pc and E.
  struct StepIn {
    float4 tb[2 * NPAIR];  // this step's table entries of the thread's states (Bt, Ct per pair)
    float2 w0, w1;         // injection weights (w_kept, w_kept), (w_other, w_other)
    float2 dv;             // (dt_kept, dt_other), for the aggregate pass
    float2 x, pc;          // (x_kept, x_other), (pc_kept, pc_other)
    float2 nk, no;         // trapezoid: the next step's dt, broadcast pairs (kept, other)
    float E;
  };
  // The output of a finished step: the NG lanes' partial sums of Re(Ct k) are combined, the
  // trapezoid correction and the D-skip added, and the lanes with g < 2 store the result.
  const bool store_one = NG > 1 && g < 2 && dvalid;
  auto finish_y = [&](float2 yp, const StepIn& sc, float* yrow, bool ok) {
    if (CKPT) return;
    if (NG == 1) {
      float o0 = fmaf(Ds.x, sc.x.x, fmaf(-sc.pc.x, sc.E, yp.x));
      float o1 = fmaf(Ds.y, sc.x.y, fmaf(-sc.pc.y, sc.E, yp.y));
      if (ACC && ok && dvalid) {   // reductions (nothing waits for them); parts run in stream order
        atomicAdd(yrow, o0);
        atomicAdd(yrow + 1, o1);
      } else if (ok && dvalid) {
        if (p.y_vec2) {
          __stcs(reinterpret_cast<float2*>(yrow), f2(o0, o1));
        } else {
          __stcs(yrow, o0);
          __stcs(yrow + 1, o1);
        }
      }
    } else {
      // lanes g and g^1 trade the partial of the channel they do not keep, then the group sums
      float keep = yp.x + __shfl_xor_sync(0xffffffffu, yp.y, 1);
#pragma unroll
      for (int o = 2; o < NG; o <<= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
      const float o = fmaf(Ds.x, sc.x.x, fmaf(-sc.pc.x, sc.E, keep));
      if (ok && store_one) {
        if (ACC) atomicAdd(yrow + g, o);   // a reduction: nothing waits for it
        else __stcs(yrow + g, o);
      }
    }
  };

  // One pass over the chunk's sub-chunks. WITH_Y: write y; otherwise accumulate the
  // aggregate's sum of dt and rotation. The time loop is software-pipelined: step t+1's
  // scalars and decays are computed during step t, and step t's output is reduced and
  // stored during step t+1; two steps per iteration with the register sets swapped, so no
  // value is copied at the loop edge.
  auto run_pass = [&](auto with_y_tag) {
    constexpr bool WITH_Y = decltype(with_y_tag)::value;
    for (int i = 0; i < n_sub; ++i, ++gstage) {
      const int slot = gstage % NST;
      if (!wait_bar_bounded(&full_bar[slot], uint32_t(gstage / NST) & 1u)) s_abort = 1;
      const unsigned char* base = smem + slot * SG::BYTES;
      const Tin* sx = reinterpret_cast<const Tin*>(base + SG::OFF_X) + cl;
      const Tin* sdtp = reinterpret_cast<const Tin*>(base + SG::OFF_DT) + cl;
      constexpr int PF4 = SG::TABW / 2;   // table float4 per state pair and step
      const float4* stab = reinterpret_cast<const float4*>(base + SG::OFF_TAB) + g * NPAIR * PF4;
      const float4* saux = reinterpret_cast<const float4*>(base + SG::OFF_AUX);
      const float4* srot = reinterpret_cast<const float4*>(base + SG::OFF_ROT);
      const int t_sub0 = (s_begin + i) * T_SUB;
      const int nt = min(T_SUB, te - t_sub0);
      // local index of the chunk's last step, where the trapezoid look-ahead p_{t+1} is left
      // to the next chunk's halo (-1 when that step lies in a later sub-chunk)
      const int t_last = te - 1 - t_sub0 < T_SUB ? te - 1 - t_sub0 : -1;
      float* yrow = p.y + (b * L + t_sub0) * D + d;

      // Table entries and scalars of step tt (rows tt of x, aux and the table; row tt of dt, or,
      // in the trapezoid mode, the pairs dd0/dd1 carried from the previous step, and row tt + 1
      // of dt; all staged), and the decays' dt broadcast pairs dd0/dd1.
      auto load_step = [&](int tt, StepIn& s, float2& dd0, float2& dd1, bool dd_given) {
        const float4* trow = stab + tt * (N / 2) * PF4;
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          s.tb[2 * q] = trow[q * PF4];
          s.tb[2 * q + 1] = trow[q * PF4 + 1];
        }
        float2 xx0, xx1;
        PairLoad<Tin>::bcast(sx + tt * DT, sel, swp, xx0, xx1);
        if (!dd_given) PairLoad<Tin>::bcast(sdtp + tt * DT, sel, swp, dd0, dd1);
        s.x = f2(xx0.x, xx1.x);
        s.dv = f2(dd0.x, dd1.x);
        if (MODE != 1) {
          s.w0 = mul2(dd0, xx0);
          s.w1 = mul2(dd1, xx1);
          s.pc = f2(0.f, 0.f);
          s.E = 0.f;
        } else {
          PairLoad<Tin>::bcast(sdtp + (tt + 1) * DT, sel, swp, s.nk, s.no);
          const float4 a = saux[2 * tt];
          const float4 e = saux[2 * tt + 1];
          const float2 lam2 = f2(a.x, a.y), mu2 = f2(a.z, a.w);
          // m = (1 - lam_{t+1}) dt_{t+1}; w = (lam_t dt_t + m) x_t; pc = m x_t
          float2 m0 = mul2(mu2, s.nk), m1 = mul2(mu2, s.no);
          if (tt == t_last) { m0 = f2(0.f, 0.f); m1 = f2(0.f, 0.f); }
          s.w0 = mul2(fma2(lam2, dd0, m0), xx0);
          s.w1 = mul2(fma2(lam2, dd1, m1), xx1);
          s.pc = f2(m0.x * xx0.x, m1.x * xx1.x);
          s.E = e.x;
        }
      };

      float2 ypend = f2(0.f, 0.f);
      // One step with this step's scalars `cur` and decays `rc`; loads step tt + 1's into
      // `nxt` / `rn` and finishes step tt - 1's output, whose scalars `nxt` held.
      auto step = [&](int tt, const StepIn& cur, const float2 (&rc)[CH][NPAIR], StepIn& nxt,
                      float2 (&rn)[CH][NPAIR]) {
        if (WITH_Y) {
          finish_y(ypend, nxt, yrow, tt > 0);
          if (tt > 0) yrow += D;
        } else {
          sdt_acc = f2(sdt_acc.x + cur.dv.x, sdt_acc.y + cur.dv.y);
        }
        float2 dd0 = cur.nk, dd1 = cur.no;
        load_step(tt + 1, nxt, dd0, dd1, MODE == 1);
        float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
        [[maybe_unused]] const float4* zrow = stab + tt * (N / 2) * PF4;   // zero-order hold: this step's row
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          rn[0][q] = ex2_pair(mul2(dd0, Ap[0][q]));
          rn[1][q] = ex2_pair(mul2(dd1, Ap[1][q]));
          const float4 bt = cur.tb[2 * q];
          const float2 btr = f2(bt.x, bt.y), bti = f2(bt.z, bt.w);
          if constexpr (MODE == 2) {
            const float4 dz = zrow[q * PF4 + 2], tz = zrow[q * PF4 + 3];
            const float2 dr = f2(dz.x, dz.y), di = f2(dz.z, dz.w);
            const float2 tq = f2(tz.x, tz.y), ntq = f2(-tz.x, -tz.y), t2 = f2(tz.z, tz.w);
            const float2 fr = mul2(f2(ZOH_TAU_LN2, ZOH_TAU_LN2), btr), fi = mul2(f2(ZOH_TAU_LN2, ZOH_TAU_LN2), bti);
            // this step's dt broadcast pairs give v = dt A log2 e, the decay's argument
            const float2 v0 = mul2(f2(cur.dv.x, cur.dv.x), Ap[0][q]);
            const float2 v1 = mul2(f2(cur.dv.y, cur.dv.y), Ap[1][q]);
            zoh_update(kr[0][q], ki[0][q], rc[0][q], v0, cur.w0, btr, bti, dr, di, tq, ntq, t2, fr, fi);
            zoh_update(kr[1][q], ki[1][q], rc[1][q], v1, cur.w1, btr, bti, dr, di, tq, ntq, t2, fr, fi);
          } else {
            kr[0][q] = fma2(rc[0][q], kr[0][q], mul2(cur.w0, btr));
            ki[0][q] = fma2(rc[0][q], ki[0][q], mul2(cur.w0, bti));
            kr[1][q] = fma2(rc[1][q], kr[1][q], mul2(cur.w1, btr));
            ki[1][q] = fma2(rc[1][q], ki[1][q], mul2(cur.w1, bti));
          }
          if (WITH_Y && !CKPT) {
            const float4 ct = cur.tb[2 * q + 1];
            const float2 ctr = f2(ct.x, ct.y), cti = f2(ct.z, ct.w);
            acc0 = fma2(cti, ki[0][q], fma2(ctr, kr[0][q], acc0));
            acc1 = fma2(cti, ki[1][q], fma2(ctr, kr[1][q], acc1));
          }
        }
        if (WITH_Y && !CKPT) ypend = f2(acc0.x + acc0.y, acc1.x + acc1.y);
      };

      StepIn sa, sb;
      float2 ra[CH][NPAIR], rb[CH][NPAIR];
      {
        float2 dd0, dd1;
        load_step(0, sa, dd0, dd1, false);
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          ra[0][q] = ex2_pair(mul2(dd0, Ap[0][q]));
          ra[1][q] = ex2_pair(mul2(dd1, Ap[1][q]));
        }
        sb = sa;
      }
      // Checkpoint variant: after local step j = 8 r + 7 the state is k_{t+1} = g_t + p_{t+1} Bt_t
      // in the frame of row r of the rotation table; h_t = e^{i Phi_t} (k - p Bt) is stored as
      // the state before the segment that starts at t + 1.
      auto store_ckpt = [&](int j, const StepIn& sc) {
        const int t1 = t_sub0 + j + 1;
        if (t1 >= p.L || !dvalid) return;
        const float4* rrow = srot + (j >> 3) * (N / 2);
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          const float4 rr = rrow[n0 / 2 + q];
          const float2 cc = f2(rr.x, rr.z), ss = f2(rr.y, rr.w), nss = f2(-rr.y, -rr.w);
          const float4 bt = sc.tb[2 * q];
          const float2 btr = f2(bt.x, bt.y), bti = f2(bt.z, bt.w);
#pragma unroll
          for (int ch = 0; ch < CH; ++ch) {
            const float pcv = ch ? sc.pc.y : sc.pc.x;
            const float2 npc = f2(-pcv, -pcv);
            const float2 ur = fma2(npc, btr, kr[ch][q]), ui = fma2(npc, bti, ki[ch][q]);
            const float2 hr = fma2(cc, ur, mul2(nss, ui)), hi = fma2(cc, ui, mul2(ss, ur));
            p.ckpt[((b * int64_t(p.S8) + t1 / 8) * D + chan(ch)) * (N / 2) + n0 / 2 + q] =
                make_float4(hr.x, hi.x, hr.y, hi.y);
          }
        }
      };
      int tt = 0;
      // 8 steps per trip: the shared-memory offsets of a trip are immediates and the loop
      // bookkeeping is paid once per 8 steps (measured 6 % faster than 2 steps per trip)
#pragma unroll 4
      for (; tt + 1 < nt; tt += 2) {
        step(tt, sa, ra, sb, rb);
        step(tt + 1, sb, rb, sa, ra);
        if (CKPT && WITH_Y && ((tt + 2) & 7) == 0) store_ckpt(tt + 1, sb);
      }
      // yrow now points at the row of the last step taken, whose output is still pending
      if (tt < nt) {
        step(tt, sa, ra, sb, rb);
        if (CKPT && WITH_Y && ((tt + 1) & 7) == 0) store_ckpt(tt, sa);
        if (WITH_Y) finish_y(ypend, sa, yrow, true);
      } else if (WITH_Y) {
        finish_y(ypend, sb, yrow, true);
      }
      // frame reset: rotate the state by e^{i Phi_last} of this sub-chunk
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) {
        const float4 rr = srot[3 * (N / 2) + n0 / 2 + q];
        const float2 cc = f2(rr.x, rr.z), ss = f2(rr.y, rr.w), nss = f2(-rr.y, -rr.w);
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) {
          const float2 nr = fma2(cc, kr[ch][q], mul2(nss, ki[ch][q]));
          const float2 ni = fma2(cc, ki[ch][q], mul2(ss, kr[ch][q]));
          kr[ch][q] = nr;
          ki[ch][q] = ni;
        }
        if (!WITH_Y) {
          const float2 r2 = fma2(cc, Rr[q], mul2(nss, Ri[q]));
          const float2 i2 = fma2(cc, Ri[q], mul2(ss, Rr[q]));
          Rr[q] = r2;
          Ri[q] = i2;
        }
      }
      __syncthreads();
      if (s_abort) { aborted = true; return; }
      if (tid == 0 && gstage + NST < total_stages) issue(gstage + NST);
    }
  };

  // ---- per-state helpers on the workspace records (float2 per state, states contiguous)
  auto rec_of = [&](float2* base, int u, int ch) { return base + (int64_t(u) * DT + cl + (ch ^ swp)) * p.N + n0; };
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
    if (tid == 0 && !silent) st_release_gpu(&p.ws.flags[unit], (epoch << 2) | status);
  };

  float2 hr[CH][NPAIR], hi[CH][NPAIR];   // carry-in h_{tc-1}
#pragma unroll
  for (int ch = 0; ch < CH; ++ch)
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) { hr[ch][q] = f2(0.f, 0.f); hi[ch][q] = f2(0.f, 0.f); }
  bool incl_published = false;
  const bool has_h0 = (p.h0 != nullptr) && dvalid;
  auto h0rec = [&](int ch) {
    return reinterpret_cast<const float2*>(p.h0) + (int64_t(b) * p.D + chan(ch)) * p.n_full + p.n_off + n0;
  };

  if (CARRY == CARRY_DECOUPLED && pass1) {
    // ---- pass 1: aggregate from a zero carry-in
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        const float hp = ch ? halo_p.y : halo_p.x;
        kr[ch][q] = mul2(f2(hp, hp), hbr[q]);
        ki[ch][q] = mul2(f2(hp, hp), hbi[q]);
      }
      Rr[q] = f2(1.f, 1.f);
      Ri[q] = f2(0.f, 0.f);
    }
    run_pass(std::false_type{});
    if (!aborted) {
      if (!silent) {
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) store_states(rec_of(p.ws.agg, unit, ch), kr[ch], ki[ch]);
        if (g == 0) __stcg(reinterpret_cast<float2*>(p.ws.sdt + int64_t(unit) * DT + cl), sdt_acc);
        if (cl == 0) store_states(p.ws.crot + int64_t(unit) * p.N + n0, Rr, Ri);
      }
      publish(ST_AGG);

      // ---- decoupled look-back over windows of 32 predecessors
      float2 Sd = f2(0.f, 0.f);
      float2 Qr[NPAIR], Qi[NPAIR];
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) { Qr[q] = f2(1.f, 1.f); Qi[q] = f2(0.f, 0.f); }
      // h_in += exp(A Sd) Q * rec   (the accumulated multiplier of the chunks seen so far)
      auto accumulate = [&](int u2, bool is_h0, bool is_incl) {
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) {
          const float2* rec = is_h0 ? h0rec(ch) : rec_of(is_incl ? p.ws.inc : p.ws.agg, u2, ch);
          const float sd = ch ? Sd.y : Sd.x;
#pragma unroll
          for (int q = 0; q < NPAIR; ++q) {
            const float4 v = is_h0 ? reinterpret_cast<const float4*>(rec)[q] : __ldcg(reinterpret_cast<const float4*>(rec) + q);
            const float2 ur = f2(v.x, v.z), ui = f2(v.y, v.w);
            const float2 e = ex2_pair(mul2(f2(sd, sd), Ap[ch][q]));
            const float2 mr = mul2(e, Qr[q]), mi = mul2(e, Qi[q]);
            hr[ch][q] = fma2(mr, ur, fma2(f2(-mi.x, -mi.y), ui, hr[ch][q]));
            hi[ch][q] = fma2(mr, ui, fma2(mi, ur, hi[ch][q]));
          }
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
              const uint32_t f = ld_acquire_gpu(&p.ws.flags[unit_of(cp)]);
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
          accumulate(u2, false, false);
          const float2 sd2 = __ldcg(reinterpret_cast<const float2*>(p.ws.sdt + int64_t(u2) * DT + cl));
          Sd = swp ? f2(Sd.x + sd2.y, Sd.y + sd2.x) : f2(Sd.x + sd2.x, Sd.y + sd2.y);
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
            if (has_h0) accumulate(0, true, false);
          } else {
            accumulate(unit_of(cp), false, true);
          }
          break;
        }
        if (tout) break;
        pred -= 32;
      }
      // ---- publish this chunk's final state: h_end = P h_in + U, P = exp(A sum dt) R
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        const float sd = ch ? sdt_acc.y : sdt_acc.x;
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          const float2 e = ex2_pair(mul2(f2(sd, sd), Ap[ch][q]));
          const float2 pr = mul2(e, Rr[q]), pi = mul2(e, Ri[q]);
          const float2 er = fma2(pr, hr[ch][q], fma2(f2(-pi.x, -pi.y), hi[ch][q], kr[ch][q]));
          const float2 ei = fma2(pr, hi[ch][q], fma2(pi, hr[ch][q], ki[ch][q]));
          kr[ch][q] = er;   // reuse as scratch for the store
          ki[ch][q] = ei;
        }
        if (!silent) store_states(rec_of(p.ws.inc, unit, ch), kr[ch], ki[ch]);
      }
      publish(ST_INCL);
      incl_published = true;
    }
  } else if (CARRY != CARRY_NONE && c > 0) {
    // ---- serial carry, or a decoupled chunk whose predecessor had already published its
    // final state when this block started: wait for (or take) that final state
    if (tid == 0) {
      const uint32_t* fp = &p.ws.flags[unit_of(c - 1)];
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
    if (!s_ctl[5]) {
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) load_states(rec_of(p.ws.inc, unit_of(c - 1), ch), hr[ch], hi[ch]);
    }
  } else if (has_h0) {
#pragma unroll
    for (int ch = 0; ch < CH; ++ch) {
      const float4* r4 = reinterpret_cast<const float4*>(h0rec(ch));
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) {
        const float4 v = r4[q];
        hr[ch][q] = f2(v.x, v.z);
        hi[ch][q] = f2(v.y, v.w);
      }
    }
  }

  if (!aborted) {
    // ---- pass 2: from the carry-in, writing y
#pragma unroll
    for (int ch = 0; ch < CH; ++ch) {
      const float hp = ch ? halo_p.y : halo_p.x;
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) {
        kr[ch][q] = fma2(f2(hp, hp), hbr[q], hr[ch][q]);
        ki[ch][q] = fma2(f2(hp, hp), hbi[q], hi[ch][q]);
      }
    }
    run_pass(std::true_type{});
  }
  if (!aborted) {
    if (CARRY != CARRY_NONE && !incl_published) {
      if (!silent) {
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) store_states(rec_of(p.ws.inc, unit, ch), kr[ch], ki[ch]);
      }
      publish(ST_INCL);
    }
    if (c == p.n_chunks - 1 && p.h_last != nullptr && dvalid) {
#pragma unroll
      for (int ch = 0; ch < CH; ++ch)
        store_states(reinterpret_cast<float2*>(p.h_last) + (int64_t(b) * p.D + chan(ch)) * p.n_full + p.n_off + n0,
                     kr[ch], ki[ch]);
    }
  } else {
    // a tile copy never arrived: report, drain what is still in flight (bounded), leave
    if (tid == 0) {
      record_error(hdr, ERR_PIPELINE, unit, -1);
      for (int gs = gstage; gs < min(gstage + NST, total_stages); ++gs)
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
