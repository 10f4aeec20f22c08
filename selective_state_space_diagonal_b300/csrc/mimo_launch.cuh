// mimo_launch.cuh -- host side of csscan_forward_mimo and csscan_backward_mimo, included by the
// per-dtype units mimo_f32.cu / mimo_bf16.cu. The forward has two kernel families:
//   mscan_kernel (mscan_kernels.cuh): staged tile copies, chunk carries as the forward scan;
//     taken for N = 8, 16, 32 with P N <= 128 when the inputs meet the tile-copy rules (16-byte
//     aligned x, dt and y, the (b, t) rows of x and dt whole multiples of 16 bytes);
//   the per-state kernels of mimo_kernels.cuh for every other supported shape.
#pragma once

#include <algorithm>
#include <cstring>

#include "forward_launch.cuh"
#include "mgrad_kernels.cuh"
#include "mimo_kernels.cuh"
#include "mscan_kernels.cuh"

namespace csscan_host {
namespace mimo_detail {

using namespace csscan;

// ----------------------------------------------------------------------------- mscan family
// States per thread: about 8 channel-state elements per thread and step (at least 2 states, at
// most 16 lanes per head). Measured on B300 on the 640-head, P = 4, N = 16 trapezoid shape: 2
// states per thread (8 lanes per head, twice the warps) 2.39 ms, 4 states 2.49 ms.
template <int N, int P>
constexpr int mscan_states() {
  int ns = 8 / P;
  if (ns > N) ns = N;
  if (ns < 2) ns = 2;
  if (N / ns > 16) ns = N / 16;
  return ns;
}

template <int N, int NS, int P, typename Tin, int MODE>
struct MScan {
  using TL = MTile<N, NS, P>;
  using SG = MStage<N, NS, P, Tin, MODE>;
  static constexpr KernelShape shape() { return KernelShape{TL::DH, SG::SMEM, 2 * P * 2 * N, MODE == 1 ? TL::AUXW : 0}; }
  static int occ(int carry, int dev, int* out) {
    if (carry == CARRY_SERIAL) return occupancy_of(mscan_kernel<N, NS, P, Tin, MODE, CARRY_SERIAL>, dev, SG::SMEM, out);
    if (carry == CARRY_DECOUPLED)
      return occupancy_of(mscan_kernel<N, NS, P, Tin, MODE, CARRY_DECOUPLED>, dev, SG::SMEM, out);
    return occupancy_of(mscan_kernel<N, NS, P, Tin, MODE, CARRY_NONE>, dev, SG::SMEM, out);
  }
  static int launch(const MimoArgs& a, cudaStream_t st) {
    int dev = 0;
    CSSCAN_CUDA(cudaGetDevice(&dev));
    // the planner sees the heads as the channels of a forward scan
    Args fa;
    std::memset(&fa, 0, sizeof(fa));
    fa.B = a.B;
    fa.L = a.L;
    fa.D = a.H;
    fa.N = N;
    fa.mode = a.mode;
    fa.dtype = a.dtype;
    const csscan_options_t o = default_options();
    Plan pl;
    int rc = make_plan(fa, o, dev, shape(), &occ, &pl);
    if (rc != CSSCAN_OK) return rc;
    WsEntry ws;
    rc = get_workspace(dev, st, size_t(pl.n_units), pl.rest_bytes, &ws);
    if (rc != CSSCAN_OK) return rc;
    char* base = static_cast<char*>(ws.base);
    char* rest = ws_rest(ws);
    const int64_t S16 = (a.L + M_SUB - 1) / M_SUB;   // the planner's rotation region holds (B, S16, N, 2)

    MTableParams tp;
    tp.Bm = a.Bm;
    tp.Cm = a.Cm;
    tp.theta = a.theta;
    tp.lam = a.lam;
    tp.tab = reinterpret_cast<float*>(rest + pl.o_tab);
    tp.aux = MODE == 1 ? reinterpret_cast<float*>(rest + pl.o_aux) : nullptr;
    tp.rot = reinterpret_cast<float*>(rest + pl.o_rot);
    tp.B = int(a.B);
    tp.L = int(a.L);
    tp.N = N;
    tp.P = P;
    tp.S = int(S16);
    tp.ng = TL::NG;
    tp.auxw = TL::AUXW;
    tp.hdr = reinterpret_cast<uint32_t*>(base);

    MScanParams mp;
    std::memset(&mp, 0, sizeof(mp));
    const CUtensorMapDataType tin = sizeof(Tin) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t s_in = sizeof(Tin);
    const uint64_t B = uint64_t(a.B), L = uint64_t(a.L), H = uint64_t(a.H), HP = H * P, S = uint64_t(S16);
    const uint64_t W = 2 * N, PL = 2 * P;
    const uint64_t tdims[4] = {W, PL, L, B};
    const uint64_t tstrides[3] = {W * 4, PL * W * 4, L * PL * W * 4};
    const uint32_t tbox[4] = {uint32_t(W), uint32_t(PL), uint32_t(SG::TAB_ROWS), 1};
    bool ok = map3(&mp.tm_x, tin, a.x, HP, L, B, HP * s_in, L * HP * s_in, TL::DH * P, SG::X_ROWS, 1) &&
              map3(&mp.tm_dt, tin, a.delta, H, L, B, H * s_in, L * H * s_in, TL::DH, SG::DT_ROWS, 1) &&
              make_map(&mp.tm_tab, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.tab, 4, tdims, tstrides, tbox) &&
              map3(&mp.tm_rot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.rot, W, S, B, W * 4, S * W * 4, uint32_t(W), 1, 1);
    if (ok && MODE == 1)
      ok = map3(&mp.tm_aux, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.aux, TL::AUXW, L, B, TL::AUXW * 4, L * TL::AUXW * 4,
                TL::AUXW, SG::AUX_ROWS, 1);
    if (!ok) {
      set_last_error("cuTensorMapEncodeTiled failed or unavailable");
      return CSSCAN_ERR_CUDA;
    }
    mp.A = a.A;
    mp.Dskip = a.Dskip;
    mp.y = a.y;
    mp.ws.hdr = reinterpret_cast<uint32_t*>(base);
    mp.ws.flags = reinterpret_cast<uint32_t*>(base + HDR_BYTES);
    mp.ws.inc = pl.carry != CARRY_NONE ? reinterpret_cast<float2*>(rest + pl.o_inc) : nullptr;
    mp.ws.agg = pl.carry == CARRY_DECOUPLED ? reinterpret_cast<float2*>(rest + pl.o_agg) : nullptr;
    mp.ws.sdt = pl.carry == CARRY_DECOUPLED ? reinterpret_cast<float*>(rest + pl.o_sdt) : nullptr;
    mp.ws.crot = pl.carry == CARRY_DECOUPLED ? reinterpret_cast<float2*>(rest + pl.o_crot) : nullptr;
    mp.B = int(a.B);
    mp.L = int(a.L);
    mp.H = int(a.H);
    mp.N = N;
    mp.n_htiles = pl.n_dtiles;
    mp.n_tiles = pl.n_tiles;
    mp.TC = pl.TC;
    mp.n_chunks = pl.n_chunks;
    mp.n_units = pl.n_units;
    mp.silent_chunk = o.silent_chunk;
    mp.poll_limit = o.poll_limit > 0 ? o.poll_limit : (int64_t(1) << 22);

    const int64_t table_threads = a.B * S16 * N;
    if (!grid_fits(table_threads)) return CSSCAN_ERR_UNSUPPORTED;
    mtable_kernel<Tin, MODE, P><<<unsigned((table_threads + 255) / 256), 256, 0, st>>>(tp);
    CSSCAN_CUDA(cudaGetLastError());
    const dim3 grid{unsigned(pl.n_units)}, block{unsigned(THREADS)};
    if (pl.carry == CARRY_NONE)
      mscan_kernel<N, NS, P, Tin, MODE, CARRY_NONE><<<grid, block, unsigned(pl.smem), st>>>(mp);
    else if (pl.carry == CARRY_SERIAL)
      mscan_kernel<N, NS, P, Tin, MODE, CARRY_SERIAL><<<grid, block, unsigned(pl.smem), st>>>(mp);
    else
      mscan_kernel<N, NS, P, Tin, MODE, CARRY_DECOUPLED><<<grid, block, unsigned(pl.smem), st>>>(mp);
    CSSCAN_CUDA(cudaGetLastError());
    return CSSCAN_OK;
  }
};

// Whether the staged kernel takes this problem (see the file comment).
inline bool mscan_takes(const MimoArgs& a) {
  const size_t s = a.dtype == CSSCAN_F32 ? 4 : 2;
  return (a.N == 8 || a.N == 16 || a.N == 32) && a.P * a.N <= 128 && (size_t(a.H * a.P) * s) % 16 == 0 &&
         (size_t(a.H) * s) % 16 == 0 && aligned(a.x, 16) && aligned(a.delta, 16) && aligned(a.y, 16);
}

// ----------------------------------------------------------------------------- per-state family
template <typename Tin, int MODE, int N, int P>
int launch_rows(const MimoArgs& a, cudaStream_t st) {
  int dev = 0, nsm = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  CSSCAN_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  // time chunks until there are SEQ_THREADS_PER_SM / P threads per SM (the recurrence is sequential
  // per thread, and a thread carries P channels' work)
  const int64_t G = mimo::GROUP;
  const int64_t S = (a.L + G - 1) / G;
  const int64_t rows = a.B * a.H * N;
  const int64_t target = int64_t(nsm) * SEQ_THREADS_PER_SM / P;
  int64_t C = std::min<int64_t>(S, std::max<int64_t>(1, (target + rows - 1) / rows));
  if (C > 65535) C = 65535;   // the output pass has one grid row per chunk
  const int64_t TC = (S + C - 1) / C * G;
  C = (a.L + TC - 1) / TC;
  const size_t rot_bytes = align_up(size_t(a.B * a.L * N) * sizeof(float2), 256);
  const size_t chunk_bytes = C > 1 ? size_t(a.B * C * a.H * N) * 2 * sizeof(float2) : 0;
  WsEntry ws;
  int rc = get_workspace(dev, st, 1, rot_bytes + chunk_bytes + rot_bytes, &ws);
  if (rc != CSSCAN_OK) return rc;
  char* rest = ws_rest(ws);
  mimo::Params p;
  p.x = a.x;
  p.dt = a.delta;
  p.Bm = a.Bm;
  p.Cm = a.Cm;
  p.lam = MODE == 1 ? a.lam : nullptr;
  p.A = a.A;
  p.Dskip = a.Dskip;
  p.y = a.y;
  p.phase = reinterpret_cast<const float2*>(rest + rot_bytes + chunk_bytes);
  p.rot = reinterpret_cast<const float2*>(rest);
  p.chunk = C > 1 ? reinterpret_cast<float2*>(rest + rot_bytes) : nullptr;
  p.B = int(a.B);
  p.L = int(a.L);
  p.H = int(a.H);
  p.N = N;
  p.P = P;
  p.TC = int(TC);
  p.C = int(C);
  const long long n_rot = (long long)a.B * a.L * N;
  const long long n_thr = (long long)a.B * C * a.H * N;
  if (!grid_fits(n_rot) || !grid_fits(n_thr)) return CSSCAN_ERR_UNSUPPORTED;
  const long long n_ph = (long long)a.B * ((a.L + G - 1) / G) * N;
  mimo::mimo_phase_kernel<Tin><<<unsigned((n_ph + 255) / 256), 256, 0, st>>>(
      a.theta, reinterpret_cast<float2*>(rest + rot_bytes + chunk_bytes), int(a.L), N, n_ph);
  CSSCAN_CUDA(cudaGetLastError());
  if (C > 1) {
    // the time-chunk pass reads e^{i theta} per step
    mimo::mimo_rot_kernel<Tin><<<unsigned((n_rot + 255) / 256), 256, 0, st>>>(a.theta, reinterpret_cast<float2*>(rest),
                                                                             n_rot);
    CSSCAN_CUDA(cudaGetLastError());
    mimo::mimo_chunk_kernel<Tin, MODE, P><<<unsigned((n_thr + 255) / 256), 256, 0, st>>>(p);
    CSSCAN_CUDA(cudaGetLastError());
    mimo::mimo_combine_kernel<<<unsigned((rows + 255) / 256), 256, 0, st>>>(p);
    CSSCAN_CUDA(cudaGetLastError());
  }
  constexpr int HB = mimo::MimoStage<N, P>::HB;
  const dim3 ogrid{unsigned((a.H + HB - 1) / HB), unsigned(C), unsigned(a.B)};
  mimo::mimo_out_kernel<Tin, MODE, N, P><<<ogrid, mimo::OUT_THREADS, 0, st>>>(p);
  CSSCAN_CUDA(cudaGetLastError());
  return CSSCAN_OK;
}

template <typename Tin, int MODE, int N, int P>
int launch_mimo(const MimoArgs& a, cudaStream_t st, bool staged) {
  if constexpr ((N == 8 || N == 16 || N == 32) && P * N <= 128) {
    if (staged) return MScan<N, mscan_states<N, P>(), P, Tin, MODE>::launch(a, st);
  }
  return launch_rows<Tin, MODE, N, P>(a, st);
}

template <typename Tin, int MODE, int P>
int dispatch_mimo_n(const MimoArgs& a, cudaStream_t st, bool staged) {
  switch (a.N) {
    case 2: return launch_mimo<Tin, MODE, 2, P>(a, st, staged);
    case 4: return launch_mimo<Tin, MODE, 4, P>(a, st, staged);
    case 8: return launch_mimo<Tin, MODE, 8, P>(a, st, staged);
    case 16: return launch_mimo<Tin, MODE, 16, P>(a, st, staged);
    case 32: return launch_mimo<Tin, MODE, 32, P>(a, st, staged);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

template <typename Tin, int MODE>
int dispatch_mimo_p(const MimoArgs& a, cudaStream_t st, bool staged) {
  switch (a.P) {
    case 1: return dispatch_mimo_n<Tin, MODE, 1>(a, st, staged);
    case 2: return dispatch_mimo_n<Tin, MODE, 2>(a, st, staged);
    case 4: return dispatch_mimo_n<Tin, MODE, 4>(a, st, staged);
    case 8: return dispatch_mimo_n<Tin, MODE, 8>(a, st, staged);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

template <typename Tin>
int mimo_dispatch(const MimoArgs& a, cudaStream_t st) {
  const bool staged = mscan_takes(a);
  return a.mode == 0 ? dispatch_mimo_p<Tin, 0>(a, st, staged) : dispatch_mimo_p<Tin, 1>(a, st, staged);
}

// ----------------------------------------------------------------------------- backward
// csscan_backward_mimo: e^{i theta} table, the checkpoint pass and the gradient pass of
// mgrad_kernels.cuh (a thread per (b, head, state); the whole sequence per thread).
template <typename Tin, int MODE, int P>
int launch_mimo_backward(const MimoBwdArgs& a, cudaStream_t st) {
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  const int64_t N = a.N, S = (a.L + mgrad::SEG - 1) / mgrad::SEG;
  const size_t rot_bytes = align_up(size_t(a.B * a.L * N) * sizeof(float2), 256);
  const size_t ckpt_bytes = align_up(size_t(a.B * S * a.H * N) * sizeof(float2), 256);
  WsEntry ws;
  int rc = get_workspace(dev, st, 1, rot_bytes + ckpt_bytes, &ws);
  if (rc != CSSCAN_OK) return rc;
  char* rest = ws_rest(ws);
  // gradients that are sums over several rows are accumulated and start at zero
  CSSCAN_CUDA(cudaMemsetAsync(a.dA, 0, size_t(a.H * N) * 4, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dBm, 0, size_t(a.B * a.L * N * a.P) * 8, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dCm, 0, size_t(a.B * a.L * N * a.P) * 8, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dtheta, 0, size_t(a.B * a.L * N) * 4, st));
  if (MODE == 1) CSSCAN_CUDA(cudaMemsetAsync(a.dlam, 0, size_t(a.B * a.L) * 4, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dDskip, 0, size_t(a.H * a.P) * 4, st));

  mgrad::Params p;
  std::memset(&p, 0, sizeof(p));
  p.x = a.x;
  p.dt = a.delta;
  p.Bm = a.Bm;
  p.Cm = a.Cm;
  p.lam = MODE == 1 ? a.lam : nullptr;
  p.A = a.A;
  p.Dskip = a.Dskip;
  p.dy = a.dy;
  p.rot = reinterpret_cast<const float2*>(rest);
  p.ckpt = reinterpret_cast<float2*>(rest + rot_bytes);
  p.dx = a.dx;
  p.ddt = a.ddelta;
  p.dA = a.dA;
  p.dBm = a.dBm;
  p.dCm = a.dCm;
  p.dtheta = a.dtheta;
  p.dlam = MODE == 1 ? a.dlam : nullptr;
  p.dD = a.dDskip;
  p.B = int(a.B);
  p.L = int(a.L);
  p.H = int(a.H);
  p.N = int(N);
  p.S = int(S);

  const long long n_rot = (long long)a.B * a.L * N;
  if (!grid_fits(n_rot)) return CSSCAN_ERR_UNSUPPORTED;
  bwd::rot_kernel<Tin><<<unsigned((n_rot + 255) / 256), 256, 0, st>>>(a.theta, reinterpret_cast<float2*>(rest), n_rot);
  CSSCAN_CUDA(cudaGetLastError());
  const int64_t heads_per_block = mgrad::THREADS / N;
  const dim3 grid{unsigned((a.H + heads_per_block - 1) / heads_per_block), unsigned(a.B)};
  if (S > 1) {
    mgrad::mckpt_kernel<Tin, MODE, P><<<grid, mgrad::THREADS, 0, st>>>(p);
    CSSCAN_CUDA(cudaGetLastError());
  }
  const int smem = mgrad::MGradSmem<P>::bytes(int(N));
  mgrad::mgrad_kernel<Tin, MODE, P><<<grid, mgrad::THREADS, unsigned(smem), st>>>(p);
  CSSCAN_CUDA(cudaGetLastError());
  return CSSCAN_OK;
}

template <typename Tin, int MODE>
int mimo_backward_p(const MimoBwdArgs& a, cudaStream_t st) {
  switch (a.P) {
    case 1: return launch_mimo_backward<Tin, MODE, 1>(a, st);
    case 2: return launch_mimo_backward<Tin, MODE, 2>(a, st);
    case 4: return launch_mimo_backward<Tin, MODE, 4>(a, st);
    case 8: return launch_mimo_backward<Tin, MODE, 8>(a, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

template <typename Tin>
int mimo_backward_dispatch(const MimoBwdArgs& a, cudaStream_t st) {
  return a.mode == 0 ? mimo_backward_p<Tin, 0>(a, st) : mimo_backward_p<Tin, 1>(a, st);
}

}  // namespace mimo_detail
}  // namespace csscan_host
