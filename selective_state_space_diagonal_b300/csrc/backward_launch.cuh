// backward_launch.cuh -- host side of csscan_backward, included by backward_f32.cu and
// backward_bf16.cu. Two paths:
//   launch_backward_rot: inputs that meet the tile-copy rules (16-byte aligned x, delta and dy
//     with 16-byte (b, t) rows, 16-byte aligned dBc and dCc, 8-byte aligned dA and dtheta): the
//     forward scan kernel's checkpoint variant, the chunk adjoints where the sequence is split,
//     and ngrad_kernel (ngrad_kernels.cuh) in the rotating frame;
//   launch_backward: every other input, and the zero-order hold (whose injection weight is
//     complex per element): checkpoints from ckpt_kernel and the absolute-frame grad_kernel
//     (backward_kernels.cuh).
#pragma once

#include "backward_kernels.cuh"
#include "forward_launch.cuh"
#include "ngrad_kernels.cuh"

namespace csscan_host {

template <typename Tin, int MODE, int N>
int launch_backward(const BwdArgs& a, cudaStream_t st) {
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  int nsm = 0;
  CSSCAN_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  const int64_t S = (a.L + bwd::SEG - 1) / bwd::SEG;
  // time chunks, only where the rows leave the GPU short of about two gradient blocks per SM;
  // then enough chunks for about four gradient blocks per SM and SEQ_THREADS_PER_SM threads of
  // the sequential per-(b, d, n) passes per SM (the two chunk passes cost about one forward each)
  const int64_t row_blocks = a.B * ((a.D + bwd::GradTile<N>::CB - 1) / bwd::GradTile<N>::CB);
  const int64_t seq_rows = a.B * a.D * N;
  int64_t C = 1;
  if (row_blocks < 2 * int64_t(nsm)) {
    const int64_t c_blocks = (4 * int64_t(nsm) + row_blocks - 1) / row_blocks;
    const int64_t c_threads = (int64_t(nsm) * SEQ_THREADS_PER_SM + seq_rows - 1) / seq_rows;
    C = std::min<int64_t>(S, std::max<int64_t>(1, std::max(c_blocks, c_threads)));
  }
  if (C > 65535) C = 65535;
  const int64_t TC = (S + C - 1) / C * bwd::SEG;
  C = (a.L + TC - 1) / TC;
  const size_t rot_bytes = align_up(size_t(a.B * a.L * N) * sizeof(float2), 256);
  const size_t ckpt_bytes = align_up(size_t(a.B * S * a.D * N) * sizeof(float2), 256);
  const size_t chunk_bytes = C > 1 ? size_t(a.B * C * a.D * N) * 5 * sizeof(float2) : 0;
  // checkpoints: the zero-order hold on inputs that meet the forward scan's tile-copy rules takes
  // them (every segment's entry state, chunk starts included) from the scan kernel's checkpoint
  // variant, one pass at forward speed; every other input from ckpt_kernel
  const int64_t s_in = a.dtype == CSSCAN_F32 ? 4 : 2;
  const bool fwd_ckpt = MODE == 2 && aligned(a.x, 16) && aligned(a.delta, 16) && (a.D * s_in) % 16 == 0;
  Args fa{a.x, a.delta, a.Bc, a.Cc, a.theta, a.lam, a.A, a.Dskip, nullptr, nullptr, nullptr, nullptr, nullptr,
          a.B, a.L, a.D, N, a.mode, a.dtype};
  const csscan_options_t fo = default_options();
  Plan fpl;
  size_t f_rest = 0, f_units = 1;
  if constexpr (MODE == 2) {
    if (fwd_ckpt) {
      const int prc = make_plan(fa, fo, dev, RScan<N, Tin, 2, true>::shape(), &RScan<N, Tin, 2, true>::occ, &fpl);
      if (prc != CSSCAN_OK) return prc;
      f_rest = align_up(fpl.rest_bytes, 256);
      f_units = size_t(fpl.n_units);
    }
  }
  WsEntry ws;
  int rc = get_workspace(dev, st, f_units, f_rest + rot_bytes + ckpt_bytes + chunk_bytes, &ws);
  if (rc != CSSCAN_OK) return rc;
  char* const ws_base = static_cast<char*>(ws.base);
  char* const f_area = ws_rest(ws);   // the checkpoint scan's tables and carries (zero-order hold)
  char* rest = f_area + f_rest;

  // gradients that are sums over several rows are accumulated and start at zero
  CSSCAN_CUDA(cudaMemsetAsync(a.dA, 0, size_t(a.D * N) * 4, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dBc, 0, size_t(a.B * a.L * N) * 8, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dCc, 0, size_t(a.B * a.L * N) * 8, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dtheta, 0, size_t(a.B * a.L * N) * 4, st));
  if (MODE == 1) CSSCAN_CUDA(cudaMemsetAsync(a.dlam, 0, size_t(a.B * a.L) * 4, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dDskip, 0, size_t(a.D) * 4, st));

  bwd::Params p;
  p.x = a.x;
  p.dt = a.delta;
  p.Bc = a.Bc;
  p.Cc = a.Cc;
  p.lam = MODE == 1 ? a.lam : nullptr;
  p.A = a.A;
  p.Dskip = a.Dskip;
  p.dy = a.dy;
  p.dx = a.dx;
  p.ddt = a.ddelta;
  p.dA = a.dA;
  p.dBc = a.dBc;
  p.dCc = a.dCc;
  p.dtheta = a.dtheta;
  p.dlam = MODE == 1 ? a.dlam : nullptr;
  p.dD = a.dDskip;
  p.rot = reinterpret_cast<const float2*>(rest);
  p.theta = a.theta;
  p.ckpt = reinterpret_cast<float2*>(rest + rot_bytes);
  p.chunk = C > 1 ? reinterpret_cast<float2*>(rest + rot_bytes + ckpt_bytes) : nullptr;
  p.B = int(a.B);
  p.L = int(a.L);
  p.D = int(a.D);
  p.N = N;
  p.S = int(S);
  p.TC = int(TC);
  p.C = int(C);
  p.fwd_ckpt = fwd_ckpt ? 1 : 0;

  if (!grid_fits((long long)a.B * a.L * N) || !grid_fits((long long)a.B * C * a.D * N)) return CSSCAN_ERR_UNSUPPORTED;
  if constexpr (MODE == 2) {
    if (fwd_ckpt) {
      rc = RScan<N, Tin, 2, true>::enqueue(fa, fo, fpl, reinterpret_cast<uint32_t*>(ws_base),
                                           reinterpret_cast<uint32_t*>(ws_base + HDR_BYTES), f_area, st,
                                           reinterpret_cast<float2*>(rest + rot_bytes), S);
      if (rc != CSSCAN_OK) return rc;
    }
  }
  const long long n_rot = (long long)a.B * a.L * N;
  bwd::rot_kernel<Tin><<<unsigned((n_rot + 255) / 256), 256, 0, st>>>(a.theta, reinterpret_cast<float2*>(rest), n_rot);
  CSSCAN_CUDA(cudaGetLastError());
  const long long n_ck = (long long)a.B * C * a.D * N;   // threads of the per-chunk passes
  const unsigned ck_blocks = unsigned((n_ck + 255) / 256);
  if (C > 1) {
    if (!fwd_ckpt) {
      bwd::chunk_fwd_kernel<Tin, MODE><<<ck_blocks, 256, 0, st>>>(p);
      CSSCAN_CUDA(cudaGetLastError());
    }
    const dim3 agrid{unsigned((a.D + 256 / N - 1) / (256 / N)), unsigned(C), unsigned(a.B)};
    bwd::chunk_adj_kernel<Tin, MODE, N><<<agrid, 256, 0, st>>>(p);
    CSSCAN_CUDA(cudaGetLastError());
    const long long n_cb = (long long)a.B * a.D * N;
    bwd::chunk_combine_kernel<<<unsigned((n_cb + 255) / 256), 256, 0, st>>>(p);
    CSSCAN_CUDA(cudaGetLastError());
  }
  if (!fwd_ckpt && TC > bwd::SEG) {   // some segments start inside a chunk: their checkpoints
    bwd::ckpt_kernel<Tin, MODE><<<ck_blocks, 256, 0, st>>>(p);
    CSSCAN_CUDA(cudaGetLastError());
  }
  const dim3 grid{unsigned((a.D + bwd::GradTile<N>::CB - 1) / bwd::GradTile<N>::CB), unsigned(a.B), unsigned(C)};
  {
    static std::mutex mu;
    static std::map<int, bool> attr_set;
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      CSSCAN_CUDA(cudaFuncSetAttribute(bwd::grad_kernel<Tin, MODE, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       bwd::GradStage<N>::BYTES));
      attr_set[dev] = true;
    }
  }
  bwd::grad_kernel<Tin, MODE, N><<<grid, bwd::THREADS, bwd::GradStage<N>::BYTES, st>>>(p);
  CSSCAN_CUDA(cudaGetLastError());
  return CSSCAN_OK;
}

// ---------------------------------------------------------------------------- rotating frame
template <typename Tin, int MODE, int N>
int launch_backward_rot(const BwdArgs& a, cudaStream_t st) {
  using GT = ngrad::GTile<N>;
  using GS = ngrad::GStage<N, Tin, MODE>;
  constexpr int SEG = ngrad::SEG;
  int dev = 0, nsm = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  CSSCAN_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  const int64_t S8 = (a.L + SEG - 1) / SEG;
  const int64_t S32 = (a.L + T_SUB - 1) / T_SUB;

  // the forward scan's checkpoint variant: one channel and 16 states (all N < 16) per thread
  constexpr int NSF = N >= 16 ? 16 : N;
  using KF = NScan<N, NSF, Tin, MODE, true>;
  Args fa{a.x, a.delta, a.Bc, a.Cc, a.theta, a.lam, a.A, a.Dskip, nullptr, nullptr, nullptr, nullptr, nullptr,
          a.B, a.L, a.D, N, a.mode, a.dtype};
  const csscan_options_t fo = default_options();
  Plan fpl;
  int rc = make_plan(fa, fo, dev, KF::shape(), &KF::occ, &fpl);
  if (rc != CSSCAN_OK) return rc;

  // gradient blocks: (channel tile, b, time chunk); time chunks of whole 32-step sub-chunks, as
  // many as make the blocks fill the resident slots in nearly whole waves (more than one chunk
  // costs the chunk-carry passes, about 0.05 of a wave)
  int occ = 0;
  rc = occupancy_of(ngrad::ngrad_kernel<Tin, MODE, N>, dev, GS::SMEM, &occ);
  if (rc != CSSCAN_OK) return rc;
  if (occ < 1) {
    set_last_error("gradient block does not fit on this device");
    return CSSCAN_ERR_CUDA;
  }
  const int64_t slots = int64_t(nsm) * occ;
  const int64_t n_dtiles = (a.D + GT::BC - 1) / GT::BC;
  const int64_t tiles = a.B * n_dtiles;
  int64_t C = 1;
  {
    double best = 1e30;
    for (int64_t cc = 1; cc <= std::min<int64_t>(S32, 256); ++cc) {
      const double t = double((tiles * cc + slots - 1) / slots) / double(cc) + (cc > 1 ? 0.05 : 0.0);
      if (t < best - 1e-9) {
        best = t;
        C = cc;
      }
    }
  }
  const int64_t TC = (S32 + C - 1) / C * T_SUB;
  C = (a.L + TC - 1) / TC;
  if (C > 65535 || n_dtiles > 0x7fffffff) return CSSCAN_ERR_UNSUPPORTED;

  // workspace: the forward plan's region (tables, carries), checkpoints, and with chunks the
  // chunk carries (V, sum dt, phase, kappa) and the chunk-start terms of ddt; G(E) sums (trapezoid)
  size_t off = align_up(fpl.rest_bytes, 256);
  auto take = [&](size_t bytes) { const size_t r = off; off = align_up(off + bytes, 256); return r; };
  const size_t o_ckpt = take(size_t(a.B * S8 * a.D * N) * sizeof(float2));
  const size_t o_V = C > 1 ? take(size_t(a.B * C * a.D * N) * sizeof(float2)) : 0;
  const size_t o_kap = C > 1 ? take(size_t(a.B * C * a.D * N) * sizeof(float2)) : 0;
  const size_t o_sdt = C > 1 ? take(size_t(a.B * C * a.D) * 4) : 0;
  const size_t o_ph = C > 1 ? take(size_t(a.B * C * N) * sizeof(float2)) : 0;
  const size_t o_xb = C > 1 && MODE == 1 ? take(size_t(a.B * C * a.D) * 4) : 0;
  const size_t o_ge = MODE == 1 ? take(size_t(a.B * a.L) * 4) : 0;
  WsEntry ws;
  rc = get_workspace(dev, st, size_t(fpl.n_units), off, &ws);
  if (rc != CSSCAN_OK) return rc;
  char* base = static_cast<char*>(ws.base);
  uint32_t* hdr = reinterpret_cast<uint32_t*>(base);
  char* rest = ws_rest(ws);
  float2* ckpt = reinterpret_cast<float2*>(rest + o_ckpt);

  // gradients that are sums over several rows are accumulated and start at zero
  CSSCAN_CUDA(cudaMemsetAsync(a.dA, 0, size_t(a.D * N) * 4, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dBc, 0, size_t(a.B * a.L * N) * 8, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dCc, 0, size_t(a.B * a.L * N) * 8, st));
  CSSCAN_CUDA(cudaMemsetAsync(a.dtheta, 0, size_t(a.B * a.L * N) * 4, st));
  if (MODE == 1) {
    CSSCAN_CUDA(cudaMemsetAsync(a.dlam, 0, size_t(a.B * a.L) * 4, st));
    CSSCAN_CUDA(cudaMemsetAsync(rest + o_ge, 0, size_t(a.B * a.L) * 4, st));
  }
  CSSCAN_CUDA(cudaMemsetAsync(a.dDskip, 0, size_t(a.D) * 4, st));

  // ---- checkpoints (and the tables the gradient pass reads)
  rc = KF::enqueue(fa, fo, fpl, hdr, reinterpret_cast<uint32_t*>(base + HDR_BYTES), rest, st, ckpt, S8);
  if (rc != CSSCAN_OK) return rc;

  // ---- chunk carries: kappa_c entering every chunk's last step
  if (C > 1) {
    using AS = ngrad::AdjStage<N, Tin>;
    ngrad::AdjParams ap;
    std::memset(&ap, 0, sizeof(ap));
    {
      const CUtensorMapDataType tin =
          sizeof(Tin) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      const uint64_t B = uint64_t(a.B), L = uint64_t(a.L), D = uint64_t(a.D), s_in = sizeof(Tin);
      const uint64_t cdims[4] = {2 * N, 2, L, B};
      const uint64_t cstrides[3] = {2 * N * 4, 4 * N * 4, L * 4 * N * 4};
      const uint32_t cbox[4] = {2 * N, 1, T_SUB, 1};
      const bool ok = map3(&ap.tm_dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.dy, D, L, B, D * 4, L * D * 4, AS::CH, T_SUB, 1) &&
                      map3(&ap.tm_dt, tin, a.delta, D, L, B, D * s_in, L * D * s_in, AS::CH, T_SUB, 1) &&
                      make_map(&ap.tm_ct, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rest + fpl.o_tab, 4, cdims, cstrides, cbox);
      if (!ok) {
        set_last_error("cuTensorMapEncodeTiled failed or unavailable");
        return CSSCAN_ERR_CUDA;
      }
    }
    ap.hdr = hdr;
    ap.rot = reinterpret_cast<const float2*>(rest + fpl.o_rot);
    ap.dy = a.dy;
    ap.dt = a.delta;
    ap.A = a.A;
    ap.V = reinterpret_cast<float2*>(rest + o_V);
    ap.Sdt = reinterpret_cast<float*>(rest + o_sdt);
    ap.P = reinterpret_cast<float2*>(rest + o_ph);
    ap.kap = reinterpret_cast<float2*>(rest + o_kap);
    ap.B = int(a.B);
    ap.L = int(a.L);
    ap.D = int(a.D);
    ap.S32 = int(S32);
    ap.TC = int(TC);
    ap.C = int(C);
    ap.tab_ng = NTile<N, NSF>::NG;
    int aocc = 0;
    rc = occupancy_of(ngrad::nadj_kernel<Tin, N>, dev, AS::SMEM, &aocc);   // raises the shared-memory limit
    if (rc != CSSCAN_OK) return rc;
    const dim3 agrid{unsigned((a.D + AS::CH - 1) / AS::CH), unsigned(C - 1), unsigned(a.B)};
    ngrad::nadj_kernel<Tin, N><<<agrid, 128, AS::SMEM, st>>>(ap);
    CSSCAN_CUDA(cudaGetLastError());
    const long long n_ph = (long long)a.B * C * N, n_cb = (long long)a.B * a.D * N;
    if (!grid_fits(n_ph) || !grid_fits(n_cb)) return CSSCAN_ERR_UNSUPPORTED;
    ngrad::nphase_kernel<<<unsigned((n_ph + 255) / 256), 256, 0, st>>>(ap, N);
    CSSCAN_CUDA(cudaGetLastError());
    ngrad::ncombine_kernel<<<unsigned((n_cb + 255) / 256), 256, 0, st>>>(ap, N);
    CSSCAN_CUDA(cudaGetLastError());
  }

  // ---- the gradient pass
  ngrad::GradParams gp;
  std::memset(&gp, 0, sizeof(gp));
  const CUtensorMapDataType tin = sizeof(Tin) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t s_in = sizeof(Tin);
  const uint64_t B = uint64_t(a.B), L = uint64_t(a.L), D = uint64_t(a.D), S = uint64_t(fpl.S);
  const uint64_t tdims[4] = {2 * N, 2, L, B};
  const uint64_t tstrides[3] = {2 * N * 4, 4 * N * 4, L * 4 * N * 4};
  const uint32_t tbox[4] = {2 * N, 2, SEG, 1};
  bool ok = map3(&gp.tm_x, tin, a.x, D, L, B, D * s_in, L * D * s_in, GT::BC, SEG, 1) &&
            map3(&gp.tm_dt, tin, a.delta, D, L, B, D * s_in, L * D * s_in, GT::BC, SEG + 1, 1) &&
            map3(&gp.tm_dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.dy, D, L, B, D * 4, L * D * 4, GT::BC, SEG, 1) &&
            make_map(&gp.tm_tab, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rest + fpl.o_tab, 4, tdims, tstrides, tbox) &&
            map3(&gp.tm_rot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rest + fpl.o_rot, 2 * N, 4 * S, B, 8 * N, 4 * S * 8 * N,
                 2 * N, 1, 1);
  if (ok && MODE == 1)
    ok = map3(&gp.tm_aux, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rest + fpl.o_aux, 4, L, B, 16, L * 16, 4, SEG, 1);
  if (!ok) {
    set_last_error("cuTensorMapEncodeTiled failed or unavailable");
    return CSSCAN_ERR_CUDA;
  }
  gp.A = a.A;
  gp.Dskip = a.Dskip;
  gp.ckpt = reinterpret_cast<const float4*>(ckpt);
  gp.kap = C > 1 ? reinterpret_cast<const float2*>(rest + o_kap) : nullptr;
  gp.dx = a.dx;
  gp.ddt = a.ddelta;
  gp.dA = a.dA;
  gp.dBc = a.dBc;
  gp.dCc = a.dCc;
  gp.dtheta = a.dtheta;
  gp.dlam = MODE == 1 ? a.dlam : nullptr;
  gp.dD = a.dDskip;
  gp.ge = MODE == 1 ? reinterpret_cast<float*>(rest + o_ge) : nullptr;
  gp.xb = o_xb ? reinterpret_cast<float*>(rest + o_xb) : nullptr;
  gp.hdr = hdr;
  gp.B = int(a.B);
  gp.L = int(a.L);
  gp.D = int(a.D);
  gp.S8 = int(S8);
  gp.TC = int(TC);
  gp.C = int(C);
  gp.tab_ng = NTile<N, NSF>::NG;
  const dim3 grid{unsigned(n_dtiles), unsigned(a.B), unsigned(C)};
  ngrad::ngrad_kernel<Tin, MODE, N><<<grid, ngrad::THREADS, GS::SMEM, st>>>(gp);
  CSSCAN_CUDA(cudaGetLastError());
  if (MODE == 1 && C > 1) {
    const long long n_fix = (long long)a.B * (C - 1) * a.D;
    if (!grid_fits(n_fix)) return CSSCAN_ERR_UNSUPPORTED;
    ngrad::ngrad_fix_kernel<<<unsigned((n_fix + 255) / 256), 256, 0, st>>>(gp.xb, a.ddelta, int(a.B), int(a.L),
                                                                          int(a.D), int(C), int(TC));
    CSSCAN_CUDA(cudaGetLastError());
  }
  const long long n_post = (long long)a.B * S32 * N;
  if (!grid_fits(n_post)) return CSSCAN_ERR_UNSUPPORTED;
  ngrad::ngrad_post_kernel<Tin, MODE><<<unsigned((n_post + 255) / 256), 256, 0, st>>>(
      a.theta, a.Bc, a.Cc, gp.ge, a.dBc, a.dCc, int(a.B), int(a.L), N, int(S32));
  CSSCAN_CUDA(cudaGetLastError());
  return CSSCAN_OK;
}

// Whether the rotating-frame path takes these arguments (see the file comment).
inline bool backward_rot_takes(const BwdArgs& a) {
  const int64_t s_in = a.dtype == CSSCAN_F32 ? 4 : 2;
  return aligned(a.x, 16) && aligned(a.delta, 16) && aligned(a.dy, 16) && (a.D * s_in) % 16 == 0 &&
         (a.D * 4) % 16 == 0 && aligned(a.dBc, 16) && aligned(a.dCc, 16) && aligned(a.dA, 8) && aligned(a.dtheta, 8);
}

template <typename Tin, int MODE>
int dispatch_backward_n(const BwdArgs& a, cudaStream_t st) {
  if constexpr (MODE != 2) {   // the zero-order hold takes the absolute-frame path only
    if (backward_rot_takes(a)) {
      switch (a.N) {
        case 2: return launch_backward_rot<Tin, MODE, 2>(a, st);
        case 4: return launch_backward_rot<Tin, MODE, 4>(a, st);
        case 8: return launch_backward_rot<Tin, MODE, 8>(a, st);
        case 16: return launch_backward_rot<Tin, MODE, 16>(a, st);
        case 32: return launch_backward_rot<Tin, MODE, 32>(a, st);
        default: return CSSCAN_ERR_UNSUPPORTED;
      }
    }
  }
  switch (a.N) {
    case 2: return launch_backward<Tin, MODE, 2>(a, st);
    case 4: return launch_backward<Tin, MODE, 4>(a, st);
    case 8: return launch_backward<Tin, MODE, 8>(a, st);
    case 16: return launch_backward<Tin, MODE, 16>(a, st);
    case 32: return launch_backward<Tin, MODE, 32>(a, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

template <typename Tin>
int backward_dispatch(const BwdArgs& a, cudaStream_t st) {
  if (a.mode == 2) return dispatch_backward_n<Tin, 2>(a, st);
  return a.mode == 0 ? dispatch_backward_n<Tin, 0>(a, st) : dispatch_backward_n<Tin, 1>(a, st);
}

}  // namespace csscan_host
