// mimo.cu -- host side of csscan_forward_mimo: time-chunk choice, workspace layout and the
// launches of the MIMO kernels (mimo_kernels.cuh), for both input dtypes.
#include <algorithm>

#include "host_common.h"
#include "mimo_kernels.cuh"

namespace csscan_host {
namespace {

using namespace csscan;

template <typename Tin, int MODE, int N, int P>
int launch_mimo(const MimoArgs& a, cudaStream_t st) {
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

template <typename Tin, int MODE, int P>
int dispatch_mimo_n(const MimoArgs& a, cudaStream_t st) {
  switch (a.N) {
    case 2: return launch_mimo<Tin, MODE, 2, P>(a, st);
    case 4: return launch_mimo<Tin, MODE, 4, P>(a, st);
    case 8: return launch_mimo<Tin, MODE, 8, P>(a, st);
    case 16: return launch_mimo<Tin, MODE, 16, P>(a, st);
    case 32: return launch_mimo<Tin, MODE, 32, P>(a, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

template <typename Tin, int MODE>
int dispatch_mimo_p(const MimoArgs& a, cudaStream_t st) {
  switch (a.P) {
    case 1: return dispatch_mimo_n<Tin, MODE, 1>(a, st);
    case 2: return dispatch_mimo_n<Tin, MODE, 2>(a, st);
    case 4: return dispatch_mimo_n<Tin, MODE, 4>(a, st);
    case 8: return dispatch_mimo_n<Tin, MODE, 8>(a, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

}  // namespace

int mimo_f32(const MimoArgs& a, cudaStream_t st) {
  return a.mode == 0 ? dispatch_mimo_p<float, 0>(a, st) : dispatch_mimo_p<float, 1>(a, st);
}
int mimo_bf16(const MimoArgs& a, cudaStream_t st) {
  return a.mode == 0 ? dispatch_mimo_p<uint16_t, 0>(a, st) : dispatch_mimo_p<uint16_t, 1>(a, st);
}

}  // namespace csscan_host
