// backward_launch.cuh -- host side of csscan_backward: time-chunk choice, workspace layout, the
// checkpoint variant of the forward scan kernel and the gradient kernels (backward_kernels.cuh).
// Included by backward_f32.cu and backward_bf16.cu.
#pragma once

#include "backward_kernels.cuh"
#include "forward_launch.cuh"

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
  // The checkpoints come from the scan kernel's checkpoint variant where its tile copies can
  // read x and delta (16-byte rows and base addresses); otherwise from ckpt_kernel.
  const size_t s_in = sizeof(Tin);
  const bool fwd_ckpt = aligned(a.x, 16) && aligned(a.delta, 16) && (a.D * int64_t(s_in)) % 16 == 0;
  using K = RScan<N, Tin, MODE, true>;
  Args fa{a.x, a.delta, a.Bc, a.Cc, a.theta, a.lam, a.A, a.Dskip, nullptr, nullptr, nullptr, nullptr, nullptr,
          a.B, a.L, a.D, N, a.mode, a.dtype};
  const csscan_options_t fo = default_options();
  Plan fpl;
  if (fwd_ckpt) {
    int rc = make_plan(fa, fo, dev, K::shape(), &K::occ, &fpl);
    if (rc != CSSCAN_OK) return rc;
  }
  const size_t fwd_bytes = fwd_ckpt ? align_up(fpl.rest_bytes, 256) : 0;
  WsEntry ws;
  int rc = get_workspace(dev, st, fwd_ckpt ? size_t(fpl.n_units) : 1, fwd_bytes + rot_bytes + ckpt_bytes + chunk_bytes,
                         &ws);
  if (rc != CSSCAN_OK) return rc;
  char* fwd_rest = ws_rest(ws);
  char* rest = fwd_rest + fwd_bytes;

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
  if (fwd_ckpt) {   // every checkpoint, chunk entries included, from the scan kernel
    uint32_t* hdr = static_cast<uint32_t*>(ws.base);
    rc = K::enqueue(fa, fo, fpl, hdr, reinterpret_cast<uint32_t*>(static_cast<char*>(ws.base) + HDR_BYTES), fwd_rest,
                    st, p.ckpt, S);
    if (rc != CSSCAN_OK) return rc;
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

template <typename Tin, int MODE>
int dispatch_backward_n(const BwdArgs& a, cudaStream_t st) {
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
  return a.mode == 0 ? dispatch_backward_n<Tin, 0>(a, st) : dispatch_backward_n<Tin, 1>(a, st);
}

}  // namespace csscan_host
