// csscan.cu -- the C ABI declared in include/csscan.h: argument checks, the per-(device,
// stream) workspace, the decode step and the no-allocation entry point. The scans themselves
// are planned and launched by the per-dtype units (forward_*.cu, backward_*.cu, mimo_*.cu).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "csscan.h"
#include "decode_kernel.cuh"
#include "host_common.h"
#include "scan_kernels.cuh"

using namespace csscan;

namespace csscan_host {

namespace {
thread_local char g_last_cuda_error[256] = "";
}  // namespace

void set_last_error(const char* msg) { std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s", msg); }

int cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", what, cudaGetErrorString(e));
  return CSSCAN_ERR_CUDA;
}

// ----------------------------------------------------------------------------- descriptors
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}
}  // namespace

bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
  return fn(m, type, cuuint32_t(rank), const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

csscan_options_t default_options() {
  csscan_options_t o;
  std::memset(&o, 0, sizeof(o));
  o.silent_chunk = -1;
  return o;
}

// ----------------------------------------------------------------------------- workspace
namespace {
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, WsEntry> g_ws;
}  // namespace

int get_workspace(int dev, cudaStream_t st, size_t units, size_t rest_bytes, WsEntry* out) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  WsEntry& e = g_ws[{dev, reinterpret_cast<uintptr_t>(st)}];
  const size_t need_cap = std::max(units, e.flag_cap);
  const size_t need = HDR_BYTES + align_up(need_cap * 4, 256) + rest_bytes;
  if (e.base == nullptr || need_cap > e.flag_cap || need > e.bytes) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CSSCAN_CUDA(cudaStreamIsCapturing(st, &cs));
    if (cs != cudaStreamCaptureStatusNone) {
      set_last_error("workspace must grow, which cannot happen during stream capture; call once before capturing");
      return CSSCAN_ERR_CUDA;
    }
    const size_t cap = std::max(need_cap, e.flag_cap * 2);
    const size_t bytes = align_up(HDR_BYTES + align_up(cap * 4, 256) + rest_bytes * 5 / 4, size_t(1) << 20);
    if (e.base) {
      CSSCAN_CUDA(cudaStreamSynchronize(st));
      CSSCAN_CUDA(cudaFree(e.base));
      e.base = nullptr;
    }
    CSSCAN_CUDA(cudaMalloc(&e.base, bytes));
    CSSCAN_CUDA(cudaMemset(e.base, 0, HDR_BYTES + align_up(cap * 4, 256)));
    e.bytes = bytes;
    e.flag_cap = cap;
  }
  *out = e;
  return CSSCAN_OK;
}

namespace {

// ----------------------------------------------------------------------------- forward checks
// One set of rules for every forward entry point and every mode: pointers, sizes, the tile
// copies' 16-byte rule on x and delta, and N.
int validate(const Args& a, const csscan_options_t& o) {
  if (a.mode != CSSCAN_MODE_EXP_EULER && a.mode != CSSCAN_MODE_EXP_TRAPEZOID && a.mode != CSSCAN_MODE_ZOH)
    return CSSCAN_ERR_INVALID_ARG;
  if (a.dtype != CSSCAN_F32 && a.dtype != CSSCAN_BF16) return CSSCAN_ERR_INVALID_ARG;
  if (a.B < 0 || a.L < 0 || a.D < 0 || a.N <= 0) return CSSCAN_ERR_INVALID_ARG;
  if (!a.x || !a.delta || !a.A || !a.Bc || !a.Cc || !a.theta || !a.Dskip || !a.y) return CSSCAN_ERR_INVALID_ARG;
  if (a.mode == CSSCAN_MODE_EXP_TRAPEZOID && !a.lam) return CSSCAN_ERR_INVALID_ARG;
  if ((a.x_prev == nullptr) != (a.Bc_prev == nullptr)) return CSSCAN_ERR_INVALID_ARG;
  if (o.cta_warps != 0 || o.carry < 0 || o.carry > 2 || o.chunk_len < 0 || (o.chunk_len % T_SUB) != 0 ||
      o.poll_limit < 0)
    return CSSCAN_ERR_INVALID_ARG;
  if (a.N != 2 && a.N != 4 && a.N != 8 && a.N != 16 && a.N != 32 && a.N != 64) return CSSCAN_ERR_UNSUPPORTED;
  if (a.B > (int64_t(1) << 31) - 1 || a.L > (int64_t(1) << 30) || a.D > (int64_t(1) << 30)) return CSSCAN_ERR_UNSUPPORTED;
  const size_t s = a.dtype == CSSCAN_F32 ? 4 : 2;
  if (!aligned(a.x, 16) || !aligned(a.delta, 16) || ((a.D * int64_t(s)) % 16) != 0) return CSSCAN_ERR_MISALIGNED;
  if (!aligned(a.Bc, s) || !aligned(a.Cc, s) || !aligned(a.theta, s) || (a.lam && !aligned(a.lam, s)) ||
      !aligned(a.A, 4) || !aligned(a.Dskip, 4) || !aligned(a.y, 4) || (a.h0 && !aligned(a.h0, 16)) ||
      (a.h_last && !aligned(a.h_last, 16)) || (a.x_prev && !aligned(a.x_prev, s)) ||
      (a.Bc_prev && !aligned(a.Bc_prev, s)))
    return CSSCAN_ERR_MISALIGNED;
  return CSSCAN_OK;
}

int forward_impl(Args a, const csscan_options_t* opts, cudaStream_t st, const FixedScratch* fixed) {
  const csscan_options_t o = opts ? *opts : default_options();
  int rc = validate(a, o);
  if (rc != CSSCAN_OK) return rc;
  if (a.mode != CSSCAN_MODE_EXP_TRAPEZOID) {   // the halo only enters the trapezoid rule
    a.x_prev = nullptr;
    a.Bc_prev = nullptr;
  }
  if (a.B == 0 || a.L == 0 || a.D == 0) return CSSCAN_OK;
  return a.dtype == CSSCAN_F32 ? forward_f32(a, o, st, fixed) : forward_bf16(a, o, st, fixed);
}

// ----------------------------------------------------------------------------- decode step
template <typename Tin, int MODE, int NP>
int launch_decode(const DecodeParams& dp, cudaStream_t st) {
  const long long threads = dp.rows * NP;
  decode_kernel<Tin, MODE, NP><<<unsigned((threads + 255) / 256), 256, 0, st>>>(dp);
  CSSCAN_CUDA(cudaGetLastError());
  return CSSCAN_OK;
}

template <typename Tin, int MODE>
int dispatch_decode(const DecodeParams& dp, cudaStream_t st) {
  switch (dp.N) {
    case 2: return launch_decode<Tin, MODE, 1>(dp, st);
    case 4: return launch_decode<Tin, MODE, 2>(dp, st);
    case 8: return launch_decode<Tin, MODE, 4>(dp, st);
    case 16: return launch_decode<Tin, MODE, 8>(dp, st);
    case 32: return launch_decode<Tin, MODE, 16>(dp, st);
    case 64: return launch_decode<Tin, MODE, 32>(dp, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

int decode_impl(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc, const void* theta,
                const void* lambda, const float* Dskip, float* y, float* h, const void* x_prev, const void* Bc_prev,
                int64_t B, int64_t D, int64_t N, int mode, int dtype, cudaStream_t stream) {
  if (mode != CSSCAN_MODE_EXP_EULER && mode != CSSCAN_MODE_EXP_TRAPEZOID && mode != CSSCAN_MODE_ZOH)
    return CSSCAN_ERR_INVALID_ARG;
  if (dtype != CSSCAN_F32 && dtype != CSSCAN_BF16) return CSSCAN_ERR_INVALID_ARG;
  if (B < 0 || D < 0 || N <= 0) return CSSCAN_ERR_INVALID_ARG;
  if (!x || !delta || !A || !Bc || !Cc || !theta || !Dskip || !y || !h) return CSSCAN_ERR_INVALID_ARG;
  if (mode == CSSCAN_MODE_EXP_TRAPEZOID && !lambda) return CSSCAN_ERR_INVALID_ARG;
  if ((x_prev == nullptr) != (Bc_prev == nullptr)) return CSSCAN_ERR_INVALID_ARG;
  if (N != 2 && N != 4 && N != 8 && N != 16 && N != 32 && N != 64) return CSSCAN_ERR_UNSUPPORTED;
  if (B > (int64_t(1) << 31) - 1 || D > (int64_t(1) << 30) || B * D > (int64_t(1) << 40)) return CSSCAN_ERR_UNSUPPORTED;
  const size_t s = dtype == CSSCAN_F32 ? 4 : 2;
  if (!aligned(h, 16) || !aligned(x, s) || !aligned(delta, s) || !aligned(Bc, s) || !aligned(Cc, s) ||
      !aligned(theta, s) || (lambda && !aligned(lambda, s)) || !aligned(A, 4) || !aligned(Dskip, 4) ||
      !aligned(y, 4) || (x_prev && !aligned(x_prev, s)) || (Bc_prev && !aligned(Bc_prev, s)))
    return CSSCAN_ERR_MISALIGNED;
  if (B == 0 || D == 0) return CSSCAN_OK;
  DecodeParams dp;
  dp.x = x;
  dp.dt = delta;
  dp.A = A;
  dp.Bc = Bc;
  dp.Cc = Cc;
  dp.theta = theta;
  dp.lam = lambda;
  dp.Dskip = Dskip;
  dp.y = y;
  dp.h = reinterpret_cast<float4*>(h);
  dp.x_prev = mode == CSSCAN_MODE_EXP_TRAPEZOID ? x_prev : nullptr;
  dp.Bc_prev = mode == CSSCAN_MODE_EXP_TRAPEZOID ? Bc_prev : nullptr;
  dp.rows = B * D;
  dp.D = int(D);
  dp.N = int(N);
  if (dtype == CSSCAN_F32)
    return mode == 0 ? dispatch_decode<float, 0>(dp, stream)
                     : (mode == 1 ? dispatch_decode<float, 1>(dp, stream) : dispatch_decode<float, 2>(dp, stream));
  return mode == 0 ? dispatch_decode<uint16_t, 0>(dp, stream)
                   : (mode == 1 ? dispatch_decode<uint16_t, 1>(dp, stream) : dispatch_decode<uint16_t, 2>(dp, stream));
}

int mimo_impl(const MimoArgs& a, cudaStream_t st) {
  if (a.mode != CSSCAN_MODE_EXP_EULER && a.mode != CSSCAN_MODE_EXP_TRAPEZOID) {
    return a.mode == CSSCAN_MODE_ZOH ? CSSCAN_ERR_UNSUPPORTED : CSSCAN_ERR_INVALID_ARG;
  }
  if (a.dtype != CSSCAN_F32 && a.dtype != CSSCAN_BF16) return CSSCAN_ERR_INVALID_ARG;
  if (a.B < 0 || a.L < 0 || a.H < 0 || a.P <= 0 || a.N <= 0) return CSSCAN_ERR_INVALID_ARG;
  const bool rows = a.B > 0 && a.L > 0, heads = a.H > 0;
  if (heads && (!a.A || !a.Dskip)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && (!a.Bm || !a.Cm || !a.theta)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && heads && (!a.x || !a.delta || !a.y)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && a.mode == CSSCAN_MODE_EXP_TRAPEZOID && !a.lam) return CSSCAN_ERR_INVALID_ARG;
  if (a.N != 2 && a.N != 4 && a.N != 8 && a.N != 16 && a.N != 32) return CSSCAN_ERR_UNSUPPORTED;
  if (a.P != 1 && a.P != 2 && a.P != 4 && a.P != 8) return CSSCAN_ERR_UNSUPPORTED;
  if (a.B > 65535 || a.L > (int64_t(1) << 30) || a.H > (int64_t(1) << 30) ||
      a.B * a.L * a.H * a.P > (int64_t(1) << 40))
    return CSSCAN_ERR_UNSUPPORTED;
  const size_t s = a.dtype == CSSCAN_F32 ? 4 : 2;
  if (!aligned(a.x, s) || !aligned(a.delta, s) || !aligned(a.Bm, 2 * s) || !aligned(a.Cm, 2 * s) ||
      !aligned(a.theta, s) || (a.lam && !aligned(a.lam, s)) || !aligned(a.A, 4) || !aligned(a.Dskip, 4) ||
      !aligned(a.y, 4))
    return CSSCAN_ERR_MISALIGNED;
  if (!rows || !heads) return CSSCAN_OK;
  return a.dtype == CSSCAN_F32 ? mimo_f32(a, st) : mimo_bf16(a, st);
}

int mimo_backward_impl(const MimoBwdArgs& a, cudaStream_t st) {
  if (a.mode != CSSCAN_MODE_EXP_EULER && a.mode != CSSCAN_MODE_EXP_TRAPEZOID) {
    return a.mode == CSSCAN_MODE_ZOH ? CSSCAN_ERR_UNSUPPORTED : CSSCAN_ERR_INVALID_ARG;
  }
  if (a.dtype != CSSCAN_F32 && a.dtype != CSSCAN_BF16) return CSSCAN_ERR_INVALID_ARG;
  if (a.B < 0 || a.L < 0 || a.H < 0 || a.P <= 0 || a.N <= 0) return CSSCAN_ERR_INVALID_ARG;
  // arrays with no elements may be NULL (an empty tensor has no storage)
  const bool rows = a.B > 0 && a.L > 0, heads = a.H > 0;
  if (heads && (!a.A || !a.Dskip || !a.dA || !a.dDskip)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && (!a.Bm || !a.Cm || !a.theta || !a.dBm || !a.dCm || !a.dtheta)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && heads && (!a.x || !a.delta || !a.dy || !a.dx || !a.ddelta)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && a.mode == CSSCAN_MODE_EXP_TRAPEZOID && (!a.lam || !a.dlam)) return CSSCAN_ERR_INVALID_ARG;
  if (a.N != 2 && a.N != 4 && a.N != 8 && a.N != 16 && a.N != 32) return CSSCAN_ERR_UNSUPPORTED;
  if (a.P != 1 && a.P != 2 && a.P != 4 && a.P != 8) return CSSCAN_ERR_UNSUPPORTED;
  if (a.B > 65535 || a.L > (int64_t(1) << 30) || a.H > (int64_t(1) << 30) ||
      a.B * a.L * a.H * a.P > (int64_t(1) << 40) || a.B * a.L * a.N * a.P > (int64_t(1) << 40))
    return CSSCAN_ERR_UNSUPPORTED;
  const size_t s = a.dtype == CSSCAN_F32 ? 4 : 2;
  if (!aligned(a.x, s) || !aligned(a.delta, s) || !aligned(a.Bm, 2 * s) || !aligned(a.Cm, 2 * s) ||
      !aligned(a.theta, s) || (a.lam && !aligned(a.lam, s)) || !aligned(a.A, 4) || !aligned(a.Dskip, 4) ||
      !aligned(a.dy, 4) || !aligned(a.dx, 4) || !aligned(a.ddelta, 4) || !aligned(a.dA, 4) || !aligned(a.dBm, 4) ||
      !aligned(a.dCm, 4) || !aligned(a.dtheta, 4) || (a.dlam && !aligned(a.dlam, 4)) || !aligned(a.dDskip, 4))
    return CSSCAN_ERR_MISALIGNED;
  if (!rows || !heads) {
    // no steps or no heads: every gradient is an empty sum
    if (heads) {
      CSSCAN_CUDA(cudaMemsetAsync(a.dA, 0, size_t(a.H * a.N) * 4, st));
      CSSCAN_CUDA(cudaMemsetAsync(a.dDskip, 0, size_t(a.H * a.P) * 4, st));
    }
    if (rows) {
      CSSCAN_CUDA(cudaMemsetAsync(a.dBm, 0, size_t(a.B * a.L * a.N * a.P) * 8, st));
      CSSCAN_CUDA(cudaMemsetAsync(a.dCm, 0, size_t(a.B * a.L * a.N * a.P) * 8, st));
      CSSCAN_CUDA(cudaMemsetAsync(a.dtheta, 0, size_t(a.B * a.L * a.N) * 4, st));
      if (a.mode == CSSCAN_MODE_EXP_TRAPEZOID) CSSCAN_CUDA(cudaMemsetAsync(a.dlam, 0, size_t(a.B * a.L) * 4, st));
    }
    return CSSCAN_OK;
  }
  return a.dtype == CSSCAN_F32 ? mimo_backward_f32(a, st) : mimo_backward_bf16(a, st);
}

int backward_impl(const BwdArgs& a, cudaStream_t st) {
  if (a.mode != CSSCAN_MODE_EXP_EULER && a.mode != CSSCAN_MODE_EXP_TRAPEZOID && a.mode != CSSCAN_MODE_ZOH)
    return CSSCAN_ERR_INVALID_ARG;
  if (a.dtype != CSSCAN_F32 && a.dtype != CSSCAN_BF16) return CSSCAN_ERR_INVALID_ARG;
  if (a.B < 0 || a.L < 0 || a.D < 0 || a.N <= 0) return CSSCAN_ERR_INVALID_ARG;
  // arrays with no elements may be NULL (an empty tensor has no storage)
  const bool rows = a.B > 0 && a.L > 0, chans = a.D > 0;
  if (chans && (!a.A || !a.Dskip || !a.dA || !a.dDskip)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && (!a.Bc || !a.Cc || !a.theta || !a.dBc || !a.dCc || !a.dtheta)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && chans && (!a.x || !a.delta || !a.dy || !a.dx || !a.ddelta)) return CSSCAN_ERR_INVALID_ARG;
  if (rows && a.mode == CSSCAN_MODE_EXP_TRAPEZOID && (!a.lam || !a.dlam)) return CSSCAN_ERR_INVALID_ARG;
  if (a.N != 2 && a.N != 4 && a.N != 8 && a.N != 16 && a.N != 32) return CSSCAN_ERR_UNSUPPORTED;
  if (a.B > 65535 || a.L > (int64_t(1) << 30) || a.D > (int64_t(1) << 30) ||
      a.B * a.L * a.D > (int64_t(1) << 40) || (a.D + 63) / 64 > 65535)
    return CSSCAN_ERR_UNSUPPORTED;
  const size_t s = a.dtype == CSSCAN_F32 ? 4 : 2;
  // Bc and Cc are read one complex entry (2 values) at a time
  if (!aligned(a.x, s) || !aligned(a.delta, s) || !aligned(a.Bc, 2 * s) || !aligned(a.Cc, 2 * s) || !aligned(a.theta, s) ||
      (a.lam && !aligned(a.lam, s)) || !aligned(a.A, 4) || !aligned(a.Dskip, 4) || !aligned(a.dy, 4) ||
      !aligned(a.dx, 4) || !aligned(a.ddelta, 4) || !aligned(a.dA, 4) || !aligned(a.dBc, 4) || !aligned(a.dCc, 4) ||
      !aligned(a.dtheta, 4) || (a.dlam && !aligned(a.dlam, 4)) || !aligned(a.dDskip, 4))
    return CSSCAN_ERR_MISALIGNED;
  if (a.B == 0 || a.L == 0 || a.D == 0) {
    // no steps or no channels: every gradient is an empty sum
    if (a.D > 0) {
      CSSCAN_CUDA(cudaMemsetAsync(a.dA, 0, size_t(a.D * a.N) * 4, st));
      CSSCAN_CUDA(cudaMemsetAsync(a.dDskip, 0, size_t(a.D) * 4, st));
    }
    if (a.B > 0 && a.L > 0) {
      CSSCAN_CUDA(cudaMemsetAsync(a.dBc, 0, size_t(a.B * a.L * a.N) * 8, st));
      CSSCAN_CUDA(cudaMemsetAsync(a.dCc, 0, size_t(a.B * a.L * a.N) * 8, st));
      CSSCAN_CUDA(cudaMemsetAsync(a.dtheta, 0, size_t(a.B * a.L * a.N) * 4, st));
      if (a.mode == CSSCAN_MODE_EXP_TRAPEZOID) CSSCAN_CUDA(cudaMemsetAsync(a.dlam, 0, size_t(a.B * a.L) * 4, st));
    }
    return CSSCAN_OK;
  }
  return a.dtype == CSSCAN_F32 ? backward_f32(a, st) : backward_bf16(a, st);
}

// ----------------------------------------------------------------------------- no-allocation entry
// csscan_forward_noalloc runs the same kernels with its scratch in one fixed array that is part
// of the library's device code, so it never calls cudaMalloc. Layout of the array:
// [header 256 B][flags: NOALLOC_FLAG_CAP words][the rest, laid out per call by the plan].
constexpr size_t NOALLOC_FLAG_CAP = 1 << 16;
constexpr size_t NOALLOC_REST_OFF = HDR_BYTES + NOALLOC_FLAG_CAP * 4;
static_assert(NOALLOC_REST_OFF < CSSCAN_NOALLOC_SCRATCH_BYTES, "scratch too small");

// The array's device address per (device, context): a context created after a device reset
// loads the library's device code afresh, and with it a new copy of the array.
std::mutex g_noalloc_mu;
std::map<std::pair<int, uintptr_t>, char*> g_noalloc_addr;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

int noalloc_scratch_address(int dev, char** out);   // defined after the array below

}  // namespace
}  // namespace csscan_host

// The fixed scratch of csscan_forward_noalloc. In host code this name is only a stand-in for
// the array, not a device address: kernels get the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CSSCAN_NOALLOC_SCRATCH_BYTES];

namespace csscan_host {
namespace {
// With `dev` current: the device address of the scratch array, looked up once per device and
// context.
int noalloc_scratch_address(int dev, char** out) {
  uintptr_t ctx = 0;
  if (auto fn = ctx_get_current_fn()) {
    CUcontext c = nullptr;
    if (fn(&c) == CUDA_SUCCESS) ctx = reinterpret_cast<uintptr_t>(c);
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  auto it = g_noalloc_addr.find({dev, ctx});
  if (it != g_noalloc_addr.end() && ctx != 0) {
    *out = it->second;
    return CSSCAN_OK;
  }
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || ptr == nullptr) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
  if (ctx != 0) g_noalloc_addr[{dev, ctx}] = static_cast<char*>(ptr);
  *out = static_cast<char*>(ptr);
  return CSSCAN_OK;
}
}  // namespace
}  // namespace csscan_host

using namespace csscan_host;

extern "C" {

int csscan_forward(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                   const void* theta, const void* lambda, const float* Dskip, float* y, int64_t B, int64_t L,
                   int64_t D, int64_t N, int mode, int dtype, cudaStream_t stream) {
  return csscan_forward_ex(x, delta, A, Bc, Cc, theta, lambda, Dskip, y, B, L, D, N, mode, dtype, nullptr, stream);
}

int csscan_forward_ex(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                      const void* theta, const void* lambda, const float* Dskip, float* y, int64_t B, int64_t L,
                      int64_t D, int64_t N, int mode, int dtype, const csscan_options_t* opts, cudaStream_t stream) {
  Args a{x, delta, Bc, Cc, theta, lambda, A, Dskip, y, nullptr, nullptr, nullptr, nullptr, B, L, D, N, mode, dtype};
  return forward_impl(a, opts, stream, nullptr);
}

int csscan_forward_state(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                         const void* theta, const void* lambda, const float* Dskip, float* y, const float* h0,
                         const void* x_prev, const void* Bc_prev, float* h_last, int64_t B, int64_t L, int64_t D,
                         int64_t N, int mode, int dtype, cudaStream_t stream) {
  Args a{x, delta, Bc, Cc, theta, lambda, A, Dskip, y, h0, h_last, x_prev, Bc_prev, B, L, D, N, mode, dtype};
  if (mode != CSSCAN_MODE_EXP_TRAPEZOID) {   // the halo only enters the trapezoid rule: not checked
    a.x_prev = nullptr;
    a.Bc_prev = nullptr;
  }
  return forward_impl(a, nullptr, stream, nullptr);
}

int csscan_decode_step(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                       const void* theta, const void* lambda, const float* Dskip, float* y, float* h,
                       const void* x_prev, const void* Bc_prev, int64_t B, int64_t D, int64_t N, int mode, int dtype,
                       cudaStream_t stream) {
  return decode_impl(x, delta, A, Bc, Cc, theta, lambda, Dskip, y, h, x_prev, Bc_prev, B, D, N, mode, dtype, stream);
}

int csscan_forward_noalloc(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                           const void* theta, const void* lambda, const float* Dskip, float* y, int64_t B, int64_t L,
                           int64_t D, int64_t N, int mode, int dtype, uint32_t* device_status, cudaStream_t stream) {
  Args a{x, delta, Bc, Cc, theta, lambda, A, Dskip, y, nullptr, nullptr, nullptr, nullptr, B, L, D, N, mode, dtype};
  const csscan_options_t o = default_options();
  int rc = validate(a, o);
  if (rc != CSSCAN_OK) return rc;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) % 4) != 0) return CSSCAN_ERR_MISALIGNED;
  if (a.B == 0 || a.L == 0 || a.D == 0) return CSSCAN_OK;
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  char* base = nullptr;
  rc = noalloc_scratch_address(dev, &base);
  if (rc != CSSCAN_OK) return rc;
  FixedScratch fx{reinterpret_cast<uint32_t*>(base), reinterpret_cast<uint32_t*>(base + HDR_BYTES),
                  base + NOALLOC_REST_OFF, NOALLOC_FLAG_CAP, CSSCAN_NOALLOC_SCRATCH_BYTES - NOALLOC_REST_OFF};
  rc = forward_impl(a, &o, stream, &fx);
  if (rc != CSSCAN_OK) return rc;
  if (device_status)
    CSSCAN_CUDA(cudaMemcpyAsync(device_status, fx.hdr + H_ERROR, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream));
  return CSSCAN_OK;
}

int csscan_forward_mimo(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm,
                        const void* theta, const void* lambda, const float* Dskip, float* y, int64_t B, int64_t L,
                        int64_t H, int64_t P, int64_t N, int mode, int dtype, cudaStream_t stream) {
  MimoArgs a{x, delta, Bm, Cm, theta, lambda, A, Dskip, y, B, L, H, P, N, mode, dtype};
  return mimo_impl(a, stream);
}

int csscan_backward(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                    const void* theta, const void* lambda, const float* Dskip, const float* dy, float* dx,
                    float* ddelta, float* dA, float* dBc, float* dCc, float* dtheta, float* dlambda, float* dDskip,
                    int64_t B, int64_t L, int64_t D, int64_t N, int mode, int dtype, cudaStream_t stream) {
  BwdArgs a{x, delta, Bc, Cc, theta, lambda, A, Dskip, dy, dx, ddelta, dA, dBc, dCc, dtheta, dlambda, dDskip,
            B, L, D, N, mode, dtype};
  return backward_impl(a, stream);
}

int csscan_backward_mimo(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm,
                         const void* theta, const void* lambda, const float* Dskip, const float* dy, float* dx,
                         float* ddelta, float* dA, float* dBm, float* dCm, float* dtheta, float* dlambda,
                         float* dDskip, int64_t B, int64_t L, int64_t H, int64_t P, int64_t N, int mode, int dtype,
                         cudaStream_t stream) {
  MimoBwdArgs a{x, delta, Bm, Cm, theta, lambda, A, Dskip, dy, dx, ddelta, dA, dBm, dCm, dtheta, dlambda, dDskip,
                B, L, H, P, N, mode, dtype};
  return mimo_backward_impl(a, stream);
}

int csscan_get_device_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    auto it = g_ws.find({dev, reinterpret_cast<uintptr_t>(stream)});
    if (it == g_ws.end() || it->second.base == nullptr) return CSSCAN_OK;
    base = it->second.base;
  }
  uint32_t hdr[8];
  CSSCAN_CUDA(cudaMemcpy(hdr, base, sizeof(hdr), cudaMemcpyDeviceToHost));
  if (hdr[H_ERROR] == 0) return CSSCAN_OK;
  CSSCAN_CUDA(cudaMemset(static_cast<uint32_t*>(base) + H_ERROR, 0, 3 * sizeof(uint32_t)));
  if (hdr[H_ERROR] & ERR_BOUNDS) return CSSCAN_ERR_BOUNDS;
  if (hdr[H_ERROR] & ERR_PIPELINE) return CSSCAN_ERR_PIPELINE_TIMEOUT;
  return CSSCAN_ERR_LOOKBACK_TIMEOUT;
}

const char* csscan_status_string(int status) {
  switch (status) {
    case CSSCAN_OK: return "ok";
    case CSSCAN_ERR_INVALID_ARG: return "invalid argument";
    case CSSCAN_ERR_MISALIGNED: return "misaligned pointer or row stride (x/delta need 16-byte alignment and D*sizeof(dtype) % 16 == 0)";
    case CSSCAN_ERR_UNSUPPORTED:
      return "unsupported size or mode for this entry point (N in {2, 4, 8, 16, 32, 64}; N <= 32 for the backward "
             "and for the MIMO scan, which does not take the zero-order hold)";
    case CSSCAN_ERR_CUDA: return g_last_cuda_error[0] ? g_last_cuda_error : "CUDA error";
    case CSSCAN_ERR_LOOKBACK_TIMEOUT: return "a chunk's carry wait timed out on the device";
    case CSSCAN_ERR_PIPELINE_TIMEOUT: return "a tile copy did not arrive within its limit on the device";
    case CSSCAN_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than csscan_forward_noalloc's fixed array (CSSCAN_NOALLOC_SCRATCH_BYTES) holds; "
             "use csscan_forward";
    case CSSCAN_ERR_BOUNDS:
      return "a kernel index fell outside its array on the device (bounds-checked build); the outputs are not valid";
    default: return "unknown status";
  }
}

int csscan_release_workspace(void) {
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    g_noalloc_addr.clear();   // looked up again on the next no-allocation call
  }
  std::lock_guard<std::mutex> lk(g_ws_mu);
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) cur = -1;
  int rc = CSSCAN_OK;
  for (auto& kv : g_ws) {
    if (!kv.second.base) continue;
    if (cudaSetDevice(kv.first.first) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaFree(kv.second.base) != cudaSuccess)
      rc = CSSCAN_ERR_CUDA;
  }
  g_ws.clear();
  if (cur >= 0) cudaSetDevice(cur);
  return rc;
}

}  // extern "C"
