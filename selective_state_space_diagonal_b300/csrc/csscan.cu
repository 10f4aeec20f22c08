// csscan.cu -- host side of the C ABI declared in include/csscan.h: argument checks,
// per-(device, stream) workspace, tile-copy descriptors, tiling choice and the launches of
// the rotation-table kernel and the scan kernel (scan_kernels.cuh).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "csscan.h"
#include "scan_kernels.cuh"

using namespace csscan;

namespace {

thread_local char g_last_cuda_error[256] = "";

int cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", what, cudaGetErrorString(e));
  return CSSCAN_ERR_CUDA;
}
#define CSSCAN_CUDA(call)                             \
  do {                                                \
    cudaError_t e_ = (call);                          \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

// ----------------------------------------------------------------------------- descriptors
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

// 3-D tiled map, dims innermost first, strides in bytes for dims 1 and 2; OOB reads give 0.
bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t n0, uint64_t n1, uint64_t n2,
              uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {n0, n1, n2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ----------------------------------------------------------------------------- workspace
// Per (device, stream): [header 256 B][flags: flag_cap words][the rest, laid out per call].
// The flags region only grows through a full reallocation, which zeroes it; records from
// earlier calls carry an older epoch and are never mistaken for this call's.
struct WsEntry {
  void* base = nullptr;
  size_t bytes = 0;
  size_t flag_cap = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, WsEntry> g_ws;

constexpr size_t HDR_BYTES = 256;
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int get_workspace(int dev, cudaStream_t st, size_t units, size_t rest_bytes, WsEntry* out) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  WsEntry& e = g_ws[{dev, reinterpret_cast<uintptr_t>(st)}];
  const size_t need_cap = std::max(units, e.flag_cap);
  const size_t need = HDR_BYTES + align_up(need_cap * 4, 256) + rest_bytes;
  if (e.base == nullptr || need_cap > e.flag_cap || need > e.bytes) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CSSCAN_CUDA(cudaStreamIsCapturing(st, &cs));
    if (cs != cudaStreamCaptureStatusNone) {
      std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                    "workspace must grow, which cannot happen during stream capture; call once before capturing");
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

// ----------------------------------------------------------------------------- dispatch
struct Args {
  const void *x, *delta, *Bc, *Cc, *theta, *lam;
  const float *A, *Dskip;
  float* y;
  const float* h0;
  float* h_last;
  const void *x_prev, *Bc_prev;
  int64_t B, L, D, N;
  int mode, dtype;
};

struct DeviceInfo {
  int nsm = 0;
};

template <int N, int NG, typename Tin, int MODE>
int launch(const Args& a, const csscan_options_t& o, cudaStream_t st) {
  using SL = StageLayout<N, NG, Tin, MODE>;
  constexpr int DT = SL::DT;
  auto kern = scan_kernel<N, NG, Tin, MODE>;
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  static std::mutex mu;
  static std::map<int, int> occ_cache;
  int nsm = 0, occ = 0;
  CSSCAN_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = occ_cache.find(dev);
    if (it == occ_cache.end()) {
      CSSCAN_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SL::SMEM));
      CSSCAN_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, THREADS, SL::SMEM));
      occ_cache[dev] = occ;
    } else {
      occ = it->second;
    }
  }
  const int64_t conc = int64_t(nsm) * std::max(occ, 1);
  const int64_t n_dtiles = (a.D + DT - 1) / DT;
  const int64_t n_tiles = a.B * n_dtiles;
  const int64_t S = (a.L + T_SUB - 1) / T_SUB;

  int carry = o.carry;
  if (carry == 0) carry = (n_tiles >= conc) ? CARRY_SERIAL : CARRY_DECOUPLED;
  int64_t TC = o.chunk_len;
  if (TC == 0) {
    const int64_t want = carry == CARRY_SERIAL ? (4 * conc + n_tiles - 1) / n_tiles : (2 * conc + n_tiles - 1) / n_tiles;
    const int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(S, want));
    TC = (S + chunks - 1) / chunks * T_SUB;
  }
  const int64_t n_chunks = (a.L + TC - 1) / TC;
  const int64_t n_units = n_tiles * n_chunks;
  if (n_units > (int64_t(1) << 30) || S > (int64_t(1) << 30)) return CSSCAN_ERR_UNSUPPORTED;

  // workspace layout after the header and flags
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t r = off; off = align_up(off + bytes, 256); return r; };
  const size_t o_inc = take(size_t(n_units) * DT * N * 8);
  const size_t o_agg = carry == CARRY_DECOUPLED ? take(size_t(n_units) * DT * N * 8) : 0;
  const size_t o_sdt = carry == CARRY_DECOUPLED ? take(size_t(n_units) * DT * 4) : 0;
  const size_t o_crot = carry == CARRY_DECOUPLED ? take(size_t(n_units) * N * 8) : 0;
  const size_t o_tab = take(size_t(a.B) * a.L * 4 * N * 4);
  const size_t o_aux = MODE == 1 ? take(size_t(a.B) * a.L * 16) : 0;
  const size_t o_rot = take(size_t(a.B) * S * 2 * N * 4);
  WsEntry ws;
  int rc = get_workspace(dev, st, size_t(n_units), off, &ws);
  if (rc != CSSCAN_OK) return rc;
  char* rest = static_cast<char*>(ws.base) + HDR_BYTES + align_up(ws.flag_cap * 4, 256);

  TableParams tp;
  tp.Bc = a.Bc;
  tp.Cc = a.Cc;
  tp.theta = a.theta;
  tp.lam = a.lam;
  tp.tab = reinterpret_cast<float*>(rest + o_tab);
  tp.aux = MODE == 1 ? reinterpret_cast<float*>(rest + o_aux) : nullptr;
  tp.rot = reinterpret_cast<float*>(rest + o_rot);
  tp.B = int(a.B);
  tp.L = int(a.L);
  tp.N = N;
  tp.S = int(S);

  ScanParams sp;
  std::memset(&sp, 0, sizeof(sp));
  const CUtensorMapDataType tin = sizeof(Tin) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t s_in = sizeof(Tin);
  bool ok = make_map(&sp.tm_x, tin, a.x, a.D, a.L, a.B, a.D * s_in, a.L * a.D * s_in, DT, T_SUB, 1) &&
            make_map(&sp.tm_dt, tin, a.delta, a.D, a.L, a.B, a.D * s_in, a.L * a.D * s_in, DT, T_SUB + 1, 1) &&
            make_map(&sp.tm_tab, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.tab, 4 * N, a.L, a.B, 16 * N, a.L * 16 * N, 4 * N,
                     T_SUB, 1) &&
            make_map(&sp.tm_rot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.rot, 2 * N, S, a.B, 8 * N, S * 8 * N, 2 * N, 1, 1);
  if (ok && MODE == 1)
    ok = make_map(&sp.tm_aux, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.aux, 4, a.L, a.B, 16, a.L * 16, 4, T_SUB, 1);
  if (!ok) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed or unavailable");
    return CSSCAN_ERR_CUDA;
  }
  sp.A = a.A;
  sp.Dskip = a.Dskip;
  sp.y = a.y;
  sp.x = a.x;
  sp.dt = a.delta;
  sp.Bc = a.Bc;
  sp.lam = a.lam;
  sp.h0 = a.h0;
  sp.h_last = a.h_last;
  sp.x_prev = a.x_prev;
  sp.Bc_prev = a.Bc_prev;
  sp.ws.hdr = static_cast<uint32_t*>(ws.base);
  sp.ws.flags = reinterpret_cast<uint32_t*>(static_cast<char*>(ws.base) + HDR_BYTES);
  sp.ws.inc = reinterpret_cast<float2*>(rest + o_inc);
  sp.ws.agg = carry == CARRY_DECOUPLED ? reinterpret_cast<float2*>(rest + o_agg) : nullptr;
  sp.ws.sdt = carry == CARRY_DECOUPLED ? reinterpret_cast<float*>(rest + o_sdt) : nullptr;
  sp.ws.crot = carry == CARRY_DECOUPLED ? reinterpret_cast<float2*>(rest + o_crot) : nullptr;
  sp.B = int(a.B);
  sp.L = int(a.L);
  sp.D = int(a.D);
  sp.N = N;
  sp.S = int(S);
  sp.n_dtiles = int(n_dtiles);
  sp.n_tiles = int(n_tiles);
  sp.TC = int(TC);
  sp.n_chunks = int(n_chunks);
  sp.n_units = int(n_units);
  sp.carry = carry;
  sp.silent_chunk = o.silent_chunk;
  sp.poll_limit = o.poll_limit > 0 ? o.poll_limit : (int64_t(1) << 22);

  const int64_t table_threads = a.B * S * N;
  table_kernel<Tin, MODE><<<unsigned((table_threads + 255) / 256), 256, 0, st>>>(tp);
  CSSCAN_CUDA(cudaGetLastError());
  if (o.scan_begin) CSSCAN_CUDA(cudaEventRecord(o.scan_begin, st));
  kern<<<unsigned(n_units), THREADS, SL::SMEM, st>>>(sp);
  CSSCAN_CUDA(cudaGetLastError());
  if (o.scan_end) CSSCAN_CUDA(cudaEventRecord(o.scan_end, st));
  return CSSCAN_OK;
}

template <typename Tin, int MODE>
int dispatch_n(const Args& a, const csscan_options_t& o, cudaStream_t st) {
  switch (a.N) {
    case 2: return launch<2, 1, Tin, MODE>(a, o, st);
    case 4: return launch<4, 1, Tin, MODE>(a, o, st);
    case 8: return launch<8, 1, Tin, MODE>(a, o, st);
    case 16: return launch<16, 1, Tin, MODE>(a, o, st);
    case 32: return launch<32, 2, Tin, MODE>(a, o, st);
    case 64: return launch<64, 4, Tin, MODE>(a, o, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int validate(const Args& a, const csscan_options_t& o) {
  if (a.mode != CSSCAN_MODE_EXP_EULER && a.mode != CSSCAN_MODE_EXP_TRAPEZOID) return CSSCAN_ERR_INVALID_ARG;
  if (a.dtype != CSSCAN_F32 && a.dtype != CSSCAN_BF16) return CSSCAN_ERR_INVALID_ARG;
  if (a.B < 0 || a.L < 0 || a.D < 0 || a.N <= 0) return CSSCAN_ERR_INVALID_ARG;
  if (!a.x || !a.delta || !a.A || !a.Bc || !a.Cc || !a.theta || !a.Dskip || !a.y) return CSSCAN_ERR_INVALID_ARG;
  if (a.mode == CSSCAN_MODE_EXP_TRAPEZOID && !a.lam) return CSSCAN_ERR_INVALID_ARG;
  if ((a.x_prev == nullptr) != (a.Bc_prev == nullptr)) return CSSCAN_ERR_INVALID_ARG;
  if (o.rows_per_cta != 0 || o.carry < 0 || o.carry > 2 || o.chunk_len < 0 || (o.chunk_len % T_SUB) != 0 ||
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

int forward_impl(const Args& a, const csscan_options_t* opts, cudaStream_t st) {
  csscan_options_t o;
  std::memset(&o, 0, sizeof(o));
  o.silent_chunk = -1;
  if (opts) o = *opts;
  int rc = validate(a, o);
  if (rc != CSSCAN_OK) return rc;
  if (a.B == 0 || a.L == 0 || a.D == 0) return CSSCAN_OK;
  if (a.dtype == CSSCAN_F32)
    return a.mode == 0 ? dispatch_n<float, 0>(a, o, st) : dispatch_n<float, 1>(a, o, st);
  return a.mode == 0 ? dispatch_n<uint16_t, 0>(a, o, st) : dispatch_n<uint16_t, 1>(a, o, st);
}


// ----------------------------------------------------------------------------- no-allocation entry
// csscan_forward_noalloc runs the same two kernels with its scratch in one fixed array that
// is part of the library's device code, so it never calls cudaMalloc. Layout of the array:
// [header 256 B][flags: NOALLOC_FLAG_CAP words][the rest, laid out per call as in launch()].
constexpr size_t NOALLOC_FLAG_CAP = 1 << 16;
constexpr size_t NOALLOC_REST_OFF = HDR_BYTES + NOALLOC_FLAG_CAP * 4;
static_assert(NOALLOC_REST_OFF < CSSCAN_NOALLOC_SCRATCH_BYTES, "scratch too small");

std::mutex g_noalloc_mu;
std::map<int, char*> g_noalloc_addr;   // device -> device address of the scratch array

int noalloc_scratch_address(int dev, char** out);   // defined after the array below

template <int N, int NG, typename Tin, int MODE>
int launch_noalloc(const Args& a, uint32_t* device_status, cudaStream_t st) {
  using SL = StageLayout<N, NG, Tin, MODE>;
  constexpr int DT = SL::DT;
  auto kern = scan_kernel<N, NG, Tin, MODE>;
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  static std::mutex mu;
  static std::map<int, int> occ_cache;
  int nsm = 0, occ = 0;
  CSSCAN_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = occ_cache.find(dev);
    if (it == occ_cache.end()) {
      CSSCAN_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SL::SMEM));
      CSSCAN_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, THREADS, SL::SMEM));
      occ_cache[dev] = occ;
    } else {
      occ = it->second;
    }
  }
  const int64_t conc = int64_t(nsm) * std::max(occ, 1);
  const int64_t n_dtiles = (a.D + DT - 1) / DT;
  const int64_t n_tiles = a.B * n_dtiles;
  const int64_t S = (a.L + T_SUB - 1) / T_SUB;
  const int carry = (n_tiles >= conc) ? CARRY_SERIAL : CARRY_DECOUPLED;
  const int64_t want = carry == CARRY_SERIAL ? (4 * conc + n_tiles - 1) / n_tiles : (2 * conc + n_tiles - 1) / n_tiles;
  const int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(S, want));
  const int64_t TC = (S + chunks - 1) / chunks * T_SUB;
  const int64_t n_chunks = (a.L + TC - 1) / TC;
  const int64_t n_units = n_tiles * n_chunks;

  size_t off = 0;
  auto take = [&](size_t bytes) { size_t r = off; off = align_up(off + bytes, 256); return r; };
  const size_t o_inc = take(size_t(n_units) * DT * N * 8);
  const size_t o_agg = carry == CARRY_DECOUPLED ? take(size_t(n_units) * DT * N * 8) : 0;
  const size_t o_sdt = carry == CARRY_DECOUPLED ? take(size_t(n_units) * DT * 4) : 0;
  const size_t o_crot = carry == CARRY_DECOUPLED ? take(size_t(n_units) * N * 8) : 0;
  const size_t o_tab = take(size_t(a.B) * a.L * 4 * N * 4);
  const size_t o_aux = MODE == 1 ? take(size_t(a.B) * a.L * 16) : 0;
  const size_t o_rot = take(size_t(a.B) * S * 2 * N * 4);
  if (size_t(n_units) > NOALLOC_FLAG_CAP || off > CSSCAN_NOALLOC_SCRATCH_BYTES - NOALLOC_REST_OFF)
    return CSSCAN_ERR_SCRATCH_LIMIT;

  char* base = nullptr;
  int rc = noalloc_scratch_address(dev, &base);
  if (rc != CSSCAN_OK) return rc;
  char* rest = base + NOALLOC_REST_OFF;
  uint32_t* hdr = reinterpret_cast<uint32_t*>(base);
  // the ticket and finished-block counters and the status words must start at zero; the
  // epoch (word 0) keeps counting so that flags left by earlier calls are never current
  CSSCAN_CUDA(cudaMemsetAsync(hdr + H_TICKET, 0, 5 * sizeof(uint32_t), st));

  TableParams tp;
  tp.Bc = a.Bc;
  tp.Cc = a.Cc;
  tp.theta = a.theta;
  tp.lam = a.lam;
  tp.tab = reinterpret_cast<float*>(rest + o_tab);
  tp.aux = MODE == 1 ? reinterpret_cast<float*>(rest + o_aux) : nullptr;
  tp.rot = reinterpret_cast<float*>(rest + o_rot);
  tp.B = int(a.B);
  tp.L = int(a.L);
  tp.N = N;
  tp.S = int(S);

  ScanParams sp;
  std::memset(&sp, 0, sizeof(sp));
  const CUtensorMapDataType tin = sizeof(Tin) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t s_in = sizeof(Tin);
  bool ok = make_map(&sp.tm_x, tin, a.x, a.D, a.L, a.B, a.D * s_in, a.L * a.D * s_in, DT, T_SUB, 1) &&
            make_map(&sp.tm_dt, tin, a.delta, a.D, a.L, a.B, a.D * s_in, a.L * a.D * s_in, DT, T_SUB + 1, 1) &&
            make_map(&sp.tm_tab, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.tab, 4 * N, a.L, a.B, 16 * N, a.L * 16 * N, 4 * N,
                     T_SUB, 1) &&
            make_map(&sp.tm_rot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.rot, 2 * N, S, a.B, 8 * N, S * 8 * N, 2 * N, 1, 1);
  if (ok && MODE == 1)
    ok = make_map(&sp.tm_aux, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.aux, 4, a.L, a.B, 16, a.L * 16, 4, T_SUB, 1);
  if (!ok) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed or unavailable");
    return CSSCAN_ERR_CUDA;
  }
  sp.A = a.A;
  sp.Dskip = a.Dskip;
  sp.y = a.y;
  sp.x = a.x;
  sp.dt = a.delta;
  sp.Bc = a.Bc;
  sp.lam = a.lam;
  sp.ws.hdr = hdr;
  sp.ws.flags = reinterpret_cast<uint32_t*>(base + HDR_BYTES);
  sp.ws.inc = reinterpret_cast<float2*>(rest + o_inc);
  sp.ws.agg = carry == CARRY_DECOUPLED ? reinterpret_cast<float2*>(rest + o_agg) : nullptr;
  sp.ws.sdt = carry == CARRY_DECOUPLED ? reinterpret_cast<float*>(rest + o_sdt) : nullptr;
  sp.ws.crot = carry == CARRY_DECOUPLED ? reinterpret_cast<float2*>(rest + o_crot) : nullptr;
  sp.B = int(a.B);
  sp.L = int(a.L);
  sp.D = int(a.D);
  sp.N = N;
  sp.S = int(S);
  sp.n_dtiles = int(n_dtiles);
  sp.n_tiles = int(n_tiles);
  sp.TC = int(TC);
  sp.n_chunks = int(n_chunks);
  sp.n_units = int(n_units);
  sp.carry = carry;
  sp.silent_chunk = -1;
  sp.poll_limit = int64_t(1) << 22;

  const int64_t table_threads = a.B * S * N;
  table_kernel<Tin, MODE><<<unsigned((table_threads + 255) / 256), 256, 0, st>>>(tp);
  CSSCAN_CUDA(cudaGetLastError());
  kern<<<unsigned(n_units), THREADS, SL::SMEM, st>>>(sp);
  CSSCAN_CUDA(cudaGetLastError());
  if (device_status)
    CSSCAN_CUDA(cudaMemcpyAsync(device_status, hdr + H_ERROR, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st));
  return CSSCAN_OK;
}

template <typename Tin, int MODE>
int dispatch_noalloc(const Args& a, uint32_t* device_status, cudaStream_t st) {
  switch (a.N) {
    case 2: return launch_noalloc<2, 1, Tin, MODE>(a, device_status, st);
    case 4: return launch_noalloc<4, 1, Tin, MODE>(a, device_status, st);
    case 8: return launch_noalloc<8, 1, Tin, MODE>(a, device_status, st);
    case 16: return launch_noalloc<16, 1, Tin, MODE>(a, device_status, st);
    case 32: return launch_noalloc<32, 2, Tin, MODE>(a, device_status, st);
    case 64: return launch_noalloc<64, 4, Tin, MODE>(a, device_status, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

}  // namespace

// The fixed scratch of csscan_forward_noalloc. In host code this name is only a stand-in for
// the array, not a device address: kernels get the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CSSCAN_NOALLOC_SCRATCH_BYTES];

namespace {
// Once per device, with that device current: the device address of the scratch array.
int noalloc_scratch_address(int dev, char** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  auto it = g_noalloc_addr.find(dev);
  if (it != g_noalloc_addr.end()) {
    *out = it->second;
    return CSSCAN_OK;
  }
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || ptr == nullptr) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
  g_noalloc_addr[dev] = static_cast<char*>(ptr);
  *out = static_cast<char*>(ptr);
  return CSSCAN_OK;
}
}  // namespace

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
  return forward_impl(a, opts, stream);
}

int csscan_forward_noalloc(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                           const void* theta, const void* lambda, const float* Dskip, float* y, int64_t B, int64_t L,
                           int64_t D, int64_t N, int mode, int dtype, uint32_t* device_status, cudaStream_t stream) {
  Args a{x, delta, Bc, Cc, theta, lambda, A, Dskip, y, nullptr, nullptr, nullptr, nullptr, B, L, D, N, mode, dtype};
  csscan_options_t o;
  std::memset(&o, 0, sizeof(o));
  o.silent_chunk = -1;
  int rc = validate(a, o);
  if (rc != CSSCAN_OK) return rc;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) % 4) != 0) return CSSCAN_ERR_MISALIGNED;
  if (a.B == 0 || a.L == 0 || a.D == 0) return CSSCAN_OK;
  if (a.dtype == CSSCAN_F32)
    return a.mode == 0 ? dispatch_noalloc<float, 0>(a, device_status, stream)
                       : dispatch_noalloc<float, 1>(a, device_status, stream);
  return a.mode == 0 ? dispatch_noalloc<uint16_t, 0>(a, device_status, stream)
                     : dispatch_noalloc<uint16_t, 1>(a, device_status, stream);
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
  if (hdr[H_ERROR] & ERR_PIPELINE) return CSSCAN_ERR_PIPELINE_TIMEOUT;
  return CSSCAN_ERR_LOOKBACK_TIMEOUT;
}

const char* csscan_status_string(int status) {
  switch (status) {
    case CSSCAN_OK: return "ok";
    case CSSCAN_ERR_INVALID_ARG: return "invalid argument";
    case CSSCAN_ERR_MISALIGNED: return "misaligned pointer or row stride (x/delta need 16-byte alignment and D*sizeof(dtype) % 16 == 0)";
    case CSSCAN_ERR_UNSUPPORTED: return "unsupported size (N must be 2, 4, 8, 16, 32 or 64)";
    case CSSCAN_ERR_CUDA: return g_last_cuda_error[0] ? g_last_cuda_error : "CUDA error";
    case CSSCAN_ERR_LOOKBACK_TIMEOUT: return "a chunk's carry wait timed out on the device";
    case CSSCAN_ERR_PIPELINE_TIMEOUT: return "a tile copy did not arrive within its limit on the device";
    case CSSCAN_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than csscan_forward_noalloc's fixed array (CSSCAN_NOALLOC_SCRATCH_BYTES) holds; "
             "use csscan_forward";
    default: return "unknown status";
  }
}

int csscan_release_workspace(void) {
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
