// csscan.cu -- host side of the C ABI declared in include/csscan.h: argument checks,
// launch planning (block width, sequence chunks, shared-memory ring), the per-(device,
// stream) workspace, tile-copy descriptors, and the launches of the rotation-table kernel
// and the scan kernel (scan_kernels.cuh; every forward mode, the zero-order hold included),
// the MIMO scan (mimo_kernels.cuh), the decode step (decode_kernel.cuh) and the backward pass
// (backward_kernels.cuh).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "csscan.h"
#include "backward_kernels.cuh"
#include "decode_kernel.cuh"
#include "mimo_kernels.cuh"
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

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
// A 1-D launch of `threads` threads in blocks of 256 stays within the grid's x limit.
bool grid_fits(long long threads) { return (threads + 255) / 256 <= 0x7fffffffLL; }
constexpr size_t HDR_BYTES = 256;

// ----------------------------------------------------------------------------- arguments
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

// ----------------------------------------------------------------------------- launch plan
// Everything a launch needs that follows from the sizes, the options and the device: sequence
// chunks and carry kind, and the workspace layout (byte offsets into the region after the
// header and the flag words). The block shape and its shared-memory ring are compile-time
// properties of the kernel (Tile, Stage in scan_kernels.cuh).
struct Plan {
  int DT = 0, n_dtiles = 0, n_tiles = 0, TC = 0, n_chunks = 0, n_units = 0, carry = 0, smem = 0;
  int64_t S = 0;
  size_t o_inc = 0, o_agg = 0, o_sdt = 0, o_crot = 0, o_tab = 0, o_aux = 0, o_rot = 0, rest_bytes = 0;
};

constexpr int MAX_DYN_SMEM = 160 * 1024;         // opt-in dynamic shared memory per block
// The MIMO path and the backward's gradient pass run one thread per (row, state) sequentially
// over time; below this many such threads per SM they also split the sequence into time chunks.
constexpr int64_t SEQ_THREADS_PER_SM = 4096;
constexpr int RESIDENT_WARPS_PER_SM = 8;         // target of the automatic chunking

// Blocks of `threads` threads and `smem` dynamic bytes resident per SM (cached per device).
template <int N, typename Tin, int MODE, int CARRY>
int occupancy(int dev, int threads, int smem, int* out) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  static std::map<int, bool> attr_set;
  std::lock_guard<std::mutex> lk(mu);
  auto kern = scan_kernel<N, Tin, MODE, CARRY>;
  if (!attr_set[dev]) {
    CSSCAN_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_DYN_SMEM));
    attr_set[dev] = true;
  }
  auto key = std::make_tuple(dev, threads, smem);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return CSSCAN_OK;
  }
  int occ = 0;
  CSSCAN_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem));
  cache[key] = occ;
  *out = occ;
  return CSSCAN_OK;
}

template <int N, typename Tin, int MODE>
int occupancy_for(int carry, int dev, int threads, int smem, int* out) {
  if (carry == CARRY_SERIAL) return occupancy<N, Tin, MODE, CARRY_SERIAL>(dev, threads, smem, out);
  if (carry == CARRY_DECOUPLED) return occupancy<N, Tin, MODE, CARRY_DECOUPLED>(dev, threads, smem, out);
  return occupancy<N, Tin, MODE, CARRY_NONE>(dev, threads, smem, out);
}

// Launch plan. Blocks are 4 warps wide (one warp per SM sub-partition, so that the warps of a
// block, which meet at a barrier once per sub-chunk, progress at the same rate). Rows with
// enough parallelism are split into a few serial-carry chunks, chosen so that the chunk-units
// fill the block slots in nearly whole waves; rows with too little parallelism are split into
// as many decoupled chunks as fill the GPU.
template <int N, typename Tin, int MODE>
int make_plan(const Args& a, const csscan_options_t& o, int dev, Plan* pl) {
  using TL = Tile<N>;
  using SG = Stage<N, Tin, MODE>;
  static_assert(SG::SMEM <= MAX_DYN_SMEM, "stage ring too large");
  int nsm = 0;
  CSSCAN_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  const int64_t S = (a.L + T_SUB - 1) / T_SUB;
  const int64_t target = int64_t(nsm) * RESIDENT_WARPS_PER_SM;
  const int w = WARPS;
  const int DT = TL::DT;
  const int smem = SG::SMEM;
  const int64_t n_dtiles = (a.D + DT - 1) / DT;
  const int64_t tiles = a.B * n_dtiles;

  int carry = o.carry;
  int64_t TC = o.chunk_len;
  if (TC == 0) {
    int64_t chunks = 1;
    // Measured on B300: the aggregate pass of decoupled chunks costs more than the extra
    // parallelism returns unless the rows alone would leave most SMs idle.
    const bool rich = 4 * tiles * w >= 3 * target;
    const bool starved = 2 * tiles < nsm;
    if (carry == CARRY_SERIAL || (carry == 0 && rich)) {
      // serial chunks: each block runs at its own pace, so the time is about
      // (waves of chunk-units) x (chunk length); pick the chunk count that minimises it, with
      // ~1 % per extra chunk for the per-unit start-up
      int occ = 0;
      int rc = occupancy_for<N, Tin, MODE>(CARRY_SERIAL, dev, w * 32, smem, &occ);
      if (rc != CSSCAN_OK) return rc;
      const int64_t slots = int64_t(nsm) * std::max(occ, 1);
      double best_t = 1e30;
      for (int64_t C = 1; C <= std::min<int64_t>(S, 16); ++C) {
        const int64_t waves = (tiles * C + slots - 1) / slots;
        const double t = double(waves) / double(C) * (1.0 + 0.01 * double(C - 1));
        if (t < best_t - 1e-12) { best_t = t; chunks = C; }
      }
      if (carry == 0) carry = CARRY_SERIAL;
    } else if (carry == CARRY_DECOUPLED || (carry == 0 && starved)) {
      // decoupled chunks: as many as fill every block slot once
      int occ = 0;
      int rc = occupancy_for<N, Tin, MODE>(CARRY_DECOUPLED, dev, w * 32, smem, &occ);
      if (rc != CSSCAN_OK) return rc;
      const int64_t slots = int64_t(nsm) * std::max(occ, 1);
      chunks = std::max<int64_t>(1, std::min<int64_t>(S, slots / tiles));
    }
    TC = (S + chunks - 1) / chunks * T_SUB;
  }
  const int64_t n_chunks = (a.L + TC - 1) / TC;
  if (n_chunks == 1) carry = CARRY_NONE;
  else if (carry == 0) carry = CARRY_DECOUPLED;
  const int64_t n_units = tiles * n_chunks;
  if (n_units > (int64_t(1) << 30) || S > (int64_t(1) << 30)) return CSSCAN_ERR_UNSUPPORTED;
  int occ = 0;
  int rc = occupancy_for<N, Tin, MODE>(carry, dev, w * 32, smem, &occ);
  if (rc != CSSCAN_OK) return rc;
  if (occ < 1) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "scan block does not fit on this device");
    return CSSCAN_ERR_CUDA;
  }
  pl->DT = DT;
  pl->n_dtiles = int(n_dtiles);
  pl->n_tiles = int(tiles);
  pl->TC = int(TC);
  pl->n_chunks = int(n_chunks);
  pl->n_units = int(n_units);
  pl->carry = carry;
  pl->S = S;
  pl->smem = smem;

  // workspace layout after the header and the flags
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t r = off; off = align_up(off + bytes, 256); return r; };
  pl->o_inc = carry != CARRY_NONE ? take(size_t(n_units) * DT * N * 8) : 0;
  pl->o_agg = carry == CARRY_DECOUPLED ? take(size_t(n_units) * DT * N * 8) : 0;
  pl->o_sdt = carry == CARRY_DECOUPLED ? take(size_t(n_units) * DT * 4) : 0;
  pl->o_crot = carry == CARRY_DECOUPLED ? take(size_t(n_units) * N * 8) : 0;
  pl->o_tab = take(size_t(a.B) * a.L * SG::TABW * N * 4);
  pl->o_aux = MODE == 1 ? take(size_t(a.B) * a.L * SG::AUX_W * 4) : 0;
  pl->o_rot = take(size_t(a.B) * S * 4 * 2 * N * 4);
  pl->rest_bytes = off;
  return CSSCAN_OK;
}

// Fill the descriptors and pointers and enqueue both kernels. `hdr` is the workspace header
// (epoch, ticket, done, status words), `flags` the per-unit flag words, `rest` the region laid
// out by the plan.
// CKPT: the checkpoint variant of the scan kernel (no y; the state before every 8-step segment
// into `ckpt`, (B, S8, D, N) complex), which the backward pass launches.
template <int N, typename Tin, int MODE, bool CKPT = false>
int enqueue(const Args& a, const csscan_options_t& o, const Plan& pl, uint32_t* hdr, uint32_t* flags, char* rest,
            cudaStream_t st, float2* ckpt = nullptr, int64_t S8 = 0) {
  TableParams tp;
  tp.Bc = a.Bc;
  tp.Cc = a.Cc;
  tp.theta = a.theta;
  tp.lam = a.lam;
  tp.tab = reinterpret_cast<float*>(rest + pl.o_tab);
  tp.aux = MODE == 1 ? reinterpret_cast<float*>(rest + pl.o_aux) : nullptr;
  tp.rot = reinterpret_cast<float*>(rest + pl.o_rot);
  tp.B = int(a.B);
  tp.L = int(a.L);
  tp.N = N;
  tp.S = int(pl.S);

  ScanParams sp;
  std::memset(&sp, 0, sizeof(sp));
  const CUtensorMapDataType tin = sizeof(Tin) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t s_in = sizeof(Tin);
  const int64_t S = pl.S;
  using SG = Stage<N, Tin, MODE>;
  bool ok = make_map(&sp.tm_x, tin, a.x, a.D, a.L, a.B, a.D * s_in, a.L * a.D * s_in, pl.DT, SG::X_ROWS, 1) &&
            make_map(&sp.tm_dt, tin, a.delta, a.D, a.L, a.B, a.D * s_in, a.L * a.D * s_in, pl.DT, SG::DT_ROWS, 1) &&
            make_map(&sp.tm_tab, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.tab, SG::TABW * N, a.L, a.B, SG::TABW * N * 4,
                     a.L * SG::TABW * N * 4, SG::TABW * N, SG::TAB_ROWS, 1) &&
            make_map(&sp.tm_rot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.rot, 2 * N, 4 * S, a.B, 8 * N, 4 * S * 8 * N, 2 * N, 4,
                     1);
  if (ok && MODE == 1)
    ok = make_map(&sp.tm_aux, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.aux, SG::AUX_W, a.L, a.B, SG::AUX_W * 4,
                  a.L * SG::AUX_W * 4, SG::AUX_W, SG::AUX_ROWS, 1);
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
  sp.ws.hdr = hdr;
  sp.ws.flags = flags;
  sp.ws.inc = pl.carry != CARRY_NONE ? reinterpret_cast<float2*>(rest + pl.o_inc) : nullptr;
  sp.ws.agg = pl.carry == CARRY_DECOUPLED ? reinterpret_cast<float2*>(rest + pl.o_agg) : nullptr;
  sp.ws.sdt = pl.carry == CARRY_DECOUPLED ? reinterpret_cast<float*>(rest + pl.o_sdt) : nullptr;
  sp.ws.crot = pl.carry == CARRY_DECOUPLED ? reinterpret_cast<float2*>(rest + pl.o_crot) : nullptr;
  sp.B = int(a.B);
  sp.L = int(a.L);
  sp.D = int(a.D);
  sp.N = N;
  sp.S = int(S);
  sp.n_dtiles = pl.n_dtiles;
  sp.n_tiles = pl.n_tiles;
  sp.TC = pl.TC;
  sp.n_chunks = pl.n_chunks;
  sp.n_units = pl.n_units;
  sp.carry = pl.carry;
  sp.y_vec2 = (reinterpret_cast<uintptr_t>(a.y) % 8) == 0;
  sp.silent_chunk = o.silent_chunk;
  sp.poll_limit = o.poll_limit > 0 ? o.poll_limit : (int64_t(1) << 22);
  sp.ckpt = reinterpret_cast<float4*>(ckpt);
  sp.S8 = int(S8);

  const int64_t table_threads = a.B * S * N;
  if (!grid_fits(table_threads)) return CSSCAN_ERR_UNSUPPORTED;
  table_kernel<Tin, MODE><<<unsigned((table_threads + 255) / 256), 256, 0, st>>>(tp);
  CSSCAN_CUDA(cudaGetLastError());
  if (o.scan_begin) CSSCAN_CUDA(cudaEventRecord(o.scan_begin, st));
  const dim3 grid{unsigned(pl.n_units)}, block{unsigned(THREADS)};
  if (pl.carry == CARRY_NONE)
    scan_kernel<N, Tin, MODE, CARRY_NONE, CKPT><<<grid, block, unsigned(pl.smem), st>>>(sp);
  else if (pl.carry == CARRY_SERIAL)
    scan_kernel<N, Tin, MODE, CARRY_SERIAL, CKPT><<<grid, block, unsigned(pl.smem), st>>>(sp);
  else
    scan_kernel<N, Tin, MODE, CARRY_DECOUPLED, CKPT><<<grid, block, unsigned(pl.smem), st>>>(sp);
  CSSCAN_CUDA(cudaGetLastError());
  if (o.scan_end) CSSCAN_CUDA(cudaEventRecord(o.scan_end, st));
  return CSSCAN_OK;
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

template <int N, typename Tin, int MODE>
int launch(const Args& a, const csscan_options_t& o, cudaStream_t st) {
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  Plan pl;
  int rc = make_plan<N, Tin, MODE>(a, o, dev, &pl);
  if (rc != CSSCAN_OK) return rc;
  WsEntry ws;
  rc = get_workspace(dev, st, size_t(pl.n_units), pl.rest_bytes, &ws);
  if (rc != CSSCAN_OK) return rc;
  char* base = static_cast<char*>(ws.base);
  return enqueue<N, Tin, MODE>(a, o, pl, reinterpret_cast<uint32_t*>(base), reinterpret_cast<uint32_t*>(base + HDR_BYTES),
                               base + HDR_BYTES + align_up(ws.flag_cap * 4, 256), st);
}

template <typename Tin, int MODE>
int dispatch_n(const Args& a, const csscan_options_t& o, cudaStream_t st) {
  switch (a.N) {
    case 2: return launch<2, Tin, MODE>(a, o, st);
    case 4: return launch<4, Tin, MODE>(a, o, st);
    case 8: return launch<8, Tin, MODE>(a, o, st);
    case 16: return launch<16, Tin, MODE>(a, o, st);
    case 32: return launch<32, Tin, MODE>(a, o, st);
    case 64:
      // the zero-order-hold table row (8 N floats) exceeds one TMA box at N = 64
      if constexpr (MODE == 2) return CSSCAN_ERR_UNSUPPORTED;
      else return launch<64, Tin, MODE>(a, o, st);
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
  if (o.cta_warps != 0 || o.carry < 0 || o.carry > 2 || o.chunk_len < 0 ||
      (o.chunk_len % T_SUB) != 0 || o.poll_limit < 0)
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

csscan_options_t default_options() {
  csscan_options_t o;
  std::memset(&o, 0, sizeof(o));
  o.silent_chunk = -1;
  return o;
}

int forward_impl(const Args& a, const csscan_options_t* opts, cudaStream_t st) {
  csscan_options_t o = opts ? *opts : default_options();
  if (a.mode == CSSCAN_MODE_ZOH) {
    // initial and final state as in exp-Euler; the trapezoid halo has no meaning here and is ignored
    Args a0 = a;
    a0.mode = CSSCAN_MODE_EXP_EULER;   // same pointer, size and alignment rules
    int rc = validate(a0, o);
    if (rc != CSSCAN_OK) return rc;
    if (a.N > 32) return CSSCAN_ERR_UNSUPPORTED;
    const size_t pair = a.dtype == CSSCAN_F32 ? 8 : 4;   // Bc, Cc are read one complex entry at a time
    if (!aligned(a.Bc, pair) || !aligned(a.Cc, pair)) return CSSCAN_ERR_MISALIGNED;
    if (a.B == 0 || a.L == 0 || a.D == 0) return CSSCAN_OK;
    return a.dtype == CSSCAN_F32 ? dispatch_n<float, 2>(a, o, st) : dispatch_n<uint16_t, 2>(a, o, st);
  }
  int rc = validate(a, o);
  if (rc != CSSCAN_OK) return rc;
  if (a.B == 0 || a.L == 0 || a.D == 0) return CSSCAN_OK;
  if (a.dtype == CSSCAN_F32)
    return a.mode == 0 ? dispatch_n<float, 0>(a, o, st) : dispatch_n<float, 1>(a, o, st);
  return a.mode == 0 ? dispatch_n<uint16_t, 0>(a, o, st) : dispatch_n<uint16_t, 1>(a, o, st);
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

// The checkpoint variants of the scan kernel need the same opt-in shared memory as the others.
template <int N, typename Tin, int MODE>
int set_ckpt_attributes(int dev) {
  static std::mutex mu;
  static std::map<int, bool> done;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev]) return CSSCAN_OK;
  CSSCAN_CUDA(cudaFuncSetAttribute(scan_kernel<N, Tin, MODE, CARRY_NONE, true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_DYN_SMEM));
  CSSCAN_CUDA(cudaFuncSetAttribute(scan_kernel<N, Tin, MODE, CARRY_SERIAL, true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_DYN_SMEM));
  CSSCAN_CUDA(cudaFuncSetAttribute(scan_kernel<N, Tin, MODE, CARRY_DECOUPLED, true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_DYN_SMEM));
  done[dev] = true;
  return CSSCAN_OK;
}

// ----------------------------------------------------------------------------- MIMO
struct MimoArgs {
  const void *x, *delta, *Bm, *Cm, *theta, *lam;
  const float *A, *Dskip;
  float* y;
  int64_t B, L, H, P, N;
  int mode, dtype;
};

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
  char* rest = static_cast<char*>(ws.base) + HDR_BYTES + align_up(ws.flag_cap * 4, 256);
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
int dispatch_mimo(const MimoArgs& a, cudaStream_t st) {
  switch (a.P) {
    case 1: return dispatch_mimo_n<Tin, MODE, 1>(a, st);
    case 2: return dispatch_mimo_n<Tin, MODE, 2>(a, st);
    case 4: return dispatch_mimo_n<Tin, MODE, 4>(a, st);
    case 8: return dispatch_mimo_n<Tin, MODE, 8>(a, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
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
  if (a.dtype == CSSCAN_F32)
    return a.mode == 0 ? dispatch_mimo<float, 0>(a, st) : dispatch_mimo<float, 1>(a, st);
  return a.mode == 0 ? dispatch_mimo<uint16_t, 0>(a, st) : dispatch_mimo<uint16_t, 1>(a, st);
}

// ----------------------------------------------------------------------------- backward
struct BwdArgs {
  const void *x, *delta, *Bc, *Cc, *theta, *lam;
  const float *A, *Dskip, *dy;
  float *dx, *ddelta, *dA, *dBc, *dCc, *dtheta, *dlam, *dDskip;
  int64_t B, L, D, N;
  int mode, dtype;
};

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
  Args fa{a.x, a.delta, a.Bc, a.Cc, a.theta, a.lam, a.A, a.Dskip, nullptr, nullptr, nullptr, nullptr, nullptr,
          a.B, a.L, a.D, N, a.mode, a.dtype};
  Plan fpl;
  if (fwd_ckpt) {
    int rc = make_plan<N, Tin, MODE>(fa, default_options(), dev, &fpl);
    if (rc != CSSCAN_OK) return rc;
    rc = set_ckpt_attributes<N, Tin, MODE>(dev);
    if (rc != CSSCAN_OK) return rc;
  }
  const size_t fwd_bytes = fwd_ckpt ? align_up(fpl.rest_bytes, 256) : 0;
  WsEntry ws;
  int rc = get_workspace(dev, st, fwd_ckpt ? size_t(fpl.n_units) : 1, fwd_bytes + rot_bytes + ckpt_bytes + chunk_bytes,
                         &ws);
  if (rc != CSSCAN_OK) return rc;
  char* fwd_rest = static_cast<char*>(ws.base) + HDR_BYTES + align_up(ws.flag_cap * 4, 256);
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
    rc = enqueue<N, Tin, MODE, true>(fa, default_options(), fpl, hdr,
                                     reinterpret_cast<uint32_t*>(static_cast<char*>(ws.base) + HDR_BYTES), fwd_rest,
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
int dispatch_backward(const BwdArgs& a, cudaStream_t st) {
  switch (a.N) {
    case 2: return launch_backward<Tin, MODE, 2>(a, st);
    case 4: return launch_backward<Tin, MODE, 4>(a, st);
    case 8: return launch_backward<Tin, MODE, 8>(a, st);
    case 16: return launch_backward<Tin, MODE, 16>(a, st);
    case 32: return launch_backward<Tin, MODE, 32>(a, st);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

int backward_impl(const BwdArgs& a, cudaStream_t st) {
  if (a.mode == CSSCAN_MODE_ZOH) return CSSCAN_ERR_UNSUPPORTED;
  if (a.mode != CSSCAN_MODE_EXP_EULER && a.mode != CSSCAN_MODE_EXP_TRAPEZOID) return CSSCAN_ERR_INVALID_ARG;
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
  if (a.dtype == CSSCAN_F32)
    return a.mode == 0 ? dispatch_backward<float, 0>(a, st) : dispatch_backward<float, 1>(a, st);
  return a.mode == 0 ? dispatch_backward<uint16_t, 0>(a, st) : dispatch_backward<uint16_t, 1>(a, st);
}

// ----------------------------------------------------------------------------- no-allocation entry
// csscan_forward_noalloc runs the same two kernels with its scratch in one fixed array that
// is part of the library's device code, so it never calls cudaMalloc. Layout of the array:
// [header 256 B][flags: NOALLOC_FLAG_CAP words][the rest, laid out per call by the plan].
constexpr size_t NOALLOC_FLAG_CAP = 1 << 16;
constexpr size_t NOALLOC_REST_OFF = HDR_BYTES + NOALLOC_FLAG_CAP * 4;
static_assert(NOALLOC_REST_OFF < CSSCAN_NOALLOC_SCRATCH_BYTES, "scratch too small");

std::mutex g_noalloc_mu;
std::map<int, char*> g_noalloc_addr;   // device -> device address of the scratch array

int noalloc_scratch_address(int dev, char** out);   // defined after the array below

template <int N, typename Tin, int MODE>
int launch_noalloc(const Args& a, uint32_t* device_status, cudaStream_t st) {
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  const csscan_options_t o = default_options();
  Plan pl;
  int rc = make_plan<N, Tin, MODE>(a, o, dev, &pl);
  if (rc != CSSCAN_OK) return rc;
  if (size_t(pl.n_units) > NOALLOC_FLAG_CAP || pl.rest_bytes > CSSCAN_NOALLOC_SCRATCH_BYTES - NOALLOC_REST_OFF)
    return CSSCAN_ERR_SCRATCH_LIMIT;

  char* base = nullptr;
  rc = noalloc_scratch_address(dev, &base);
  if (rc != CSSCAN_OK) return rc;
  uint32_t* hdr = reinterpret_cast<uint32_t*>(base);
  // the ticket and finished-block counters and the status words must start at zero; the
  // epoch (word 0) keeps counting so that flags left by earlier calls are never current
  CSSCAN_CUDA(cudaMemsetAsync(hdr + H_TICKET, 0, 5 * sizeof(uint32_t), st));
  rc = enqueue<N, Tin, MODE>(a, o, pl, hdr, reinterpret_cast<uint32_t*>(base + HDR_BYTES), base + NOALLOC_REST_OFF, st);
  if (rc != CSSCAN_OK) return rc;
  if (device_status)
    CSSCAN_CUDA(cudaMemcpyAsync(device_status, hdr + H_ERROR, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st));
  return CSSCAN_OK;
}

template <typename Tin, int MODE>
int dispatch_noalloc(const Args& a, uint32_t* device_status, cudaStream_t st) {
  switch (a.N) {
    case 2: return launch_noalloc<2, Tin, MODE>(a, device_status, st);
    case 4: return launch_noalloc<4, Tin, MODE>(a, device_status, st);
    case 8: return launch_noalloc<8, Tin, MODE>(a, device_status, st);
    case 16: return launch_noalloc<16, Tin, MODE>(a, device_status, st);
    case 32: return launch_noalloc<32, Tin, MODE>(a, device_status, st);
    case 64:
      if constexpr (MODE == 2) return CSSCAN_ERR_UNSUPPORTED;
      else return launch_noalloc<64, Tin, MODE>(a, device_status, st);
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

int csscan_forward_state(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                         const void* theta, const void* lambda, const float* Dskip, float* y, const float* h0,
                         const void* x_prev, const void* Bc_prev, float* h_last, int64_t B, int64_t L, int64_t D,
                         int64_t N, int mode, int dtype, cudaStream_t stream) {
  if (mode == CSSCAN_MODE_EXP_EULER) {   // the halo only enters the trapezoid rule
    x_prev = nullptr;
    Bc_prev = nullptr;
  }
  Args a{x, delta, Bc, Cc, theta, lambda, A, Dskip, y, h0, h_last, x_prev, Bc_prev, B, L, D, N, mode, dtype};
  return forward_impl(a, nullptr, stream);
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
  Args av = a;
  if (mode == CSSCAN_MODE_ZOH) av.mode = CSSCAN_MODE_EXP_EULER;   // same pointer, size and alignment rules
  int rc = validate(av, o);
  if (rc != CSSCAN_OK) return rc;
  if (mode == CSSCAN_MODE_ZOH && N > 32) return CSSCAN_ERR_UNSUPPORTED;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) % 4) != 0) return CSSCAN_ERR_MISALIGNED;
  if (a.B == 0 || a.L == 0 || a.D == 0) return CSSCAN_OK;
  if (a.dtype == CSSCAN_F32)
    return a.mode == 0 ? dispatch_noalloc<float, 0>(a, device_status, stream)
                       : (a.mode == 1 ? dispatch_noalloc<float, 1>(a, device_status, stream)
                                      : dispatch_noalloc<float, 2>(a, device_status, stream));
  return a.mode == 0 ? dispatch_noalloc<uint16_t, 0>(a, device_status, stream)
                     : (a.mode == 1 ? dispatch_noalloc<uint16_t, 1>(a, device_status, stream)
                                    : dispatch_noalloc<uint16_t, 2>(a, device_status, stream));
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
    case CSSCAN_ERR_UNSUPPORTED:
      return "unsupported size or mode for this entry point (N in {2, 4, 8, 16, 32, 64}; N <= 32 for the backward and "
             "for the zero-order-hold scan, which the backward does not take)";
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
