// forward_launch.cuh -- host side of the forward scan: launch planning (sequence chunks, carry
// kind, workspace layout), tile-copy descriptors and the launches of the table and scan kernels.
// Two kernel families: nscan_kernel (nscan_kernels.cuh; the exp-Euler and trapezoid modes) and
// scan_kernel (scan_kernels.cuh; the zero-order-hold mode, and the checkpoint variant the
// backward pass launches). Included by the per-dtype forward and backward units.
#pragma once

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "host_common.h"
#include "nscan_kernels.cuh"
#include "scan_kernels.cuh"

namespace csscan_host {

using namespace csscan;

// Everything a launch needs that follows from the sizes, the options and the device: sequence
// chunks and carry kind, and the workspace layout (byte offsets into the region after the
// header and the flag words).
struct Plan {
  int DT = 0, n_dtiles = 0, n_tiles = 0, TC = 0, n_chunks = 0, n_units = 0, carry = 0, smem = 0;
  int64_t S = 0;
  size_t o_inc = 0, o_agg = 0, o_sdt = 0, o_crot = 0, o_tab = 0, o_aux = 0, o_rot = 0, rest_bytes = 0;
};

// What the planner needs to know of a scan kernel: its channel tile, shared memory, the table
// and aux floats per (b, t), and its residency for a carry kind.
struct KernelShape {
  int DT;
  int smem;
  int tab_floats;   // table floats per (b, t)
  int aux_floats;   // aux floats per (b, t)
};
using OccFn = int (*)(int carry, int dev, int* occ);

// Blocks of THREADS threads with `smem` dynamic bytes resident per SM (cached per kernel and
// device; the opt-in shared-memory limit is raised once per kernel and device).
template <typename PT>
int occupancy_of(void (*kern)(PT), int dev, int smem, int* out) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int>, int> cache;
  static std::map<std::pair<const void*, int>, bool> attr_set;
  std::lock_guard<std::mutex> lk(mu);
  const void* kp = reinterpret_cast<const void*>(kern);
  if (!attr_set[{kp, dev}]) {
    CSSCAN_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_DYN_SMEM));
    attr_set[{kp, dev}] = true;
  }
  auto key = std::make_tuple(kp, dev, smem);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return CSSCAN_OK;
  }
  int occ = 0;
  CSSCAN_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, THREADS, smem));
  cache[key] = occ;
  *out = occ;
  return CSSCAN_OK;
}

// Launch plan. Blocks are 4 warps wide (one warp per SM sub-partition, so that the warps of a
// block, which meet at a barrier once per sub-chunk, progress at the same rate). Rows with
// enough parallelism are split into a few serial-carry chunks, chosen so that the chunk-units
// fill the block slots in nearly whole waves; rows with too little parallelism are split into
// as many decoupled chunks as fill the GPU.
inline int make_plan(const Args& a, const csscan_options_t& o, int dev, const KernelShape& ks, OccFn occ_fn,
                     Plan* pl) {
  int nsm = 0;
  CSSCAN_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  const int64_t S = (a.L + T_SUB - 1) / T_SUB;
  const int64_t target = int64_t(nsm) * RESIDENT_WARPS_PER_SM;
  const int w = WARPS;
  const int64_t n_dtiles = (a.D + ks.DT - 1) / ks.DT;
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
      // serial chunks, only when the tiles exceed the block slots (otherwise every tile runs
      // at once and chunking would only add blocks that wait for their predecessors): each
      // block runs at its own pace, so the time is about (waves of chunk-units) x (chunk
      // length); pick the chunk count that minimises it, with ~1 % per extra chunk for the
      // per-unit start-up
      int occ = 0;
      int rc = occ_fn(CARRY_SERIAL, dev, &occ);
      if (rc != CSSCAN_OK) return rc;
      const int64_t slots = int64_t(nsm) * std::max(occ, 1);
      if (carry == CARRY_SERIAL || tiles > slots) {
        double best_t = 1e30;
        for (int64_t C = 1; C <= std::min<int64_t>(S, 16); ++C) {
          const int64_t waves = (tiles * C + slots - 1) / slots;
          const double t = double(waves) / double(C) * (1.0 + 0.01 * double(C - 1));
          if (t < best_t - 1e-12) { best_t = t; chunks = C; }
        }
      }
      if (carry == 0) carry = CARRY_SERIAL;
    } else if (carry == CARRY_DECOUPLED || (carry == 0 && starved)) {
      // decoupled chunks: as many as fill every block slot once
      int occ = 0;
      int rc = occ_fn(CARRY_DECOUPLED, dev, &occ);
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
  int rc = occ_fn(carry, dev, &occ);
  if (rc != CSSCAN_OK) return rc;
  if (occ < 1) {
    set_last_error("scan block does not fit on this device");
    return CSSCAN_ERR_CUDA;
  }
  pl->DT = ks.DT;
  pl->n_dtiles = int(n_dtiles);
  pl->n_tiles = int(tiles);
  pl->TC = int(TC);
  pl->n_chunks = int(n_chunks);
  pl->n_units = int(n_units);
  pl->carry = carry;
  pl->S = S;
  pl->smem = ks.smem;

  // workspace layout after the header and the flags
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t r = off; off = align_up(off + bytes, 256); return r; };
  const size_t N = size_t(a.N);
  pl->o_inc = carry != CARRY_NONE ? take(size_t(n_units) * ks.DT * N * 8) : 0;
  pl->o_agg = carry == CARRY_DECOUPLED ? take(size_t(n_units) * ks.DT * N * 8) : 0;
  pl->o_sdt = carry == CARRY_DECOUPLED ? take(size_t(n_units) * ks.DT * 4) : 0;
  pl->o_crot = carry == CARRY_DECOUPLED ? take(size_t(n_units) * N * 8) : 0;
  pl->o_tab = take(size_t(a.B) * a.L * ks.tab_floats * 4);
  pl->o_aux = ks.aux_floats ? take(size_t(a.B) * a.L * ks.aux_floats * 4) : 0;
  pl->o_rot = take(size_t(a.B) * S * 4 * 2 * N * 4);
  pl->rest_bytes = off;
  return CSSCAN_OK;
}

inline bool map3(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t n0, uint64_t n1, uint64_t n2,
                 uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2) {
  const uint64_t dims[3] = {n0, n1, n2};
  const uint64_t strides[2] = {stride1, stride2};
  const uint32_t box[3] = {b0, b1, b2};
  return make_map(m, type, base, 3, dims, strides, box);
}

// Fill the pointers of ScanParams that both kernel families share.
inline void fill_common(ScanParams& sp, const Args& a, const Plan& pl, uint32_t* hdr, uint32_t* flags, char* rest,
                        const csscan_options_t& o) {
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
  sp.N = int(a.N);
  sp.S = int(pl.S);
  sp.n_dtiles = pl.n_dtiles;
  sp.n_tiles = pl.n_tiles;
  sp.TC = pl.TC;
  sp.n_chunks = pl.n_chunks;
  sp.n_units = pl.n_units;
  sp.carry = pl.carry;
  sp.y_vec2 = (reinterpret_cast<uintptr_t>(a.y) % 8) == 0;
  sp.silent_chunk = o.silent_chunk;
  sp.poll_limit = o.poll_limit > 0 ? o.poll_limit : (int64_t(1) << 22);
  sp.n_full = int(a.n_full ? a.n_full : a.N);
  sp.n_off = int(a.n_off);
}

inline TableParams table_params(const Args& a, const Plan& pl, char* rest, int N) {
  TableParams tp;
  tp.Bc = a.Bc;
  tp.Cc = a.Cc;
  tp.theta = a.theta;
  tp.lam = a.lam;
  tp.tab = reinterpret_cast<float*>(rest + pl.o_tab);
  tp.aux = pl.o_aux ? reinterpret_cast<float*>(rest + pl.o_aux) : nullptr;
  tp.rot = reinterpret_cast<float*>(rest + pl.o_rot);
  tp.B = int(a.B);
  tp.L = int(a.L);
  tp.N = N;
  tp.S = int(pl.S);
  tp.ng = 1;
  tp.planes = 2;
  tp.plane_w = 2 * N;
  tp.hdr = nullptr;
  tp.n_full = int(a.n_full ? a.n_full : a.N);
  tp.n_off = int(a.n_off);
  return tp;
}

// ============================================================================ nscan family
// CKPT: the checkpoint variant (no y; the rotated-frame state before every 8-step segment into
// `ckpt`), which the backward pass launches.
template <int N, int NS, typename Tin, int MODE, bool CKPT = false>
struct NScan {
  using SG = NStage<N, NS, Tin, MODE>;
  static constexpr KernelShape shape() {
    return KernelShape{NTile<N, NS>::DT, SG::SMEM, NTile<N, NS>::PLANES * NTile<N, NS>::W, MODE == 1 ? 4 : 0};
  }
  static int occ(int carry, int dev, int* out) {
    if (carry == CARRY_SERIAL)
      return occupancy_of(nscan_kernel<N, NS, Tin, MODE, CARRY_SERIAL, CKPT>, dev, SG::SMEM, out);
    if (carry == CARRY_DECOUPLED)
      return occupancy_of(nscan_kernel<N, NS, Tin, MODE, CARRY_DECOUPLED, CKPT>, dev, SG::SMEM, out);
    return occupancy_of(nscan_kernel<N, NS, Tin, MODE, CARRY_NONE, CKPT>, dev, SG::SMEM, out);
  }
  static int enqueue(const Args& a, const csscan_options_t& o, const Plan& pl, uint32_t* hdr, uint32_t* flags,
                     char* rest, cudaStream_t st, float2* ckpt = nullptr, int64_t S8 = 0) {
    TableParams tp = table_params(a, pl, rest, N);
    using TL = NTile<N, NS>;
    tp.ng = TL::NG;
    tp.planes = TL::PLANES;
    tp.plane_w = TL::W;
    tp.hdr = hdr;
    ScanParams sp;
    std::memset(&sp, 0, sizeof(sp));
    const CUtensorMapDataType tin = sizeof(Tin) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t s_in = sizeof(Tin);
    const uint64_t B = uint64_t(a.B), L = uint64_t(a.L), D = uint64_t(a.D), S = uint64_t(pl.S);
    const uint64_t tdims[4] = {TL::W, TL::PLANES, L, B};
    const uint64_t tstrides[3] = {TL::W * 4, TL::PLANES * TL::W * 4, L * TL::PLANES * TL::W * 4};
    const uint32_t tbox[4] = {TL::W, TL::PLANES, SG::TAB_ROWS, 1};
    bool ok = map3(&sp.tm_x, tin, a.x, D, L, B, D * s_in, L * D * s_in, pl.DT, SG::X_ROWS, 1) &&
              map3(&sp.tm_dt, tin, a.delta, D, L, B, D * s_in, L * D * s_in, pl.DT, SG::DT_ROWS, 1) &&
              make_map(&sp.tm_tab, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.tab, 4, tdims, tstrides, tbox) &&
              map3(&sp.tm_rot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.rot, 2 * N, 4 * S, B, 8 * N, 4 * S * 8 * N, 2 * N, 1, 1);
    if (ok && MODE == 1)
      ok = map3(&sp.tm_aux, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.aux, 4, L, B, 16, L * 16, 4, SG::AUX_ROWS, 1);
    if (!ok) {
      set_last_error("cuTensorMapEncodeTiled failed or unavailable");
      return CSSCAN_ERR_CUDA;
    }
    fill_common(sp, a, pl, hdr, flags, rest, o);
    sp.ckpt = reinterpret_cast<float4*>(ckpt);
    sp.S8 = int(S8);
    const int64_t table_threads = a.B * pl.S * N;
    if (!grid_fits(table_threads)) return CSSCAN_ERR_UNSUPPORTED;
    ntable_kernel<Tin, MODE><<<unsigned((table_threads + 255) / 256), 256, 0, st>>>(tp);
    CSSCAN_CUDA(cudaGetLastError());
    if (o.scan_begin) CSSCAN_CUDA(cudaEventRecord(o.scan_begin, st));
    const dim3 grid{unsigned(pl.n_units)}, block{unsigned(THREADS)};
    if (pl.carry == CARRY_NONE)
      nscan_kernel<N, NS, Tin, MODE, CARRY_NONE, CKPT><<<grid, block, unsigned(pl.smem), st>>>(sp);
    else if (pl.carry == CARRY_SERIAL)
      nscan_kernel<N, NS, Tin, MODE, CARRY_SERIAL, CKPT><<<grid, block, unsigned(pl.smem), st>>>(sp);
    else
      nscan_kernel<N, NS, Tin, MODE, CARRY_DECOUPLED, CKPT><<<grid, block, unsigned(pl.smem), st>>>(sp);
    CSSCAN_CUDA(cudaGetLastError());
    if (o.scan_end) CSSCAN_CUDA(cudaEventRecord(o.scan_end, st));
    return CSSCAN_OK;
  }
};

// ============================================================================ scan family
// ACC: the kernel variant of a later part of a zero-order-hold state split (adds to y)
template <int N, typename Tin, int MODE, bool CKPT = false, bool ACC = false>
struct RScan {
  using SG = Stage<N, Tin, MODE>;
  // the table's tile-copy descriptor: rows of TABW N floats, one box each (a box is at most 256
  // elements wide: the zero-order hold runs N > 16 as 16-state parts)
  static bool table_map(CUtensorMap* m, const float* tab, uint64_t L, uint64_t B) {
    constexpr uint64_t W = uint64_t(SG::TABW) * N;
    static_assert(W <= 256, "table row wider than one tile-copy box");
    return map3(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tab, W, L, B, W * 4, L * W * 4, uint32_t(W), SG::TAB_ROWS, 1);
  }
  static_assert(SG::SMEM <= MAX_DYN_SMEM, "stage ring too large");
  static constexpr KernelShape shape() { return KernelShape{Tile<N>::DT, SG::SMEM, SG::TABW * N, MODE == 1 ? SG::AUX_W : 0}; }
  static int occ(int carry, int dev, int* out) {
    if (carry == CARRY_SERIAL) return occupancy_of(scan_kernel<N, Tin, MODE, CARRY_SERIAL, CKPT, ACC>, dev, SG::SMEM, out);
    if (carry == CARRY_DECOUPLED) return occupancy_of(scan_kernel<N, Tin, MODE, CARRY_DECOUPLED, CKPT, ACC>, dev, SG::SMEM, out);
    return occupancy_of(scan_kernel<N, Tin, MODE, CARRY_NONE, CKPT, ACC>, dev, SG::SMEM, out);
  }
  // CKPT: the checkpoint variant (no y; the state before every 8-step segment into `ckpt`,
  // (B, S8, D, N) complex), which the backward pass launches.
  static int enqueue(const Args& a, const csscan_options_t& o, const Plan& pl, uint32_t* hdr, uint32_t* flags,
                     char* rest, cudaStream_t st, float2* ckpt = nullptr, int64_t S8 = 0) {
    const TableParams tp = table_params(a, pl, rest, N);
    ScanParams sp;
    std::memset(&sp, 0, sizeof(sp));
    const CUtensorMapDataType tin = sizeof(Tin) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t s_in = sizeof(Tin);
    const uint64_t B = uint64_t(a.B), L = uint64_t(a.L), D = uint64_t(a.D), S = uint64_t(pl.S);
    bool ok = map3(&sp.tm_x, tin, a.x, D, L, B, D * s_in, L * D * s_in, pl.DT, SG::X_ROWS, 1) &&
              map3(&sp.tm_dt, tin, a.delta, D, L, B, D * s_in, L * D * s_in, pl.DT, SG::DT_ROWS, 1) &&
              table_map(&sp.tm_tab, tp.tab, L, B) &&
              map3(&sp.tm_rot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.rot, 2 * N, 4 * S, B, 8 * N, 4 * S * 8 * N, 2 * N, 4, 1);
    if (ok && MODE == 1)
      ok = map3(&sp.tm_aux, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tp.aux, SG::AUX_W, L, B, SG::AUX_W * 4, L * SG::AUX_W * 4,
                SG::AUX_W, SG::AUX_ROWS, 1);
    if (!ok) {
      set_last_error("cuTensorMapEncodeTiled failed or unavailable");
      return CSSCAN_ERR_CUDA;
    }
    fill_common(sp, a, pl, hdr, flags, rest, o);
    sp.ckpt = reinterpret_cast<float4*>(ckpt);
    sp.S8 = int(S8);
    const int64_t table_threads = a.B * pl.S * N;
    if (!grid_fits(table_threads)) return CSSCAN_ERR_UNSUPPORTED;
    table_kernel<Tin, MODE><<<unsigned((table_threads + 255) / 256), 256, 0, st>>>(tp);
    CSSCAN_CUDA(cudaGetLastError());
    if (o.scan_begin) CSSCAN_CUDA(cudaEventRecord(o.scan_begin, st));
    const dim3 grid{unsigned(pl.n_units)}, block{unsigned(THREADS)};
    if (pl.carry == CARRY_NONE)
      scan_kernel<N, Tin, MODE, CARRY_NONE, CKPT, ACC><<<grid, block, unsigned(pl.smem), st>>>(sp);
    else if (pl.carry == CARRY_SERIAL)
      scan_kernel<N, Tin, MODE, CARRY_SERIAL, CKPT, ACC><<<grid, block, unsigned(pl.smem), st>>>(sp);
    else
      scan_kernel<N, Tin, MODE, CARRY_DECOUPLED, CKPT, ACC><<<grid, block, unsigned(pl.smem), st>>>(sp);
    CSSCAN_CUDA(cudaGetLastError());
    if (o.scan_end) CSSCAN_CUDA(cudaEventRecord(o.scan_end, st));
    return CSSCAN_OK;
  }
};

// Plan, find scratch (the per-stream workspace or a fixed region) and enqueue one forward.
template <class K>
int launch_forward(const Args& a, const csscan_options_t& o, cudaStream_t st, const FixedScratch* fixed) {
  int dev = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  Plan pl;
  int rc = make_plan(a, o, dev, K::shape(), &K::occ, &pl);
  if (rc != CSSCAN_OK) return rc;
  if (fixed) {
    if (size_t(pl.n_units) > fixed->flag_cap || pl.rest_bytes > fixed->rest_cap) return CSSCAN_ERR_SCRATCH_LIMIT;
    // the ticket and finished-block counters and the status words must start at zero; the
    // epoch (word 0) keeps counting so that flags left by earlier calls are never current
    CSSCAN_CUDA(cudaMemsetAsync(fixed->hdr + H_TICKET, 0, 5 * sizeof(uint32_t), st));
    return K::enqueue(a, o, pl, fixed->hdr, fixed->flags, fixed->rest, st);
  }
  WsEntry ws;
  rc = get_workspace(dev, st, size_t(pl.n_units), pl.rest_bytes, &ws);
  if (rc != CSSCAN_OK) return rc;
  char* base = static_cast<char*>(ws.base);
  return K::enqueue(a, o, pl, reinterpret_cast<uint32_t*>(base), reinterpret_cast<uint32_t*>(base + HDR_BYTES),
                    ws_rest(ws), st);
}

// Zero-order hold with N > 16: the states are independent recurrences that meet only in the
// sum over n of y, so the scan runs as N / 16 scans of 16 states each, in stream order, the first
// writing y (with the Dskip term) and the others adding to it with reductions that no thread
// waits for. Measured on B300 on the large-batch shape (B=16 L=8192 D=2560, bf16): N = 32 in
// 9.8 ms and N = 64 in 19.7 ms, against 18.9 ms and 76.4 ms for one scan over all N states, whose
// table stage (8 N floats per step) leaves room for too few resident warps. The options'
// scan_begin event goes with the first part and scan_end with the last.
template <typename Tin>
int zoh_by_parts(const Args& a, const csscan_options_t& o, cudaStream_t st, const FixedScratch* fx) {
  constexpr int64_t PART = 16;
  const int64_t parts = a.N / PART;
  for (int64_t j = 0; j < parts; ++j) {
    Args pa = a;
    pa.N = PART;
    pa.n_full = a.N;
    pa.n_off = j * PART;
    csscan_options_t po = o;
    if (j > 0) po.scan_begin = nullptr;
    if (j + 1 < parts) po.scan_end = nullptr;
    const int rc = j == 0 ? launch_forward<RScan<16, Tin, 2>>(pa, po, st, fx)
                          : launch_forward<RScan<16, Tin, 2, false, true>>(pa, po, st, fx);
    if (rc != CSSCAN_OK) return rc;
  }
  return CSSCAN_OK;
}

template <typename Tin>
int forward_dispatch(const Args& a, const csscan_options_t& o, cudaStream_t st, const FixedScratch* fx) {
  if (a.mode == CSSCAN_MODE_ZOH) {
    switch (a.N) {
      case 2: return launch_forward<RScan<2, Tin, 2>>(a, o, st, fx);
      case 4: return launch_forward<RScan<4, Tin, 2>>(a, o, st, fx);
      case 8: return launch_forward<RScan<8, Tin, 2>>(a, o, st, fx);
      case 16: return launch_forward<RScan<16, Tin, 2>>(a, o, st, fx);
      case 32:
      case 64: return zoh_by_parts<Tin>(a, o, st, fx);
      default: return CSSCAN_ERR_UNSUPPORTED;
    }
  }
  int dev = 0, nsm = 0;
  CSSCAN_CUDA(cudaGetDevice(&dev));
  CSSCAN_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  // states per thread: 16 where the (b, d) rows give enough threads or the sequence is long
  // enough for decoupled chunks to supply them; 8 (two lanes per channel, twice the threads) for
  // N = 32 rows that would leave the SMs under 8 warps each, and for N = 16 rows under 2 warps per
  // SM, on sequences whose decoupled chunks would otherwise be too short to amortise their
  // look-back (measured on B, L, D = 1, 131072, 1024: N = 32 at 16 states per thread 2.5 ms, at 8
  // states 3.4 ms)
  const int64_t rows = a.B * a.D;
  const bool wide32 = 2 * rows >= int64_t(nsm) * 32 * RESIDENT_WARPS_PER_SM || a.L > 16384;
  const bool wide16 = rows >= int64_t(nsm) * 64 || a.L > 16384;
  if (a.mode == CSSCAN_MODE_EXP_EULER) {
    switch (a.N) {
      case 2: return launch_forward<NScan<2, 2, Tin, 0>>(a, o, st, fx);
      case 4: return launch_forward<NScan<4, 4, Tin, 0>>(a, o, st, fx);
      case 8: return launch_forward<NScan<8, 8, Tin, 0>>(a, o, st, fx);
      case 16: return wide16 ? launch_forward<NScan<16, 16, Tin, 0>>(a, o, st, fx)
                             : launch_forward<NScan<16, 8, Tin, 0>>(a, o, st, fx);
      case 32: return wide32 ? launch_forward<NScan<32, 16, Tin, 0>>(a, o, st, fx)
                             : launch_forward<NScan<32, 8, Tin, 0>>(a, o, st, fx);
      case 64: return launch_forward<NScan<64, 16, Tin, 0>>(a, o, st, fx);
      default: return CSSCAN_ERR_UNSUPPORTED;
    }
  }
  switch (a.N) {
    case 2: return launch_forward<NScan<2, 2, Tin, 1>>(a, o, st, fx);
    case 4: return launch_forward<NScan<4, 4, Tin, 1>>(a, o, st, fx);
    case 8: return launch_forward<NScan<8, 8, Tin, 1>>(a, o, st, fx);
    case 16: return wide16 ? launch_forward<NScan<16, 16, Tin, 1>>(a, o, st, fx)
                           : launch_forward<NScan<16, 8, Tin, 1>>(a, o, st, fx);
    case 32: return wide32 ? launch_forward<NScan<32, 16, Tin, 1>>(a, o, st, fx)
                           : launch_forward<NScan<32, 8, Tin, 1>>(a, o, st, fx);
    case 64: return launch_forward<NScan<64, 16, Tin, 1>>(a, o, st, fx);
    default: return CSSCAN_ERR_UNSUPPORTED;
  }
}

}  // namespace csscan_host
