// host_common.h -- host-side pieces shared by the translation units of the library: error
// reporting, tile-copy descriptors, the argument records of the entry points, the per-(device,
// stream) workspace, and the per-dtype launch functions each unit defines (csscan.cu holds the
// C ABI and calls them).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "csscan.h"

namespace csscan_host {

// ----------------------------------------------------------------------------- errors
// The message csscan_status_string returns for CSSCAN_ERR_CUDA (per host thread).
void set_last_error(const char* msg);
int cuda_fail(cudaError_t e, const char* what);
#define CSSCAN_CUDA(call)                                              \
  do {                                                                 \
    cudaError_t e_ = (call);                                           \
    if (e_ != cudaSuccess) return ::csscan_host::cuda_fail(e_, #call); \
  } while (0)

// ----------------------------------------------------------------------------- helpers
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
// A 1-D launch of `threads` threads in blocks of 256 stays within the grid's x limit.
inline bool grid_fits(long long threads) { return (threads + 255) / 256 <= 0x7fffffffLL; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
constexpr size_t HDR_BYTES = 256;
constexpr int MAX_DYN_SMEM = 160 * 1024;         // opt-in dynamic shared memory per block
// The MIMO path and the backward's gradient pass run one thread per (row, state) sequentially
// over time; below this many such threads per SM they also split the sequence into time chunks.
constexpr int64_t SEQ_THREADS_PER_SM = 4096;
constexpr int RESIDENT_WARPS_PER_SM = 8;         // target of the automatic chunking

// Tiled tile-copy descriptor over `rank` dimensions (innermost first), byte strides of dims 1..;
// reads outside the tensor give 0. False if the driver entry point is missing or refuses.
bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box);

csscan_options_t default_options();

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
  // the zero-order-hold scan of a part of the states (forward_launch.cuh splits N > 16 into
  // 16-state parts): N of the whole problem (0: N) and the part's first state
  int64_t n_full = 0, n_off = 0;
};

struct MimoArgs {
  const void *x, *delta, *Bm, *Cm, *theta, *lam;
  const float *A, *Dskip;
  float* y;
  int64_t B, L, H, P, N;
  int mode, dtype;
};

struct MimoBwdArgs {
  const void *x, *delta, *Bm, *Cm, *theta, *lam;
  const float *A, *Dskip, *dy;
  float *dx, *ddelta, *dA, *dBm, *dCm, *dtheta, *dlam, *dDskip;
  int64_t B, L, H, P, N;
  int mode, dtype;
};

struct BwdArgs {
  const void *x, *delta, *Bc, *Cc, *theta, *lam;
  const float *A, *Dskip, *dy;
  float *dx, *ddelta, *dA, *dBc, *dCc, *dtheta, *dlam, *dDskip;
  int64_t B, L, D, N;
  int mode, dtype;
};

// ----------------------------------------------------------------------------- workspace
// Per (device, stream): [header 256 B][flags: flag_cap words][the rest, laid out per call].
// The flags region only grows through a full reallocation, which zeroes it; records from
// earlier calls carry an older epoch and are never mistaken for this call's.
struct WsEntry {
  void* base = nullptr;
  size_t bytes = 0;
  size_t flag_cap = 0;
};
int get_workspace(int dev, cudaStream_t st, size_t units, size_t rest_bytes, WsEntry* out);
inline char* ws_rest(const WsEntry& e) { return static_cast<char*>(e.base) + HDR_BYTES + align_up(e.flag_cap * 4, 256); }

// A fixed scratch region (the no-allocation entry point): header, flag words and the rest, with
// their capacities; a forward launch that needs more returns CSSCAN_ERR_SCRATCH_LIMIT.
struct FixedScratch {
  uint32_t* hdr;
  uint32_t* flags;
  char* rest;
  size_t flag_cap;
  size_t rest_cap;
};

// ----------------------------------------------------------------------------- launches
// Forward scan of a validated, non-empty problem (every mode); `fixed` = NULL uses the
// per-stream workspace. Defined in forward_f32.cu / forward_bf16.cu.
int forward_f32(const Args& a, const csscan_options_t& o, cudaStream_t st, const FixedScratch* fixed);
int forward_bf16(const Args& a, const csscan_options_t& o, cudaStream_t st, const FixedScratch* fixed);
// Backward of a validated, non-empty problem. Defined in backward_f32.cu / backward_bf16.cu.
int backward_f32(const BwdArgs& a, cudaStream_t st);
int backward_bf16(const BwdArgs& a, cudaStream_t st);
// MIMO scan of a validated, non-empty problem. Defined in mimo_f32.cu / mimo_bf16.cu.
int mimo_f32(const MimoArgs& a, cudaStream_t st);
int mimo_bf16(const MimoArgs& a, cudaStream_t st);
// Backward of a validated, non-empty MIMO problem. Defined in mimo_f32.cu / mimo_bf16.cu.
int mimo_backward_f32(const MimoBwdArgs& a, cudaStream_t st);
int mimo_backward_bf16(const MimoBwdArgs& a, cudaStream_t st);

}  // namespace csscan_host
