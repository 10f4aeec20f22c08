// device_util.cuh -- small sm_103a device helpers: tile copies (TMA) tracked by mbarriers,
// gpu-scope acquire/release flag accesses, packed float32x2 arithmetic and the hardware
// base-2 exponential. Every wait here is bounded by its caller.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csscan {

// ---------------------------------------------------------------------------- arithmetic
// Hardware 2^x (MUFU.EX2); inputs below the float32 range flush to +0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Hardware reciprocal (MUFU.RCP, about 1 ulp); denormal inputs and results flush to zero.
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
// Packed float32x2 fused multiply-add / multiply (one instruction for two lanes).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
// 2^z for both halves of a pair.
__device__ __forceinline__ float2 ex2_pair(float2 z) { return make_float2(ex2_approx(z.x), ex2_approx(z.y)); }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

template <typename Tin> __device__ __forceinline__ float load_in(const Tin* p, int64_t i);
template <> __device__ __forceinline__ float load_in<float>(const float* p, int64_t i) { return p[i]; }
template <> __device__ __forceinline__ float load_in<uint16_t>(const uint16_t* p, int64_t i) {
  return bf16_bits_to_float(p[i]);
}
// The two values at p[2 i], p[2 i + 1] (a complex entry), with one load (needs 2 * sizeof(Tin)
// alignment).
template <typename Tin> __device__ __forceinline__ float2 load_pair(const Tin* p, int64_t i);
template <> __device__ __forceinline__ float2 load_pair<float>(const float* p, int64_t i) {
  return reinterpret_cast<const float2*>(p)[i];
}
template <> __device__ __forceinline__ float2 load_pair<uint16_t>(const uint16_t* p, int64_t i) {
  const uint32_t v = reinterpret_cast<const uint32_t*>(p)[i];
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
template <typename Tin> __device__ __forceinline__ float smem_in(const Tin* p, int i);
template <> __device__ __forceinline__ float smem_in<float>(const float* p, int i) { return p[i]; }
template <> __device__ __forceinline__ float smem_in<uint16_t>(const uint16_t* p, int i) {
  return bf16_bits_to_float(p[i]);
}

// The K consecutive values p[0 .. K-1] widened to float, with vector loads (p aligned to
// K * sizeof(Tin) bytes; K = 1, 2, 4 or 8).
template <typename Tin, int K>
__device__ __forceinline__ void smem_row(const Tin* p, float (&v)[K]) {
  if constexpr (sizeof(Tin) == 4) {
    if constexpr (K % 4 == 0) {
#pragma unroll
      for (int i = 0; i < K / 4; ++i) {
        const float4 f = reinterpret_cast<const float4*>(p)[i];
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
      }
    } else if constexpr (K == 2) {
      const float2 f = *reinterpret_cast<const float2*>(p);
      v[0] = f.x; v[1] = f.y;
    } else {
      v[0] = p[0];
    }
  } else {
    uint32_t w[(K + 1) / 2];
    if constexpr (K == 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else if constexpr (K == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      w[0] = u.x; w[1] = u.y;
    } else if constexpr (K == 2) {
      w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else {
      w[0] = uint32_t(p[0]);
    }
#pragma unroll
    for (int i = 0; i < K; ++i)
      v[i] = __uint_as_float((i & 1) ? (w[i / 2] & 0xffff0000u) : (w[i / 2] << 16));
  }
}

// ---------------------------------------------------------------------------- lane sums
// Reduce-scatter of NARR arrays v[k][0 .. LEN-1] over the N lanes of a lane group (lane bits
// below N; N and LEN powers of two): rounds with the high masks halve the arrays (each lane
// keeps one half and adds its partner's copy of it), rounds with the remaining masks add whole
// values. Afterwards a lane holds the group sums for entries base .. base + max(1, LEN/N) - 1 in
// v[k][0 ..]; lanes that differ only in bits below max(1, N/LEN) hold the same entries.
// Returns base. `lane` is the lane's index within its group; the group's lanes are STRIDE apart
// in the warp (partners differ by m * STRIDE).
template <int N, int NARR, int LEN, int STRIDE = 1>
__device__ __forceinline__ int butterfly(float (&v)[NARR][LEN], int lane) {
  int base = 0;
  int len = LEN;
#pragma unroll
  for (int m = N / 2; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
    if (len > 1) {
      const int half = len / 2;
#pragma unroll
      for (int k = 0; k < NARR; ++k)
#pragma unroll
        for (int i = 0; i < LEN / 2; ++i)
          if (i < half) {
            const float send = upper ? v[k][i] : v[k][i + half];
            const float keep = upper ? v[k][i + half] : v[k][i];
            v[k][i] = keep + __shfl_xor_sync(0xffffffffu, send, m * STRIDE);
          }
      if (upper) base += half;
      len = half;
    } else {
#pragma unroll
      for (int k = 0; k < NARR; ++k) v[k][0] += __shfl_xor_sync(0xffffffffu, v[k][0], m * STRIDE);
    }
  }
  return base;
}
// The base butterfly<N, NARR, LEN> returns for a lane, without the sums.
template <int N, int LEN>
__device__ __forceinline__ int butterfly_base(int lane) {
  int base = 0, len = LEN;
#pragma unroll
  for (int m = N / 2; m >= 1; m >>= 1)
    if (len > 1) {
      if (lane & m) base += len / 2;
      len /= 2;
    }
  return base;
}

// ---------------------------------------------------------------------------- flags
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------------------- TMA
// 3-D tiled copy global -> shared, completion counted on `bar` (bytes of the whole box).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}
// 4-D tiled copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace csscan
