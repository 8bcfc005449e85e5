// common.cuh — device helpers shared by the engine's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kConvK = 4;        // depthwise conv taps
constexpr int kWinRows = kConvK - 1;

// ---- element access ------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// SiLU in fp32 with the accurate expf.
__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// First error wins; later faults keep the first code.
__device__ __forceinline__ void set_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// ---- pool addressing -----------------------------------------------------
struct Pool {
  char* base;
  int64_t page_bytes;
  int32_t num_pages;
  int64_t state_bytes;   // Hv*dv*dk*4, window starts here
};

__device__ __forceinline__ float* page_state(const Pool& p, int32_t page) {
  return reinterpret_cast<float*>(p.base + (int64_t)page * p.page_bytes);
}
template <typename TIN>
__device__ __forceinline__ TIN* page_window(const Pool& p, int32_t page) {
  return reinterpret_cast<TIN*>(p.base + (int64_t)page * p.page_bytes + p.state_bytes);
}
__device__ __forceinline__ bool page_ok(const Pool& p, int32_t page) {
  return page >= 0 && page < p.num_pages;
}

// ---- warp reductions (fixed xor order: deterministic) ----------------------
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace gdn

namespace gdn {

// ---- Ampere-style asynchronous copies global -> shared (LDGSTS).  A
// src_bytes of 0 zero-fills the destination without reading the source.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(dst)), "l"(src));
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// SiLU with the fast exponential and division intrinsics (a few ulp).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

}  // namespace gdn

namespace gdn {

// ---- packed fp32 pairs (Blackwell f32x2 instructions): one instruction does
// two IEEE fp32 operations, halving the issue slots of the scan's FMAs.
typedef unsigned long long f32x2;  // low 32 bits = first element

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float sum2(f32x2 v) {
  const float2 f = unpack2(v);
  return f.x + f.y;
}

}  // namespace gdn
