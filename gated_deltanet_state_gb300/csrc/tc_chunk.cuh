// tc_chunk.cuh — device helpers of the tensor-core prefill kernels: named
// barriers of the worker warps, the fresh read-only load, and the inverse
// T = (I + A)^{-1} of a chunk's strictly lower triangular 64 x 64 A.
// Included by the fused prefill (tc_prefill.cu) and by the chunk / chain
// pair (tc_chain.cu); each translation unit gets its own internal copy.
#pragma once

#include "tc.cuh"

namespace gdn {
namespace {

// Which piece of which chain a CTA runs.  A launch takes consecutive
// (level, sequence) pairs of the level-major order, at most nseqs of them,
// each with all value heads: CTA (h, b) runs head h of sequence s0 + b at
// level0, or past the last sequence, of sequence s0 + b - nseqs at level0 + 1;
// its chunks are [level * piece, +piece) of the chain (the last level: to the
// sequence's end).
struct PieceMap {
  int32_t s0, level0, nseqs, piece, last_level;
};

// Four floats through the read-only path by an asm load that the compiler
// keeps where it stands (a loop-invariant plain load would be hoisted and
// its registers held through the whole loop).
__device__ __forceinline__ float4 ldg_f4_fresh(const float* src) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(src));
  return v;
}

// Named barrier `id` over `count` threads: wait for the others, or only mark
// this warp's arrival (a producer that does not wait for its consumers).
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// Barrier of the sixteen worker warps alone (threads 0..511).
__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 2, 512;\n" ::: "memory"); }

// The same barrier, returning whether `v` holds on every worker.
__device__ __forceinline__ bool workers_sync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 2, 512, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Barrier of the threads that build T (256..511).
__device__ __forceinline__ void tgrp_sync() { asm volatile("bar.sync 1, 256;\n" ::: "memory"); }

// Row-major A with 16-byte slots XOR-swizzled by row (conflict-free stores
// of a row per lane, loads of a row segment per warp).
__device__ __forceinline__ int am_index(int i, int j) { return i * 64 + (j ^ ((i & 7) << 2)); }

// Block pair (p, k), p > k, of the 4 x 4 grid of 16 x 16 blocks:
// (1,0) (2,0) (2,1) (3,0) (3,1) (3,2) -> 0..5.
__device__ __forceinline__ int pair_index(int p, int k) { return p * (p - 1) / 2 + k; }

// T = (I + A)^{-1} for the 64 x 64 strictly lower triangular A (at: A^T,
// at[j * 64 + i] = A_ij; am: A row-major, am_index), by 256 threads t, in
// 16 x 16 blocks.  With D_b = (I + A_bb)^{-1} and N_pk = -D_p A_pk (p > k),
// T_bb = D_b and T_pq = sum_{k=q}^{p-1} N_pk T_kq, so after the diagonal
// blocks (forward substitution, a column per thread) and all six N blocks (one
// phase), each distance from the diagonal takes one product.  Register tiles
// keep the shared-memory loads at one 16-byte vector per four to eight FMAs.
// tf[i * 64 + j] receives T on and below the diagonal (the blocks above it
// are left unwritten); dt holds D_b^T ([4][16][20]), nt the N_pk^T ([6][16][16]).
__device__ void tri_inverse64(const float* at, const float* am, float* tf, float* dt, float* nt, int t) {
  if (t < 64) {
    // column sweep: once x_k is final, x_i -= A_ik x_k for every i > k (A^T
    // row o+k holds A_{o+i, o+k} contiguously in i; zero for i <= k)
    const int b = t >> 4, o = 16 * b, l = t & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = i == l ? 1.f : 0.f;
#pragma unroll
    for (int k = 0; k < 15; ++k) {
      const float xk = x[k];
#pragma unroll
      for (int i4 = (k + 1) / 4; i4 < 4; ++i4) {
        const float4 a4 = *reinterpret_cast<const float4*>(at + (o + k) * 64 + o + 4 * i4);
        x[4 * i4] = fmaf(-a4.x, xk, x[4 * i4]);
        x[4 * i4 + 1] = fmaf(-a4.y, xk, x[4 * i4 + 1]);
        x[4 * i4 + 2] = fmaf(-a4.z, xk, x[4 * i4 + 2]);
        x[4 * i4 + 3] = fmaf(-a4.w, xk, x[4 * i4 + 3]);
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) tf[(o + i) * 64 + o + l] = x[i];
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4)
      *reinterpret_cast<float4*>(dt + (o + l) * 20 + 4 * i4) =
          make_float4(x[4 * i4], x[4 * i4 + 1], x[4 * i4 + 2], x[4 * i4 + 3]);
  }
  tgrp_sync();
  // N_pk^T[j][i] = -sum_m A_{16p+m, 16k+j} D_p[i][m]: 6 pairs x 16 tiles of 4 j x 4 i
  if (t < 96) {
    const int pr = t >> 4, tile = t & 15;
    const int p = pr == 0 ? 1 : pr < 3 ? 2 : 3;
    const int k = pr - pair_index(p, 0);
    const int j0 = 4 * (tile >> 2), i0 = 4 * (tile & 3);
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float4 a4 = *reinterpret_cast<const float4*>(am + am_index(16 * p + m, 16 * k + j0));
      const float4 d4 = *reinterpret_cast<const float4*>(dt + (16 * p + m) * 20 + i0);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        acc[r][0] = fmaf(a[r], d4.x, acc[r][0]); acc[r][1] = fmaf(a[r], d4.y, acc[r][1]);
        acc[r][2] = fmaf(a[r], d4.z, acc[r][2]); acc[r][3] = fmaf(a[r], d4.w, acc[r][3]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
      *reinterpret_cast<float4*>(nt + (pr * 16 + j0 + r) * 16 + i0) =
          make_float4(-acc[r][0], -acc[r][1], -acc[r][2], -acc[r][3]);
  }
  tgrp_sync();
  // distances 1 and 2: blocks (p, q = p - d) in tiles of 2 rows x 4 columns
#pragma unroll
  for (int d = 1; d < 3; ++d) {
    if (t < (4 - d) * 32) {
      const int q = t >> 5, p = q + d, tile = t & 31;
      const int i0 = 2 * (tile >> 2), j0 = 4 * (tile & 3);
      float acc[2][4];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll
      for (int kk = 0; kk < d; ++kk) {
        const int k = q + kk;
        const float* n = nt + pair_index(p, k) * 256;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float2 n2 = *reinterpret_cast<const float2*>(n + m * 16 + i0);
          const float4 b4 = *reinterpret_cast<const float4*>(tf + (16 * k + m) * 64 + 16 * q + j0);
          acc[0][0] = fmaf(n2.x, b4.x, acc[0][0]); acc[0][1] = fmaf(n2.x, b4.y, acc[0][1]);
          acc[0][2] = fmaf(n2.x, b4.z, acc[0][2]); acc[0][3] = fmaf(n2.x, b4.w, acc[0][3]);
          acc[1][0] = fmaf(n2.y, b4.x, acc[1][0]); acc[1][1] = fmaf(n2.y, b4.y, acc[1][1]);
          acc[1][2] = fmaf(n2.y, b4.z, acc[1][2]); acc[1][3] = fmaf(n2.y, b4.w, acc[1][3]);
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
        *reinterpret_cast<float4*>(tf + (16 * p + i0 + r) * 64 + 16 * q + j0) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
    tgrp_sync();
  }
  // distance 3: block (3, 0) in tiles of 2 x 2 (64 threads)
  if (t < 64) {
    const int i0 = 2 * (t >> 3), j0 = 2 * (t & 7);
    float2 s0 = make_float2(0.f, 0.f), s1 = s0;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const float* n = nt + pair_index(3, k) * 256;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float2 n2 = *reinterpret_cast<const float2*>(n + m * 16 + i0);
        const float2 b2 = *reinterpret_cast<const float2*>(tf + (16 * k + m) * 64 + j0);
        s0.x = fmaf(n2.x, b2.x, s0.x); s0.y = fmaf(n2.x, b2.y, s0.y);
        s1.x = fmaf(n2.y, b2.x, s1.x); s1.y = fmaf(n2.y, b2.y, s1.y);
      }
    }
    *reinterpret_cast<float2*>(tf + (48 + i0) * 64 + j0) = s0;
    *reinterpret_cast<float2*>(tf + (48 + i0 + 1) * 64 + j0) = s1;
  }
  tgrp_sync();
}

}  // namespace
}  // namespace gdn
