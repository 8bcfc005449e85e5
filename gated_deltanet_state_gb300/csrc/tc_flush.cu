// tc_flush.cu — replay flush on the tensor cores ("Caching less to serve
// more requests", section "What we changed": the flush applies the accepted
// tokens as one block of matrix operations, one launch per layer).
//
// One CTA folds the n <= 32 logged rows of one request into one value head's
// checkpoint state S0 (dv x dk = 128 x 128, fp32) with the chunk (UT) form of
// the gated delta rule, all rows at once:
//   k^_i = k_i / |k_i|,  G_i = sum_{l<=i} g_l,  gam_i = exp(G_i)
//   A_ij = b_i exp(G_i - G_j) k^_i.k^_j (j < i)
//   D1   = S0 K^T                                  (tensor cores, 128 x n x 128)
//   (I + A) U = diag(b) V - diag(b gam) D1^T       (CUDA cores: each thread solves
//                                                   its state row by forward substitution)
//   W    = U^T diag(exp(G_{n-1} - G))
//   S    = gam_{n-1} S0 + W K^                     (tensor cores, 128 x 128 x n,
//                                                   accumulated onto gam S0 in tensor memory)
// The two tensor-core products read bf16 operands split into hi + lo parts
// (three passes: hi*hi + hi*lo + lo*hi), which keeps ~16 bits per operand and
// fp32 accumulation in tensor memory: the state stays within ~1e-5 of fp32.
// The conv + SiLU of the CTA's k and v channels and the L2 norms of k are
// computed in the kernel from the checkpoint's window and the log; the
// window itself is rewritten afterwards by window_kernel (other heads of the
// qk group still read it here).
#include "launch.h"
#include "tc.cuh"

namespace gdn {

constexpr int kTcThreads = 128;
constexpr int kTcD = 128;             // dk = dv
constexpr int kTcMaxRows = GDN_REPLAY_LOG_SLOTS;
constexpr uint32_t kTcCols = 256;     // tensor-memory columns: D1 at 0 (32), D2 at 32 (128), V at 160 (32)
constexpr uint32_t kColV = 160;
constexpr long long kWaitCycles = 4000000000LL;

// Shared-memory plan (byte offsets from a 1024-byte aligned base).
struct TcSmem {
  static constexpr uint32_t A1 = 0;                    // S0 hi | lo: 2 x [2 kb][128][64] bf16 (64 KB)
  static constexpr uint32_t A1_LO = 32768;
  static constexpr uint32_t A2 = 0;                    // W hi | lo: 2 x [128][64] bf16 (reuses A1)
  static constexpr uint32_t A2_LO = 16384;
  static constexpr uint32_t B2 = 32768;                // K^T hi | lo: 2 x [128][64] bf16 (reuses A1)
  static constexpr uint32_t B2_LO = 49152;
  static constexpr uint32_t B1 = 65536;                // K^ hi | lo: 2 x [2 kb][32][64] bf16 (16 KB)
  static constexpr uint32_t B1_LO = 65536 + 8192;
  static constexpr uint32_t XLOG = B1;                 // staging: bf16 [32][k 128 | v 128] log rows
  static constexpr uint32_t KF = 81920;                // K^ fp32 [32][128] (16 KB)
  static constexpr uint32_t AM = KF + 16384;           // fp32 [32][32]: A (strictly lower)
  static constexpr uint32_t XWIN = AM;                 // staging: bf16 [3][256] window rows
  static constexpr uint32_t PART = AM + 4096;          // fp32 [4][32]: partial squared norms
  static constexpr uint32_t GATE = PART + 512;         // fp32 [5][32]: G, gam, b, fk, exp(G_n-1 - G)
  static constexpr uint32_t MBAR = GATE + 640;         // uint64 mbarrier: MMA completion
  static constexpr uint32_t MBAR_TMA = MBAR + 8;       // uint64 mbarrier: state tile arrival
  static constexpr uint32_t TSLOT = MBAR_TMA + 8;      // uint32 tensor-memory base
  static constexpr uint32_t BYTES = TSLOT + 8;
  static constexpr uint32_t ALLOC = BYTES + 1024;      // + alignment slack
};

// NMAX bounds the logged rows at compile time (16 or 32), so per-row loops
// and register arrays are as short as the log allows.
// The state of (page, head h) is the box set {x: 0..127 in 32-column boxes,
// y: h*128 .. +127, z: page} of a 3-D tensor map over the pool:
// [page][head row][column] fp32, boxes of 128 rows x 32 columns (128 B) in the
// 128-byte swizzled shared layout.
__device__ __forceinline__ uint32_t state_smem_offset(int row, int col) {
  return (uint32_t)((col >> 5) * 16384 + row * 128 + ((((col & 31) >> 2) ^ (row & 7)) << 4) + ((col & 3) << 2));
}

template <int NMAX>
__device__ __forceinline__ void tc_flush_body(const ScanParams& p, const CUtensorMap* tmap, int h, int r,
                                              int32_t page, int n) {
  using TIN = __nv_bfloat16;
  constexpr int D = kTcD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  float* kf = reinterpret_cast<float*>(sm + TcSmem::KF);
  float* am = reinterpret_cast<float*>(sm + TcSmem::AM);
  float* Gs = reinterpret_cast<float*>(sm + TcSmem::GATE);
  float* gam = Gs + 32;
  float* bs = Gs + 64;
  float* fk = Gs + 96;
  float* dec = Gs + 128;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + TcSmem::MBAR);
  uint64_t* mbar_tma = reinterpret_cast<uint64_t*>(sm + TcSmem::MBAR_TMA);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + TcSmem::TSLOT);
  TIN* xlog = reinterpret_cast<TIN*>(sm + TcSmem::XLOG);
  TIN* xwin = reinterpret_cast<TIN*>(sm + TcSmem::XWIN);

  // (0) async copies of this CTA's pre-conv rows (k | v channels: the window's
  // three rows and the n logged rows) and of the gates
  const int G = p.Hv / p.Hqk, jq = h / G;
  const int ck0 = p.Hqk * D + jq * D, cv0 = 2 * p.Hqk * D + h * D;
  {
    const TIN* win = page_window<TIN>(p.pool, page);
    const TIN* lx = reinterpret_cast<const TIN*>(p.log_x) + (int64_t)r * kTcMaxRows * p.conv_dim;
    constexpr int RC = 2 * D / 8;                     // 16-byte chunks per staged row
    for (int i = tid; i < (3 + n) * RC; i += kTcThreads) {
      const int row = i / RC, col = (i - row * RC) * 8;
      const int ch = col < D ? ck0 + col : cv0 + col - D;
      const TIN* src = row < 3 ? win + (int64_t)row * p.conv_dim + ch : lx + (int64_t)(row - 3) * p.conv_dim + ch;
      TIN* dst = row < 3 ? xwin + row * 2 * D + col : xlog + (row - 3) * 2 * D + col;
      cp_async16(dst, src, 16);
    }
    for (int i = tid; i < 2 * n; i += kTcThreads) {
      const int row = i >> 1;
      const int64_t lrow = (int64_t)r * kTcMaxRows + row;
      cp_async4((i & 1) ? bs + row : Gs + row, ((i & 1) ? p.log_beta : p.log_g) + lrow * p.Hv + h, 4);
    }
    cp_async_commit();
  }

  if (warp == 0) {
    tc::tmem_alloc(tslot, kTcCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(mbar, 1);
    tc::mbar_init(mbar_tma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    // (1) the state, 64 KB of fp32, arrives by four TMA tile loads into the A1 region
    tc::mbar_expect_tx(mbar_tma, D * D * 4);
#pragma unroll
    for (int cb = 0; cb < 4; ++cb)
      tc::tma_load_3d(sm + TcSmem::A1 + cb * 16384, tmap, 32 * cb, h * D, page, mbar_tma);
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tlane = (uint32_t)(warp * 32) << 16;
  bool ok = tc::mbar_wait_bounded(mbar_tma, 0, kWaitCycles);
  ok = __syncthreads_and(ok);
  if (!ok) {   // the state never arrived: report, give the copy one more bounded wait, leave
    if (tid == 0) set_error(p.err, GDN_ERR_TIMEOUT);
    tc::mbar_wait_bounded(mbar_tma, 0, kWaitCycles);
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, kTcCols);
    return;
  }
  // state row `tid` (= tensor-memory lane tid) into registers; once every
  // thread holds its row the region takes the bf16 hi / lo operand A1
  float sv[D];
#pragma unroll
  for (int c = 0; c < D; c += 4) {
    const float4 f = *reinterpret_cast<const float4*>(sm + TcSmem::A1 + state_smem_offset(tid, c));
    sv[c] = f.x; sv[c + 1] = f.y; sv[c + 2] = f.z; sv[c + 3] = f.w;
  }
  __syncthreads();
  // bf16 hi / lo into A1 (for D1 = S0 K^T); raw S0 into the D2 columns
#pragma unroll
  for (int c8 = 0; c8 < D / 8; ++c8) {
    __nv_bfloat16 hi[8], lo[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) tc::split_bf16(sv[8 * c8 + e], hi[e], lo[e]);
    const uint32_t off = tc::sw128_offset(tid, 8 * c8, D);
    *reinterpret_cast<uint4*>(sm + TcSmem::A1 + off) = *reinterpret_cast<const uint4*>(hi);
    *reinterpret_cast<uint4*>(sm + TcSmem::A1_LO + off) = *reinterpret_cast<const uint4*>(lo);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float v[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] = sv[32 * q + c];
    tc::tmem_st32(tbase + tlane + 32 + 32 * q, v);
  }
  tc::tmem_st_wait();

  // (2) conv + SiLU of k channel `tid` (qk head of h) and v channel `tid` (head h)
  cp_async_wait<0>();
  __syncthreads();
  const float4 wk = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)(ck0 + tid) * kConvK);
  const float4 wv = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)(cv0 + tid) * kConvK);
  float k0 = to_f32(xwin[tid]), k1 = to_f32(xwin[2 * D + tid]), k2 = to_f32(xwin[4 * D + tid]);
  float v0 = to_f32(xwin[D + tid]), v1 = to_f32(xwin[3 * D + tid]), v2 = to_f32(xwin[5 * D + tid]);
  float vr[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) vr[i] = 0.f;
#pragma unroll
  for (int i = 0; i < NMAX; ++i) {
    const float xk = i < n ? to_f32(xlog[i * 2 * D + tid]) : 0.f;
    const float xv = i < n ? to_f32(xlog[i * 2 * D + D + tid]) : 0.f;
    float zk = wk.x * k0;
    zk = fmaf(wk.y, k1, zk);
    zk = fmaf(wk.z, k2, zk);
    zk = fmaf(wk.w, xk, zk);
    float zv = wv.x * v0;
    zv = fmaf(wv.y, v1, zv);
    zv = fmaf(wv.z, v2, zv);
    zv = fmaf(wv.w, xv, zv);
    k0 = k1; k1 = k2; k2 = xk;
    v0 = v1; v1 = v2; v2 = xv;
    kf[i * D + tid] = i < n ? silu_fast(zk) : 0.f;
    vr[i] = i < n ? silu_fast(zv) : 0.f;
  }
  for (int i = NMAX; i < kTcMaxRows; ++i) kf[i * D + tid] = 0.f;
  tc::tmem_st32(tbase + tlane + kColV, vr);   // park v (lane = state row) until the epilogue
  tc::tmem_st_wait();
  __syncthreads();
  // squared norms of the k rows: warp w reduces rows w, w+4, ... (fixed order)
  for (int i = warp; i < n; i += kTcThreads / 32) {
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < D / 32; ++m) {
      const float y = kf[i * D + lane + 32 * m];
      ss = fmaf(y, y, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) fk[i] = 1.0f / sqrtf(ss + p.eps);
  }
  if (warp == 1) {   // cumulative log decay and the decay factors
    float g = lane < n ? Gs[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, g, o);
      if (lane >= o) g += t;
    }
    const float gn = __shfl_sync(0xffffffffu, g, n - 1);
    if (lane < n) { Gs[lane] = g; gam[lane] = expf(g); dec[lane] = expf(gn - g); }
  }
  __syncthreads();

  // (3) k^ = k / |k| (this thread's column); B1 = K^ hi / lo (rows i < NB1);
  // D2 <- gam_{n-1} * S0 in tensor memory
  for (int i = 0; i < n; ++i) kf[i * D + tid] *= fk[i];
  const int NB1 = n <= 16 ? 16 : 32;
  for (int i = 0; i < NB1; ++i) {
    __nv_bfloat16 hi, lo;
    tc::split_bf16(i < n ? kf[i * D + tid] : 0.f, hi, lo);
    const uint32_t off = tc::sw128_offset(i, tid, NB1);
    *reinterpret_cast<__nv_bfloat16*>(sm + TcSmem::B1 + off) = hi;
    *reinterpret_cast<__nv_bfloat16*>(sm + TcSmem::B1_LO + off) = lo;
  }
  {
    const float gN = gam[n - 1];
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      float v[32];
      tc::tmem_ld32(tbase + tlane + 32 + 32 * q, v);
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] *= gN;
      tc::tmem_st32(tbase + tlane + 32 + 32 * q, v);
    }
    tc::tmem_st_wait();
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // (4) D1 = S0 K^T on the tensor cores (three bf16 passes, K = 128)
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(D, NB1);
    for (int pass = 0; pass < 3; ++pass) {
      const uint32_t a = sbase + (pass == 2 ? TcSmem::A1_LO : TcSmem::A1);
      const uint32_t b = sbase + (pass == 1 ? TcSmem::B1_LO : TcSmem::B1);
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t kb = ks >> 2, koff = (ks & 3) * 32;
        tc::mma_bf16(tbase, tc::desc_sw128(a + kb * D * 128 + koff), tc::desc_sw128(b + kb * NB1 * 128 + koff),
                     idesc, (pass | ks) != 0);
      }
    }
    tc::mma_commit(mbar);
  }

  // (5) meanwhile: A_ij = b_i exp(G_i - G_j) k^_i.k^_j for j < i < n
  for (int e = tid; e < n * n; e += kTcThreads) {
    const int i = e / n, j = e % n;
    if (j < i) {
      float acc = 0.f;
      for (int c = 0; c < D; c += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(kf + i * D + c);
        const float4 b4 = *reinterpret_cast<const float4*>(kf + j * D + c);
        acc = fmaf(a4.x, b4.x, acc);
        acc = fmaf(a4.y, b4.y, acc);
        acc = fmaf(a4.z, b4.z, acc);
        acc = fmaf(a4.w, b4.w, acc);
      }
      am[i * 32 + j] = bs[i] * expf(Gs[i] - Gs[j]) * acc;
    }
  }
  __syncthreads();

  // (6) wait for D1; this thread's state row r: R_i = b_i (v_i[r] - gam_i D1[r][i]),
  // (I + A) U = R by forward substitution, W_i = U_i exp(G_{n-1} - G_i)
  ok = tc::mbar_wait_bounded(mbar, 0, kWaitCycles);
  ok = __syncthreads_and(ok);
  tc::fence_after_sync();
  if (ok) {
    float d1[32], vr[32];
    tc::tmem_ld32(tbase + tlane, d1);
    tc::tmem_ld32(tbase + tlane + kColV, vr);
    float u[NMAX];
#pragma unroll
    for (int i = 0; i < NMAX; ++i) u[i] = i < n ? bs[i] * fmaf(-gam[i], d1[i], vr[i]) : 0.f;
#pragma unroll
    for (int j = 0; j < NMAX; ++j)
#pragma unroll
      for (int i = j + 1; i < NMAX; ++i) u[i] = fmaf(-am[i * 32 + j], u[j], u[i]);
    __nv_bfloat16 whi[64], wlo[64];
#pragma unroll
    for (int i = 0; i < NMAX; ++i) tc::split_bf16(i < n ? u[i] * dec[i] : 0.f, whi[i], wlo[i]);
#pragma unroll
    for (int i = NMAX; i < 64; ++i) whi[i] = wlo[i] = __float2bfloat16_rn(0.f);
    // A2 row `tid` = W (K = 64, zeros past n); B2 row `tid` = column tid of K^
    // (both in the A1 region, which MMA1 no longer reads)
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint32_t off = tc::sw128_offset(tid, 8 * c8, D);
      *reinterpret_cast<uint4*>(sm + TcSmem::A2 + off) = *reinterpret_cast<const uint4*>(whi + 8 * c8);
      *reinterpret_cast<uint4*>(sm + TcSmem::A2_LO + off) = *reinterpret_cast<const uint4*>(wlo + 8 * c8);
      __nv_bfloat16 khi[8], klo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = 8 * c8 + e;
        if (i < NMAX) tc::split_bf16(i < n ? kf[i * D + tid] : 0.f, khi[e], klo[e]);
        else khi[e] = klo[e] = __float2bfloat16_rn(0.f);
      }
      *reinterpret_cast<uint4*>(sm + TcSmem::B2 + off) = *reinterpret_cast<const uint4*>(khi);
      *reinterpret_cast<uint4*>(sm + TcSmem::B2_LO + off) = *reinterpret_cast<const uint4*>(klo);
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // (7) D2 += W K^ on the tensor cores (three bf16 passes, K = n rounded to 16)
  if (ok && tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(D, D);
    const int nks = (n + 15) / 16;
    for (int pass = 0; pass < 3; ++pass) {
      const uint32_t a = sbase + (pass == 2 ? TcSmem::A2_LO : TcSmem::A2);
      const uint32_t b = sbase + (pass == 1 ? TcSmem::B2_LO : TcSmem::B2);
      for (int ks = 0; ks < nks; ++ks)   // D2 already holds gam_{n-1} S0
        tc::mma_bf16(tbase + 32, tc::desc_sw128(a + ks * 32), tc::desc_sw128(b + ks * 32), idesc, 1u);
    }
    tc::mma_commit(mbar);
  }
  if (ok) {
    const bool ok2 = tc::mbar_wait_bounded(mbar, 1, kWaitCycles);
    ok = __syncthreads_and(ok2);
  }
  tc::fence_after_sync();

  // (8) D2 = gam_{n-1} S0 + W K^ is the new state: each thread parks its row
  // in the A1 region (free once the second product has completed) in the
  // tensor map's swizzled layout, then four TMA tile stores write it back
  if (ok) {
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      float d2[32];
      tc::tmem_ld32(tbase + tlane + 32 + 32 * q, d2);
#pragma unroll
      for (int c = 0; c < 32; c += 4)
        *reinterpret_cast<float4*>(sm + TcSmem::A1 + state_smem_offset(tid, 32 * q + c)) =
            make_float4(d2[c], d2[c + 1], d2[c + 2], d2[c + 3]);
    }
    tc::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::tma_store_3d(tmap, 32 * cb, h * D, page, sm + TcSmem::A1 + cb * 16384);
      tc::bulk_commit();
      tc::bulk_wait_all();
    }
  } else {
    // a wait ran out: report it, give the tensor core one more bounded wait
    // for the work it may still hold, then release the tensor memory
    if (tid == 0) set_error(p.err, GDN_ERR_TIMEOUT);
    tc::mbar_wait_bounded(mbar, 1, kWaitCycles);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, kTcCols);
}

__global__ void __launch_bounds__(kTcThreads, 2) tc_flush_kernel(const ScanParams p,
                                                                 const __grid_constant__ CUtensorMap tmap) {
  const int h = blockIdx.x, r = blockIdx.y;
  // uniform validation (the window / log_len kernels repeat it)
  const int32_t page = p.ckpt_slot[r];
  const int32_t n = p.log_len[r];
  if (!page_ok(p.pool, page) || n < 0 || n > kTcMaxRows) {
    if (h == 0 && threadIdx.x == 0)
      set_error(p.err, page_ok(p.pool, page) ? GDN_ERR_INVALID_ARG : GDN_ERR_PAGE_RANGE);
    return;
  }
  if (n == 0) return;   // nothing logged: the state stays as it is
  if (n <= 16) tc_flush_body<16>(p, &tmap, h, r, page, n);
  else tc_flush_body<32>(p, &tmap, h, r, page, n);
}

bool tc_flush_supported(int dk, int dv, int in_dtype) {
  return dk == kTcD && dv == kTcD && in_dtype == GDN_BF16;   // staging sized for bf16 rows
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

cudaError_t launch_tc_flush(const ScanParams& p, int in_dtype, cudaStream_t st) {
  (void)in_dtype;
  if (p.num_seqs == 0) return cudaSuccess;
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  // pool states as [page][Hv * 128 rows][128 columns] fp32
  CUtensorMap tmap;
  const cuuint64_t dims[3] = {(cuuint64_t)kTcD, (cuuint64_t)p.Hv * kTcD, (cuuint64_t)p.pool.num_pages};
  const cuuint64_t strides[2] = {(cuuint64_t)kTcD * 4, (cuuint64_t)p.pool.page_bytes};
  const cuuint32_t box[3] = {32, (cuuint32_t)kTcD, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.pool.base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const size_t smem = TcSmem::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(tc_flush_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_flush_kernel<<<dim3(p.Hv, p.num_seqs), kTcThreads, smem, st>>>(p, tmap);
  return cudaGetLastError();
}

}  // namespace gdn
