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

constexpr int kTcThreads = 256;   // two threads per state row (64 columns each)
constexpr int kTcD = 128;             // dk = dv
constexpr int kTcMaxRows = GDN_REPLAY_LOG_SLOTS;
constexpr uint32_t kTcCols = 256;     // tensor-memory columns: D1 at 0 (32), D2 at 32 (128), V at 160 (32)
constexpr uint32_t kColV = 160;
constexpr long long kWaitCycles = 4000000000LL;

// Shared-memory plan (byte offsets from a 1024-byte aligned base).
struct TcSmem {
  static constexpr uint32_t A1 = 0;                    // S0 fp32 (TMA) | S0 hi | lo: 2 x [2 kb][128][64] bf16 (64 KB)
  static constexpr uint32_t A1_LO = 32768;
  static constexpr uint32_t A2 = 0;                    // W hi | lo: 2 x [128][64] bf16 (reuses A1)
  static constexpr uint32_t A2_LO = 16384;
  static constexpr uint32_t B2 = 32768;                // K^T hi | lo: 2 x [128][64] bf16 (reuses A1)
  static constexpr uint32_t B2_LO = 49152;
  static constexpr uint32_t B1 = 65536;                // K^ hi | lo: 2 x [2 kb][32][64] bf16 (16 KB)
  static constexpr uint32_t B1_LO = 65536 + 8192;
  static constexpr uint32_t XLOG = B1;                 // staging: bf16 [32][k 128 | v 128] log rows
  static constexpr uint32_t KF = 81920;                // K^ fp32 [32][132] (rows padded: distinct banks)
  static constexpr int KF_LD = 132;
  static constexpr uint32_t AM = KF + 32 * KF_LD * 4;  // fp32 [32][32]: A (strictly lower)
  static constexpr uint32_t XWIN = AM;                 // staging: bf16 [3][256] window rows
  static constexpr uint32_t GATE = AM + 4096;          // fp32 [5][32]: G, gam, b, fk, exp(G_n-1 - G)
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

// Eight fp32 values as bf16 hi and lo parts (x ~= hi + lo), converted in
// pairs, each part stored as one 16-byte vector.
__device__ __forceinline__ void flush_split8(uint8_t* hi, uint8_t* lo, const float* e) {
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(e[2 * u], e[2 * u + 1]);
    const float2 hf = __bfloat1622float2(hb);
    const __nv_bfloat162 lb = __floats2bfloat162_rn(e[2 * u] - hf.x, e[2 * u + 1] - hf.y);
    hw[u] = *reinterpret_cast<const uint32_t*>(&hb);
    lw[u] = *reinterpret_cast<const uint32_t*>(&lb);
  }
  *reinterpret_cast<uint4*>(hi) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4*>(lo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

template <int NMAX>
__device__ __forceinline__ void tc_flush_body(const ScanParams& p, const CUtensorMap* tmap, int h, int r,
                                              int32_t page, int n) {
  using TIN = __nv_bfloat16;
  constexpr int D = kTcD;
  constexpr int LD = TcSmem::KF_LD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127;                 // state row / channel of this thread
  const int half = tid >> 7;                 // which 64 columns (and which conv channel) it takes
  const uint32_t tlane = (uint32_t)((warp & 3) * 32) << 16;

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

  // (0) the state, 64 KB of fp32, starts arriving by four TMA tile loads into
  // the A1 region; everything up to step (5) needs no state and overlaps it
  if (warp == 0) {
    tc::tmem_alloc(tslot, kTcCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(mbar, 1);
    tc::mbar_init(mbar_tma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tc::mbar_expect_tx(mbar_tma, D * D * 4);
#pragma unroll
    for (int cb = 0; cb < 4; ++cb)
      tc::tma_load_3d(sm + TcSmem::A1 + cb * 16384, tmap, 32 * cb, h * D, page, mbar_tma);
  }
  // (1) async copies of this CTA's pre-conv rows (k | v channels: the
  // window's three rows and the log's NMAX rows, zeros past n) and of the
  // gates (zeros past n)
  const int G = p.Hv / p.Hqk, jq = h / G;
  const int ck0 = p.Hqk * D + jq * D, cv0 = 2 * p.Hqk * D + h * D;
  TIN* win = page_window<TIN>(p.pool, page);
  {
    const TIN* lx = reinterpret_cast<const TIN*>(p.log_x) + (int64_t)r * kTcMaxRows * p.conv_dim;
    constexpr int RC = 2 * D / 8;                     // 16-byte chunks per staged row
    for (int i = tid; i < (3 + NMAX) * RC; i += kTcThreads) {
      const int srow = i / RC, col = (i - srow * RC) * 8;
      const int ch = col < D ? ck0 + col : cv0 + col - D;
      const bool in = srow < 3 + n;
      const TIN* src = srow < 3 ? win + (int64_t)srow * p.conv_dim + ch
                                : lx + (int64_t)(in ? srow - 3 : 0) * p.conv_dim + ch;
      TIN* dst = srow < 3 ? xwin + srow * 2 * D + col : xlog + (srow - 3) * 2 * D + col;
      cp_async16(dst, src, in ? 16 : 0);
    }
    if (tid < 2 * NMAX) {
      const int lr = tid >> 1;
      const bool in = lr < n;
      const int64_t lrow = (int64_t)r * kTcMaxRows + (in ? lr : 0);
      cp_async4((tid & 1) ? bs + lr : Gs + lr, ((tid & 1) ? p.log_beta : p.log_g) + lrow * p.Hv + h, in ? 4 : 0);
    }
    cp_async_commit();
  }
  // conv taps: the first half of the CTA takes k channel `row`, the second v channel `row`
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)((half ? cv0 : ck0) + row) * kConvK);
  cp_async_wait<0>();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;

  // (2) conv + SiLU over all NMAX rows (zero inputs past n), masked to zero
  // past n: k channel -> kf; v channel -> tensor memory (lane = state row),
  // and its new conv window (the last three rows of window || log), written
  // to the page here: this CTA alone reads this head's v channels
  {
    const TIN* xw = xwin + half * D + row;
    const TIN* xl = xlog + half * D + row;
    float x[NMAX + 3];
#pragma unroll
    for (int i = 0; i < 3; ++i) x[i] = to_f32(xw[i * 2 * D]);
#pragma unroll
    for (int i = 0; i < NMAX; ++i) x[i + 3] = to_f32(xl[i * 2 * D]);
    float y[32];
#pragma unroll
    for (int i = 0; i < NMAX; ++i) {
      float z = w.x * x[i];
      z = fmaf(w.y, x[i + 1], z);
      z = fmaf(w.z, x[i + 2], z);
      z = fmaf(w.w, x[i + 3], z);
      y[i] = (i < n ? 1.f : 0.f) * silu_fast(z);
    }
    if (half == 0) {
#pragma unroll
      for (int i = 0; i < NMAX; ++i) kf[i * LD + row] = y[i];
#pragma unroll
      for (int i = NMAX; i < kTcMaxRows; ++i) kf[i * LD + row] = 0.f;
    } else {
#pragma unroll
      for (int i = NMAX; i < 32; ++i) y[i] = 0.f;
      tc::tmem_st32(tbase + tlane + kColV, y);
      TIN* wdst = win + cv0 + row;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int t = n + j;   // position in window || log
        wdst[(int64_t)j * p.conv_dim] = t < 3 ? xw[t * 2 * D] : xl[(t - 3) * 2 * D];
      }
      tc::tmem_st_wait();
    }
  }
  __syncthreads();
  // (3) squared norms of the k rows: warp w reduces rows w, w+8, ...
  // (interleaved, fixed order); cumulative log decay and the decay factors
  // (gates are zero past n)
  {
    constexpr int RPW = NMAX / 8;
    float ss[RPW];
#pragma unroll
    for (int it = 0; it < RPW; ++it) {
      const int i = warp + 8 * it;
      float a = 0.f;
#pragma unroll
      for (int m = 0; m < D / 32; ++m) {
        const float y = kf[i * LD + lane + 32 * m];
        a = fmaf(y, y, a);
      }
      ss[it] = a;
    }
#pragma unroll
    for (int it = 0; it < RPW; ++it) ss[it] = warp_sum(ss[it]);
    if (lane == 0) {
#pragma unroll
      for (int it = 0; it < RPW; ++it) fk[warp + 8 * it] = 1.0f / sqrtf(ss[it] + p.eps);
    }
  }
  if (warp == 1) {
    float g = lane < NMAX ? Gs[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, g, o);
      if (lane >= o) g += t;
    }
    const float gn = __shfl_sync(0xffffffffu, g, n - 1);
    if (lane < NMAX) { Gs[lane] = g; gam[lane] = expf(g); dec[lane] = expf(gn - g); }
  }
  __syncthreads();

  // (4) k^ = k / |k| (channel `row`, rows of this thread's half) and
  // B1 = K^ hi / lo (rows i < NMAX)
  const int NB1 = NMAX;
  {
    constexpr int HR = NMAX / 2;
    float kv[HR];
#pragma unroll
    for (int u = 0; u < HR; ++u) kv[u] = kf[(half * HR + u) * LD + row] * fk[half * HR + u];
#pragma unroll
    for (int u = 0; u < HR; ++u) {
      const int i = half * HR + u;
      kf[i * LD + row] = kv[u];
      __nv_bfloat16 hi, lo;
      tc::split_bf16(kv[u], hi, lo);
      const uint32_t off = tc::sw128_offset(i, row, NB1);
      *reinterpret_cast<__nv_bfloat16*>(sm + TcSmem::B1 + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(sm + TcSmem::B1_LO + off) = lo;
    }
  }
  __syncthreads();
  // A_ij = b_i exp(G_i - G_j) k^_i.k^_j for j < i < NMAX (rows past n are
  // zero), one pair per thread and round; padded rows put the two operand
  // rows of a warp's lanes on distinct banks
  for (int q = tid; q < NMAX * (NMAX - 1) / 2; q += kTcThreads) {
    int i = (int)((1.0f + sqrtf(1.0f + 8.0f * (float)q)) * 0.5f);
    if (i * (i - 1) / 2 > q) --i;
    if ((i + 1) * i / 2 <= q) ++i;
    const int j = q - i * (i - 1) / 2;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 4
    for (int c = 0; c < D; c += 8) {
      const float4 x0 = *reinterpret_cast<const float4*>(kf + i * LD + c);
      const float4 y0 = *reinterpret_cast<const float4*>(kf + j * LD + c);
      const float4 x1 = *reinterpret_cast<const float4*>(kf + i * LD + c + 4);
      const float4 y1 = *reinterpret_cast<const float4*>(kf + j * LD + c + 4);
      a0 = fmaf(x0.x, y0.x, a0); a1 = fmaf(x0.y, y0.y, a1); a2 = fmaf(x0.z, y0.z, a2); a3 = fmaf(x0.w, y0.w, a3);
      a0 = fmaf(x1.x, y1.x, a0); a1 = fmaf(x1.y, y1.y, a1); a2 = fmaf(x1.z, y1.z, a2); a3 = fmaf(x1.w, y1.w, a3);
    }
    am[i * 32 + j] = bs[i] * __expf(fminf(Gs[i] - Gs[j], 0.f)) * ((a0 + a1) + (a2 + a3));
  }

  // (5) the state: columns [64 half, +64) of row `row` into registers; once
  // every thread holds its part the region takes the bf16 hi / lo operand
  // A1, and gam_{n-1} S0 goes to the D2 columns
  bool ok = tc::mbar_wait_bounded(mbar_tma, 0, kWaitCycles);
  ok = __syncthreads_and(ok);
  if (!ok) {   // the state never arrived: report, give the copy one more bounded wait, leave
    if (tid == 0) set_error(p.err, GDN_ERR_TIMEOUT);
    tc::mbar_wait_bounded(mbar_tma, 0, kWaitCycles);
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, kTcCols);
    return;
  }
  {
    float sv[64];
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      const float4 f = *reinterpret_cast<const float4*>(sm + TcSmem::A1 + state_smem_offset(row, 64 * half + c));
      sv[c] = f.x; sv[c + 1] = f.y; sv[c + 2] = f.z; sv[c + 3] = f.w;
    }
    __syncthreads();
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint32_t off = tc::sw128_offset(row, 64 * half + 8 * c8, D);
      flush_split8(sm + TcSmem::A1 + off, sm + TcSmem::A1_LO + off, sv + 8 * c8);
    }
    const float gN = gam[n - 1];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float v[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] = gN * sv[32 * q + c];
      tc::tmem_st32(tbase + tlane + 32 + 64 * half + 32 * q, v);
    }
    tc::tmem_st_wait();
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // (6) D1 = S0 K^T on the tensor cores (three bf16 passes, K = 128)
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

  // (7) wait for D1.  First half, state row `row`: R_i = b_i (v_i[r] - gam_i
  // D1[r][i]), (I + A) U = R by forward substitution, W_i = U_i exp(G_{n-1} -
  // G_i) -> A2 row `row`.  Second half: K^T (row = k channel) -> B2.  Both go
  // to the A1 region, which D1's product no longer reads; the second product
  // reads K = NMAX <= 32 columns of them.
  ok = tc::mbar_wait_bounded(mbar, 0, kWaitCycles);
  ok = __syncthreads_and(ok);
  tc::fence_after_sync();
  if (ok) {
    if (half == 0) {
      float d1[32], vr[32];
      tc::tmem_ld32x2(tbase + tlane, tbase + tlane + kColV, d1, vr);
      float u[NMAX];
#pragma unroll
      for (int i = 0; i < NMAX; ++i) u[i] = bs[i] * fmaf(-gam[i], d1[i], vr[i]);
#pragma unroll
      for (int j = 0; j < NMAX; ++j)
#pragma unroll
        for (int i = j + 1; i < NMAX; ++i) u[i] = fmaf(-am[i * 32 + j], u[j], u[i]);
#pragma unroll
      for (int i = 0; i < NMAX; ++i) u[i] *= dec[i];
#pragma unroll
      for (int c8 = 0; c8 < NMAX / 8; ++c8) {
        const uint32_t off = tc::sw128_offset(row, 8 * c8, D);
        flush_split8(sm + TcSmem::A2 + off, sm + TcSmem::A2_LO + off, u + 8 * c8);
      }
    } else {
      float kt[NMAX];
#pragma unroll
      for (int i = 0; i < NMAX; ++i) kt[i] = kf[i * LD + row];
#pragma unroll
      for (int c8 = 0; c8 < NMAX / 8; ++c8) {
        const uint32_t off = tc::sw128_offset(row, 8 * c8, D);
        flush_split8(sm + TcSmem::B2 + off, sm + TcSmem::B2_LO + off, kt + 8 * c8);
      }
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // (8) D2 += W K^ on the tensor cores (three bf16 passes, K = NMAX)
  if (ok && tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(D, D);
    constexpr int nks = NMAX / 16;
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

  // (9) D2 = gam_{n-1} S0 + W K^ is the new state: each thread parks its 64
  // columns in the A1 region (free once the second product has completed) in
  // the tensor map's swizzled layout, then four TMA tile stores write it back
  if (ok) {
    float d2[32], d3[32];
    tc::tmem_ld32x2(tbase + tlane + 32 + 64 * half, tbase + tlane + 64 + 64 * half, d2, d3);
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      *reinterpret_cast<float4*>(sm + TcSmem::A1 + state_smem_offset(row, 64 * half + c)) =
          make_float4(d2[c], d2[c + 1], d2[c + 2], d2[c + 3]);
      *reinterpret_cast<float4*>(sm + TcSmem::A1 + state_smem_offset(row, 64 * half + 32 + c)) =
          make_float4(d3[c], d3[c + 1], d3[c + 2], d3[c + 3]);
    }
    tc::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::tma_store_3d(tmap, 32 * cb, h * D, page, sm + TcSmem::A1 + cb * 16384);
      tc::bulk_commit();
      tc::bulk_wait_read();
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

// After the tensor-core flush (which read the k windows and rewrote the v
// windows): the q and k channels of every request's conv window (the last
// three rows of window || log), then log_len = 0.  One CTA per request; a
// thread moves 16-byte chunks (8 channels) and reads a chunk's three source
// rows before it writes them; log_len is cleared once every thread of the
// request has read it.
constexpr int kQkWinThreads = 512;
__global__ void __launch_bounds__(kQkWinThreads) flush_qk_window_kernel(const ScanParams p) {
  using TIN = __nv_bfloat16;
  const int r = blockIdx.x;
  const int32_t page = p.ckpt_slot[r];
  const int32_t n = p.log_len[r];
  if (!page_ok(p.pool, page) || n < 0 || n > kTcMaxRows) return;   // reported by the flush kernel
  if (n > 0) {
    TIN* win = page_window<TIN>(p.pool, page);
    const TIN* lx = reinterpret_cast<const TIN*>(p.log_x) + (int64_t)r * kTcMaxRows * p.conv_dim;
    const int chunks = 2 * p.Hqk * kTcD / 8;
    for (int c = threadIdx.x; c < chunks; c += kQkWinThreads) {
      uint4 keep[kWinRows];
#pragma unroll
      for (int j = 0; j < kWinRows; ++j) {
        const int t = n + j;   // position in window || log
        const TIN* src = t < kWinRows ? win + (int64_t)t * p.conv_dim : lx + (int64_t)(t - kWinRows) * p.conv_dim;
        keep[j] = *reinterpret_cast<const uint4*>(src + 8 * c);
      }
#pragma unroll
      for (int j = 0; j < kWinRows; ++j) *reinterpret_cast<uint4*>(win + (int64_t)j * p.conv_dim + 8 * c) = keep[j];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) const_cast<int32_t*>(p.log_len)[r] = 0;
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
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  flush_qk_window_kernel<<<p.num_seqs, kQkWinThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
