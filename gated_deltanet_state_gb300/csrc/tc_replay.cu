// tc_replay.cu — replay verification (append) and flush on the tensor cores
// ("Caching less to serve more requests", section "What we changed": one
// checkpoint state per request plus a log of the per-token inputs since it;
// a step's outputs are computed from the two, and the flush applies the kept
// rows to the state as one block of matrix operations, one launch per layer).
//
// One CTA takes one (value head h, request r) pair and L <= 32 rows at once:
// the n logged rows (flush), or the n logged rows followed by the m new rows
// (append, L = n + m).  From the checkpoint state S0 (dv x dk = 128 x 128,
// fp32), in the chunk (UT) form of the gated delta rule:
//   G_i = sum_{l<=i} g_l,  gam_i = exp(G_i),  k^_i = fk_i k_i,  q^_i = fq_i q_i
//   A_ij = b_i exp(G_i - G_j) k^_i.k^_j  (j < i),    T = (I + A)^-1
//   R_i  = b_i (v_i - gam_i S0 k^_i),                U = T R
// flush:   S = gam_{L-1} S0 + sum_i exp(G_{L-1} - G_i) u_i k^_i^T
//            = gam_{L-1} S0 + R^T Kt,   Kt = T^T diag(exp(G_{L-1} - G)) K^
// append:  o_i = gam_i S0 q^_i + sum_{j<=i} exp(G_i - G_j) (q^_i.k^_j) u_j
//              = gam_i fq_i (S0 q_i) + (Pt R)_i,  Pt = P T,
//          P_ij = exp(G_i - G_j) q^_i.k^_j  (j <= i), for the m new rows i.
// Whatever does not involve S0 is formed while the state's TMA load is in
// flight: the Gram matrix of the raw [K; Q] rows on the tensor cores (its
// diagonal gives the L2 norms), A and P from it, and Kt or Pt by triangular
// solves.  The state then meets D1 = S0 [K; Q]^T on the tensor cores, R is
// elementwise, and the flush ends with S += R^T Kt on the tensor cores.
// Every product reads bf16 operands split into hi + lo parts (three passes:
// hi*hi + hi*lo + lo*hi), about 16 bits per operand, fp32 accumulation in
// tensor memory.
#include "launch.h"
#include "tc.cuh"

namespace gdn {

constexpr int kRpThreads = 256;        // two threads per state row
constexpr int kRpD = 128;              // dk = dv
constexpr int kRpMaxRows = GDN_REPLAY_LOG_SLOTS;
constexpr uint32_t kRpCols = 256;      // tensor-memory columns of one CTA
constexpr long long kRpWait = 4000000000LL;

// Shared-memory plan (byte offsets from a 1024-byte aligned base).  NB1 rows
// of raw operand rows: the k rows (flush), or the k rows then the q rows
// (append).
template <int NMAX, bool APPEND>
struct RpSmem {
  static constexpr int NB1 = APPEND ? 2 * NMAX : NMAX;
  static constexpr int CH = APPEND ? 3 * kRpD : 2 * kRpD;     // staged channels: [q |] k | v
  static constexpr uint32_t A1 = 0;         // S0 fp32 (TMA) -> S0 hi | lo [2 kb][128][64] bf16 (64 KB)
  static constexpr uint32_t A1_LO = 32768;
  static constexpr uint32_t A2 = 0;         // flush: R^T hi | lo [128][64] bf16 (after D1)
  static constexpr uint32_t A2_LO = 16384;
  static constexpr uint32_t B2 = 32768;     // flush: Kt^T hi | lo [128][64] bf16 (after D1)
  static constexpr uint32_t B2_LO = 49152;
  static constexpr uint32_t B1 = 65536;     // raw rows hi | lo [2 kb][NB1][64] bf16
  static constexpr uint32_t B1_LO = B1 + 2 * NB1 * 128;
  static constexpr uint32_t B1_END = B1_LO + 2 * NB1 * 128;
  // staging of the pre-conv rows: append: [3 + NMAX][q | k | v] in the B1
  // region; flush: log rows [NMAX][k | v] in B1, window rows [3][k | v] in AM
  static constexpr uint32_t XS = B1;
  static constexpr uint32_t KF = B1_END;    // flush: raw k fp32 [NMAX][KF_LD]
  static constexpr int KF_LD = 132;
  static constexpr int AM_LD = 36;          // rows of A: 16-byte aligned, distinct banks
  static constexpr uint32_t AM = APPEND ? B1_END : KF + NMAX * KF_LD * 4;   // A fp32 [32][AM_LD]
  static constexpr uint32_t XWIN = AM;      // flush staging of the window rows
  static constexpr uint32_t PT = AM + 32 * AM_LD * 4;                          // append: P T fp32 [32][32]
  static constexpr uint32_t GATE = PT + (APPEND ? 4096 : 0);   // fp32 [8][32]: G, gam, b, fk, fq, dec
  static constexpr uint32_t MBAR = GATE + 1024;                // 4 mbarriers: state, Gram, D1, S
  static constexpr uint32_t TSLOT = MBAR + 32;
  // the Gram product reads 128 rows of 128 B from each start in B1: rows past
  // NB1 are other data of this CTA (their results are not used), in bounds
  static constexpr uint32_t GRAM_READ_END = B1_LO + NB1 * 128 + 16384;
  static constexpr uint32_t BYTES = TSLOT + 16 > GRAM_READ_END ? TSLOT + 16 : GRAM_READ_END;
  static_assert(APPEND ? (3 + NMAX) * CH * 2 <= 4 * NB1 * 128 : NMAX * CH * 2 <= 4 * NB1 * 128,
                "staged log rows fit the B1 region");
  static_assert(APPEND || 3 * CH * 2 <= 32 * AM_LD * 4, "staged window rows fit the A region");
  static constexpr uint32_t ALLOC = BYTES + 1024;
};
// tensor-memory columns
template <bool APPEND>
struct RpCols {
  static constexpr uint32_t D1 = 0;                        // S0 [K; Q]^T: NB1 columns
  static constexpr uint32_t D2 = 32;                       // flush: the new state (128)
  static constexpr uint32_t V = APPEND ? 64 : 160;         // conv'd v (lane = channel), 32
  static constexpr uint32_t G = APPEND ? 96 : 192;         // Gram [K; Q][K; Q]^T, NB1 columns
};

// The state of (page, head h) is the box set {x: 0..127 in 32-column boxes,
// y: h*128 .. +127, z: page} of a 3-D tensor map over the pool:
// [page][head row][column] fp32, boxes of 128 rows x 32 columns (128 B) in the
// 128-byte swizzled shared layout.
__device__ __forceinline__ uint32_t rp_state_offset(int row, int col) {
  return (uint32_t)((col >> 5) * 16384 + row * 128 + ((((col & 31) >> 2) ^ (row & 7)) << 4) + ((col & 3) << 2));
}

// Diagonal entry `lane` of a register row (a select chain: no local memory).
template <int N>
__device__ __forceinline__ float rp_pick(const float (&v)[N], int idx) {
  float d = 0.f;
#pragma unroll
  for (int c = 0; c < N; ++c) d = c == idx ? v[c] : d;
  return d;
}

// x_l = rhs_l - sum_{j > l} A_jl x_j for l = NMAX-1 .. 0 (A strictly lower
// triangular, am[j][l] = A_jl, rows AM_LD apart), right-looking: once x_j is
// final, every x_l (l < j) takes its term, so the chain is one FMA per row.
// Used for Kt columns ((I + A^T) x = dec k^) and for rows of P T
// (x (I + A) = P_i.).
template <int NMAX, int LD>
__device__ __forceinline__ void rp_back_solve(float (&x)[NMAX], const float* am) {
#pragma unroll
  for (int j = NMAX - 1; j > 0; --j) {
    float a[NMAX];
#pragma unroll
    for (int l4 = 0; l4 < j; l4 += 4) {
      const float4 v = *reinterpret_cast<const float4*>(am + j * LD + l4);   // same address in every thread
      a[l4] = v.x; a[l4 + 1] = v.y; a[l4 + 2] = v.z; a[l4 + 3] = v.w;
    }
#pragma unroll
    for (int l = 0; l < j; ++l) x[l] = fmaf(-a[l], x[j], x[l]);
  }
}

// BND: a flush that also writes a block-boundary checkpoint after its first
// bj kept rows (a separate instantiation: the common path compiles as if the
// boundary code did not exist).
template <int NMAX, bool APPEND, bool BND = false>
__device__ __forceinline__ void replay_body(const ScanParams& p, const CUtensorMap* tmap, int h, int r,
                                            int32_t page, int n, int L, int bj_arg = 0, int32_t bpage = -1) {
  const int bj = BND ? bj_arg : 0;
  using TIN = __nv_bfloat16;
  using S = RpSmem<NMAX, APPEND>;
  using C = RpCols<APPEND>;
  constexpr int D = kRpD;
  constexpr int NB1 = S::NB1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127;                 // state row / channel of this thread
  const int half = tid >> 7;
  const uint32_t tlane = (uint32_t)((warp & 3) * 32) << 16;

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  float* Gs = reinterpret_cast<float*>(sm + S::GATE);
  float* gam = Gs + 32;
  float* bs = Gs + 64;
  float* fk = Gs + 96;
  float* fq = Gs + 128;
  float* dec = Gs + 160;
  float* am = reinterpret_cast<float*>(sm + S::AM);
  float* pt = reinterpret_cast<float*>(sm + S::PT);
  float* kf = reinterpret_cast<float*>(sm + S::KF);
  uint64_t* mbar_tma = reinterpret_cast<uint64_t*>(sm + S::MBAR);
  uint64_t* mbar_g = mbar_tma + 1;
  uint64_t* mbar_1 = mbar_tma + 2;
  uint64_t* mbar_2 = mbar_tma + 3;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::TSLOT);
  TIN* xs = reinterpret_cast<TIN*>(sm + S::XS);
  TIN* xwin = reinterpret_cast<TIN*>(sm + (APPEND ? S::XS : S::XWIN));
  TIN* xlog = APPEND ? xs + 3 * S::CH : xs;

  // (0) the state (64 KB of fp32) starts arriving by four TMA tile loads into
  // A1; nothing before step (4) needs it
  if (warp == 0) {
    tc::tmem_alloc(tslot, kRpCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(mbar_tma, 1);
    tc::mbar_init(mbar_g, 1);
    tc::mbar_init(mbar_1, 1);
    tc::mbar_init(mbar_2, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tc::mbar_expect_tx(mbar_tma, D * D * 4);
#pragma unroll
    for (int cb = 0; cb < 4; ++cb)
      tc::tma_load_3d(sm + S::A1 + cb * 16384, tmap, 32 * cb, h * D, page, mbar_tma);
  }
  // (1) async copies of this CTA's pre-conv channels ([q |] k | v) of the
  // window's three rows and of the L rows (the log, then the new rows), zeros
  // past L, and of the gates (zeros past L)
  const int G = p.Hv / p.Hqk, jq = h / G;
  const int cq0 = jq * D, ck0 = p.Hqk * D + jq * D, cv0 = 2 * p.Hqk * D + h * D;
  TIN* win = page_window<TIN>(p.pool, page);
  const TIN* lx = reinterpret_cast<const TIN*>(p.log_x) + (int64_t)r * kRpMaxRows * p.conv_dim;
  const TIN* nx = APPEND ? reinterpret_cast<const TIN*>(p.x_new) + (int64_t)r * p.num_new * p.conv_dim : nullptr;
  {
    constexpr int RC = S::CH / 8;                     // 16-byte chunks per staged row
    for (int i = tid; i < (3 + NMAX) * RC; i += kRpThreads) {
      const int srow = i / RC, col = (i - srow * RC) * 8;
      const int part = col / D;                       // append: 0 q, 1 k, 2 v; flush: 0 k, 1 v
      const int ch = (APPEND ? (part == 0 ? cq0 : part == 1 ? ck0 : cv0) : (part == 0 ? ck0 : cv0)) + col - part * D;
      const int t = srow - 3;                         // row of the L rows (negative: window)
      const bool in = t < L;                          // past L: zero fill from a valid address
      const TIN* src = (t < 0 || !in) ? win + (int64_t)(in ? srow : 0) * p.conv_dim + ch
                     : (!APPEND || t < n) ? lx + (int64_t)t * p.conv_dim + ch
                                          : nx + (int64_t)(t - n) * p.conv_dim + ch;
      TIN* dst = t < 0 ? xwin + srow * S::CH + col : xlog + t * S::CH + col;
      cp_async16(dst, src, in ? 16 : 0);
    }
    if (tid < 2 * 32) {
      const int t = tid >> 1;
      const bool in = t < L;
      const bool logged = !in || !APPEND || t < n;
      const float* base = (tid & 1) ? (logged ? p.log_beta : p.beta_new) : (logged ? p.log_g : p.g_new);
      const int64_t grow = logged ? (int64_t)r * kRpMaxRows + (in ? t : 0) : (int64_t)r * p.num_new + (t - n);
      cp_async4((tid & 1) ? bs + t : Gs + t, base + grow * p.Hv + h, in ? 4 : 0);
    }
    cp_async_commit();
  }
  // conv taps of the channels this thread convolves
  const int cc = APPEND ? (half ? ck0 + row : cq0 + row) : (half ? cv0 + row : ck0 + row);
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)cc * kConvK);
  const float4 wv = APPEND ? *reinterpret_cast<const float4*>(p.conv_w + (int64_t)(cv0 + row) * kConvK) : w;
  cp_async_wait<0>();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;

  // (2) conv + SiLU of one channel over the NMAX rows (zero past L).  The
  // staged rows share their region with B1, so every thread first takes what
  // it needs from them into registers (and tensor memory), then, after a
  // barrier, writes the operand rows.
  // append: every thread one q (first half) or k channel -> raw rows of B1;
  //   the first half first one v channel -> tensor memory; the second half
  //   then copies the new rows into the log.
  // flush: first half one k channel -> B1 and kf; second half one v channel
  //   -> tensor memory, and its new conv window (the last three rows of
  //   window || log) to the page (this CTA alone reads this head's v channels).
  float y[32];
  TIN wv3[3], wb3[3];
  {
    auto conv_col = [&](int sc, const float4& cw) {
      float x[NMAX + 3];
#pragma unroll
      for (int i = 0; i < 3; ++i) x[i] = to_f32(xwin[i * S::CH + sc]);
#pragma unroll
      for (int i = 0; i < NMAX; ++i) x[i + 3] = to_f32(xlog[i * S::CH + sc]);
#pragma unroll
      for (int i = 0; i < NMAX; ++i) {
        float z = cw.x * x[i];
        z = fmaf(cw.y, x[i + 1], z);
        z = fmaf(cw.z, x[i + 2], z);
        z = fmaf(cw.w, x[i + 3], z);
        y[i] = (i < L ? 1.f : 0.f) * silu_fast(z);
      }
#pragma unroll
      for (int i = NMAX; i < 32; ++i) y[i] = 0.f;
    };
    if (APPEND && half == 0) {
      conv_col(2 * D + row, wv);                       // v channel -> tensor memory
      tc::tmem_st32(tbase + tlane + C::V, y);
      tc::tmem_st_wait();
    }
    conv_col(half * D + row, w);                       // append: q | k; flush: k | v
    if (!APPEND && half == 1) {
      tc::tmem_st32(tbase + tlane + C::V, y);
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int t = n + j, tb = bj + j;   // positions in window || log
        wv3[j] = t < 3 ? xwin[t * S::CH + D + row] : xlog[(t - 3) * S::CH + D + row];
        if (BND) wb3[j] = tb < 3 ? xwin[tb * S::CH + D + row] : xlog[(tb - 3) * S::CH + D + row];
      }
      tc::tmem_st_wait();
    }
  }
  __syncthreads();   // the staged rows have been read
  if (APPEND || half == 0) {
    // raw operand row: k rows at 0..NMAX-1, q rows (append) at NMAX..
    const int brow0 = (APPEND && half == 0) ? NMAX : 0;
#pragma unroll
    for (int i = 0; i < NMAX; ++i) {
      __nv_bfloat16 hi, lo;
      tc::split_bf16(y[i], hi, lo);
      const uint32_t off = tc::sw128_offset(brow0 + i, row, NB1);
      *reinterpret_cast<__nv_bfloat16*>(sm + S::B1 + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(sm + S::B1_LO + off) = lo;
      if (!APPEND) kf[i * S::KF_LD + row] = y[i];
    }
  } else {
    TIN* wdst = win + cv0 + row;
#pragma unroll
    for (int j = 0; j < 3; ++j) wdst[(int64_t)j * p.conv_dim] = wv3[j];
    if (BND) {
      TIN* bdst = page_window<TIN>(p.pool, bpage) + cv0 + row;
#pragma unroll
      for (int j = 0; j < 3; ++j) bdst[(int64_t)j * p.conv_dim] = wb3[j];
    }
  }
  if (APPEND && half == 1) {
    // the m new rows join the log after the n logged ones: this head's v
    // channels and gates; the first head of a qk group also its q and k
    // channels (rows n.. are read by no CTA of this launch)
    const int m = L - n;
    TIN* ldst = const_cast<TIN*>(lx) + (int64_t)n * p.conv_dim;
    const int t2 = tid - 128;
    for (int i = t2; i < m * (D / 8); i += 128) {
      const int t = i / (D / 8), c8 = (i - t * (D / 8)) * 8;
      *reinterpret_cast<uint4*>(ldst + (int64_t)t * p.conv_dim + cv0 + c8) =
          *reinterpret_cast<const uint4*>(nx + (int64_t)t * p.conv_dim + cv0 + c8);
    }
    if (h % G == 0) {
      for (int i = t2; i < m * (2 * D / 8); i += 128) {
        const int t = i / (2 * D / 8), c8 = (i - t * (2 * D / 8)) * 8;
        const int ch = c8 < D ? cq0 + c8 : ck0 + c8 - D;
        *reinterpret_cast<uint4*>(ldst + (int64_t)t * p.conv_dim + ch) =
            *reinterpret_cast<const uint4*>(nx + (int64_t)t * p.conv_dim + ch);
      }
    }
    if (t2 < m) {
      const int64_t lrow = (int64_t)r * kRpMaxRows + n + t2, nrow = (int64_t)r * m + t2;
      const_cast<float*>(p.log_g)[lrow * p.Hv + h] = p.g_new[nrow * p.Hv + h];
      const_cast<float*>(p.log_beta)[lrow * p.Hv + h] = p.beta_new[nrow * p.Hv + h];
    }
  }
  // cumulative log decay and the decay factors (gates are zero past L)
  if (warp == 1) {
    float g = Gs[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, g, o);
      if (lane >= o) g += t;
    }
    const float gn = __shfl_sync(0xffffffffu, g, L - 1);
    __syncwarp();
    Gs[lane] = g;
    gam[lane] = expf(g);
    dec[lane] = expf(gn - g);
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // (3) the Gram matrix of the raw rows: D_G = B1 B1^T (M = 128: rows past
  // NB1 are other data of this CTA and their lanes are not read).  The
  // products are issued by one thread of warp 7, which has no other work
  // while they run.
  constexpr int kIssue = 224;
  if (tid == kIssue) {
    const uint32_t idesc = tc::idesc_bf16_f32(128, NB1);
    for (int pass = 0; pass < 3; ++pass) {
      const uint32_t a = sbase + (pass == 2 ? S::B1_LO : S::B1);
      const uint32_t b = sbase + (pass == 1 ? S::B1_LO : S::B1);
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t kb = ks >> 2, koff = (ks & 3) * 32;
        tc::mma_bf16(tbase + C::G, tc::desc_sw128(a + kb * NB1 * 128 + koff),
                     tc::desc_sw128(b + kb * NB1 * 128 + koff), idesc, (pass | ks) != 0);
      }
    }
    tc::mma_commit(mbar_g);
  }
  // (4) the state: columns [64 half, +64) of row `row` into registers; the
  // region then takes the bf16 hi / lo operand A1; the flush puts
  // gam_{L-1} S0 in the D2 columns
  const bool ok_tma = tc::mbar_wait_bounded(mbar_tma, 0, kRpWait);
  bool ok = __syncthreads_and(ok_tma);
  if (!ok) {   // a wait ran out: report, give the copies and products one more bounded wait, leave
    if (tid == 0) set_error(p.err, GDN_ERR_TIMEOUT);
    tc::mbar_wait_bounded(mbar_tma, 0, kRpWait);
    tc::mbar_wait_bounded(mbar_g, 0, kRpWait);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, kRpCols);
    return;
  }
  {
    float sv[64];
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      const float4 f = *reinterpret_cast<const float4*>(sm + S::A1 + rp_state_offset(row, 64 * half + c));
      sv[c] = f.x; sv[c + 1] = f.y; sv[c + 2] = f.z; sv[c + 3] = f.w;
    }
    __syncthreads();
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint32_t off = tc::sw128_offset(row, 64 * half + 8 * c8, D);
      tc::store_split8(sm + S::A1 + off, sm + S::A1_LO + off, sv + 8 * c8);
    }
    if (!APPEND) {
      const float gN = gam[(BND ? bj : L) - 1];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = gN * sv[32 * q + c];
        tc::tmem_st32(tbase + tlane + C::D2 + 64 * half + 32 * q, v);
      }
      tc::tmem_st_wait();
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // (5) D1 = S0 B1^T on the tensor cores (K = 128)
  if (tid == kIssue) {
    const uint32_t idesc = tc::idesc_bf16_f32(D, NB1);
    for (int pass = 0; pass < 3; ++pass) {
      const uint32_t a = sbase + (pass == 2 ? S::A1_LO : S::A1);
      const uint32_t b = sbase + (pass == 1 ? S::B1_LO : S::B1);
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t kb = ks >> 2, koff = (ks & 3) * 32;
        tc::mma_bf16(tbase + C::D1, tc::desc_sw128(a + kb * D * 128 + koff),
                     tc::desc_sw128(b + kb * NB1 * 128 + koff), idesc, (pass | ks) != 0);
      }
    }
    tc::mma_commit(mbar_1);
  }
  // while D1 runs: norms, A and (append) P T from the Gram rows: k rows in
  // lanes 0..NMAX-1, q rows in lanes NMAX.. (warp 4 reads lanes 0-31, warp 5
  // lanes 32-63); the barrier after them publishes fk, fq, A^T and P T
  const bool gram_warp = warp == 4 || (APPEND && NMAX == 32 && warp == 5);
  bool okg = true;
  if (gram_warp) {
    okg = tc::mbar_wait_bounded(mbar_g, 0, kRpWait);
    okg = __all_sync(0xffffffffu, okg);
    tc::fence_after_sync();
    const int grow = (warp - 4) * 32 + lane;          // Gram row of this lane
    const bool is_k = grow < NMAX;
    const int i = is_k ? grow : grow - NMAX;          // row index among the L rows
    float gk[32], gq[32];
    if (okg) {
      if (APPEND && NMAX == 32) tc::tmem_ld32x2(tbase + tlane + C::G, tbase + tlane + C::G + 32, gk, gq);
      else {
        tc::tmem_ld32(tbase + tlane + C::G, gk);
#pragma unroll
        for (int c = 0; c < 32; ++c) gq[c] = 0.f;
      }
      // the diagonal: |k_i|^2 or |q_i|^2 (the q block sits at columns NMAX..)
      float dg;
      if (APPEND && NMAX == 16) dg = rp_pick(gk, grow);
      else dg = is_k ? rp_pick(gk, i) : rp_pick(gq, i);
      if (is_k) fk[i] = 1.0f / sqrtf(dg + p.eps);
      else if (APPEND) fq[i] = p.q_scale / sqrtf(dg + p.eps);
    }
    // the two Gram warps meet here whatever their waits returned
    if (APPEND && NMAX == 32) asm volatile("bar.sync 3, 64;\n" ::: "memory");
    else __syncwarp();
    if (okg && is_k) {
      // row i of A (A_ij, j < i) into registers first (no store may come
      // between the loads), then as 16-byte vectors into am
      const float ci = bs[i] * fk[i], Gi = Gs[i];
#pragma unroll
      for (int j4 = 0; j4 < NMAX; j4 += 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(Gs + j4);
        const float4 f4 = *reinterpret_cast<const float4*>(fk + j4);
        const float gj[4] = {g4.x, g4.y, g4.z, g4.w}, fj[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          // branch-free: every term is computed (all finite), the triangle is a 0 / 1 factor
          const int j = j4 + u;
          const float keep = j < i ? 1.f : 0.f;
          gk[j] = keep * (ci * __expf(fminf(Gi - gj[u], 0.f)) * fj[u] * gk[j]);
        }
      }
#pragma unroll
      for (int j4 = 0; j4 < NMAX; j4 += 4)
        *reinterpret_cast<float4*>(am + i * S::AM_LD + j4) = make_float4(gk[j4], gk[j4 + 1], gk[j4 + 2], gk[j4 + 3]);
    }
    if (APPEND && NMAX == 32) asm volatile("bar.sync 3, 64;\n" ::: "memory");
    else __syncwarp();
    if (APPEND && okg && !is_k) {
      // P_il = exp(G_i - G_l) q^_i.k^_l (l <= i), then row i of P T
      float x[NMAX];
      const float fi = fq[i], Gi = Gs[i];
#pragma unroll
      for (int l = 0; l < NMAX; ++l) {
        const float keep = (l <= i && i < L) ? 1.f : 0.f;   // branch-free, as for A
        x[l] = keep * (__expf(fminf(Gi - Gs[l], 0.f)) * fi * fk[l] * gk[l]);
      }
      rp_back_solve<NMAX, S::AM_LD>(x, am);
#pragma unroll
      for (int l = 0; l < NMAX; ++l) pt[i * 32 + l] = x[l];
    }
  }

  okg = __syncthreads_and(okg);
  ok = ok && okg;
  if (APPEND) {
    const bool ok1 = tc::mbar_wait_bounded(mbar_1, 0, kRpWait);
    ok = __syncthreads_and(ok && ok1);
    tc::fence_after_sync();
    // (6a) R_l = b_l (v_l - gam_l fk_l (S0 k_l)) for state row `row`, then the
    // outputs of the new rows i: o_i = gam_i fq_i (S0 q_i) + sum_{l<=i} Pt_il R_l
    // (rows of the first half of the CTA even i, of the second odd i)
    if (ok) {
      float rr[32], d1[32];
      tc::tmem_ld32x2(tbase + tlane + C::D1, tbase + tlane + C::V, d1, rr);
#pragma unroll
      for (int l4 = 0; l4 < NMAX; l4 += 4) {
        const float4 b4 = *reinterpret_cast<const float4*>(bs + l4);
        const float4 g4 = *reinterpret_cast<const float4*>(gam + l4);
        const float4 f4 = *reinterpret_cast<const float4*>(fk + l4);
        const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, cg[4] = {g4.x * f4.x, g4.y * f4.y, g4.z * f4.z, g4.w * f4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) rr[l4 + u] = bb[u] * fmaf(-cg[u], d1[l4 + u], rr[l4 + u]);
      }
      // S0 q_i: columns NMAX.. of D1 (loads start on 32-column boundaries)
      float dq[32];
      if (NMAX == 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) dq[i] = d1[16 + i];
      } else {
        tc::tmem_ld32(tbase + tlane + C::D1 + 32, dq);
      }
      const int m = L - n;
#pragma unroll
      for (int i = 0; i < NMAX; ++i) {
        if (i >= n && i < L && (i & 1) == half) {
          const float* prow = pt + i * 32;
          float acc = gam[i] * fq[i] * dq[i];
#pragma unroll
          for (int l = 0; l <= i; ++l) acc = fmaf(prow[l], rr[l], acc);
          const int64_t orow = ((int64_t)r * m + (i - n)) * p.Hv + h;
          reinterpret_cast<__nv_bfloat16*>(p.o)[orow * D + row] = __float2bfloat16_rn(acc);
        }
      }
    } else {
      // a wait ran out: report it, give the products one more bounded wait
      if (tid == 0) set_error(p.err, GDN_ERR_TIMEOUT);
      tc::mbar_wait_bounded(mbar_g, 0, kRpWait);
      tc::mbar_wait_bounded(mbar_1, 0, kRpWait);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, kRpCols);
    return;
  }

  // (6) flush.  First half, while D1 runs: column `row` of Kt, by back
  // substitution through (I + A^T) from dec_l k^_l, then (D1 done) Kt^T ->
  // B2.  Second half (D1 done): R^T -> A2 for state row `row`.  Both go to
  // A1, which D1's product has finished reading once its barrier fires.
  bool ok1;
  float kt[NMAX];
  if (ok && half == 0) {
    if (BND) {
      const float Gb = Gs[bj - 1];
#pragma unroll
      for (int l = 0; l < NMAX; ++l) kt[l] = l < bj ? __expf(Gb - Gs[l]) * fk[l] * kf[l * S::KF_LD + row] : 0.f;
    } else {
#pragma unroll
      for (int l = 0; l < NMAX; ++l) kt[l] = dec[l] * fk[l] * kf[l * S::KF_LD + row];
    }
    rp_back_solve<NMAX, S::AM_LD>(kt, am);
    ok1 = tc::mbar_wait_bounded(mbar_1, 0, kRpWait);
    if (ok1) {
#pragma unroll
      for (int c8 = 0; c8 < NMAX / 8; ++c8) {
        const uint32_t off = tc::sw128_offset(row, 8 * c8, D);
        tc::store_split8(sm + S::B2 + off, sm + S::B2_LO + off, kt + 8 * c8);
      }
    }
  } else if (ok && half == 1) {
    ok1 = tc::mbar_wait_bounded(mbar_1, 0, kRpWait);
    tc::fence_after_sync();
    if (ok1) {
      float rr[32], d1[32];
      tc::tmem_ld32x2(tbase + tlane + C::D1, tbase + tlane + C::V, d1, rr);
#pragma unroll
      for (int l4 = 0; l4 < NMAX; l4 += 4) {
        const float4 b4 = *reinterpret_cast<const float4*>(bs + l4);
        const float4 g4 = *reinterpret_cast<const float4*>(gam + l4);
        const float4 f4 = *reinterpret_cast<const float4*>(fk + l4);
        const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, cg[4] = {g4.x * f4.x, g4.y * f4.y, g4.z * f4.z, g4.w * f4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) rr[l4 + u] = bb[u] * fmaf(-cg[u], d1[l4 + u], rr[l4 + u]);
      }
#pragma unroll
      for (int c8 = 0; c8 < NMAX / 8; ++c8) {
        const uint32_t off = tc::sw128_offset(row, 8 * c8, D);
        tc::store_split8(sm + S::A2 + off, sm + S::A2_LO + off, rr + 8 * c8);
      }
    }
  } else {
    ok1 = tc::mbar_wait_bounded(mbar_1, 0, kRpWait);
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  ok = __syncthreads_and(ok && ok1);
  tc::fence_after_sync();

  // (7) D2 += R^T Kt on the tensor cores (K = NMAX); D2 holds gam_{L-1} S0
  if (ok && tid == kIssue) {
    const uint32_t idesc = tc::idesc_bf16_f32(D, D);
    constexpr int nks = NMAX / 16;
    for (int pass = 0; pass < 3; ++pass) {
      const uint32_t a = sbase + (pass == 2 ? S::A2_LO : S::A2);
      const uint32_t b = sbase + (pass == 1 ? S::B2_LO : S::B2);
      for (int ks = 0; ks < nks; ++ks)
        tc::mma_bf16(tbase + C::D2, tc::desc_sw128(a + ks * 32), tc::desc_sw128(b + ks * 32), idesc, 1u);
    }
    tc::mma_commit(mbar_2);
  }
  if (BND) {
    // a block boundary after the first bj rows: D2 now holds that state.
    // The first half solves for the remaining rows meanwhile; every thread
    // writes its 64 columns of the boundary state to the boundary page,
    // scales them to the end of the log, and the second product adds the
    // rows from bj on: S = exp(G_{L-1} - G_{bj-1}) S_bj + R^T Kt_b.
    if (ok && half == 0) {
#pragma unroll
      for (int l = 0; l < NMAX; ++l) kt[l] = l >= bj ? dec[l] * fk[l] * kf[l * S::KF_LD + row] : 0.f;
      rp_back_solve<NMAX, S::AM_LD>(kt, am);
    }
    if (ok) {
      const bool okb = tc::mbar_wait_bounded(mbar_2, 0, kRpWait);
      ok = __syncthreads_and(okb);
    }
    tc::fence_after_sync();
    if (ok) {
      if (half == 0) {   // the first product has read B2: the remaining rows' Kt^T replace it
#pragma unroll
        for (int c8 = 0; c8 < NMAX / 8; ++c8) {
          const uint32_t off = tc::sw128_offset(row, 8 * c8, D);
          tc::store_split8(sm + S::B2 + off, sm + S::B2_LO + off, kt + 8 * c8);
        }
      }
      const float scale = __expf(Gs[L - 1] - Gs[bj - 1]);
      float* bst = page_state(p.pool, bpage) + ((int64_t)h * D + row) * D + 64 * half;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float v[32];
        tc::tmem_ld32(tbase + tlane + C::D2 + 64 * half + 32 * q, v);
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<float4*>(bst + 32 * q + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] *= scale;
        tc::tmem_st32(tbase + tlane + C::D2 + 64 * half + 32 * q, v);
      }
      tc::tmem_st_wait();
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    ok = __syncthreads_and(ok);
    tc::fence_after_sync();
    if (ok && tid == kIssue) {
      const uint32_t idesc = tc::idesc_bf16_f32(D, D);
      constexpr int nks = NMAX / 16;
      for (int pass = 0; pass < 3; ++pass) {
        const uint32_t a = sbase + (pass == 2 ? S::A2_LO : S::A2);
        const uint32_t b = sbase + (pass == 1 ? S::B2_LO : S::B2);
        for (int ks = 0; ks < nks; ++ks)
          tc::mma_bf16(tbase + C::D2, tc::desc_sw128(a + ks * 32), tc::desc_sw128(b + ks * 32), idesc, 1u);
      }
      tc::mma_commit(mbar_2);
    }
  }
  if (ok) {
    const bool ok2 = tc::mbar_wait_bounded(mbar_2, BND ? 1 : 0, kRpWait);
    ok = __syncthreads_and(ok2);
  }
  tc::fence_after_sync();

  // (8) the new state: each thread parks its 64 columns in A1 (free once the
  // second product has completed) in the tensor map's swizzled layout, then
  // four TMA tile stores write it back
  if (ok) {
    float d2[32], d3[32];
    tc::tmem_ld32x2(tbase + tlane + C::D2 + 64 * half, tbase + tlane + C::D2 + 32 + 64 * half, d2, d3);
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      *reinterpret_cast<float4*>(sm + S::A1 + rp_state_offset(row, 64 * half + c)) =
          make_float4(d2[c], d2[c + 1], d2[c + 2], d2[c + 3]);
      *reinterpret_cast<float4*>(sm + S::A1 + rp_state_offset(row, 64 * half + 32 + c)) =
          make_float4(d3[c], d3[c + 1], d3[c + 2], d3[c + 3]);
    }
    tc::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::tma_store_3d(tmap, 32 * cb, h * D, page, sm + S::A1 + cb * 16384);
      tc::bulk_commit();
      tc::bulk_wait_read();
    }
  } else {
    // a wait ran out: report it, give the tensor core one more bounded wait
    // for the work it may still hold, then release the tensor memory
    if (tid == 0) set_error(p.err, GDN_ERR_TIMEOUT);
    tc::mbar_wait_bounded(mbar_1, 0, kRpWait);
    tc::mbar_wait_bounded(mbar_2, BND ? 1 : 0, kRpWait);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, kRpCols);
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
  // the flush kernel's validation (it reports the errors)
  if (!page_ok(p.pool, page) || n < 0 || n > kRpMaxRows) return;
  const int bj = (p.boundary_rows && n > 0) ? p.boundary_rows[r] : 0;
  const int32_t bpage = bj > 0 ? p.boundary_page[r] : -1;
  if (bj > 0 && (bj > n || bpage == page || !page_ok(p.pool, bpage))) return;
  if (n > 0) {
    TIN* win = page_window<TIN>(p.pool, page);
    TIN* bwin = bj > 0 ? page_window<TIN>(p.pool, bpage) : nullptr;
    const TIN* lx = reinterpret_cast<const TIN*>(p.log_x) + (int64_t)r * kRpMaxRows * p.conv_dim;
    const int chunks = 2 * p.Hqk * kRpD / 8;
    auto src = [&](int t) {   // row t of window || log
      return t < kWinRows ? win + (int64_t)t * p.conv_dim : lx + (int64_t)(t - kWinRows) * p.conv_dim;
    };
    for (int c = threadIdx.x; c < chunks; c += kQkWinThreads) {
      uint4 keep[kWinRows], kb[kWinRows];
#pragma unroll
      for (int j = 0; j < kWinRows; ++j) {
        keep[j] = *reinterpret_cast<const uint4*>(src(n + j) + 8 * c);
        if (bwin) kb[j] = *reinterpret_cast<const uint4*>(src(bj + j) + 8 * c);
      }
#pragma unroll
      for (int j = 0; j < kWinRows; ++j) {
        *reinterpret_cast<uint4*>(win + (int64_t)j * p.conv_dim + 8 * c) = keep[j];
        if (bwin) *reinterpret_cast<uint4*>(bwin + (int64_t)j * p.conv_dim + 8 * c) = kb[j];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) const_cast<int32_t*>(p.log_len)[r] = 0;
}

// After the tensor-core append: log_len += m for every request that passed
// validation (all CTAs of the append have read the old value).
__global__ void append_len_kernel(const ScanParams p) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= p.num_seqs) return;
  const int32_t len = p.log_len[r];
  if (!page_ok(p.pool, p.ckpt_slot[r]) || len < 0 || len + p.num_new > kRpMaxRows) return;
  const_cast<int32_t*>(p.log_len)[r] = len + p.num_new;
}

__global__ void __launch_bounds__(kRpThreads, 2) tc_flush_kernel(const ScanParams p,
                                                                 const __grid_constant__ CUtensorMap tmap) {
  const int h = blockIdx.x, r = blockIdx.y;
  // uniform validation (the window / log_len kernel repeats it)
  const int32_t page = p.ckpt_slot[r];
  const int32_t n = p.log_len[r];
  if (!page_ok(p.pool, page) || n < 0 || n > kRpMaxRows) {
    if (h == 0 && threadIdx.x == 0)
      set_error(p.err, page_ok(p.pool, page) ? GDN_ERR_INVALID_ARG : GDN_ERR_PAGE_RANGE);
    return;
  }
  if (n == 0) return;   // nothing logged: the state stays as it is
  if (p.boundary_rows && p.boundary_rows[r] > 0) return;   // tc_flush_boundary_kernel's request
  if (n <= 16) replay_body<16, false>(p, &tmap, h, r, page, n, n);
  else replay_body<32, false>(p, &tmap, h, r, page, n, n);
}

// The requests of a flush whose kept rows cross a block boundary (prefix
// caching): also the state and conv window after the first bj rows, to the
// boundary page.  A kernel of its own, launched only when the call passes
// boundary rows, so that the common flush compiles without this path.
__global__ void __launch_bounds__(kRpThreads, 2) tc_flush_boundary_kernel(const ScanParams p,
                                                                          const __grid_constant__ CUtensorMap tmap) {
  const int h = blockIdx.x, r = blockIdx.y;
  const int bj = p.boundary_rows[r];
  if (bj <= 0) return;
  const int32_t page = p.ckpt_slot[r];
  const int32_t n = p.log_len[r];
  if (!page_ok(p.pool, page) || n < 0 || n > kRpMaxRows) return;   // reported by tc_flush_kernel
  const int32_t bpage = p.boundary_page[r];
  if (bj > n || bpage == page || !page_ok(p.pool, bpage)) {
    if (h == 0 && threadIdx.x == 0)
      set_error(p.err, page_ok(p.pool, bpage) ? GDN_ERR_INVALID_ARG : GDN_ERR_PAGE_RANGE);
    return;
  }
  if (n <= 16) replay_body<16, false, true>(p, &tmap, h, r, page, n, n, bj, bpage);
  else replay_body<32, false, true>(p, &tmap, h, r, page, n, n, bj, bpage);
}

__global__ void __launch_bounds__(kRpThreads, 2) tc_append_kernel(const ScanParams p,
                                                                  const __grid_constant__ CUtensorMap tmap) {
  const int h = blockIdx.x, r = blockIdx.y;
  const int32_t page = p.ckpt_slot[r];
  const int32_t n = p.log_len[r];
  int32_t code = 0;
  if (!page_ok(p.pool, page)) code = GDN_ERR_PAGE_RANGE;
  else if (n < 0 || n > kRpMaxRows) code = GDN_ERR_INVALID_ARG;
  else if (n + p.num_new > kRpMaxRows) code = GDN_ERR_LOG_OVERFLOW;
  if (code) {
    if (h == 0 && threadIdx.x == 0) set_error(p.err, code);
    return;
  }
  const int L = n + p.num_new;
  if (L <= 16) replay_body<16, true>(p, &tmap, h, r, page, n, L);
  else replay_body<32, true>(p, &tmap, h, r, page, n, L);
}

bool tc_replay_supported(int dk, int dv, int in_dtype) {
  return dk == kRpD && dv == kRpD && in_dtype == GDN_BF16;   // bf16 rows in and out (in = out)
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

// The pool's states as [page][Hv * 128 rows][128 columns] fp32, boxes of 128
// rows x 32 columns.
static cudaError_t state_tensor_map(const ScanParams& p, CUtensorMap* tmap) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kRpD, (cuuint64_t)p.Hv * kRpD, (cuuint64_t)p.pool.num_pages};
  const cuuint64_t strides[2] = {(cuuint64_t)kRpD * 4, (cuuint64_t)p.pool.page_bytes};
  const cuuint32_t box[3] = {32, (cuuint32_t)kRpD, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (encode(tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.pool.base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

cudaError_t launch_tc_flush(const ScanParams& p, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  CUtensorMap tmap;
  cudaError_t e = state_tensor_map(p, &tmap);
  if (e != cudaSuccess) return e;
  const size_t smem = RpSmem<32, false>::ALLOC;
  static_assert(RpSmem<16, false>::ALLOC <= RpSmem<32, false>::ALLOC, "launch size covers both variants");
  e = cudaFuncSetAttribute(tc_flush_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_flush_kernel<<<dim3(p.Hv, p.num_seqs), kRpThreads, smem, st>>>(p, tmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.boundary_rows) {
    e = cudaFuncSetAttribute(tc_flush_boundary_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tc_flush_boundary_kernel<<<dim3(p.Hv, p.num_seqs), kRpThreads, smem, st>>>(p, tmap);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  flush_qk_window_kernel<<<p.num_seqs, kQkWinThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tc_append(const ScanParams& p, cudaStream_t st) {
  if (p.num_seqs == 0 || p.num_new == 0) return cudaSuccess;
  CUtensorMap tmap;
  cudaError_t e = state_tensor_map(p, &tmap);
  if (e != cudaSuccess) return e;
  const size_t smem = RpSmem<32, true>::ALLOC;
  static_assert(RpSmem<16, true>::ALLOC <= RpSmem<32, true>::ALLOC, "launch size covers both variants");
  e = cudaFuncSetAttribute(tc_append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_append_kernel<<<dim3(p.Hv, p.num_seqs), kRpThreads, smem, st>>>(p, tmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  append_len_kernel<<<(p.num_seqs + 255) / 256, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
