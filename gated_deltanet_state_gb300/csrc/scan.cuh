// scan.cuh — token-sequential scan of the gated delta rule on CUDA cores.
//
// One CTA owns ROWS = 32*RPT rows of one value head's state for one sequence
// (or replay request) and keeps them in registers for the whole token stream,
// so the state crosses HBM once on the way in and once per checkpoint / at the
// end.  Rows of S evolve independently under
//     S_t = a_t S_{t-1} + c_t k_t^T,  c_t = b_t (v_t - a_t S_{t-1} k_t),  o_t = S_t q_t
// (the gated delta rule, expanded), so splitting dv across CTAs needs no
// communication and does not change any result bit.
//
// Deferred decay: inside a tile of 16 tokens the registers hold R = S / A with
// A = prod a (a per-head scalar), so a token costs three FMAs per element
// (issued as packed fp32 pairs, fma.rn.f32x2, two elements per instruction):
// R += (c/A) k_t, o += R q_t, u += R k_{t+1}.  At each tile end R is scaled
// back (R *= A, A = 1).  A token whose running product would fall below 2^-64
// applies its decay directly instead (R = (A a) R + c k, A = 1), so R never
// overflows whatever the gates are.
//
// Tiles start at absolute positions that are multiples of 16 and every tile
// recomputes u for its first token from the renormalised state.  Block
// boundaries (multiples of the block size, itself a multiple of 16) are tile
// ends, so a checkpoint holds exactly the register state there and a resume
// from it replays the cold run's arithmetic bit for bit.
//
// Thread layout: four lanes share a row, each owning DK/4 columns as float4
// chunks 4*(4m+cq) (interleaved so a group's shared-memory reads hit distinct
// banks); a 128-thread CTA covers 32 row groups x RPT rows.  All sums run in a
// fixed order, with two partial sums per dot product for instruction-level
// parallelism.
//
// Inputs: a pre-pass kernel computes SiLU(conv) of every channel once (plus
// the q / k norm factors and the gates) into a workspace; the scan streams its
// q, k and v-slice rows from there into two shared-memory stages with
// cp.async, loading tile j+1 while it scans tile j.  q and k stay
// unnormalised; their norm factors are applied as per-token scalars, which is
// the same product reassociated.
#pragma once

#include "common.cuh"

namespace gdn {

enum ScanMode { kPrefill = 0, kAppend = 1, kFlush = 2 };

struct ScanParams {
  Pool pool;
  int32_t Hqk, Hv, conv_dim, block_size;
  float q_scale, eps;
  int32_t num_seqs;
  const float* conv_w;
  void* o;
  int32_t* err;
  // prefill
  const int32_t* cu_seqlens;
  const int64_t* start_pos;
  const int32_t* init_page;
  const int32_t* block_table;
  int32_t max_blocks;
  const int32_t* out_slot;
  const void* x;
  const float* g;
  const float* beta;
  int64_t total_rows;   // rows of x, g, beta and o (all sequences)
  const int8_t* skip;   // mixed batches: nonzero = a decode sequence, not prefilled here
  int32_t x_ld;         // elements from one x row to the next (conv_dim; packed q|k|v|z rows: more)
  const float* norm_w;  // packed core: gated-norm scale [dv] (nullptr: plain outputs)
  float norm_eps2;      // packed core: gated-norm epsilon
  long long wait_cycles;   // bound of a tensor-core kernel's waits in SM clocks (0: the default;
                           // < 0: every wait reports a timeout at once)
  // replay
  const int32_t* ckpt_slot;
  const void* log_x;
  const float* log_g;
  const float* log_beta;
  const int32_t* log_len;
  int32_t num_new;
  const void* x_new;
  const float* g_new;
  const float* beta_new;
  const int32_t* boundary_rows;   // flush: kept rows up to a block boundary ([N], optional)
  const int32_t* boundary_page;   // flush: the boundary checkpoint's page ([N])
  // workspace written by the conv pre-pass, read by the scan
  float* ws_y;     // [rows][conv_dim]   SiLU(conv) of every channel
  float* ws_nrm;   // [rows][2*Hqk]      q (times q_scale) and k norm factors
  float* ws_ab;    // [rows][Hv][2]      a = exp(g), b
};

// Per-sequence view of the token stream: relative token t >= -3; negative t
// reads the carried conv window (or zeros on a cold start).
template <typename TIN>
struct TokenView {
  const TIN* win;        // [3][conv_dim] or nullptr (zeros)
  const TIN* seg0;       // rows [0, n0)
  const TIN* seg1;       // rows [n0, n)
  const float* g0; const float* g1;
  const float* b0; const float* b1;
  int64_t n0, n;
  int64_t wrow0;         // workspace row of token 0
  int32_t conv_dim, Hv;
  int32_t ld;            // elements from one token row to the next (the window's rows: conv_dim)

  __device__ __forceinline__ float x(int64_t t, int c) const {
    if (t < 0) return win ? to_f32(win[(kWinRows + t) * conv_dim + c]) : 0.0f;
    if (t < n0) return to_f32(seg0[t * ld + c]);
    return to_f32(seg1[(t - n0) * ld + c]);
  }
  // Raw element (bit-exact copies of window rows).
  __device__ __forceinline__ TIN raw(int64_t t, int c) const {
    if (t < 0) return win ? win[(kWinRows + t) * conv_dim + c] : from_f32<TIN>(0.0f);
    if (t < n0) return seg0[t * ld + c];
    return seg1[(t - n0) * ld + c];
  }
  // Pointer to pre-conv row t, or nullptr where the row is zero (a cold
  // start's history, or past the end).
  __device__ __forceinline__ const TIN* row(int64_t t) const {
    if (t < 0) return win ? win + (kWinRows + t) * conv_dim : nullptr;
    if (t >= n) return nullptr;
    return t < n0 ? seg0 + t * ld : seg1 + (t - n0) * ld;
  }
  __device__ __forceinline__ const float* gptr(int64_t t, int h) const {
    return t < n0 ? g0 + t * Hv + h : g1 + (t - n0) * Hv + h;
  }
  __device__ __forceinline__ const float* bptr(int64_t t, int h) const {
    return t < n0 ? b0 + t * Hv + h : b1 + (t - n0) * Hv + h;
  }
  __device__ __forceinline__ float g(int64_t t, int h) const {
    return t < n0 ? g0[t * Hv + h] : g1[(t - n0) * Hv + h];
  }
  __device__ __forceinline__ float b(int64_t t, int h) const {
    return t < n0 ? b0[t * Hv + h] : b1[(t - n0) * Hv + h];
  }
};

// Validates sequence s for the mode and fills its view.  Returns false (after
// recording the error when there is one) if the sequence must be skipped.
// Every CTA and the window kernels evaluate the same conditions, so a bad
// sequence is skipped consistently.
template <typename TIN, int MODE>
__device__ __forceinline__ bool make_view(const ScanParams& p, int s, TokenView<TIN>& v,
                                          int64_t& start, int32_t& init, int32_t& final_page,
                                          int64_t& n_log, bool report) {
  v.conv_dim = p.conv_dim;
  v.ld = p.conv_dim;
  v.Hv = p.Hv;
  if (MODE == kPrefill) {
    if (p.skip && p.skip[s]) return false;   // decoded by the mixed step's decode kernel
    const int64_t t0 = p.cu_seqlens[s], t1 = p.cu_seqlens[s + 1];
    start = p.start_pos[s];
    init = p.init_page[s];
    final_page = p.out_slot[s];
    n_log = 0;
    int32_t code = 0;
    if (t1 < t0 || start < 0) code = GDN_ERR_INVALID_ARG;
    else if (init == -1 ? start != 0 : (start <= 0 || start % p.block_size != 0))
      code = GDN_ERR_NOT_BLOCK_ALIGNED;
    else if ((init != -1 && !page_ok(p.pool, init)) || !page_ok(p.pool, final_page))
      code = GDN_ERR_PAGE_RANGE;
    if (code) { if (report) set_error(p.err, code); return false; }
    v.win = init >= 0 ? page_window<TIN>(p.pool, init) : nullptr;
    v.ld = p.x_ld;
    v.seg0 = reinterpret_cast<const TIN*>(p.x) + t0 * p.x_ld;
    v.seg1 = v.seg0;
    v.g0 = v.g1 = p.g + t0 * p.Hv;
    v.b0 = v.b1 = p.beta + t0 * p.Hv;
    v.n0 = v.n = t1 - t0;
    v.wrow0 = t0;
    return true;
  } else {
    init = p.ckpt_slot[s];
    final_page = MODE == kFlush ? init : -1;
    start = 0;
    const int32_t len = p.log_len[s];
    const int32_t m = MODE == kAppend ? p.num_new : 0;
    int32_t code = 0;
    if (!page_ok(p.pool, init)) code = GDN_ERR_PAGE_RANGE;
    else if (len < 0 || len > GDN_REPLAY_LOG_SLOTS) code = GDN_ERR_INVALID_ARG;
    else if (len + m > GDN_REPLAY_LOG_SLOTS) code = GDN_ERR_LOG_OVERFLOW;
    if (code) { if (report) set_error(p.err, code); return false; }
    n_log = len;
    v.win = page_window<TIN>(p.pool, init);
    const int64_t lrow = (int64_t)s * GDN_REPLAY_LOG_SLOTS;
    v.seg0 = reinterpret_cast<const TIN*>(p.log_x) + lrow * p.conv_dim;
    v.g0 = p.log_g + lrow * p.Hv;
    v.b0 = p.log_beta + lrow * p.Hv;
    const int64_t nrow = (int64_t)s * (MODE == kAppend ? p.num_new : 0);
    v.seg1 = MODE == kAppend ? reinterpret_cast<const TIN*>(p.x_new) + nrow * p.conv_dim : v.seg0;
    v.g1 = MODE == kAppend ? p.g_new + nrow * p.Hv : v.g0;
    v.b1 = MODE == kAppend ? p.beta_new + nrow * p.Hv : v.b0;
    v.n0 = len;
    v.n = len + m;
    v.wrow0 = lrow;
    return true;
  }
}

// ---------------------------------------------------------------------------
// Conv pre-pass: SiLU(depthwise causal conv) of every channel of every token,
// once, into the workspace, with the L2-norm factors of each q and k head and
// the gates of each value head.  It is bound by HBM (reads x once, writes fp32
// rows), so each thread owns VEC consecutive channels and moves 16 bytes per
// load; a head's D channels are D / VEC adjacent lanes, which reduce the
// squared norm with shuffles.  SiLU uses the fast exponential and division
// (a few ulp); the gates keep the accurate expf.
constexpr int kConvTokens = 32;
constexpr int kConvThreads = 128;

template <typename TIN>
struct Vec16 {                      // 16 bytes of TIN
  static constexpr int N = 16 / sizeof(TIN);
  TIN v[N];
};
template <typename TIN>
__device__ __forceinline__ void load16(Vec16<TIN>& d, const TIN* src) {
  *reinterpret_cast<uint4*>(d.v) = *reinterpret_cast<const uint4*>(src);
}

template <typename TIN, int MODE, int D>
__global__ void __launch_bounds__(kConvThreads) conv_kernel(const ScanParams p) {
  constexpr int VEC = Vec16<TIN>::N;          // channels per thread
  constexpr int TPH = D / VEC;                // lanes per head
  static_assert(TPH >= 1 && TPH <= 32 && (TPH & (TPH - 1)) == 0, "head must map to a lane group");
  const int s = blockIdx.z, tid = threadIdx.x;
  TokenView<TIN> V;
  int64_t start, n_log;
  int32_t init, final_page;
  if (!make_view<TIN, MODE>(p, s, V, start, init, final_page, n_log, false)) return;
  const int64_t t0 = (int64_t)blockIdx.y * kConvTokens;
  if (t0 >= V.n) return;
  const int cnt = (int)(V.n - t0 < kConvTokens ? V.n - t0 : kConvTokens);
  const int c0 = (blockIdx.x * kConvThreads + tid) * VEC;   // first channel of this thread
  const bool valid = c0 < p.conv_dim;
  const int head = valid ? c0 / D : 0;        // channel head: q heads, k heads, v heads
  const bool qk = head < 2 * p.Hqk;
  const bool leader = (tid & (TPH - 1)) == 0;

  float w[VEC][4];
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    const float4 w4 = valid ? *reinterpret_cast<const float4*>(p.conv_w + (int64_t)(c0 + e) * kConvK)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    w[e][0] = w4.x; w[e][1] = w4.y; w[e][2] = w4.z; w[e][3] = w4.w;
  }
  // history rows t0-3 .. t0-1
  float hist[3][VEC];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const TIN* row = V.row(t0 - 3 + r);
    Vec16<TIN> x;
    if (valid && row) load16(x, row + c0);
#pragma unroll
    for (int e = 0; e < VEC; ++e) hist[r][e] = (valid && row) ? to_f32(x.v[e]) : 0.f;
  }
  // rows are loaded GRP at a time, the next group in flight while this one computes
  constexpr int GRP = 4;
  Vec16<TIN> xr[GRP], xn[GRP];
#pragma unroll
  for (int u = 0; u < GRP; ++u)
    if (valid && u < cnt) load16(xr[u], V.row(t0 + u) + c0);
  for (int g0 = 0; g0 < cnt; g0 += GRP) {
#pragma unroll
    for (int u = 0; u < GRP; ++u)
      if (valid && g0 + GRP + u < cnt) load16(xn[u], V.row(t0 + g0 + GRP + u) + c0);
#pragma unroll
    for (int u = 0; u < GRP; ++u) {
      const int tt = g0 + u;
      if (tt < cnt) {                         // uniform across the CTA
        float y[VEC];
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float xv = to_f32(xr[u].v[e]);
          float z = w[e][0] * hist[0][e];
          z = fmaf(w[e][1], hist[1][e], z);
          z = fmaf(w[e][2], hist[2][e], z);
          z = fmaf(w[e][3], xv, z);
          y[e] = silu_fast(z);
          ss = fmaf(y[e], y[e], ss);
          hist[0][e] = hist[1][e]; hist[1][e] = hist[2][e]; hist[2][e] = xv;
        }
        const int64_t wr = V.wrow0 + t0 + tt;
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(p.ws_y + wr * p.conv_dim + c0);
#pragma unroll
          for (int e = 0; e < VEC; e += 4) dst[e / 4] = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
        }
        // squared norm of the head: sum over its TPH lanes (fixed xor order)
#pragma unroll
        for (int o = 1; o < TPH; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (valid && leader) {
          if (qk) {
            const float scale = head < p.Hqk ? p.q_scale : 1.0f;
            p.ws_nrm[wr * 2 * p.Hqk + head] = scale / sqrtf(ss + p.eps);
          } else {
            const int h = head - 2 * p.Hqk;
            float* ab = p.ws_ab + (wr * p.Hv + h) * 2;
            ab[0] = expf(V.g(t0 + tt, h));
            ab[1] = V.b(t0 + tt, h);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < GRP; ++u) xr[u] = xn[u];
  }
}

// ---------------------------------------------------------------------------
// The scan.
constexpr int kScanTile = 16;
// Lanes that share one state row (each owns DK / kLanesPerRow columns) and the
// CTA size that gives 32 row groups.
constexpr int kLanesPerRow = 4;
constexpr int kScanThreads = 32 * kLanesPerRow;

// Sum over the kLanesPerRow lanes of a row group (fixed xor order; every lane
// of the group ends with the same bits).
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int o = 1; o < kLanesPerRow; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Shared-memory plan of one scan CTA (byte offsets): two tile stages.
template <int DK, int DV, int RPT>
struct ScanSmem {
  static constexpr int TT = kScanTile, ROWS = 32 * RPT;
  static constexpr size_t q = 0;                                    // f32 [TT][DK] SiLU(conv) q
  static constexpr size_t k = q + sizeof(float) * TT * DK;          // f32 [TT][DK] SiLU(conv) k
  static constexpr size_t vo = k + sizeof(float) * TT * DK;         // f32 [TT][ROWS] v in, o out
  static constexpr size_t sc = vo + sizeof(float) * TT * ROWS;      // float4 [TT]: a, b, fq, fk
  static constexpr size_t stage = sc + sizeof(float4) * TT;
  static constexpr size_t bytes = 2 * stage;
  static_assert(stage % 16 == 0, "stages must stay 16-byte aligned");
};

template <int DK, int DV, int RPT>
constexpr size_t scan_smem_bytes() { return ScanSmem<DK, DV, RPT>::bytes; }

// Asynchronous copies of one tile from the workspace into a stage.
template <int DK, int DV, int RPT, typename TIN>
__device__ __forceinline__ void stage_tile(const ScanParams& p, const TokenView<TIN>& V, char* st,
                                           int64_t t0, int cnt, int jq, int h, int row0, int tid) {
  using L = ScanSmem<DK, DV, RPT>;
  constexpr int QC = DK / 4, VC = L::ROWS / 4, RC = 2 * QC + VC;  // 16-byte chunks per token
  float* q_s = reinterpret_cast<float*>(st + L::q);
  float* k_s = reinterpret_cast<float*>(st + L::k);
  float* v_s = reinterpret_cast<float*>(st + L::vo);
  float* sc_s = reinterpret_cast<float*>(st + L::sc);
  const int cq = jq * DK, ck = p.Hqk * DK + jq * DK, cv = 2 * p.Hqk * DK + h * DV + row0;
  for (int i = tid; i < cnt * RC; i += kScanThreads) {
    const int tt = i / RC, c = i - tt * RC;
    const float* row = p.ws_y + (V.wrow0 + t0 + tt) * p.conv_dim;
    if (c < QC) cp_async16(q_s + tt * DK + 4 * c, row + cq + 4 * c, 16);
    else if (c < 2 * QC) cp_async16(k_s + tt * DK + 4 * (c - QC), row + ck + 4 * (c - QC), 16);
    else cp_async16(v_s + tt * L::ROWS + 4 * (c - 2 * QC), row + cv + 4 * (c - 2 * QC), 16);
  }
  for (int i = tid; i < 3 * cnt; i += kScanThreads) {
    const int tt = i / 3, c = i - tt * 3;
    const int64_t wr = V.wrow0 + t0 + tt;
    if (c == 0) cp_async8(sc_s + 4 * tt, p.ws_ab + (wr * p.Hv + h) * 2);
    else cp_async4(sc_s + 4 * tt + 1 + c, p.ws_nrm + wr * 2 * p.Hqk + (c - 1) * p.Hqk + jq, 4);
  }
  cp_async_commit();
}

template <int DK, int DV, int RPT, typename TIN, typename TOUT, int MODE>
__global__ void __launch_bounds__(kScanThreads, 3) scan_kernel(const ScanParams p) {
  using L = ScanSmem<DK, DV, RPT>;
  constexpr int TT = L::TT;
  constexpr int ROWS = L::ROWS;
  constexpr int LPR = kLanesPerRow;
  constexpr int NCH = DK / (4 * LPR);   // float4 chunks per thread
  static_assert(NCH >= 1, "dk too small for the lane layout");
  static_assert(DV % ROWS == 0, "row slices must tile dv");
  static_assert(DK % 32 == 0, "dk must be a multiple of 32");

  const int slice = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = lane & (LPR - 1);                   // column group of this lane
  const int rg = warp * (32 / LPR) + lane / LPR;     // row group 0..31
  const int row0 = slice * ROWS;
  const int grp = p.Hv / p.Hqk, jq = h / grp;

  TokenView<TIN> V;
  int64_t start, n_log;
  int32_t init, final_page;
  const bool report = (slice == 0 && h == 0 && tid == 0);
  if (!make_view<TIN, MODE>(p, s, V, start, init, final_page, n_log, report)) return;
  const int64_t n = V.n;
  const int64_t ntiles = (n + TT - 1) / TT;

  extern __shared__ float4 smem4[];
  char* sm = reinterpret_cast<char*>(smem4);
  if (ntiles > 0) stage_tile<DK, DV, RPT, TIN>(p, V, sm, 0, (int)(n < TT ? n : TT), jq, h, row0, tid);

  // initial state rows (zeros on a cold start: the pool is not read); each
  // float4 chunk of a row is held as two packed pairs
  f32x2 S[RPT][NCH][2];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = row0 + rg + 32 * i;
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      ulonglong2 v2 = make_ulonglong2(0ull, 0ull);
      if (init >= 0)
        v2 = *reinterpret_cast<const ulonglong2*>(page_state(p.pool, init) +
                                                  ((int64_t)h * DV + row) * DK + 4 * (LPR * m + cq));
      S[i][m][0] = v2.x;
      S[i][m][1] = v2.y;
    }
  }

  for (int64_t j = 0; j < ntiles; ++j) {
    const int64_t t0 = j * TT;
    const int cnt = (int)(n - t0 < TT ? n - t0 : TT);
    cp_async_wait<0>();
    __syncthreads();   // stage j is visible and every thread is done with tile j-1
    if (j + 1 < ntiles) {
      const int64_t t1 = t0 + TT;
      stage_tile<DK, DV, RPT, TIN>(p, V, sm + ((j + 1) & 1) * L::stage, t1,
                                   (int)(n - t1 < TT ? n - t1 : TT), jq, h, row0, tid);
    }
    const char* st = sm + (j & 1) * L::stage;
    const float* q_s = reinterpret_cast<const float*>(st + L::q);
    const float* k_s = reinterpret_cast<const float*>(st + L::k);
    float* vo_s = reinterpret_cast<float*>(const_cast<char*>(st) + L::vo);
    const float4* sc_s = reinterpret_cast<const float4*>(st + L::sc);

    // tile prologue: h = R k_0 (k before its norm factor) with R = S, A = 1
    float hk[RPT];
    ulonglong2 kc[NCH];
    {
      f32x2 acc[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) acc[i] = 0ull;
#pragma unroll
      for (int m = 0; m < NCH; ++m) {
        const ulonglong2 k2 = *reinterpret_cast<const ulonglong2*>(k_s + 4 * (LPR * m + cq));
        kc[m] = k2;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          acc[i] = fma2(S[i][m][0], k2.x, acc[i]);
          acc[i] = fma2(S[i][m][1], k2.y, acc[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < RPT; ++i) hk[i] = row_sum(sum2(acc[i]));
    }
    float A = 1.0f;

    for (int tt = 0; tt < cnt; ++tt) {
      const float4 scl = sc_s[tt];                      // a, b, fq, fk of token tt
      const float a = scl.x, b = scl.y, fq = scl.z, fk = scl.w;
      const float An = A * a;
      const bool direct = An < 0x1p-64f;                // uniform across the CTA
      const float inv = direct ? 1.0f : 1.0f / An;
      const bool nxt = tt + 1 < cnt;
      f32x2 d2[RPT], o2[RPT][2], u2[RPT][2];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float u = (A * fk) * hk[i];               // u_t = S_{t-1} k_t (normalised k)
        const float coef = b * fmaf(-a, u, vo_s[tt * ROWS + rg + 32 * i]);
        const float d = (coef * fk) * inv;
        d2[i] = pack2(d, d);
        o2[i][0] = o2[i][1] = 0ull;
        u2[i][0] = u2[i][1] = 0ull;
      }
      // The decay branch is uniform across the CTA; each variant is one loop.
      // kc holds k_t (loaded as the previous token's k_{t+1}).
#define GDN_SCAN_TOKEN(UPDATE)                                                                     \
  _Pragma("unroll") for (int m = 0; m < NCH; ++m) {                                               \
    const ulonglong2 q2 = *reinterpret_cast<const ulonglong2*>(q_s + tt * DK + 4 * (LPR * m + cq)); \
    ulonglong2 n2 = make_ulonglong2(0ull, 0ull);                                                  \
    if (nxt) n2 = *reinterpret_cast<const ulonglong2*>(k_s + (tt + 1) * DK + 4 * (LPR * m + cq)); \
    _Pragma("unroll") for (int i = 0; i < RPT; ++i) {                                             \
      S[i][m][0] = UPDATE(S[i][m][0], kc[m].x);                                                   \
      S[i][m][1] = UPDATE(S[i][m][1], kc[m].y);                                                   \
      o2[i][m & 1] = fma2(S[i][m][0], q2.x, o2[i][m & 1]);                                        \
      u2[i][m & 1] = fma2(S[i][m][0], n2.x, u2[i][m & 1]);                                        \
      o2[i][m & 1] = fma2(S[i][m][1], q2.y, o2[i][m & 1]);                                        \
      u2[i][m & 1] = fma2(S[i][m][1], n2.y, u2[i][m & 1]);                                        \
    }                                                                                             \
    kc[m] = n2;                                                                                   \
  }
      if (!direct) {
#define GDN_UPD(SV, KV) fma2(d2[i], KV, SV)
        GDN_SCAN_TOKEN(GDN_UPD)
#undef GDN_UPD
      } else {
        const f32x2 an2 = pack2(An, An);
#define GDN_UPD(SV, KV) fma2(d2[i], KV, mul2(an2, SV))
        GDN_SCAN_TOKEN(GDN_UPD)
#undef GDN_UPD
      }
#undef GDN_SCAN_TOKEN
      A = direct ? 1.0f : An;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float o = (A * fq) * row_sum(sum2(o2[i][0]) + sum2(o2[i][1]));
        hk[i] = row_sum(sum2(u2[i][0]) + sum2(u2[i][1]));
        // every lane of the quad has read v (the shuffles above synchronise it)
        if (cq == 0) vo_s[tt * ROWS + rg + 32 * i] = o;
      }
    }

    // tile end: back to the plain state (exact when A == 1)
    {
      const f32x2 a2 = pack2(A, A);
#pragma unroll
      for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int m = 0; m < NCH; ++m) {
          S[i][m][0] = mul2(a2, S[i][m][0]);
          S[i][m][1] = mul2(a2, S[i][m][1]);
        }
    }

    if (MODE == kPrefill) {
      const int64_t pos = start + t0 + cnt;   // a multiple of B only at a full tile's end
      if (pos % p.block_size == 0) {
        const int64_t jb = pos / p.block_size - 1;
        int32_t page = -1;
        if (jb < p.max_blocks) page = p.block_table[(int64_t)s * p.max_blocks + jb];
        else if (report) set_error(p.err, GDN_ERR_INVALID_ARG);
        if (page >= 0) {
          if (page_ok(p.pool, page)) {
            float* dstS = page_state(p.pool, page);
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
              const int row = row0 + rg + 32 * i;
#pragma unroll
              for (int m = 0; m < NCH; ++m)
                *reinterpret_cast<ulonglong2*>(dstS + ((int64_t)h * DV + row) * DK + 4 * (LPR * m + cq)) =
                    make_ulonglong2(S[i][m][0], S[i][m][1]);
            }
          } else if (report) {
            set_error(p.err, GDN_ERR_PAGE_RANGE);
          }
        }
      }
    }

    // outputs of the tile, coalesced along dv
    if (MODE != kFlush) {
      __syncthreads();
      TOUT* out = reinterpret_cast<TOUT*>(p.o);
      for (int idx = tid; idx < cnt * ROWS; idx += kScanThreads) {
        const int tt = idx / ROWS, r = idx % ROWS;
        const int64_t t = t0 + tt;
        if (MODE == kPrefill) {
          const int64_t trow = p.cu_seqlens[s] + t;
          out[(trow * p.Hv + h) * DV + row0 + r] = from_f32<TOUT>(vo_s[idx]);
        } else if (t >= n_log) {
          const int64_t trow = (int64_t)s * p.num_new + (t - n_log);
          out[(trow * p.Hv + h) * DV + row0 + r] = from_f32<TOUT>(vo_s[idx]);
        }
      }
    }
  }

  // final state
  if (final_page >= 0) {
    float* dstS = page_state(p.pool, final_page);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int row = row0 + rg + 32 * i;
#pragma unroll
      for (int m = 0; m < NCH; ++m)
        *reinterpret_cast<ulonglong2*>(dstS + ((int64_t)h * DV + row) * DK + 4 * (LPR * m + cq)) =
            make_ulonglong2(S[i][m][0], S[i][m][1]);
    }
  }
}

// Conv windows after the scan: every crossed boundary (prefill) and the final
// window (prefill: out_slot, flush: the checkpoint page).  One thread owns one
// channel of one sequence and reads all three rows before writing them, so an
// in-place update (out_slot == init_page, or the flush) is safe.  The grid's
// z CTAs of a (channel block, sequence) share its boundaries (boundary b goes
// to z = b mod gridDim.z; their rows lie a block or more after the call's
// first token, so none of them reads the carried window) and z = 0 writes
// the final window.  log_len is only read here; the flush clears it in
// log_len_kernel afterwards.
template <typename TIN, int MODE>
__global__ void __launch_bounds__(256) window_kernel(const ScanParams p) {
  const int s = blockIdx.y;
  TokenView<TIN> V;
  int64_t start, n_log;
  int32_t init, final_page;
  if (!make_view<TIN, MODE>(p, s, V, start, init, final_page, n_log, false)) return;
  // a prefill whose device wait ran out wrote no states: no windows either
  if (MODE == kPrefill && *reinterpret_cast<volatile const int32_t*>(p.err) == GDN_ERR_TIMEOUT) return;
  const int64_t n = V.n;
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < p.conv_dim; c += gridDim.x * blockDim.x) {
    if (MODE == kPrefill) {
      const int64_t step = (int64_t)gridDim.z * p.block_size;
      for (int64_t P = (start / p.block_size + 1 + blockIdx.z) * p.block_size; P <= start + n; P += step) {
        const int64_t jb = P / p.block_size - 1;
        if (jb >= p.max_blocks) break;
        const int32_t page = p.block_table[(int64_t)s * p.max_blocks + jb];
        if (!page_ok(p.pool, page)) continue;
        TIN* w = page_window<TIN>(p.pool, page);
        const int64_t rel = P - start;
#pragma unroll
        for (int r = 0; r < kWinRows; ++r)
          w[(int64_t)r * p.conv_dim + c] = V.raw(rel - kWinRows + r, c);
      }
    }
    if (final_page >= 0 && blockIdx.z == 0) {
      TIN keep[kWinRows];
#pragma unroll
      for (int r = 0; r < kWinRows; ++r) keep[r] = V.raw(n - kWinRows + r, c);
      TIN* w = page_window<TIN>(p.pool, final_page);
#pragma unroll
      for (int r = 0; r < kWinRows; ++r) w[(int64_t)r * p.conv_dim + c] = keep[r];
    }
  }
}

// log_len bookkeeping after every reader of the old value has finished:
// append publishes n + m, flush clears the log.  Requests that failed
// validation keep their log_len.
template <int MODE>
__global__ void log_len_kernel(const ScanParams p) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= p.num_seqs) return;
  const int32_t len = p.log_len[r];
  const int32_t m = MODE == kAppend ? p.num_new : 0;
  if (!page_ok(p.pool, p.ckpt_slot[r]) || len < 0 || len + m > GDN_REPLAY_LOG_SLOTS) return;
  const_cast<int32_t*>(p.log_len)[r] = MODE == kAppend ? len + m : 0;
}

}  // namespace gdn
