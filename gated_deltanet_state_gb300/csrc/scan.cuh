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
// A = prod a (a per-head scalar), so a token costs three FMAs per element:
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
// chunks 4*(4m+cq) (interleaved so a quad's shared-memory reads hit distinct
// banks).  All sums run in a fixed order.
//
// Input staging: the CTA's q, k and v-slice channels of the pre-conv rows of
// the next tile are copied into shared memory with cp.async while the current
// tile is scanned (double buffer); conv + SiLU and the L2 norms of q and k are
// then computed from shared memory.
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
  int32_t conv_dim, Hv;

  __device__ __forceinline__ float x(int64_t t, int c) const {
    if (t < 0) return win ? to_f32(win[(kWinRows + t) * conv_dim + c]) : 0.0f;
    if (t < n0) return to_f32(seg0[t * conv_dim + c]);
    return to_f32(seg1[(t - n0) * conv_dim + c]);
  }
  // Raw element (bit-exact copies of window rows).
  __device__ __forceinline__ TIN raw(int64_t t, int c) const {
    if (t < 0) return win ? win[(kWinRows + t) * conv_dim + c] : from_f32<TIN>(0.0f);
    if (t < n0) return seg0[t * conv_dim + c];
    return seg1[(t - n0) * conv_dim + c];
  }
  // Pointer to pre-conv row t, or nullptr where the row is zero (a cold
  // start's history, or past the end).
  __device__ __forceinline__ const TIN* row(int64_t t) const {
    if (t < 0) return win ? win + (kWinRows + t) * conv_dim : nullptr;
    if (t >= n) return nullptr;
    return t < n0 ? seg0 + t * conv_dim : seg1 + (t - n0) * conv_dim;
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
  v.Hv = p.Hv;
  if (MODE == kPrefill) {
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
    v.seg0 = reinterpret_cast<const TIN*>(p.x) + t0 * p.conv_dim;
    v.seg1 = v.seg0;
    v.g0 = v.g1 = p.g + t0 * p.Hv;
    v.b0 = v.b1 = p.beta + t0 * p.Hv;
    v.n0 = v.n = t1 - t0;
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
    return true;
  }
}

constexpr int kScanTile = 16;
constexpr int kScanThreads = 128;

// Shared-memory plan of one scan CTA (byte offsets).
template <int DK, int DV, int RPT, typename TIN>
struct ScanSmem {
  static constexpr int TT = kScanTile, ROWS = 32 * RPT, NC = 2 * DK + ROWS;
  static constexpr int XROWS = TT + 3;  // pre-conv rows t0-3 .. t0+TT-1
  static constexpr size_t q = 0;                                      // f32 [TT][DK]
  static constexpr size_t k = q + sizeof(float) * TT * DK;            // f32 [TT][DK]
  static constexpr size_t vo = k + sizeof(float) * TT * DK;           // f32 [TT][ROWS]: v in, o out
  static constexpr size_t ab = vo + sizeof(float) * TT * ROWS;        // f32 [2][TT]: a, b
  static constexpr size_t xs = (ab + sizeof(float) * 2 * TT + 15) / 16 * 16;  // TIN [2][XROWS][NC]
  static constexpr size_t gb = xs + 2 * sizeof(TIN) * XROWS * NC;     // f32 [2][2][TT]: g, beta
  static constexpr size_t bytes = gb + sizeof(float) * 2 * 2 * TT;
};

template <int DK, int DV, int RPT, typename TIN>
constexpr size_t scan_smem_bytes() { return ScanSmem<DK, DV, RPT, TIN>::bytes; }

// Issues the asynchronous copies of one tile: the CTA's q, k and v-slice
// channels of pre-conv rows t0-3 .. t0+TT-1 (window rows before the sequence,
// zeros on a cold start or past the end), and g, beta of tokens t0 .. t0+TT-1.
template <int DK, int DV, int RPT, typename TIN>
__device__ __forceinline__ void stage_tile(const ScanParams& p, const TokenView<TIN>& V, TIN* xs,
                                           float* gb, int64_t t0, int cqk, int ckk, int cvv, int h,
                                           int tid) {
  using L = ScanSmem<DK, DV, RPT, TIN>;
  constexpr int CH = 16 / sizeof(TIN);            // elements per 16-byte chunk
  constexpr int QC = DK / CH, VC = L::ROWS / CH;  // chunks per channel segment
  constexpr int RC = 2 * QC + VC;                 // chunks per row
  const void* dummy = p.conv_w;                   // any valid address for zero-fill
  for (int i = tid; i < L::XROWS * RC; i += kScanThreads) {
    const int rr = i / RC, ch = i - rr * RC;
    const int64_t t = t0 - 3 + rr;
    int col, cidx;
    if (ch < QC) { col = ch * CH; cidx = cqk + ch * CH; }
    else if (ch < 2 * QC) { col = DK + (ch - QC) * CH; cidx = ckk + (ch - QC) * CH; }
    else { col = 2 * DK + (ch - 2 * QC) * CH; cidx = cvv + (ch - 2 * QC) * CH; }
    const TIN* row = V.row(t);
    const bool ok = row != nullptr;
    cp_async16(xs + rr * L::NC + col, ok ? static_cast<const void*>(row + cidx) : dummy, ok ? 16 : 0);
  }
  for (int i = tid; i < 2 * L::TT; i += kScanThreads) {
    const int which = i / L::TT, tt = i - which * L::TT;
    const int64_t t = t0 + tt;
    const bool ok = t < V.n;
    const float* src = ok ? (which ? V.bptr(t, h) : V.gptr(t, h)) : static_cast<const float*>(dummy);
    cp_async4(gb + i, src, ok ? 4 : 0);
  }
}

template <int DK, int DV, int RPT, typename TIN, typename TOUT, int MODE>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const ScanParams p) {
  using L = ScanSmem<DK, DV, RPT, TIN>;
  constexpr int TT = L::TT;
  constexpr int ROWS = L::ROWS;
  constexpr int NC = L::NC;
  constexpr int NCH = DK / 16;   // float4 chunks per thread
  constexpr int NW = (NC + kScanThreads - 1) / kScanThreads;
  static_assert(DV % ROWS == 0, "row slices must tile dv");
  static_assert(DK % 32 == 0, "dk must be a multiple of 32");

  const int slice = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = lane & 3;
  const int rg = warp * 8 + (lane >> 2);
  const int row0 = slice * ROWS;
  const int grp = p.Hv / p.Hqk, jq = h / grp;

  TokenView<TIN> V;
  int64_t start, n_log;
  int32_t init, final_page;
  const bool report = (slice == 0 && h == 0 && tid == 0);
  if (!make_view<TIN, MODE>(p, s, V, start, init, final_page, n_log, report)) return;
  const int64_t n = V.n;

  extern __shared__ float4 smem4[];
  char* sm = reinterpret_cast<char*>(smem4);
  float* q_s = reinterpret_cast<float*>(sm + L::q);
  float* k_s = reinterpret_cast<float*>(sm + L::k);
  float* vo_s = reinterpret_cast<float*>(sm + L::vo);
  float* a_s = reinterpret_cast<float*>(sm + L::ab);
  float* b_s = a_s + TT;
  TIN* xs_s = reinterpret_cast<TIN*>(sm + L::xs);
  float* gb_s = reinterpret_cast<float*>(sm + L::gb);

  const int cqk = jq * DK;                         // q channels of this qk head
  const int ckk = p.Hqk * DK + jq * DK;            // k channels
  const int cvv = 2 * p.Hqk * DK + h * DV + row0;  // v channels of this slice

  const int64_t ntiles = (n + TT - 1) / TT;
  if (ntiles > 0) {
    stage_tile<DK, DV, RPT, TIN>(p, V, xs_s, gb_s, 0, cqk, ckk, cvv, h, tid);
    cp_async_commit();
  }

  // ---- initial state rows (zeros on a cold start: the pool is not read)
  float S[RPT][NCH][4];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = row0 + rg + 32 * i;
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (init >= 0)
        v4 = *reinterpret_cast<const float4*>(page_state(p.pool, init) +
                                              ((int64_t)h * DV + row) * DK + 4 * (4 * m + cq));
      S[i][m][0] = v4.x; S[i][m][1] = v4.y; S[i][m][2] = v4.z; S[i][m][3] = v4.w;
    }
  }

  // conv taps of the channels this thread computes
  float4 wreg[NW];
#pragma unroll
  for (int u = 0; u < NW; ++u) {
    const int idx = tid + u * kScanThreads;
    wreg[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (idx < NC) {
      const int c = idx < DK ? cqk + idx : (idx < 2 * DK ? ckk + idx - DK : cvv + idx - 2 * DK);
      wreg[u] = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)c * kConvK);
    }
  }

  for (int64_t it = 0; it < ntiles; ++it) {
    const int64_t t0 = it * TT;
    const int cnt = (int)(n - t0 < TT ? n - t0 : TT);
    if (it + 1 < ntiles) {
      stage_tile<DK, DV, RPT, TIN>(p, V, xs_s + ((it + 1) & 1) * L::XROWS * NC,
                                   gb_s + ((it + 1) & 1) * 2 * TT, t0 + TT, cqk, ckk, cvv, h, tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // this tile's rows are in shared memory; last tile's readers are done

    // ---- conv + SiLU for the tile's tokens on this CTA's channels
    const TIN* xb = xs_s + (it & 1) * L::XROWS * NC;
#pragma unroll
    for (int uu = 0; uu < NW; ++uu) {
      const int idx = tid + uu * kScanThreads;
      if (idx < NC) {
        const float4 w = wreg[uu];
        float* dst;
        int ld;
        if (idx < DK) { dst = q_s + idx; ld = DK; }
        else if (idx < 2 * DK) { dst = k_s + idx - DK; ld = DK; }
        else { dst = vo_s + idx - 2 * DK; ld = ROWS; }
        float h0 = to_f32(xb[idx]), h1 = to_f32(xb[NC + idx]), h2 = to_f32(xb[2 * NC + idx]);
        for (int tt = 0; tt < cnt; ++tt) {
          const float xv = to_f32(xb[(tt + 3) * NC + idx]);
          float z = w.x * h0;
          z = fmaf(w.y, h1, z);
          z = fmaf(w.z, h2, z);
          z = fmaf(w.w, xv, z);
          dst[tt * ld] = silu_fast(z);
          h0 = h1; h1 = h2; h2 = xv;
        }
      }
    }
    if (tid < cnt) {
      const float* gbb = gb_s + (it & 1) * 2 * TT;
      a_s[tid] = expf(gbb[tid]);
      b_s[tid] = gbb[TT + tid];
    }
    __syncthreads();

    // ---- L2 norms of q and k, one warp per token, fixed reduction order
    for (int tt = warp; tt < cnt; tt += kScanThreads / 32) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int jj = 0; jj < DK / 32; ++jj) {
        const float qv = q_s[tt * DK + lane + 32 * jj];
        const float kv = k_s[tt * DK + lane + 32 * jj];
        sq = fmaf(qv, qv, sq);
        sk = fmaf(kv, kv, sk);
      }
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      const float fq = p.q_scale / sqrtf(sq + p.eps);
      const float fk = 1.0f / sqrtf(sk + p.eps);
#pragma unroll
      for (int jj = 0; jj < DK / 32; ++jj) {
        q_s[tt * DK + lane + 32 * jj] *= fq;
        k_s[tt * DK + lane + 32 * jj] *= fk;
      }
    }
    __syncthreads();

    // ---- tile prologue: u = R k_0 with R = S (A = 1)
    float uh[RPT];
    {
      float acc0[RPT], acc1[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) { acc0[i] = 0.f; acc1[i] = 0.f; }
#pragma unroll
      for (int m = 0; m < NCH; ++m) {
        const float4 k4 = *reinterpret_cast<const float4*>(k_s + 4 * (4 * m + cq));
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          float& acc = (m & 1) ? acc1[i] : acc0[i];
          acc = fmaf(S[i][m][0], k4.x, acc);
          acc = fmaf(S[i][m][1], k4.y, acc);
          acc = fmaf(S[i][m][2], k4.z, acc);
          acc = fmaf(S[i][m][3], k4.w, acc);
        }
      }
#pragma unroll
      for (int i = 0; i < RPT; ++i) uh[i] = quad_sum(acc0[i] + acc1[i]);
    }
    float A = 1.0f;

    // ---- scan the tile
    for (int tt = 0; tt < cnt; ++tt) {
      const float a = a_s[tt], b = b_s[tt];
      const float An = A * a;
      const bool direct = An < 0x1p-64f;  // uniform across the CTA
      const float inv = direct ? 1.0f : 1.0f / An;
      const bool nxt = tt + 1 < cnt;
      float d[RPT], o0[RPT], o1[RPT], un0[RPT], un1[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float coef = b * fmaf(-a, A * uh[i], vo_s[tt * ROWS + rg + 32 * i]);
        d[i] = coef * inv;
        o0[i] = 0.f; o1[i] = 0.f; un0[i] = 0.f; un1[i] = 0.f;
      }
      // The decay branch is uniform across the CTA; each variant is one loop.
#define GDN_SCAN_TOKEN(UPDATE)                                                                 \
  _Pragma("unroll") for (int m = 0; m < NCH; ++m) {                                           \
    const float4 k4 = *reinterpret_cast<const float4*>(k_s + tt * DK + 4 * (4 * m + cq));     \
    const float4 q4 = *reinterpret_cast<const float4*>(q_s + tt * DK + 4 * (4 * m + cq));     \
    float4 n4 = make_float4(0.f, 0.f, 0.f, 0.f);                                              \
    if (nxt) n4 = *reinterpret_cast<const float4*>(k_s + (tt + 1) * DK + 4 * (4 * m + cq));   \
    const float kv[4] = {k4.x, k4.y, k4.z, k4.w};                                             \
    const float qv[4] = {q4.x, q4.y, q4.z, q4.w};                                             \
    const float kn[4] = {n4.x, n4.y, n4.z, n4.w};                                             \
    _Pragma("unroll") for (int i = 0; i < RPT; ++i) {                                         \
      float& oa = (m & 1) ? o1[i] : o0[i];                                                    \
      float& ua = (m & 1) ? un1[i] : un0[i];                                                  \
      _Pragma("unroll") for (int e = 0; e < 4; ++e) {                                         \
        const float sn = UPDATE;                                                              \
        S[i][m][e] = sn;                                                                      \
        oa = fmaf(sn, qv[e], oa);                                                             \
        ua = fmaf(sn, kn[e], ua);                                                             \
      }                                                                                       \
    }                                                                                         \
  }
      if (!direct) {
        GDN_SCAN_TOKEN(fmaf(d[i], kv[e], S[i][m][e]))
      } else {
        GDN_SCAN_TOKEN(fmaf(d[i], kv[e], An * S[i][m][e]))
      }
#undef GDN_SCAN_TOKEN
      A = direct ? 1.0f : An;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float o = A * quad_sum(o0[i] + o1[i]);
        uh[i] = quad_sum(un0[i] + un1[i]);
        // every lane of the quad has read v (the shuffles above synchronise it)
        if (cq == 0) vo_s[tt * ROWS + rg + 32 * i] = o;
      }
    }

    // ---- tile end: back to the plain state (exact when A == 1)
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
      for (int m = 0; m < NCH; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) S[i][m][e] *= A;

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
                *reinterpret_cast<float4*>(dstS + ((int64_t)h * DV + row) * DK + 4 * (4 * m + cq)) =
                    make_float4(S[i][m][0], S[i][m][1], S[i][m][2], S[i][m][3]);
            }
          } else if (report) {
            set_error(p.err, GDN_ERR_PAGE_RANGE);
          }
        }
      }
    }
    __syncthreads();

    // ---- outputs of the tile, coalesced along dv
    if (MODE != kFlush) {
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

  // ---- final state
  if (final_page >= 0) {
    float* dstS = page_state(p.pool, final_page);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int row = row0 + rg + 32 * i;
#pragma unroll
      for (int m = 0; m < NCH; ++m)
        *reinterpret_cast<float4*>(dstS + ((int64_t)h * DV + row) * DK + 4 * (4 * m + cq)) =
            make_float4(S[i][m][0], S[i][m][1], S[i][m][2], S[i][m][3]);
    }
  }
}

// Conv windows after the scan: every crossed boundary (prefill) and the final
// window (prefill: out_slot, flush: the checkpoint page).  One thread owns one
// channel of one sequence and reads all three rows before writing them, so an
// in-place update (out_slot == init_page, or the flush) is safe.  log_len is
// only read here; the flush clears it in log_len_kernel afterwards.
template <typename TIN, int MODE>
__global__ void __launch_bounds__(256) window_kernel(const ScanParams p) {
  const int s = blockIdx.y;
  TokenView<TIN> V;
  int64_t start, n_log;
  int32_t init, final_page;
  if (!make_view<TIN, MODE>(p, s, V, start, init, final_page, n_log, false)) return;
  const int64_t n = V.n;
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < p.conv_dim; c += gridDim.x * blockDim.x) {
    if (MODE == kPrefill) {
      for (int64_t P = (start / p.block_size + 1) * p.block_size; P <= start + n; P += p.block_size) {
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
    if (final_page >= 0) {
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
