// scan.cuh — token-sequential scan of the gated delta rule on CUDA cores.
//
// One CTA owns ROWS = 32*RPT rows of one value head's state for one sequence
// (or replay request) and keeps them in registers for the whole token stream,
// so the state crosses HBM once on the way in and once per checkpoint / at the
// end.  Rows of S evolve independently under
//     S_t = a_t S_{t-1} + b_t (v_t - a_t S_{t-1} k_t) k_t^T,   o_t = S_t q_t
// (the gated delta rule, expanded), so splitting dv across CTAs needs no
// communication and does not change any result bit.
//
// Thread layout: four lanes share a row, each owning DK/4 columns as float4
// chunks 4*(4m+cq) (interleaved so a quad's shared-memory reads hit distinct
// banks).  Per token one pass over the registers both applies the update and
// accumulates o_t = S_t q_t and u_{t+1} = S_t k_{t+1}, so each token costs one
// quad reduction round.  All sums run in a fixed order, so results depend only
// on a sequence's own data: a resume from a checkpoint replays the cold run's
// arithmetic exactly (the prologue computes u with the same order).
//
// Tokens are processed in tiles of TT: the CTA first computes conv + SiLU and
// the L2 norms of q and k for the tile (plus one look-ahead token) into shared
// memory, then scans the tile.
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

constexpr int kScanTile = 32;
constexpr int kScanThreads = 128;

template <int DK, int DV, int RPT>
constexpr size_t scan_smem_bytes() {
  return sizeof(float) * (2 * (kScanTile + 1) * DK + 2 * kScanTile * 32 * RPT + 2 * (kScanTile + 1));
}

template <int DK, int DV, int RPT, typename TIN, typename TOUT, int MODE>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const ScanParams p) {
  constexpr int TT = kScanTile;
  constexpr int ROWS = 32 * RPT;
  constexpr int NCH = DK / 16;   // float4 chunks per thread
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
  float* q_s = reinterpret_cast<float*>(smem4);  // [TT+1][DK]
  float* k_s = q_s + (TT + 1) * DK;              // [TT+1][DK]
  float* v_s = k_s + (TT + 1) * DK;              // [TT][ROWS]
  float* o_s = v_s + TT * ROWS;                  // [TT][ROWS]
  float* a_s = o_s + TT * ROWS;                  // [TT+1]
  float* b_s = a_s + (TT + 1);                   // [TT+1]

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

  const int cqk = jq * DK;                       // q channels of this qk head
  const int ckk = p.Hqk * DK + jq * DK;          // k channels
  const int cvv = 2 * p.Hqk * DK + h * DV + row0;  // v channels of this slice
  constexpr int NC = 2 * DK + ROWS;

  float kc[NCH][4];
  float u[RPT];

  for (int64_t t0 = 0; t0 < n; t0 += TT) {
    const int cnt = (int)(n - t0 < TT ? n - t0 : TT);
    const int ntok = cnt + (t0 + cnt < n ? 1 : 0);
    __syncthreads();  // the previous tile's readers are done

    // ---- conv + SiLU for ntok tokens on this CTA's channels
    for (int idx = tid; idx < NC; idx += kScanThreads) {
      const int c = idx < DK ? cqk + idx : (idx < 2 * DK ? ckk + idx - DK : cvv + idx - 2 * DK);
      const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)c * kConvK);
      float* dst;
      int ld;
      if (idx < DK) { dst = q_s + idx; ld = DK; }
      else if (idx < 2 * DK) { dst = k_s + idx - DK; ld = DK; }
      else { dst = v_s + idx - 2 * DK; ld = ROWS; }
      const int lim = idx < 2 * DK ? ntok : cnt;
      float h0 = V.x(t0 - 3, c), h1 = V.x(t0 - 2, c), h2 = V.x(t0 - 1, c);
      float xr[TT + 1];
#pragma unroll
      for (int tt = 0; tt < TT + 1; ++tt) xr[tt] = tt < lim ? V.x(t0 + tt, c) : 0.0f;
#pragma unroll
      for (int tt = 0; tt < TT + 1; ++tt) {
        if (tt < lim) {
          float z = w.x * h0;
          z = fmaf(w.y, h1, z);
          z = fmaf(w.z, h2, z);
          z = fmaf(w.w, xr[tt], z);
          dst[tt * ld] = silu(z);
        }
        h0 = h1; h1 = h2; h2 = xr[tt];
      }
    }
    if (tid < cnt) {
      a_s[tid] = expf(V.g(t0 + tid, h));
      b_s[tid] = V.b(t0 + tid, h);
    }
    __syncthreads();

    // ---- L2 norms of q and k, one warp per token, fixed reduction order
    for (int tt = warp; tt < ntok; tt += kScanThreads / 32) {
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

    // ---- prologue at the first token: u = S k_0 in the scan's summation order
    if (t0 == 0) {
#pragma unroll
      for (int m = 0; m < NCH; ++m) {
        const float4 k4 = *reinterpret_cast<const float4*>(k_s + 4 * (4 * m + cq));
        kc[m][0] = k4.x; kc[m][1] = k4.y; kc[m][2] = k4.z; kc[m][3] = k4.w;
      }
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < NCH; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc = fmaf(S[i][m][e], kc[m][e], acc);
        u[i] = quad_sum(acc);
      }
    }

    // ---- scan the tile
    for (int tt = 0; tt < cnt; ++tt) {
      const float a = a_s[tt], b = b_s[tt];
      const bool nxt = tt + 1 < ntok;
      float coef[RPT], o[RPT], un[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        coef[i] = b * fmaf(-a, u[i], v_s[tt * ROWS + rg + 32 * i]);
        o[i] = 0.f;
        un[i] = 0.f;
      }
#pragma unroll
      for (int m = 0; m < NCH; ++m) {
        const float4 q4 = *reinterpret_cast<const float4*>(q_s + tt * DK + 4 * (4 * m + cq));
        float4 k4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (nxt) k4 = *reinterpret_cast<const float4*>(k_s + (tt + 1) * DK + 4 * (4 * m + cq));
        const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
        const float kn[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float sn = fmaf(coef[i], kc[m][e], a * S[i][m][e]);
            S[i][m][e] = sn;
            o[i] = fmaf(sn, qv[e], o[i]);
            un[i] = fmaf(sn, kn[e], un[i]);
          }
#pragma unroll
        for (int e = 0; e < 4; ++e) kc[m][e] = kn[e];
      }
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        o[i] = quad_sum(o[i]);
        u[i] = quad_sum(un[i]);
        if (cq == 0) o_s[tt * ROWS + rg + 32 * i] = o[i];
      }
      if (MODE == kPrefill) {
        const int64_t pos = start + t0 + tt + 1;
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
          out[(trow * p.Hv + h) * DV + row0 + r] = from_f32<TOUT>(o_s[idx]);
        } else if (t >= n_log) {
          const int64_t trow = (int64_t)s * p.num_new + (t - n_log);
          out[(trow * p.Hv + h) * DV + row0 + r] = from_f32<TOUT>(o_s[idx]);
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
// in-place update (out_slot == init_page, or the flush) is safe.  The flush
// variant also clears log_len once every channel is done.
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
  if (MODE == kFlush) {
    __syncthreads();
    if (threadIdx.x == 0) const_cast<int32_t*>(p.log_len)[s] = 0;
  }
}

}  // namespace gdn
