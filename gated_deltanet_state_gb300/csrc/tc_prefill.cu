// tc_prefill.cu — the chunked prefill on the tensor cores (dk = dv = 128, bf16
// inputs and outputs).
//
// The gated delta rule ("Gated DeltaNet", the recurrence
// S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t) taken a
// chunk of C = 64 tokens at a time in its chunk (UT) form.  With k^, q^ the
// L2-normalised rows of a chunk, G_i the running sum of the log decays inside
// the chunk, gam_i = exp(G_i), S0 the state entering the chunk and row r of S
// one value channel:
//   u_i   = b_i (v_i - gam_i S0 k^_i) - sum_{j<i} A_ij u_j,
//   A_ij  = b_i exp(G_i - G_j) k^_i.k^_j                        (j < i)
//   o_i   = gam_i S0 q^_i + sum_{j<=i} exp(G_i - G_j) (q^_i.k^_j) u_j
//   S_C   = gam_C S0 + sum_j exp(G_C - G_j) u_j k^_j^T
// which is the token recurrence regrouped (u_i is the rank-one update of token
// i, the triangular system collects the (I - b k k^T) factors of the tokens
// before it).
//
// One CTA owns one (sequence, value head) and walks its tokens in chunks that
// start at absolute multiples of 64, so a block boundary (a multiple of the
// block size, itself a multiple of 64) is always a chunk end: a checkpoint is
// the state between two chunks and a resume replays the cold run's arithmetic
// bit for bit.  The fp32 state lives in tensor memory from the CTA's first
// chunk to its last.  When the chains outnumber the SMs, a CTA walks one
// piece of its chain (an even number of chunks) and the next piece runs in a
// later launch from the state this one leaves in the final slot's page
// (tc_prefill_schedule).  Per chunk:
//   (A) conv + SiLU of the chunk's q, k, v channels from pre-conv rows staged
//       in shared memory (prefetched during the previous chunk; packed fp32
//       pairs), L2 norms; meanwhile the issuing warp forms the cumulative
//       gates; operands [K^; Q^] and K^T diag(exp(G_C - G)).
//   (B) S0 from tensor memory into a bf16 operand (and gam_C S0 back);
//       tensor cores: [K^K^T; Q^K^T] and S0 [K^; Q^]^T.
//   (C) A and P = exp(G_i - G_j) q^_i.k^_j (j <= i) (computed while the
//       tensor core forms S0 [K^; Q^]^T); T = (I + A)^{-1} by two warpgroups
//       (16 x 16 blocks: diagonal inverses, the blocks N = -D A below them,
//       then one product per distance from the diagonal) while the others form
//       R_i = b_i (v_i - gam_i S0 k^_i);
//       tensor cores: U^T = R T^T.
//   (D) tensor cores: S += U^T (K^T diag(exp(G_C - G)))^T in tensor memory and
//       U^T P^T; outputs o_i = gam_i (S0 q^_i) + (U^T P^T)_i.
// Every product reads bf16 operands split into hi + lo parts and runs three
// passes (hi*hi + hi*lo + lo*hi) into fp32 accumulators: each operand keeps
// ~16 significant bits, so the chunk stays within ~1e-5 of an fp32 evaluation.
// Every mbarrier wait is bounded; a wait that runs out sets GDN_ERR_TIMEOUT
// (over any earlier code), lets the tensor core and the copy engine drain
// (bounded again, by the default limit) and releases tensor memory; later
// pieces of the call and the window pass then write nothing.
#include "launch.h"
#include "tc.cuh"
#include "tc_chunk.cuh"

namespace gdn {

namespace {

constexpr int kPfWorkers = 512;         // sixteen warps of CUDA-core work
constexpr int kPfThreads = kPfWorkers + 32;   // + one warp that issues the tensor-core products
constexpr int kMmaTid = kPfWorkers;      // the issuing thread (lane 0 of the seventeenth warp)
constexpr int kPfC = 64;                 // chunk rows
constexpr int kPfD = 128;                // dk = dv
constexpr int kPfXRows = kPfC + kWinRows;
constexpr uint32_t kPfCols = 512;        // tensor-memory columns (the whole SM's)
// tensor-memory column map (lane = state row r, or chunk row i for D_KK / D_QK)
constexpr uint32_t kColS = 0;            // S, fp32 128 x 128
constexpr uint32_t kColSK = 128;         // S0 K^T, 128 x 64
constexpr uint32_t kColSQ = 192;         // S0 Q^T, 128 x 64
constexpr uint32_t kColKK = 256;         // [K^ K^T; Q^ K^T], 128 x 64
constexpr uint32_t kColV = 320;          // v of the chunk, row r = channel r, 128 x 64
constexpr uint32_t kColU = 384;          // U^T = R T^T, then U^T P^T, 128 x 64
constexpr long long kPfWait = 4000000000LL;

// Shared-memory plan (byte offsets from a 1024-byte aligned base).  The
// 128-byte swizzled operands are K-major bf16 tiles (sw128_offset), hi part
// then lo part.  Regions are reused phase by phase:
//   R1: (A) y | (B) S0 operand | (C) T fp32, its blocks, T operand, A row-major
//   R2: (A-B) [K^; Q^] operand | (C-D) R^T then U^T operand, P operand, A^T fp32
struct PfSmem {
  static constexpr uint32_t R1 = 0;
  static constexpr uint32_t YF = R1;                  // fp32 [64][256] (q | k)
  static constexpr uint32_t S0 = R1;                  // S0 hi [2 kb][128][64], lo at +32 KB
  static constexpr uint32_t S0_LO = R1 + 32768;
  static constexpr uint32_t TF = R1;                  // T fp32 [64 i][64 j]
  static constexpr uint32_t DT = R1 + 16384;          // fp32 [4][16][20]: diagonal inverses, transposed
  static constexpr uint32_t NT = R1 + 21504;          // fp32 [6][16][16]: N_pk^T
  static constexpr uint32_t TB = R1 + 32768;          // T hi [64][64], lo at +8 KB
  static constexpr uint32_t TB_LO = R1 + 40960;
  static constexpr uint32_t AM = R1 + 49152;          // A fp32 [64][64] row-major, slots swizzled
  static constexpr uint32_t R2 = 65536;
  static constexpr uint32_t KQ = R2;                  // [K^; Q^] hi [2 kb][128][64], lo at +32 KB
  static constexpr uint32_t KQ_LO = R2 + 32768;
  static constexpr uint32_t UT = R2;                  // R^T, then U^T: hi [128][64], lo at +16 KB
  static constexpr uint32_t UT_LO = R2 + 16384;
  static constexpr uint32_t PB = R2 + 32768;          // P hi [64][64], lo at +8 KB
  static constexpr uint32_t PB_LO = R2 + 40960;
  static constexpr uint32_t AT = R2 + 49152;          // A^T fp32 [64 j][64 i]
  static constexpr uint32_t KT = 131072;              // K^T diag(dec) hi [128][64], lo at +16 KB
  static constexpr uint32_t KT_LO = KT + 16384;
  static constexpr uint32_t OT = R1;                  // (D) outputs bf16 [64 rows][128 dv]
  static constexpr uint32_t OF = R1 + 16384;          // (D) packed core: outputs fp32 [64][128]
  // pre-conv rows t0-3 .. t0+63 of the chunk, bf16 [67][128] per tile: q, k, v
  static constexpr uint32_t XS = 163840;
  static constexpr uint32_t XTILE = 17408;            // tile stride (1024-aligned)
  static constexpr uint32_t GT = XS + 2 * XTILE + kPfXRows * kPfD * 2;
  // fp32 [64] each at GT: G, gam, dec = exp(G_C - G), b of even chunks, the
  // same of odd chunks (the issuing warp fills the next set while the workers
  // still read the current one), q factor, k factor
  static constexpr uint32_t MBAR = GT + 10 * 256;      // mbarriers: K^K^T, S0[K^;Q^]^T, U, U^T P^T, staged rows, state update
  static constexpr uint32_t TSLOT = MBAR + 48;
  static constexpr uint32_t BYTES = TSLOT + 8;
  static constexpr uint32_t ALLOC = BYTES + 1024;     // + alignment slack
};
static_assert(PfSmem::GT % 16 == 0, "gate staging must be 16-byte aligned");
static_assert(PfSmem::ALLOC <= 232448, "shared memory plan exceeds the per-CTA limit");


// A bounded wait of the chunk loop: at most `lim` SM clocks, or (lim < 0)
// none at all, reporting a timeout at once (how the run-out path is tested).
// The drain after a run-out always takes the default bound.
__device__ __forceinline__ bool work_wait(uint64_t* m, uint32_t parity, long long lim) {
  return lim >= 0 && tc::mbar_wait_bounded(m, parity, lim);
}

// A worker's bounded wait for a tensor-core product; a wait that runs out
// clears `ok`, which the next whole-CTA barrier turns into a common exit.
__device__ __forceinline__ void mma_wait(uint64_t* m, uint32_t parity, bool& ok, long long lim) {
  ok = work_wait(m, parity, lim) && ok;
  tc::fence_after_sync();
}

// Whole-CTA barrier (workers and the issuing warp) that also agrees on `ok`.
__device__ __forceinline__ bool cta_sync_ok(bool ok) {
  tc::fence_before_sync();
  ok = __syncthreads_and(ok);
  tc::fence_after_sync();
  return ok;
}

}  // namespace

__global__ void __launch_bounds__(kPfThreads, 1)
    tc_prefill_kernel(const ScanParams p, const __grid_constant__ CUtensorMap xmap,
                      const __grid_constant__ CUtensorMap omap, int tma_out, const PieceMap pm) {
  using TIN = __nv_bfloat16;
  using TOUT = __nv_bfloat16;
  constexpr int D = kPfD, C = kPfC;
  // this CTA's piece: chain (sequence s, value head h), chunks [cb, ce)
  const int h = blockIdx.x;
  int s = pm.s0 + (int)blockIdx.y, level = pm.level0;
  if (s >= pm.nseqs) {
    s -= pm.nseqs;
    ++level;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool worker = tid < kPfWorkers;
  const int row = tid & 127;                  // state row = tensor-memory lane of this thread
  const int quarter = (tid >> 7) & 3;         // column quarter handled in tensor-memory phases
  const uint32_t tlane = (uint32_t)((warp & 3) * 32) << 16;

  TokenView<TIN> V;
  int64_t start, n_log;
  int32_t init, final_page;
  // errors are recorded first-wins, so every piece of head 0 may report
  const bool report = (h == 0 && tid == 0);
  if (!make_view<TIN, kPrefill>(p, s, V, start, init, final_page, n_log, report)) return;
  const int64_t n = V.n;
  const int64_t nch = (n + C - 1) / C;
  // the first piece of a chain starts from the resumed page (or zeros) and
  // always runs (it also writes the state of an empty sequence); a later one
  // starts from the state the previous piece left in the final slot, and the
  // last level runs to the sequence's end
  const int64_t cb = (int64_t)level * pm.piece;   // even: a piece is an even number of chunks
  if (level > 0 && cb >= nch) return;
  const int64_t ce = level == pm.last_level || cb + pm.piece > nch ? nch : cb + pm.piece;
  const int32_t from = level > 0 ? final_page : init;
  // a later piece continues from the state the chain's previous piece left in
  // the final slot; if a wait of an earlier launch of this call ran out, that
  // state may be stale, so no later piece runs (the error word says so)
  if (level > 0 &&
      __syncthreads_or(tid == 0 && *reinterpret_cast<volatile const int32_t*>(p.err) == GDN_ERR_TIMEOUT))
    return;
  const long long wlim = p.wait_cycles > 0 ? p.wait_cycles : p.wait_cycles < 0 ? -1 : kPfWait;
  const int grp = p.Hv / p.Hqk, jq = h / grp;
  const int cq0 = jq * D, ck0 = p.Hqk * D + jq * D, cv0 = 2 * p.Hqk * D + h * D;
  const int64_t row0 = p.cu_seqlens[s];      // first row of this sequence in x, g, beta, o

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  float* yf = reinterpret_cast<float*>(sm + PfSmem::YF);
  TIN* xq = reinterpret_cast<TIN*>(sm + PfSmem::XS);
  TIN* xk = reinterpret_cast<TIN*>(sm + PfSmem::XS + PfSmem::XTILE);
  TIN* xv = reinterpret_cast<TIN*>(sm + PfSmem::XS + 2 * PfSmem::XTILE);
  float* gbuf = reinterpret_cast<float*>(sm + PfSmem::GT);   // two gate sets (by chunk parity)
  float* rq = gbuf + 512;
  float* rk = gbuf + 576;
  float* at = reinterpret_cast<float*>(sm + PfSmem::AT);
  float* tf = reinterpret_cast<float*>(sm + PfSmem::TF);
  TOUT* ot = reinterpret_cast<TOUT*>(sm + PfSmem::OT);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + PfSmem::MBAR);   // [0] K^K^T [1] S0 [K^;Q^]^T [2] U [3] U^T P^T [4] rows [5] S update
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + PfSmem::TSLOT);

  if (warp == 0) {
    tc::tmem_alloc(tslot, kPfCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
#pragma unroll
    for (int b = 0; b < 6; ++b) tc::mbar_init(mbar + b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tS = tbase + tlane + kColS + 32 * quarter;   // this thread's 32 state columns

  // chunk c's pre-conv rows t0-3 .. t0+63 (three TMA tiles: q, k, v channels;
  // rows outside x read as zeros).  The rows before a sequence's first token
  // are fixed up after they land (they belong to the previous sequence).
  auto stage = [&](int64_t c) {
    const int64_t t0 = c * C;
    if (tid == 0) {
      tc::mbar_expect_tx(mbar + 4, 3 * kPfXRows * D * 2);
      const int y = (int)(row0 + t0 - kWinRows);
      tc::tma_load_2d(xq, &xmap, cq0, y, mbar + 4);
      tc::tma_load_2d(xk, &xmap, ck0, y, mbar + 4);
      tc::tma_load_2d(xv, &xmap, cv0, y, mbar + 4);
    }
  };
  int64_t x_issued = -1;   // chunk whose rows are in flight (every worker tracks it)
  if (worker && cb < ce) {
    stage(cb);
    x_issued = cb;
  }

  // conv taps of this thread's q | k channel pair and v channel (row),
  // re-read from L1 / L2 at every chunk (an asm load the compiler does not
  // hoist) rather than held in registers through the chunk's other phases
  const int qkp = 2 * (tid & 127);   // this thread's q | k channel pair in the conv
  const float* wqk_src = p.conv_w + (int64_t)(qkp < D ? cq0 + qkp : ck0 + qkp - D) * kConvK;   // two tap sets
  const float* wv_src = p.conv_w + (int64_t)(cv0 + row) * kConvK;
  if (worker) {
    // initial state (zeros on a cold start: the pool is not read)
    const float* src = from >= 0 ? page_state(p.pool, from) + ((int64_t)h * D + row) * D + 32 * quarter : nullptr;
    float v[32];
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4) {
      const float4 f = src ? reinterpret_cast<const float4*>(src)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
      v[4 * c4] = f.x; v[4 * c4 + 1] = f.y; v[4 * c4 + 2] = f.z; v[4 * c4 + 3] = f.w;
    }
    tc::tmem_st32(tS, v);
    tc::tmem_st_wait();
  }

  int32_t pend = -1;    // checkpoint page due at the next read of S
  bool ok = true;
  uint32_t issued = 0;  // tensor-core products committed in the current chunk (bit b: mbar[b])
  bool s_pending = false;   // the previous chunk's state update may still be running
  int64_t ci = cb;          // the chunk `issued` refers to
  int64_t c = cb;
  for (; c < ce; ++c) {
    // each mbarrier completes once per chunk; a piece starts at an even chunk,
    // so the parity of its first wait is 0
    const uint32_t par = (uint32_t)(c & 1);
    const int64_t t0 = c * C;
    const int cnt = (int)(n - t0 < C ? n - t0 : C);
    issued = 0;
    ci = c;
    // this chunk's gate set: G (running sum of the log decays), gam = exp(G),
    // dec = exp(G_C - G), b; rows past the end have g = b = 0
    float* const Gs = gbuf + 256 * (int)(c & 1);
    float* const gam = Gs + 64;
    float* const dec = Gs + 128;
    float* const bv = Gs + 192;
    if (!worker) {
      // the issuing warp forms the gate set while the workers convolve (the
      // set it overwrites was last read two chunks ago); the workers meet it
      // at named barrier 3 before their first use
      float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
      if (t0 + lane < n) { g0 = *V.gptr(t0 + lane, h); b0 = *V.bptr(t0 + lane, h); }
      if (t0 + lane + 32 < n) { g1 = *V.gptr(t0 + lane + 32, h); b1 = *V.bptr(t0 + lane + 32, h); }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float a0 = __shfl_up_sync(0xffffffffu, g0, o);
        const float a1 = __shfl_up_sync(0xffffffffu, g1, o);
        if (lane >= o) { g0 += a0; g1 += a1; }
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      const float gC = __shfl_sync(0xffffffffu, g1, 31);
      Gs[lane] = g0; Gs[lane + 32] = g1;
      gam[lane] = expf(g0); gam[lane + 32] = expf(g1);
      dec[lane] = expf(gC - g0); dec[lane + 32] = expf(gC - g1);
      bv[lane] = b0; bv[lane + 32] = b1;
      named_arrive(3, kPfThreads);
    }

    if (worker) {
      const float4 wqa = ldg_f4_fresh(wqk_src), wqb = ldg_f4_fresh(wqk_src + kConvK), wv = ldg_f4_fresh(wv_src);
      // ---- the chunk's rows and gates have landed; the previous output tile
      // has been read out
      if (tid == 0) tc::bulk_wait_read();
      // the workers agree on the outcome: rows still landing are never
      // staged over (a run-out skips the next chunk's rows and leaves at the
      // next whole-CTA barrier)
      ok = workers_sync_and(work_wait(mbar + 4, par, wlim) && ok);
      if (ok) x_issued = -1;
      if (c == 0) {
        // history rows of the first chunk: the resumed window, or zeros
        const TIN* win = V.win;
        for (int e = tid; e < 3 * kWinRows * (D / 2); e += kPfWorkers) {
          const int tile = e / (kWinRows * (D / 2)), r = (e / (D / 2)) % kWinRows, c2 = e % (D / 2);
          const int ch = (tile == 0 ? cq0 : tile == 1 ? ck0 : cv0) + 2 * c2;
          uint32_t v = 0;
          if (win) v = *reinterpret_cast<const uint32_t*>(win + (int64_t)r * p.conv_dim + ch);
          TIN* dst = tile == 0 ? xq : tile == 1 ? xk : xv;
          *reinterpret_cast<uint32_t*>(dst + r * D + 2 * c2) = v;
        }
        workers_sync();
      }

      // ---- (A) conv + SiLU.  q | k channels qkp, qkp + 1 for rows [16 rh, +16)
      // -> y, the two channels as packed fp32 pairs (one 32-bit load of the two
      // bf16 inputs, one f32x2 instruction per tap, one 8-byte store; each
      // element's arithmetic as in a scalar evaluation).  Rows past the end are
      // computed too and masked later: their norm factors and b are zero, so
      // they contribute nothing (no data-dependent branch around the SiLU)
      {
        const int tb = 16 * (tid >> 7);
        const TIN* xp = (qkp < D ? xq + qkp : xk + qkp - D) + tb * D;
        const f32x2 w0 = pack2(wqa.x, wqb.x), w1 = pack2(wqa.y, wqb.y), w2 = pack2(wqa.z, wqb.z),
                    w3 = pack2(wqa.w, wqb.w);
        f32x2 x[19];
#pragma unroll
        for (int u = 0; u < 19; ++u) {
          // a bf16 is the upper half of its fp32: shift the first channel up, mask the second
          const uint32_t v = *reinterpret_cast<const uint32_t*>(xp + u * D);
          x[u] = pack2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
        }
        float* yrow = yf + tb * 256 + qkp;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          f32x2 z = mul2(w0, x[i]);
          z = fma2(w1, x[i + 1], z);
          z = fma2(w2, x[i + 2], z);
          z = fma2(w3, x[i + 3], z);
          const float2 zz = unpack2(z);
          *reinterpret_cast<float2*>(yrow + i * 256) = make_float2(silu_fast(zz.x), silu_fast(zz.y));
        }
      }
      // v channel `row` for rows [16 quarter, +16) -> tensor memory (lane = channel)
      {
        // rows i and i + 8 as one packed pair (their windows do not overlap)
        const int tb = 16 * quarter;
        float xr[19], vr[16];
#pragma unroll
        for (int u = 0; u < 19; ++u) xr[u] = to_f32(xv[(tb + u) * D + row]);
        const f32x2 w0 = pack2(wv.x, wv.x), w1 = pack2(wv.y, wv.y), w2 = pack2(wv.z, wv.z), w3 = pack2(wv.w, wv.w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          f32x2 z = mul2(w0, pack2(xr[i], xr[i + 8]));
          z = fma2(w1, pack2(xr[i + 1], xr[i + 9]), z);
          z = fma2(w2, pack2(xr[i + 2], xr[i + 10]), z);
          z = fma2(w3, pack2(xr[i + 3], xr[i + 11]), z);
          const float2 zz = unpack2(z);
          vr[i] = silu_fast(zz.x);
          vr[i + 8] = silu_fast(zz.y);
        }
        tc::tmem_st16(tbase + tlane + kColV + 16 * quarter, vr);
      }
      tc::tmem_st_wait();
      workers_sync();
      // the staged rows are consumed: prefetch the next chunk
      if (ok && c + 1 < ce) {
        stage(c + 1);
        x_issued = c + 1;
      }
      // L2 norm factors: warp w reduces (row, q | k) pairs w, w+16, ... in a
      // fixed order; rows past the end get factor 0
      {
        constexpr int NP = 128 / (kPfWorkers / 32);
        float ss[NP];
#pragma unroll
        for (int it = 0; it < NP; ++it) {
          const int k = warp + (kPfWorkers / 32) * it, t = k >> 1, isk = k & 1;
          const float* yr = yf + t * 256 + isk * D;
          float a = 0.f;
#pragma unroll
          for (int m = 0; m < D / 32; ++m) {
            const float y = yr[lane + 32 * m];
            a = fmaf(y, y, a);
          }
          ss[it] = a;
        }
        // the eight sums over the warp at once: lanes 16 apart swap half of
        // their partial sums and add (four sums left per lane), then lanes 8
        // apart (two), 4 apart (one), and two more levels finish it; lane l
        // ends with the total of pair (l >> 2) (9 shuffles instead of 40)
        static_assert(NP == 8, "the halving reduction is written for eight sums");
        float h4[4], h2[2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool up = lane & 16;
          const float send = up ? ss[j] : ss[j + 4];
          h4[j] = (up ? ss[j + 4] : ss[j]) + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const bool up = lane & 8;
          const float send = up ? h4[j] : h4[j + 2];
          h2[j] = (up ? h4[j + 2] : h4[j]) + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        float a;
        {
          const bool up = lane & 4;
          a = (up ? h2[1] : h2[0]) + __shfl_xor_sync(0xffffffffu, up ? h2[0] : h2[1], 4);
        }
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        if ((lane & 3) == 0) {
          const int k = warp + (kPfWorkers / 32) * (lane >> 2), t = k >> 1, isk = k & 1;
          (isk ? rk : rq)[t] = t < cnt ? (isk ? 1.0f : p.q_scale) / sqrtf(a + p.eps) : 0.f;
        }
      }
      named_sync(3, kPfThreads);   // the norm factors, and the issuing warp's gate set
      // operands: [K^; Q^] (rows 0-63 k^, 64-127 q^) and K^T diag(dec) (row =
      // k channel); each thread loads all of its inputs before it stores.
      // The previous chunk's state update reads U^T and K^T diag(dec): it
      // has finished first.
      if (s_pending) mma_wait(mbar + 5, (uint32_t)((c - 1) & 1), ok, wlim);
      {
        constexpr int NKQ = 2048 / kPfWorkers, NKT = 1024 / kPfWorkers;
        float4 ya[NKQ], yb[NKQ];
        float fv[NKQ];
#pragma unroll
        for (int it = 0; it < NKQ; ++it) {
          const int i = tid + kPfWorkers * it, r = i >> 4, c8 = i & 15;
          const int t = r & (C - 1);
          const bool isq = r >= C;
          fv[it] = isq ? rq[t] : rk[t];
          const float4* src = reinterpret_cast<const float4*>(yf + t * 256 + (isq ? 0 : D) + 8 * c8);
          ya[it] = src[0];
          yb[it] = src[1];
        }
#pragma unroll
        for (int it = 0; it < NKQ; ++it) {
          const int i = tid + kPfWorkers * it, r = i >> 4, c8 = i & 15;
          const float f = fv[it];
          const f32x2 f2 = pack2(f, f);
          const float2 e01 = unpack2(mul2(pack2(ya[it].x, ya[it].y), f2));
          const float2 e23 = unpack2(mul2(pack2(ya[it].z, ya[it].w), f2));
          const float2 e45 = unpack2(mul2(pack2(yb[it].x, yb[it].y), f2));
          const float2 e67 = unpack2(mul2(pack2(yb[it].z, yb[it].w), f2));
          const float e[8] = {e01.x, e01.y, e23.x, e23.y, e45.x, e45.y, e67.x, e67.y};
          const uint32_t off = tc::sw128_offset(r, 8 * c8, 128);
          tc::store_split8(sm + PfSmem::KQ + off, sm + PfSmem::KQ_LO + off, e);
        }
        float kt[NKT][8];
#pragma unroll
        for (int it = 0; it < NKT; ++it) {
          const int i = tid + kPfWorkers * it, k = i & 127, j8 = i >> 7;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = 8 * j8 + u;
            kt[it][u] = (yf[j * 256 + D + k] * rk[j]) * dec[j];
          }
        }
#pragma unroll
        for (int it = 0; it < NKT; ++it) {
          const int i = tid + kPfWorkers * it, k = i & 127, j8 = i >> 7;
          const uint32_t off = tc::sw128_offset(k, 8 * j8, 128);
          tc::store_split8(sm + PfSmem::KT + off, sm + PfSmem::KT_LO + off, kt[it]);
        }
      }
      tc::fence_async_smem();
    }
    ok = cta_sync_ok(ok);   // y is consumed; [K^; Q^] and K^T diag(dec) are in place
    if (!ok) break;
    s_pending = false;
    // [K^ K^T; Q^ K^T] (M 128, N 64, K 128) needs no state: it runs during the split
    if (tid == kMmaTid) {
      tc::mma3_sw128<D / 16, 16384, 16384>(tbase + kColKK, sbase + PfSmem::KQ, sbase + PfSmem::KQ_LO, sbase + PfSmem::KQ,
           sbase + PfSmem::KQ_LO, tc::idesc_bf16_f32(128, 64), false);
      tc::mma_commit(mbar + 0);
    }
    issued |= 1u;

    // ---- (B) S0 -> bf16 operand; checkpoint due at this boundary; gam_C S0 back
    if (worker) {
      const float gC = gam[C - 1];
      float* ck = pend >= 0 ? page_state(p.pool, pend) + ((int64_t)h * D + row) * D + 32 * quarter : nullptr;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v0[16];
        tc::tmem_ld16(tS + 16 * hh, v0);
        if (ck) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            reinterpret_cast<float4*>(ck + 16 * hh)[c4] =
                make_float4(v0[4 * c4], v0[4 * c4 + 1], v0[4 * c4 + 2], v0[4 * c4 + 3]);
        }
#pragma unroll
        for (int c8 = 0; c8 < 2; ++c8) {
          const uint32_t off = tc::sw128_offset(row, 32 * quarter + 16 * hh + 8 * c8, 128);
          tc::store_split8(sm + PfSmem::S0 + off, sm + PfSmem::S0_LO + off, v0 + 8 * c8);
        }
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float2 g = unpack2(mul2(pack2(v0[e], v0[e + 1]), pack2(gC, gC)));
          v0[e] = g.x;
          v0[e + 1] = g.y;
        }
        tc::tmem_st16(tS + 16 * hh, v0);
      }
      tc::tmem_st_wait();
      pend = -1;
      tc::fence_async_smem();
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == kMmaTid) {
      // S0 [K^; Q^]^T (M 128, N 128, K 128)
      tc::mma3_sw128<D / 16, 16384, 16384>(tbase + kColSK, sbase + PfSmem::S0, sbase + PfSmem::S0_LO, sbase + PfSmem::KQ,
           sbase + PfSmem::KQ_LO, tc::idesc_bf16_f32(128, 128), false);
      tc::mma_commit(mbar + 1);
    }
    issued |= 2u;

    // ---- (C) A^T (lanes 0-63: k^_i.k^_j) and P (lanes 64-127: q^_i.k^_j) for
    // columns j in [16 quarter, +16), computed while S0 [K^; Q^]^T runs
    if (worker) {
      mma_wait(mbar + 0, par, ok, wlim);
      const int q4 = warp & 3;
      const int ir = (q4 & 1) * 32 + lane;   // chunk row i of this thread's lane
      float ap[16];
      {
        tc::tmem_ld16(tbase + tlane + kColKK + 16 * quarter, ap);
        const float Gi = Gs[ir];
        const float bi = q4 < 2 ? bv[ir] : 1.0f;
        const int lim = q4 < 2 ? ir : ir + 1;        // A: j < i; P: j <= i
        // exp(G_i - G_j) <= 1 where it is kept; the clamp keeps the masked
        // entries finite, the 0/1 mask avoids a branch around the exponential
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = 16 * quarter + e;
          const float m = j < lim ? bi : 0.f;
          ap[e] = m * __expf(fminf(Gi - Gs[j], 0.f)) * ap[e];
        }
      }
      mma_wait(mbar + 1, par, ok, wlim);
      workers_sync();   // every worker is past the S0 [K^; Q^]^T wait: [K^; Q^] is free
      if (q4 < 2) {
        float* am = reinterpret_cast<float*>(sm + PfSmem::AM);
#pragma unroll
        for (int e = 0; e < 16; ++e) at[(16 * quarter + e) * C + ir] = ap[e];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          *reinterpret_cast<float4*>(am + am_index(ir, 16 * quarter + 4 * c4)) =
              make_float4(ap[4 * c4], ap[4 * c4 + 1], ap[4 * c4 + 2], ap[4 * c4 + 3]);
      } else {
#pragma unroll
        for (int c8 = 0; c8 < 2; ++c8) {
          const uint32_t off = tc::sw128_offset(ir, 16 * quarter + 8 * c8, 64);
          tc::store_split8(sm + PfSmem::PB + off, sm + PfSmem::PB_LO + off, ap + 8 * c8);
        }
      }
      workers_sync();
      if (tid >= 256) {
        // T = (I + A)^{-1}, then T as the B operand (rows i, K = j; zero above the diagonal)
        tri_inverse64(at, reinterpret_cast<const float*>(sm + PfSmem::AM), tf, reinterpret_cast<float*>(sm + PfSmem::DT),
                      reinterpret_cast<float*>(sm + PfSmem::NT), tid - 256);
        for (int e = tid - 256; e < 512; e += 256) {
          const int i = e >> 3, c8 = e & 7;
          const float4 a = *reinterpret_cast<const float4*>(tf + i * C + 8 * c8);
          const float4 b = *reinterpret_cast<const float4*>(tf + i * C + 8 * c8 + 4);
          float v8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (8 * c8 + u > i) v8[u] = 0.f;
          const uint32_t off = tc::sw128_offset(i, 8 * c8, 64);
          tc::store_split8(sm + PfSmem::TB + off, sm + PfSmem::TB_LO + off, v8);
        }
      } else {
        // R_i = b_i (v_i - gam_i (S0 k^_i)) of state row `row` for rows i in
        // [32 qh, +32) -> the A operand of U^T = R T^T
        const int qh = tid >> 7;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i0 = 32 * qh + 16 * hh;
          float a[16], b[16];
          tc::tmem_ld16x2(tbase + tlane + kColSK + i0, tbase + tlane + kColV + i0, a, b);
#pragma unroll
          for (int e = 0; e < 16; ++e) a[e] = bv[i0 + e] * fmaf(-gam[i0 + e], a[e], b[e]);
#pragma unroll
          for (int c8 = 0; c8 < 2; ++c8) {
            const uint32_t off = tc::sw128_offset(row, i0 + 8 * c8, 128);
            tc::store_split8(sm + PfSmem::UT + off, sm + PfSmem::UT_LO + off, a + 8 * c8);
          }
        }
      }
      tc::fence_async_smem();
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == kMmaTid) {
      // U^T = R T^T (M 128, N 64, K 64)
      tc::mma3_sw128<C / 16, 0, 0>(tbase + kColU, sbase + PfSmem::UT, sbase + PfSmem::UT_LO, sbase + PfSmem::TB,
           sbase + PfSmem::TB_LO, tc::idesc_bf16_f32(128, 64), false);
      tc::mma_commit(mbar + 2);
    }
    issued |= 4u;
    // U^T (rows r, K = i) as the A operand of the state update and the outputs
    if (worker) {
      mma_wait(mbar + 2, par, ok, wlim);
      float u[16];
      tc::tmem_ld16(tbase + tlane + kColU + 16 * quarter, u);
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {
        const uint32_t off = tc::sw128_offset(row, 16 * quarter + 8 * c8, 128);
        tc::store_split8(sm + PfSmem::UT + off, sm + PfSmem::UT_LO + off, u + 8 * c8);
      }
      tc::fence_async_smem();
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;

    // ---- (D) U^T P^T first (the outputs wait for it), then S += U^T
    // (K^T diag(dec))^T onto gam_C S0, which finishes while the next chunk's
    // conv and norms run
    if (tid == kMmaTid) {
      tc::mma3_sw128<C / 16, 0, 0>(tbase + kColU, sbase + PfSmem::UT, sbase + PfSmem::UT_LO, sbase + PfSmem::PB,
           sbase + PfSmem::PB_LO, tc::idesc_bf16_f32(128, 64), false);
      tc::mma_commit(mbar + 3);
      tc::mma3_sw128<C / 16, 0, 0>(tbase + kColS, sbase + PfSmem::UT, sbase + PfSmem::UT_LO, sbase + PfSmem::KT,
           sbase + PfSmem::KT_LO, tc::idesc_bf16_f32(128, 128), true);
      tc::mma_commit(mbar + 5);
    }
    issued |= 8u | 32u;
    s_pending = true;
    if (worker) {
      mma_wait(mbar + 3, par, ok, wlim);
      // outputs o_i = gam_i (S0 q^_i) + (U^T P^T)_i for rows i in [16 quarter, +16):
      // a full chunk goes out as one TMA tile through shared memory, a
      // partial one (the sequence's last) by plain stores
      float sq[16], up[16];
      tc::tmem_ld16x2(tbase + tlane + kColSQ + 16 * quarter, tbase + tlane + kColU + 16 * quarter, sq, up);
      if (p.norm_w) {
        // packed core: a token's 128 outputs are normalised together, so they
        // meet in shared memory; warp w then takes tokens w, w+16, ...: RMS
        // over dv, the norm scale, the silu(z) gate from the packed row
        float* of = reinterpret_cast<float*>(sm + PfSmem::OF);
#pragma unroll
        for (int e = 0; e < 16; ++e) of[(16 * quarter + e) * D + row] = fmaf(gam[16 * quarter + e], sq[e], up[e]);
        workers_sync();
        const TIN* zrow = reinterpret_cast<const TIN*>(p.x) + (row0 + t0) * p.x_ld + p.conv_dim + h * D;
        TOUT* orow = reinterpret_cast<TOUT*>(p.o) + ((row0 + t0) * p.Hv + h) * D;
        for (int i = warp; i < cnt; i += kPfWorkers / 32) {
          float v[4];
          float ss = 0.f;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            v[m] = of[i * D + lane + 32 * m];
            ss = fmaf(v[m], v[m], ss);
          }
          ss = warp_sum(ss);
          const float inv = 1.0f / sqrtf(ss * (1.0f / D) + p.norm_eps2);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float z = to_f32(zrow[(int64_t)i * p.x_ld + lane + 32 * m]);
            orow[(int64_t)i * p.Hv * D + lane + 32 * m] = from_f32<TOUT>(v[m] * inv * p.norm_w[lane + 32 * m] * silu_fast(z));
          }
        }
      } else if (tma_out && cnt == C) {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          ot[(16 * quarter + e) * D + row] = from_f32<TOUT>(fmaf(gam[16 * quarter + e], sq[e], up[e]));
        tc::fence_async_smem();
        workers_sync();
        if (tid == 0) {
          tc::tma_store_2d(&omap, h * D, (int)(row0 + t0), ot);
          tc::bulk_commit();
        }
      } else {
        TOUT* out = reinterpret_cast<TOUT*>(p.o) + ((row0 + t0) * p.Hv + h) * D + row;
        const int64_t tstride = (int64_t)p.Hv * D;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i = 16 * quarter + e;
          if (i < cnt) out[i * tstride] = from_f32<TOUT>(fmaf(gam[i], sq[e], up[e]));
        }
      }
      // a block boundary at this chunk's end: the state is checkpointed when
      // it is next read
      const int64_t pos = start + t0 + cnt;
      if (pos % p.block_size == 0) {
        const int64_t jb = pos / p.block_size - 1;
        int32_t page = -1;
        if (jb < p.max_blocks) page = p.block_table[(int64_t)s * p.max_blocks + jb];
        else if (report) set_error(p.err, GDN_ERR_INVALID_ARG);
        if (page >= 0) {
          if (page_ok(p.pool, page)) pend = page;
          else if (report) set_error(p.err, GDN_ERR_PAGE_RANGE);
        }
      }
    }
  }

  if (ok && worker && s_pending) mma_wait(mbar + 5, (uint32_t)((c - 1) & 1), ok, wlim);
  ok = cta_sync_ok(ok);
  if (ok) {
    if (worker) {
      // final state (and a checkpoint due at the last chunk's end)
      float* dst = page_state(p.pool, final_page) + ((int64_t)h * D + row) * D + 32 * quarter;
      float* ck = pend >= 0 ? page_state(p.pool, pend) + ((int64_t)h * D + row) * D + 32 * quarter : nullptr;
      float v0[32];
      tc::tmem_ld32(tS, v0);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 f0 = make_float4(v0[4 * c4], v0[4 * c4 + 1], v0[4 * c4 + 2], v0[4 * c4 + 3]);
        reinterpret_cast<float4*>(dst)[c4] = f0;
        if (ck) reinterpret_cast<float4*>(ck)[c4] = f0;
      }
    }
  } else {
    // a wait ran out: report it, give the tensor core and the copy engine one
    // more bounded wait for each piece of work they may still hold, then
    // release the tensor memory
    if (tid == 0) atomicExch(p.err, GDN_ERR_TIMEOUT);   // overrides an earlier code
    const uint32_t par = (uint32_t)(ci & 1);
#pragma unroll 1
    for (int b = 0; b < 4; ++b)
      if (issued & (1u << b)) tc::mbar_wait_bounded(mbar + b, par, kPfWait);
    // the last state update issued: chunk ci's, or else the one before it
    if (issued & 32u) tc::mbar_wait_bounded(mbar + 5, par, kPfWait);
    else if (s_pending && ci > 0) tc::mbar_wait_bounded(mbar + 5, (uint32_t)((ci - 1) & 1), kPfWait);
    if (worker && x_issued >= 0) tc::mbar_wait_bounded(mbar + 4, (uint32_t)(x_issued & 1), kPfWait);
  }
  if (tid == 0) tc::bulk_wait_all();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, kPfCols);
}

int tc_prefill_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// One CTA holds an SM for a whole chain, so the Hv x N chains of maxc chunks
// take ceil(Hv N / sms) rounds of maxc chunk times in one launch: 192 chains
// on 152 SMs take two, the second with 40 SMs busy.  A chain's chunks must
// run in order, but its state can move between launches exactly (fp32
// through the final slot's page), so the chains are cut into pieces of P
// chunks and run level by level: (level, sequence) pairs in level-major order
// (every sequence's first pieces, then every second piece, ...), floor(sms /
// Hv) pairs of Hv CTAs a launch.  With N >= that many pairs, consecutive
// pieces of a chain are N pairs apart, so each lands in a later launch than
// the one before it, and no launch holds two pieces of one chain.  Each
// chunk's arithmetic is the same as in one launch, so the results are
// bitwise the same.  A launch costs about 1.5 chunk times more than its
// pieces' chunks (state in and out, the first rows' load, the slowest CTA,
// the launch gap: measured 21 us a launch against 13 us a chunk); P is the
// even piece length >= 4 with the least estimated time, kept only when it
// saves 5 % over one launch and needs at most 64 launches.  A piece starts at
// an even chunk, which keeps the kernel's mbarrier parities (chunk & 1)
// valid.
PrefillSchedule tc_prefill_schedule(int Hv, int num_seqs, int64_t max_len, int sms) {
  return tc_prefill_schedule_cost(Hv, num_seqs, max_len, sms, 1.5);
}

PrefillSchedule tc_prefill_schedule_cost(int Hv, int num_seqs, int64_t max_len, int sms, double kLaunchCost) {
  constexpr int64_t kMinPiece = 4, kMaxLaunches = 64;
  PrefillSchedule sc;
  sc.nchains = (int64_t)Hv * num_seqs;
  const int64_t maxc = max_len > 0 ? (max_len + kPfC - 1) / kPfC : 0;
  sc.piece = maxc > 0 ? (maxc < (1 << 30) ? maxc : (1 << 30)) : 1;
  sc.levels = 1;
  sc.width = sc.nchains;
  sc.launches = sc.nchains > 0 ? 1 : 0;
  sc.chunk_launches = 0;
  const int64_t per = Hv > 0 && sms > 0 ? sms / Hv : 0;   // pairs a launch
  if (per < 1 || num_seqs < per || sc.nchains < sms || maxc < 2 * kMinPiece) return sc;
  const double single = (double)((sc.nchains + sms - 1) / sms) * ((double)maxc + kLaunchCost);
  double best = 0.95 * single;
  for (int64_t P = kMinPiece; P < maxc; P += 2) {
    const int64_t levels = (maxc + P - 1) / P;
    const int64_t launches = (levels * num_seqs + per - 1) / per;
    if (launches > kMaxLaunches) continue;
    const double cost = (double)launches * ((double)P + kLaunchCost);
    if (cost < best) {
      best = cost;
      sc.piece = P;
      sc.levels = levels;
      sc.width = per * Hv;
      sc.launches = launches;
    }
  }
  return sc;
}

bool tc_prefill_supported(int dk, int dv, int in_dtype, int out_dtype, int block_size) {
  return dk == kPfD && dv == kPfD && in_dtype == GDN_BF16 && out_dtype == GDN_BF16 && block_size % kPfC == 0;
}

cudaError_t launch_tc_prefill(const ScanParams& p, int64_t max_len, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  if ((int64_t)p.Hv * p.num_seqs > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
  CUtensorMap xmap, omap;
  memset(&xmap, 0, sizeof(xmap));
  memset(&omap, 0, sizeof(omap));
  int tma_out = 0;
  if (p.total_rows > 0) {
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint32_t estr[2] = {1, 1};
    // x as [rows][x_ld] bf16 (x_ld = conv_dim, or the packed q | k | v | z
    // row); a box is 128 channels x 67 rows
    {
      const cuuint64_t dims[2] = {(cuuint64_t)p.x_ld, (cuuint64_t)p.total_rows};
      const cuuint64_t strides[1] = {(cuuint64_t)p.x_ld * 2};
      const cuuint32_t box[2] = {(cuuint32_t)kPfD, (cuuint32_t)kPfXRows};
      if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    // o as [rows][Hv * dv] bf16; a box is one head's 128 channels x 64 rows
    // (used for full chunks when o is 16-byte aligned)
    if ((reinterpret_cast<uintptr_t>(p.o) & 15) == 0) {
      const cuuint64_t dims[2] = {(cuuint64_t)p.Hv * kPfD, (cuuint64_t)p.total_rows};
      const cuuint64_t strides[1] = {(cuuint64_t)p.Hv * kPfD * 2};
      const cuuint32_t box[2] = {(cuuint32_t)kPfD, (cuuint32_t)kPfC};
      if (encode(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.o, dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
        tma_out = 1;
    }
  }
  const size_t smem = PfSmem::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(tc_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const PrefillSchedule sc = tc_prefill_schedule(p.Hv, p.num_seqs, max_len, tc_prefill_sm_count());
  PieceMap pm;
  pm.nseqs = p.num_seqs;
  pm.piece = (int32_t)sc.piece;
  pm.last_level = (int32_t)(sc.levels - 1);
  const int64_t pairs = sc.levels * p.num_seqs, per = sc.width / p.Hv;   // (level, sequence) pairs
  for (int64_t t = 0; t < sc.launches; ++t) {
    const int64_t base = t * per;
    pm.s0 = (int32_t)(base % p.num_seqs);
    pm.level0 = (int32_t)(base / p.num_seqs);
    const int64_t cnt = pairs - base < per ? pairs - base : per;
    tc_prefill_kernel<<<dim3(p.Hv, (unsigned)cnt), kPfThreads, smem, st>>>(p, xmap, omap, tma_out, pm);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // conv windows of every crossed boundary and of the final slot
  window_kernel<__nv_bfloat16, kPrefill><<<dim3((p.conv_dim + 255) / 256, p.num_seqs, window_slices(p, max_len)), 256, 0,
                                            st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
