// tc_chain.cu — the chunked prefill as two kernels on the tensor cores (dk =
// dv = 128, bf16 inputs and outputs, block size a multiple of 64), with the
// same arithmetic as the fused kernel (tc_prefill.cu), bit for bit.
//
// The chunk (UT) form of the gated delta rule ("Gated DeltaNet",
// S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t) over a
// chunk of C = 64 tokens, with k^, q^ the L2-normalised rows, G_i the running
// sum of the log decays inside the chunk, gam_i = exp(G_i), dec_i =
// exp(G_C - G_i), S0 the state entering the chunk:
//   A_ij = b_i exp(G_i - G_j) k^_i.k^_j (j < i),  T = (I + A)^{-1}
//   P_ij = exp(G_i - G_j) q^_i.k^_j (j <= i)
//   R_i  = b_i (v_i - gam_i S0 k^_i),  U = T R
//   o_i  = gam_i S0 q^_i + (P U)_i,    S_C = gam_C S0 + U^T diag(dec) K^
// Everything left of R depends only on the chunk's rows; the rest needs S0.
//
// tc_chunk_kernel: one CTA per (sequence, chunk, qk head).  The conv + SiLU of
//   the q and k channels, their norms, the operand [K^; Q^] and the Gram
//   products [K^ K^T; Q^ K^T] run once for the qk head's group of value heads;
//   then per value head the gates, A, P, T and K^T diag(dec).  It leaves, per
//   chunk slot of the workspace, the fused kernel's own operand images:
//   [K^; Q^] per qk head; T, P and K^T diag(dec) (bf16 hi / lo, 128-byte
//   swizzled) and the gates per value head.  No chunk waits for another, so
//   the whole call's chunks fill every SM.
// tc_chain_kernel: one CTA per (sequence, value head) chain, or a piece of
//   one: a chain's chunks run in order, and a call cut into pieces passes the
//   state between launches through the final page, exactly.  The fp32 state
//   stays in tensor memory; per chunk, the fused kernel's state steps:
//   S0 [K^; Q^]^T, R, U^T = R T^T, then S += U^T (K^T diag(dec))^T and U^T P^T,
//   and the outputs.  v comes from the conv + SiLU of the pre-conv rows, in
//   the fused kernel's expression, while the first product runs.  The next
//   chunk's images and rows load as soon as their readers are done.
// With no more chains than SMs the two kernels overlap: the chains are cut
// into levels, and level l of every chain runs on a second stream once the
// chunk kernel's launch l has written that level's images, while launch
// l + 1 takes the SMs the chains leave (tc_chain_schedule picks the level
// length, or none, from a cost model of both paths).  The chain is then the
// call's critical path, so in this mode (VIMG) the chunk kernel convolves v
// and writes it as an fp32 image instead.
// Every operand is split and every product issued exactly as in the fused
// kernel (the same bf16 hi / lo parts, the same M x N x K shapes and passes in
// the same order), so the two paths give the same bits and a call may take
// either.  Chunks start at absolute multiples of 64, so a block boundary is a
// chunk end and a checkpoint is the tensor-memory state between two chunks.
// Every mbarrier wait is bounded (gdn_prefill_args.wait_cycles).
#include <cmath>
#include <mutex>

#include "launch.h"
#include "tc.cuh"
#include "tc_chunk.cuh"

namespace gdn {

namespace {

constexpr int kD = 128, kC = 64;
constexpr int kWorkers = 512;                 // sixteen worker warps
constexpr int kThreads = kWorkers + 32;       // + the issuing warp
constexpr int kMma = kWorkers;                // the issuing thread
constexpr int kXRows = kC + kWinRows;
constexpr long long kWaitDefault = 4000000000LL;

// ---- workspace: per chunk slot, the fused kernel's operand images ----------
constexpr uint32_t kImgKQ = 65536;   // [K^; Q^] hi | lo: 128 rows x 128 k, two 64-wide k-blocks each (per qk head)
constexpr uint32_t kImgT = 16384;    // T hi | lo: 64 rows (i) x 64 k (j)
constexpr uint32_t kImgP = 16384;    // P hi | lo: 64 rows (i) x 64 k (j)
constexpr uint32_t kImgK = 32768;    // K^T diag(dec) hi | lo: 128 rows (c) x 64 k (j)
constexpr uint32_t kImgV = 32768;    // v fp32 [64 rows][128 channels] (image mode only)
constexpr uint32_t kImgG = 1024;     // G, gam, dec, b fp32 [4][64]

struct ChunkWs {
  uint8_t* kq;     // [slots][Hqk] kImgKQ
  uint8_t* t;      // [slots][Hv] kImgT
  uint8_t* pm;     // [slots][Hv] kImgP
  uint8_t* k;      // [slots][Hv] kImgK
  float* v;        // [slots][Hv] kImgV (image mode)
  float* g;        // [slots][Hv] kImgG
  float* core_o;   // packed core: fp32 outputs [rows][Hv][dv] before the gated norm (else null)
  int64_t slots;
};

// A sequence's chunk c lives in slot floor(cu[s] / 64) + s + c: chunks of
// consecutive sequences never share a slot, and the slots of a call number
// at most floor(T / 64) + N + 1.
__device__ __forceinline__ int64_t chunk_slot(const ScanParams& p, int s, int64_t c) {
  return (int64_t)p.cu_seqlens[s] / kC + s + c;
}

// ---- shared memory of the chunk kernel (offsets from a 1024-aligned base) ----
struct CkSmem {
  static constexpr uint32_t XQ = 0;                  // (A) pre-conv rows t0-3 .. t0+63, bf16 [67][128]
  static constexpr uint32_t XK = 17408;
  static constexpr uint32_t TB = 0;                  // (B) T hi [64][64], lo at +8 KB
  static constexpr uint32_t TB_LO = 8192;
  static constexpr uint32_t PB = 16384;              //     P hi [64][64], lo at +8 KB
  static constexpr uint32_t PB_LO = 24576;
  static constexpr uint32_t XV = 34816;              // (image mode) v rows of the current value head
  static constexpr uint32_t YQ = 53248;              // (A) SiLU(conv) of the q channels, fp32 [64][128]
  static constexpr uint32_t KT = YQ;                 // (B) K^T diag(dec) hi [128][64], lo at +16 KB
  static constexpr uint32_t KT_LO = YQ + 16384;
  static constexpr uint32_t YK = 86016;              // SiLU(conv) of the k channels, fp32 [64][128] (kept)
  static constexpr uint32_t KQ = 118784;             // (A) [K^; Q^] hi [2 kb][128][64], lo at +32 KB
  static constexpr uint32_t KQ_LO = KQ + 32768;
  static constexpr uint32_t VS = KQ;                 // (B, image mode) v fp32 [64 rows][128 channels], stored with K~
  static constexpr uint32_t TF = KQ + 32768;         // (B) T fp32 [64][64]
  static constexpr uint32_t DT = KQ + 49152;         //     diagonal inverses [4][16][20]
  static constexpr uint32_t NT = KQ + 54272;         //     N blocks [6][16][16]
  static constexpr uint32_t GT = KQ + 65536;         // gate sets [4][4][64] fp32 (G, gam, dec, b), then rq, rk
  static constexpr uint32_t AT = GT + 4096 + 512;    // A^T fp32 [64 j][64 i]
  static constexpr uint32_t AM = AT + 16384;         // A fp32 row-major, slots swizzled
  // (B, conv mode) a second A^T / A / P set: the K group forms the next
  // value head's while the T group inverts this one's (regions the image
  // mode uses for v)
  static constexpr uint32_t AT1 = KQ;
  static constexpr uint32_t AM1 = KQ + 16384;
  static constexpr uint32_t PB1 = XV;               //     (P hi, lo at +8 KB)
  static constexpr uint32_t MBAR = AM + 16384;       // [0] Gram [1] q / k rows [2] v rows (image mode)
  static constexpr uint32_t TSLOT = MBAR + 24;
  static constexpr uint32_t BYTES = TSLOT + 8;
  static constexpr uint32_t ALLOC = BYTES + 1024;
};
static_assert(CkSmem::PB_LO + 8192 <= CkSmem::XV && CkSmem::XV + 17408 <= CkSmem::YQ, "chunk kernel regions overlap");
static_assert(CkSmem::ALLOC <= 232448, "chunk kernel shared memory exceeds the per-CTA limit");

constexpr int kGateSets = 4;        // gate sets of the chunk kernel (value heads formed ahead)
constexpr uint32_t kCkCols = 128;   // tensor memory of the chunk kernel
constexpr uint32_t kCkGram = 0;     // [K^ K^T; Q^ K^T]: lanes 0-63 k^_i.k^_j, 64-127 q^_i.k^_j
constexpr uint32_t kCkV = 64;       // (image mode) v of the chunk, lane = channel, column = row

// ---- shared memory of the chain kernel: T and P (with the gates) in two
// buffers, the others in one, each reloaded as soon as its reader is done -------
struct ChSmem {
  static constexpr uint32_t KQ = 0;                  // [K^; Q^] hi | lo
  static constexpr uint32_t KT = KQ + kImgKQ;        // K^T diag(dec) hi | lo
  static constexpr uint32_t TB = KT + kImgK;         // T hi | lo [2]
  static constexpr uint32_t PB = TB + 2 * kImgT;     // P hi | lo [2]
  static constexpr uint32_t XV = PB + 2 * kImgP;     // v: the image fp32 [64 rows][128 channels] (image mode), or
                                                     // the pre-conv rows t0-3 .. t0+63 of the head, bf16 [67][128]
  static constexpr uint32_t OT = XV + kImgV;         // outputs bf16 [64 rows][128 dv]
  static constexpr uint32_t G = OT + 16384;          // gate sets [2][4][64]
  static constexpr uint32_t MBAR = G + 2 * kImgG;
  // mbarriers: the images [K^; Q^], K~, T [2], P | gates [2], v; then the
  // products S0 [K^; Q^]^T, R T^T, the state update, U^T P^T
  // (kZ: the packed core's z rows of a chunk, in the output tile's region)
  static constexpr int kKQ = 0, kKT = 1, kTb = 2, kPG = 4, kVb = 6, kSK = 7, kU = 8, kS = 9, kUP = 10, kZ = 11,
                       kBars = 12;
  static constexpr uint32_t ARMED = MBAR + 8 * kBars;    // int64 [kBars]: last chunk each was armed for
  static constexpr uint32_t NW = ARMED + 8 * kBars;      // the packed core's norm scale fp32 [128]
  static constexpr uint32_t TSLOT = NW + 512;
  static constexpr uint32_t BYTES = TSLOT + 8;
  static constexpr uint32_t ALLOC = BYTES + 1024;
  static constexpr bool two_buffers(int k) { return k == kTb || k == kTb + 1 || k == kPG || k == kPG + 1; }
};
static_assert(ChSmem::KT % 1024 == 0 && ChSmem::TB % 1024 == 0 && ChSmem::PB % 1024 == 0 && ChSmem::OT % 1024 == 0,
              "operand images must be 1024-byte aligned");
static_assert(ChSmem::ALLOC <= 232448, "chain kernel shared memory exceeds the per-CTA limit");

// tensor-memory columns of the chain kernel (lane = state row r)
constexpr uint32_t kChCols = 512;
constexpr uint32_t kChS = 0;        // S fp32 [128][128]
constexpr uint32_t kChSK = 128;     // S0 K^T fp32 [128][64] (then S0 Q^T: one product)
constexpr uint32_t kChSQ = 192;     // S0 Q^T
constexpr uint32_t kChU = 256;      // U^T = R T^T, then U^T P^T
constexpr uint32_t kChS0H = 320;    // S0 hi, bf16 pairs [128][64] (the A operand of S0 [K^; Q^]^T)
constexpr uint32_t kChS0L = 384;    // S0 lo
constexpr uint32_t kChUH = 448;     // R^T, then U^T: hi, bf16 pairs [128][32] (the A operand of the rest)
constexpr uint32_t kChUL = 480;     // lo

__device__ __forceinline__ bool work_wait(uint64_t* m, uint32_t parity, long long lim) {
  return lim >= 0 && tc::mbar_wait_bounded_fast(m, parity, lim);
}
__device__ __forceinline__ void mma_wait(uint64_t* m, uint32_t parity, bool& ok, long long lim) {
  ok = work_wait(m, parity, lim) && ok;
  tc::fence_after_sync();
}
__device__ __forceinline__ bool cta_sync_ok(bool ok) {
  tc::fence_before_sync();
  ok = __syncthreads_and(ok);
  tc::fence_after_sync();
  return ok;
}
// Barrier of the chunk kernel's K group (threads 0..255), and the same
// barrier returning whether `v` holds on every one of them.
__device__ __forceinline__ void kgrp_sync() { asm volatile("bar.sync 4, 256;\n" ::: "memory"); }
__device__ __forceinline__ bool kgrp_sync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 4, 256, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ long long wait_limit(const ScanParams& p) {
  return p.wait_cycles > 0 ? p.wait_cycles : p.wait_cycles < 0 ? -1 : kWaitDefault;
}

// The issuing warp's gate set of value head h for the chunk's rows [t0, t0 +
// 64) (the fused kernel's expressions): G, gam = exp(G), dec = exp(G_C - G),
// b; rows past the end have g = b = 0.
__device__ __forceinline__ void chunk_gates(const TokenView<__nv_bfloat16>& V, int64_t t0, int64_t n, int h,
                                            int lane, float* Gs) {
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
  Gs[64 + lane] = expf(g0); Gs[96 + lane] = expf(g1);
  Gs[128 + lane] = expf(gC - g0); Gs[160 + lane] = expf(gC - g1);
  Gs[192 + lane] = b0; Gs[224 + lane] = b1;
}

}  // namespace

// ============================================================================
// Chunk kernel: grid (Hqk, chunks, N), one CTA per (qk head, chunk c0 + y, sequence)
// ============================================================================
// VIMG (image mode): the chunk kernel also convolves v and writes it as an
// image; otherwise the chain kernel convolves v from the rows itself.
template <bool VIMG>
__global__ void __launch_bounds__(kThreads, 1)
    tc_chunk_kernel(const ScanParams p, const __grid_constant__ CUtensorMap xmap, const ChunkWs ws, int64_t c0) {
  using TIN = __nv_bfloat16;
  constexpr int D = kD, C = kC;
  const int jq = blockIdx.x;
  const int64_t c = c0 + blockIdx.y;
  const int s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool worker = tid < kWorkers;
  const int row = tid & 127;
  const int quarter = (tid >> 7) & 3;
  const uint32_t tlane = (uint32_t)((warp & 3) * 32) << 16;

  TokenView<TIN> V;
  int64_t start, n_log;
  int32_t init, final_page;
  if (!make_view<TIN, kPrefill>(p, s, V, start, init, final_page, n_log, false)) return;
  const int64_t n = V.n;
  if (c * C >= n) return;
  const int64_t t0 = c * C;
  const int cnt = (int)(n - t0 < C ? n - t0 : C);
  const int G = p.Hv / p.Hqk;
  const int cq0 = jq * D, ck0 = p.Hqk * D + jq * D;
  const int64_t row0 = p.cu_seqlens[s];
  const int64_t slot = chunk_slot(p, s, c);
  const long long wlim = wait_limit(p);

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  float* yq = reinterpret_cast<float*>(sm + CkSmem::YQ);
  float* yk = reinterpret_cast<float*>(sm + CkSmem::YK);
  TIN* xq = reinterpret_cast<TIN*>(sm + CkSmem::XQ);
  TIN* xk = reinterpret_cast<TIN*>(sm + CkSmem::XK);
  TIN* xv = reinterpret_cast<TIN*>(sm + CkSmem::XV);
  float* gbuf = reinterpret_cast<float*>(sm + CkSmem::GT);
  float* rq = gbuf + 256 * kGateSets;
  float* rk = rq + 64;
  float* tf = reinterpret_cast<float*>(sm + CkSmem::TF);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + CkSmem::MBAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + CkSmem::TSLOT);

  if (warp == 0) {
    tc::tmem_alloc(tslot, kCkCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
#pragma unroll
    for (int b = 0; b < 3; ++b) tc::mbar_init(mbar + b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;

  const int y = (int)(row0 + t0 - kWinRows);
  auto stage_v = [&](int g) {
    tc::mbar_expect_tx(mbar + 2, kXRows * D * 2);
    tc::tma_load_2d(xv, &xmap, 2 * p.Hqk * D + (jq * G + g) * D, y, mbar + 2);
  };
  // copies and products in flight, for the drain after a run-out
  bool qk_pending = true, gram_pending = false;
  int v_pending = VIMG ? 0 : -1;   // value head whose rows are in flight (-1: none)
  if (tid == 0) {
    tc::mbar_expect_tx(mbar + 1, 2 * kXRows * D * 2);
    tc::tma_load_2d(xq, &xmap, cq0, y, mbar + 1);
    tc::tma_load_2d(xk, &xmap, ck0, y, mbar + 1);
    if (VIMG) stage_v(0);
  }

  // history rows of a sequence's first chunk: the resumed window, or zeros
  auto fix_history = [&](TIN* dst, int ch0, int t, int nthreads) {
    for (int e = t; e < kWinRows * (D / 2); e += nthreads) {
      const int r = e / (D / 2), c2 = e % (D / 2);
      uint32_t v = 0;
      if (V.win) v = *reinterpret_cast<const uint32_t*>(V.win + (int64_t)r * p.conv_dim + ch0 + 2 * c2);
      *reinterpret_cast<uint32_t*>(dst + r * D + 2 * c2) = v;
    }
  };
  // (image mode) v conv of a value head with taps wv (v_taps): channel `row`,
  // rows [16 qtr, +16) -> tensor memory (rows i and i + 8 as one packed pair)
  auto v_taps = [&](int h) { return ldg_f4_fresh(p.conv_w + (int64_t)(2 * p.Hqk * D + h * D + row) * kConvK); };
  auto v_conv = [&](const float4 wv, int qtr) {
    const int tb = 16 * qtr;
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
    tc::tmem_st16(tbase + tlane + kCkV + 16 * qtr, vr);
    tc::tmem_st_wait();
  };
  bool ok = true;
  // ---------------------------------------------------------------- (A) q / k
  if (worker) {
    // the conv taps of this thread's q | k channel pair (and of its first
    // head's v channel), requested before the rows' wait (their latency
    // hides behind it)
    const int qkp = 2 * (tid & 127);
    const float* wsrc = p.conv_w + (int64_t)(qkp < D ? cq0 + qkp : ck0 + qkp - D) * kConvK;
    const float4 wqa = ldg_f4_fresh(wsrc), wqb = ldg_f4_fresh(wsrc + kConvK);
    const float4 wv0 = VIMG ? v_taps(jq * G) : make_float4(0.f, 0.f, 0.f, 0.f);
    ok = workers_sync_and(work_wait(mbar + 1, 0, wlim) && (!VIMG || work_wait(mbar + 2, 0, wlim)));
    if (ok) { qk_pending = false; v_pending = -1; }
    if (c == 0) {
      fix_history(xq, cq0, tid, kWorkers);
      fix_history(xk, ck0, tid, kWorkers);
      if (VIMG) fix_history(xv, 2 * p.Hqk * D + jq * G * D, tid, kWorkers);
      workers_sync();
    }
    // conv + SiLU of the q | k channel pair qkp, qkp + 1, rows [16 rh, +16)
    {
      const int tb = 16 * (tid >> 7);
      const TIN* xp = (qkp < D ? xq + qkp : xk + qkp - D) + tb * D;
      const f32x2 w0 = pack2(wqa.x, wqb.x), w1 = pack2(wqa.y, wqb.y), w2 = pack2(wqa.z, wqb.z),
                  w3 = pack2(wqa.w, wqb.w);
      f32x2 x[19];
#pragma unroll
      for (int u = 0; u < 19; ++u) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(xp + u * D);
        x[u] = pack2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
      }
      float* yrow = (qkp < D ? yq + qkp : yk + qkp - D) + tb * D;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        f32x2 z = mul2(w0, x[i]);
        z = fma2(w1, x[i + 1], z);
        z = fma2(w2, x[i + 2], z);
        z = fma2(w3, x[i + 3], z);
        const float2 zz = unpack2(z);
        *reinterpret_cast<float2*>(yrow + i * D) = make_float2(silu_fast(zz.x), silu_fast(zz.y));
      }
    }
    if (VIMG) v_conv(wv0, quarter);
    workers_sync();
    if (VIMG) {
      // the first head's v rows are consumed: the next head's rows
      if (tid == 0 && ok && G > 1) stage_v(1);
      if (ok && G > 1) v_pending = 1;
    }
    // L2 norm factors: warp w reduces (row, q | k) pairs w, w+16, ... in a
    // fixed order (the fused kernel's); rows past the end get factor 0
    {
      constexpr int NP = 128 / (kWorkers / 32);
      float ss[NP];
#pragma unroll
      for (int it = 0; it < NP; ++it) {
        const int k = warp + (kWorkers / 32) * it, t = k >> 1, isk = k & 1;
        const float* yr = (isk ? yk : yq) + t * D;
        float a = 0.f;
#pragma unroll
        for (int m = 0; m < D / 32; ++m) {
          const float yv = yr[lane + 32 * m];
          a = fmaf(yv, yv, a);
        }
        ss[it] = a;
      }
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
        const int k = warp + (kWorkers / 32) * (lane >> 2), t = k >> 1, isk = k & 1;
        (isk ? rk : rq)[t] = t < cnt ? (isk ? 1.0f : p.q_scale) / sqrtf(a + p.eps) : 0.f;
      }
    }
    workers_sync();
    // the operand [K^; Q^] (rows 0-63 k^, 64-127 q^)
    {
      constexpr int NKQ = 2048 / kWorkers;
      float4 ya[NKQ], yb[NKQ];
      float fv[NKQ];
#pragma unroll
      for (int it = 0; it < NKQ; ++it) {
        const int i = tid + kWorkers * it, r = i >> 4, c8 = i & 15;
        const int t = r & (C - 1);
        const bool isq = r >= C;
        fv[it] = isq ? rq[t] : rk[t];
        const float4* src = reinterpret_cast<const float4*>((isq ? yq : yk) + t * D + 8 * c8);
        ya[it] = src[0];
        yb[it] = src[1];
      }
#pragma unroll
      for (int it = 0; it < NKQ; ++it) {
        const int i = tid + kWorkers * it, r = i >> 4, c8 = i & 15;
        const float f = fv[it];
        const f32x2 f2 = pack2(f, f);
        const float2 e01 = unpack2(mul2(pack2(ya[it].x, ya[it].y), f2));
        const float2 e23 = unpack2(mul2(pack2(ya[it].z, ya[it].w), f2));
        const float2 e45 = unpack2(mul2(pack2(yb[it].x, yb[it].y), f2));
        const float2 e67 = unpack2(mul2(pack2(yb[it].z, yb[it].w), f2));
        const float e[8] = {e01.x, e01.y, e23.x, e23.y, e45.x, e45.y, e67.x, e67.y};
        const uint32_t off = tc::sw128_offset(r, 8 * c8, 128);
        tc::store_split8(sm + CkSmem::KQ + off, sm + CkSmem::KQ_LO + off, e);
      }
    }
    tc::fence_async_smem();
  }
  if (!worker) {
    // the q, k and first v rows of the CTA one round of SMs ahead (it starts
    // about when this one ends) into L2, so that its first wait is short
    if (tid == kMma) {
      uint32_t nsm;
      asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
      const int64_t gx = gridDim.x, gy = gridDim.y;
      const int64_t nxt = (int64_t)blockIdx.x + gx * ((int64_t)blockIdx.y + gy * blockIdx.z) + nsm;
      const int64_t s2 = nxt / (gx * gy);
      if (s2 < p.num_seqs) {
        const int j2 = (int)(nxt % gx);
        const int64_t y2 = (int64_t)p.cu_seqlens[s2] + (c0 + (nxt / gx) % gy) * C - kWinRows;
        if (y2 >= 0 && y2 + kXRows <= p.total_rows) {
          tc::tma_prefetch_2d(&xmap, j2 * D, (int)y2);
          tc::tma_prefetch_2d(&xmap, p.Hqk * D + j2 * D, (int)y2);
          tc::tma_prefetch_2d(&xmap, 2 * p.Hqk * D + j2 * G * D, (int)y2);
        }
      }
    }
    // the value heads' gate sets (up to four) while the workers convolve
    for (int g = 0; g < G && g < kGateSets; ++g) chunk_gates(V, t0, n, jq * G + g, lane, gbuf + 256 * g);
    tc::fence_async_smem();
  }
  ok = cta_sync_ok(ok);
  if (ok && tid == kMma) {
    // [K^ K^T; Q^ K^T] (M 128, N 64, K 128), and [K^; Q^] for the chain
    tc::mma3_sw128<D / 16, 16384, 16384>(tbase + kCkGram, sbase + CkSmem::KQ, sbase + CkSmem::KQ_LO,
                                         sbase + CkSmem::KQ, sbase + CkSmem::KQ_LO, tc::idesc_bf16_f32(128, 64),
                                         false);
    tc::mma_commit(mbar + 0);
    tc::bulk_store(ws.kq + (slot * p.Hqk + jq) * (int64_t)kImgKQ, sm + CkSmem::KQ, kImgKQ);
    tc::bulk_commit();
  }
  if (ok) gram_pending = true;

  // ---------------------------------------------------------- (B) value heads
  const bool kgrp = tid < 256;
  // A^T (lanes 0-63: k^_i.k^_j) and P (lanes 64-127: q^_i.k^_j) of one value
  // head, columns j in [16 cb, +16) of this warp's Gram lanes, into A^T / A /
  // P set `set` (the second set: conv mode only)
  auto form_ap = [&](int cb, const float* Gs, int set) {
    float* atp = reinterpret_cast<float*>(sm + (set ? CkSmem::AT1 : CkSmem::AT));
    float* amp = reinterpret_cast<float*>(sm + (set ? CkSmem::AM1 : CkSmem::AM));
    const uint32_t pb = set ? CkSmem::PB1 : CkSmem::PB;
    const float* bv = Gs + 192;
    const int q4 = warp & 3;
    const int ir = (q4 & 1) * 32 + lane;
    float ap[16];
    tc::tmem_ld16(tbase + tlane + kCkGram + 16 * cb, ap);
    const float Gi = Gs[ir];
    const float bi = q4 < 2 ? bv[ir] : 1.0f;
    const int lim = q4 < 2 ? ir : ir + 1;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int j = 16 * cb + e;
      const float m = j < lim ? bi : 0.f;
      ap[e] = m * __expf(fminf(Gi - Gs[j], 0.f)) * ap[e];
    }
    if (q4 < 2) {
#pragma unroll
      for (int e = 0; e < 16; ++e) atp[(16 * cb + e) * C + ir] = ap[e];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        *reinterpret_cast<float4*>(amp + am_index(ir, 16 * cb + 4 * c4)) =
            make_float4(ap[4 * c4], ap[4 * c4 + 1], ap[4 * c4 + 2], ap[4 * c4 + 3]);
    } else {
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {
        const uint32_t off = tc::sw128_offset(ir, 16 * cb + 8 * c8, 64);
        tc::store_split8(sm + pb + off, sm + pb + 8192 + off, ap + 8 * c8);
      }
    }
  };
  // K^T diag(dec) (row = k channel) into the KT region: the fused kernel's
  // elements and expression, four of its eight-row groups per K-group thread
  auto form_kt = [&](const float* dec) {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int i = tid + 256 * it, k = i & 127, j8 = i >> 7;
      float kt[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = 8 * j8 + u;
        kt[u] = (yk[j * D + k] * rk[j]) * dec[j];
      }
      const uint32_t off = tc::sw128_offset(k, 8 * j8, 128);
      tc::store_split8(sm + CkSmem::KT + off, sm + CkSmem::KT_LO + off, kt);
    }
  };
  // T = (I + A)^{-1} by the T group, then (its region free) T as the B
  // operand (rows i, K = j; zero above the diagonal)
  auto form_t = [&](int set) {
    const float* atp = reinterpret_cast<const float*>(sm + (set ? CkSmem::AT1 : CkSmem::AT));
    const float* amp = reinterpret_cast<const float*>(sm + (set ? CkSmem::AM1 : CkSmem::AM));
    tri_inverse64(atp, amp, tf, reinterpret_cast<float*>(sm + CkSmem::DT), reinterpret_cast<float*>(sm + CkSmem::NT),
                  tid - 256);
    named_sync(6, 288);
    for (int e = tid - 256; e < 512; e += 256) {
      const int i = e >> 3, c8 = e & 7;
      const float4 a = *reinterpret_cast<const float4*>(tf + i * C + 8 * c8);
      const float4 b = *reinterpret_cast<const float4*>(tf + i * C + 8 * c8 + 4);
      float v8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (8 * c8 + u > i) v8[u] = 0.f;
      const uint32_t off = tc::sw128_offset(i, 8 * c8, 64);
      tc::store_split8(sm + CkSmem::TB + off, sm + CkSmem::TB_LO + off, v8);
    }
  };
  int g = 0;
  if (!VIMG) {
    // ------------------------------------------------------------ conv mode
    // A and P of head 0 by every worker; then, head by head, the T group
    // inverts head g's A while the K group forms head g's K~ and head g + 1's
    // A and P (into the other A^T / A / P set).  The issuing warp stores P
    // at the head's start, K~ when the K group has formed it, T and the gates
    // at its end.
    for (; ok && g < G; ++g) {
      const int h = jq * G + g;
      const int b = g & 1;
      float* const Gs = gbuf + 256 * (g % kGateSets);
      const int64_t hv = slot * p.Hv + h;
      if (!worker) {
        if (g == 0) {
          __syncwarp();
          named_arrive(3, kThreads);        // (the gates of the first heads were formed during the conv)
          if (tid == kMma) tc::bulk_wait_read();   // [K^; Q^] (T's work region, the second A set) read out
          __syncwarp();
          named_sync(5, kThreads);          // head 0's A and P are formed
        }
        if (tid == kMma) {
          tc::bulk_store(ws.pm + hv * kImgP, sm + (b ? CkSmem::PB1 : CkSmem::PB), kImgP);
          tc::bulk_commit();
          // all but this P: the head before's K~, T and gates, and the P before
          if (g > 0) tc::bulk_wait_read_but<1>();
        }
        __syncwarp();
        named_arrive(6, 288);               // the T image region is free
        if (g > 0) named_arrive(9, 288);    // the K~ region is free
        if (g + 1 < G) {
          if (g + 1 >= kGateSets) {
            // the set was last stored by head g + 1 - kGateSets
            if (tid == kMma) tc::bulk_wait_read();
            __syncwarp();
            chunk_gates(V, t0, n, h + 1, lane, gbuf + 256 * ((g + 1) % kGateSets));
            tc::fence_async_smem();
          }
          __syncwarp();
          named_arrive(8, 288);             // the next head's gates; its P region is free
        }
        named_sync(7, 288);                 // K~ is formed
        if (tid == kMma) {
          tc::bulk_store(ws.k + hv * kImgK, sm + CkSmem::KT, kImgK);
          tc::bulk_commit();
        }
      } else {
        if (g == 0) {
          named_sync(3, kThreads);
          mma_wait(mbar + 0, 0, ok, wlim);
          if (ok) gram_pending = false;
          form_ap(quarter, Gs, 0);
          tc::fence_async_smem();
          named_sync(5, kThreads);
        }
        if (!kgrp) {
          form_t(b);
        } else {
          if (g > 0) named_sync(9, 288);
          form_kt(Gs + 128);
          tc::fence_async_smem();
          named_arrive(7, 288);
          if (g + 1 < G) {
            named_sync(8, 288);
            const float* Gn = gbuf + 256 * ((g + 1) % kGateSets);
#pragma unroll 1
            for (int cb = quarter; cb < 4; cb += 2) form_ap(cb, Gn, b ^ 1);
          }
        }
        tc::fence_async_smem();
      }
      ok = cta_sync_ok(ok);
      if (!ok) break;
      if (tid == kMma) {
        tc::bulk_store(ws.t + hv * kImgT, sm + CkSmem::TB, kImgT);
        tc::bulk_store(ws.g + hv * (kImgG / 4), Gs, kImgG);
        tc::bulk_commit();
      }
    }
  }
  // ----------------------------------------------------------- image mode
  // After A and P, threads 0-255 (the K group) form K^T diag(dec) and v, then
  // the next head's v conv; threads 256-511 (the T group) form T.  The issuing
  // warp stores each image once it is complete: P after A and P, K~ and v
  // when the K group is done, T and the gates at the head's end, and waits
  // for a store to have left shared memory only before that region is
  // written again.
  for (; VIMG && ok && g < G; ++g) {
    const int h = jq * G + g;
    float* const Gs = gbuf + 256 * (g % kGateSets);
    const int64_t hv = slot * p.Hv + h;
    if (!worker) {
      if (g >= kGateSets) {
        // the set was last stored by head g - kGateSets
        if (tid == kMma) tc::bulk_wait_read();
        __syncwarp();
        chunk_gates(V, t0, n, h, lane, Gs);
        tc::fence_async_smem();
      } else if (g > 0 && tid == kMma) {
        tc::bulk_wait_read_but<2>();      // P of the head before
      }
      __syncwarp();
      named_arrive(3, kThreads);          // the gates; the P region is free
      // [K^; Q^] (T's work region and v's image) or the head before's K~ and
      // v have been read out
      if (tid == kMma) {
        if (g == 0) tc::bulk_wait_read();
        else tc::bulk_wait_read_but<1>();
      }
      __syncwarp();
      named_sync(5, kThreads);            // A and P are formed
      if (tid == kMma) {
        tc::bulk_store(ws.pm + hv * kImgP, sm + CkSmem::PB, kImgP);
        tc::bulk_commit();
        if (g > 0) tc::bulk_wait_read_but<1>();   // T and the gates of the head before
      }
      __syncwarp();
      named_arrive(6, 288);               // the T image region is free
      named_sync(7, 288);                 // K~ and v are formed
      if (tid == kMma) {
        tc::bulk_store(ws.k + hv * kImgK, sm + CkSmem::KT, kImgK);
        tc::bulk_store(ws.v + hv * (kImgV / 4), sm + CkSmem::VS, kImgV);
        tc::bulk_commit();
      }
    } else {
      named_sync(3, kThreads);
      if (g == 0) {
        mma_wait(mbar + 0, 0, ok, wlim);
        if (ok) gram_pending = false;
      }
      form_ap(quarter, Gs, 0);
      tc::fence_async_smem();
      named_sync(5, kThreads);
      if (!kgrp) {
        form_t(0);
      } else {
        // the next head's conv taps (their load's latency hides behind K~ and v)
        const float4 wv = g + 1 < G ? v_taps(h + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        form_kt(Gs + 128);
        // v of channel `row`, rows [32 (tid >> 7), +32) -> its image ([i][r]:
        // a warp's stores of one row are 128 contiguous bytes), which leaves
        // by a bulk copy (per-thread global stores of every CTA at once would
        // back up the load / store pipe that shared-memory loads also use)
        float* vs = reinterpret_cast<float*>(sm + CkSmem::VS) + 32 * (tid >> 7) * D + row;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[16];
          tc::tmem_ld16(tbase + tlane + kCkV + 32 * (tid >> 7) + 16 * hh, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) vs[(16 * hh + e) * D] = v[e];
        }
        tc::fence_async_smem();
        named_arrive(7, 288);
        if (g + 1 < G) {
          // the next head's v rows (requested after this head's v conv) -> its v conv
          ok = kgrp_sync_and(work_wait(mbar + 2, (uint32_t)((g + 1) & 1), wlim) && ok);
          if (ok) v_pending = -1;
          if (c == 0) {
            fix_history(xv, 2 * p.Hqk * D + (h + 1) * D, tid, 256);
            kgrp_sync();
          }
          v_conv(wv, 2 * (tid >> 7));
          v_conv(wv, 2 * (tid >> 7) + 1);
          kgrp_sync();
          if (tid == 0 && ok && g + 2 < G) stage_v(g + 2);
          if (ok && g + 2 < G) v_pending = g + 2;
        }
      }
      tc::fence_async_smem();
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == kMma) {
      tc::bulk_store(ws.t + hv * kImgT, sm + CkSmem::TB, kImgT);
      tc::bulk_store(ws.g + hv * (kImgG / 4), Gs, kImgG);
      tc::bulk_commit();
    }
  }

  if (!ok) {
    // a wait ran out: report it, let the copies and products in flight finish
    // (default bound), release the tensor memory
    if (tid == 0) atomicExch(p.err, GDN_ERR_TIMEOUT);
    if (worker) {
      // (the K group alone tracks the v rows once the value heads start)
      if (qk_pending) tc::mbar_wait_bounded(mbar + 1, 0, kWaitDefault);
      if ((kgrp || g == 0) && v_pending >= 0) tc::mbar_wait_bounded(mbar + 2, (uint32_t)(v_pending & 1), kWaitDefault);
      if (gram_pending) tc::mbar_wait_bounded(mbar + 0, 0, kWaitDefault);
    }
  }
  // the images' shared memory has been read out (their global writes finish
  // on their own; the chain kernel reads them only after this launch ends)
  if (tid == kMma) tc::bulk_wait_read();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, kCkCols);
}

// ============================================================================
// Chain kernel: grid (Hv, pieces), one CTA per (value head, (level, sequence))
// ============================================================================
// Per chunk c: (1) the state after chunk c - 1 (checkpointed at a block
// boundary) split into tensor memory as the A operand, gam_C S0 back; then
// S0 [K^; Q^]^T.  (2) The outputs of chunk c - 1; R into the tensor-memory
// operand; then U^T = R T^T.  (3) U into that operand; then the state update
// S += U^T (K^T diag(dec))^T and U^T P^T.  Every image of chunk c + 1 is
// requested as soon as the reader of chunk c's (or c - 1's, for the two
// buffers of T, P and the gates) is done.
template <bool VIMG, bool POST>
__global__ void __launch_bounds__(kThreads, 1)
    tc_chain_kernel(const ScanParams p, const __grid_constant__ CUtensorMap xmap,
                    const __grid_constant__ CUtensorMap omap, int tma_out, const ChunkWs ws, const PieceMap pm,
                    int64_t max_chunks) {
  // xmap: the pre-conv rows ([rows][x_ld], 128 x 67 boxes), of which the
  // chain takes its head's v channels; omap: the outputs as [rows][Hv * dv]
  // in 64-row tiles (tma_out), or for the packed core the z columns of the
  // packed rows (128 x 64 boxes), loaded a chunk ahead into the tile's shared
  // memory
  using TOUT = __nv_bfloat16;
  constexpr int D = kD, C = kC;
  const int h = blockIdx.x;
  int s = pm.s0 + (int)blockIdx.y, level = pm.level0;
  if (s >= pm.nseqs) {
    s -= pm.nseqs;
    ++level;
  }
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool worker = tid < kWorkers;
  const int row = tid & 127;
  const int quarter = (tid >> 7) & 3;
  const uint32_t tlane = (uint32_t)((warp & 3) * 32) << 16;

  TokenView<__nv_bfloat16> V;
  int64_t start, n_log;
  int32_t init, final_page;
  const bool report = (h == 0 && tid == 0);
  if (!make_view<__nv_bfloat16, kPrefill>(p, s, V, start, init, final_page, n_log, report)) return;
  const int64_t n = V.n;
  const int64_t nch = (n + C - 1) / C;
  if (nch > max_chunks) {   // the call's max_seq_len was below this sequence's length
    if (report) set_error(p.err, GDN_ERR_INVALID_ARG);
    return;
  }
  const int64_t cb = (int64_t)level * pm.piece;
  if (level > 0 && cb >= nch) return;
  const int64_t ce = level == pm.last_level || cb + pm.piece > nch ? nch : cb + pm.piece;
  const int32_t from = level > 0 ? final_page : init;
  // a wait that ran out in an earlier launch of the call (the chunk kernel or
  // an earlier piece) leaves images or a state that cannot be trusted
  if (__syncthreads_or(tid == 0 && *reinterpret_cast<volatile const int32_t*>(p.err) == GDN_ERR_TIMEOUT))
    return;
  const long long wlim = wait_limit(p);
  const int64_t row0 = p.cu_seqlens[s];
  const int hq = h / (p.Hv / p.Hqk);

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + ChSmem::MBAR);
  int64_t* armed = reinterpret_cast<int64_t*>(sm + ChSmem::ARMED);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + ChSmem::TSLOT);
  TOUT* ot = reinterpret_cast<TOUT*>(sm + ChSmem::OT);

  if (warp == 0) {
    tc::tmem_alloc(tslot, kChCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
#pragma unroll
    for (int k = 0; k < ChSmem::kBars; ++k) {
      tc::mbar_init(mbar + k, 1);
      armed[k] = -1;
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (p.norm_w && tid < D) reinterpret_cast<float*>(sm + ChSmem::NW)[tid] = p.norm_w[tid];
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tS = tbase + tlane + kChS + 32 * quarter;

  // the issuing thread's loads of chunk c's images (each arms its mbarrier)
  // the chunk slots of this sequence start at slot0 (chunk_slot without the
  // global load of cu_seqlens on the issuing thread's path)
  const int64_t slot0 = row0 / kC + s;
  auto hv_of = [&](int64_t c) { return (slot0 + c) * p.Hv + h; };
  auto load_kq = [&](int64_t c) {
    tc::mbar_expect_tx(mbar + ChSmem::kKQ, kImgKQ);
    const uint8_t* src = ws.kq + ((slot0 + c) * p.Hqk + hq) * kImgKQ;
    tc::bulk_load(sm + ChSmem::KQ, src, 32768, mbar + ChSmem::kKQ);
    tc::bulk_load(sm + ChSmem::KQ + 32768, src + 32768, 32768, mbar + ChSmem::kKQ);
    armed[ChSmem::kKQ] = c;
  };
  auto load_kt = [&](int64_t c) {
    tc::mbar_expect_tx(mbar + ChSmem::kKT, kImgK);
    tc::bulk_load(sm + ChSmem::KT, ws.k + hv_of(c) * kImgK, kImgK, mbar + ChSmem::kKT);
    armed[ChSmem::kKT] = c;
  };
  auto load_t = [&](int64_t c) {
    const int b = (int)(c & 1);
    tc::mbar_expect_tx(mbar + ChSmem::kTb + b, kImgT);
    tc::bulk_load(sm + ChSmem::TB + b * kImgT, ws.t + hv_of(c) * kImgT, kImgT, mbar + ChSmem::kTb + b);
    armed[ChSmem::kTb + b] = c;
  };
  auto load_pg = [&](int64_t c) {   // P and the gates
    const int b = (int)(c & 1);
    const int64_t hv = hv_of(c);
    tc::mbar_expect_tx(mbar + ChSmem::kPG + b, kImgG + kImgP);
    tc::bulk_load(sm + ChSmem::G + b * kImgG, ws.g + hv * (kImgG / 4), kImgG, mbar + ChSmem::kPG + b);
    tc::bulk_load(sm + ChSmem::PB + b * kImgP, ws.pm + hv * kImgP, kImgP, mbar + ChSmem::kPG + b);
    armed[ChSmem::kPG + b] = c;
  };
  // v of chunk c: its image (image mode), or the head's pre-conv v rows of
  // chunk c and the three before it (for the first chunk of a sequence those
  // three are another sequence's or out of range: the conv takes the carried
  // window or zeros instead)
  auto load_v = [&](int64_t c) {
    if (VIMG) {
      tc::mbar_expect_tx(mbar + ChSmem::kVb, kImgV);
      tc::bulk_load(sm + ChSmem::XV, ws.v + hv_of(c) * (kImgV / 4), kImgV, mbar + ChSmem::kVb);
    } else {
      tc::mbar_expect_tx(mbar + ChSmem::kVb, kXRows * D * 2);
      tc::tma_load_2d(sm + ChSmem::XV, &xmap, 2 * p.Hqk * D + h * D, (int)(row0 + c * C - kWinRows),
                      mbar + ChSmem::kVb);
    }
    armed[ChSmem::kVb] = c;
  };
  auto gates_of = [&](int64_t c) { return reinterpret_cast<const float*>(sm + ChSmem::G + (int)(c & 1) * kImgG); };
  // the checkpoint page of a block boundary at absolute position pos (-1: none)
  auto boundary_page = [&](int64_t pos) {
    int32_t page = -1;
    if (pos % p.block_size == 0) {
      const int64_t jb = pos / p.block_size - 1;
      if (jb < p.max_blocks) page = p.block_table[(int64_t)s * p.max_blocks + jb];
      else if (report) set_error(p.err, GDN_ERR_INVALID_ARG);
      if (page >= 0 && !page_ok(p.pool, page)) {
        if (report) set_error(p.err, GDN_ERR_PAGE_RANGE);
        page = -1;
      }
    }
    return page;
  };
  auto full_chunk = [&](int64_t c) { return n - c * C >= C; };
  // outputs of chunk c: o_i = gam_i (S0 q^_i) + (U^T P^T)_i for rows i in
  // [16 quarter, +16), from S0 Q^T kept in registers and U^T P^T in tensor
  // memory; a full chunk into the tile (one TMA store), a partial one by plain stores
  auto outputs = [&](int64_t c, const float (&sq)[16]) {
    const float* gam = gates_of(c) + 64;
    float up[16];
    tc::tmem_ld16(tbase + tlane + kChU + 16 * quarter, up);
    if (tma_out && full_chunk(c)) {
#pragma unroll
      for (int e = 0; e < 16; ++e)
        ot[(16 * quarter + e) * D + row] = from_f32<TOUT>(fmaf(gam[16 * quarter + e], sq[e], up[e]));
    } else {
      const int64_t t0 = c * C;
      const int cnt = (int)(n - t0 < C ? n - t0 : C);
      TOUT* out = reinterpret_cast<TOUT*>(p.o) + ((row0 + t0) * p.Hv + h) * D + row;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int i = 16 * quarter + e;
        if (i < cnt) out[(int64_t)i * p.Hv * D] = from_f32<TOUT>(fmaf(gam[i], sq[e], up[e]));
      }
    }
  };
  // packed core: the outputs of chunk c gated-normalised as the fused kernel
  // does it (a token's 128 outputs meet in shared memory, v's region, free
  // once R or the conv has read it: all 64 tokens in the image mode, 32 at a
  // time in the rows' smaller region; warp w then takes tokens w, w + 16, ...:
  // RMS over dv, the norm scale, the silu(z) gate from the packed row).  Every
  // worker calls it (two or four worker barriers).
  const bool core = p.norm_w != nullptr;
  auto load_z = [&](int64_t c) {
    tc::mbar_expect_tx(mbar + ChSmem::kZ, 16384);
    tc::tma_load_2d(ot, &omap, p.conv_dim + h * D, (int)(row0 + c * C), mbar + ChSmem::kZ);
    armed[ChSmem::kZ] = c;
  };
  // (POST: the packed core's outputs leave fp32, into the workspace, for the
  // gated-norm pass after the chains, core_gate_norm_kernel, which takes a
  // token's 128 values together in the same expression)
  auto outputs_f32 = [&](int64_t c, const float (&sq)[16]) {
    const float* gam = gates_of(c) + 64;
    float up[16];
    tc::tmem_ld16(tbase + tlane + kChU + 16 * quarter, up);
    const int64_t t0 = c * C;
    const int cnt = (int)(n - t0 < C ? n - t0 : C);
    float* out = ws.core_o + ((row0 + t0) * p.Hv + h) * D + row;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int i = 16 * quarter + e;
      if (i < cnt) out[(int64_t)i * p.Hv * D] = fmaf(gam[i], sq[e], up[e]);
    }
  };
  auto outputs_core = [&](int64_t c, const float (&sq)[16], bool& okc) {
    const float* gam = gates_of(c) + 64;
    float up[16];
    tc::tmem_ld16(tbase + tlane + kChU + 16 * quarter, up);
    // the tokens' outputs, all 64 at once (image mode: the 32 KB region) or
    // 32 at a time (the rows' region)
    constexpr int kTok = VIMG ? 64 : 32;
    float* of = reinterpret_cast<float*>(sm + ChSmem::XV);
    okc = work_wait(mbar + ChSmem::kZ, (uint32_t)((c - cb) & 1), wlim) && okc;   // the z rows
    const int64_t t0 = c * C;
    const int cnt = (int)(n - t0 < C ? n - t0 : C);
    const int lane = tid & 31;
    const __nv_bfloat16* zs = ot;
    const float* nw = reinterpret_cast<const float*>(sm + ChSmem::NW);
    TOUT* orow = reinterpret_cast<TOUT*>(p.o) + ((row0 + t0) * p.Hv + h) * D;
#pragma unroll 1
    for (int hf = 0; hf < 64 / kTok; ++hf) {
      workers_sync();   // every worker has read v (R, the conv); the tokens before are done
      if ((16 * quarter) / kTok == hf) {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          of[(16 * quarter - kTok * hf + e) * D + row] = fmaf(gam[16 * quarter + e], sq[e], up[e]);
      }
      workers_sync();
      const int iend = cnt < kTok * hf + kTok ? cnt : kTok * hf + kTok;
      for (int i = kTok * hf + warp; i < iend; i += kWorkers / 32) {
        const float* orw = of + (i - kTok * hf) * D;
        float v[4];
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          v[m] = orw[lane + 32 * m];
          ss = fmaf(v[m], v[m], ss);
        }
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss * (1.0f / D) + p.norm_eps2);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float z = to_f32(zs[i * D + lane + 32 * m]);
          orow[(int64_t)i * p.Hv * D + lane + 32 * m] = from_f32<TOUT>(v[m] * inv * nw[lane + 32 * m] * silu_fast(z));
        }
      }
    }
  };
  // 16 fp32 values (rows [16 quarter, +16) of state row `row`) as bf16 hi / lo
  // pairs into the tensor-memory A operand
  auto split_to_tmem = [&](const float (&a)[16]) {
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) tc::split_pair(a[2 * e], a[2 * e + 1], hi[e], lo[e]);
    tc::tmem_st8(tbase + tlane + kChUH + 8 * quarter, hi);
    tc::tmem_st8(tbase + tlane + kChUL + 8 * quarter, lo);
    tc::tmem_st_wait();
  };

  if (tid == kMma && cb < ce) {
    load_pg(cb);
    load_kq(cb);
    load_v(cb);
    load_t(cb);
    load_kt(cb);
  }
  // the conv taps of this worker's v channel (state row `row`)
  const float* vtaps = p.conv_w + (int64_t)(2 * p.Hqk * D + h * D + row) * kConvK;
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

  float sq[16];             // S0 Q^T of the chunk before, until its outputs
  bool ok = true;
  int64_t c = cb;
  for (; c < ce; ++c) {
    const int b = (int)(c & 1);
    const uint32_t par = (uint32_t)((c - cb) & 1);
    const uint32_t bpar = (uint32_t)(((c - cb) >> 1) & 1);
    if (worker) {
      // ---- (1) the state after chunk c - 1: checkpoint, split into tensor
      // memory (gam_C S0 goes back in step 2, while the first product runs)
      if (c > cb) mma_wait(mbar + ChSmem::kS, par ^ 1u, ok, wlim);
      const int32_t ck = c > cb ? boundary_page(start + c * C) : -1;
      float* ckp = ck >= 0 ? page_state(p.pool, ck) + ((int64_t)h * D + row) * D + 32 * quarter : nullptr;
      float v0[32];
      tc::tmem_ld32(tS, v0);
      if (ckp) {
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          reinterpret_cast<float4*>(ckp)[c4] = make_float4(v0[4 * c4], v0[4 * c4 + 1], v0[4 * c4 + 2], v0[4 * c4 + 3]);
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) tc::split_pair(v0[16 * hh + 2 * e], v0[16 * hh + 2 * e + 1], hi[e], lo[e]);
        tc::tmem_st8(tbase + tlane + kChS0H + 16 * quarter + 8 * hh, hi);
        tc::tmem_st8(tbase + tlane + kChS0L + 16 * quarter + 8 * hh, lo);
      }
      tc::tmem_st_wait();
      if (tid == 0) tc::bulk_wait_read();   // the output tile, before this chunk's step 2 rewrites it
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == kMma) {
      // S0 [K^; Q^]^T (M 128, N 128, K 128) -> [S0 K^T | S0 Q^T]
      ok = work_wait(mbar + ChSmem::kKQ, par, wlim) && ok;
      tc::mma3_ts<D / 16, 16384>(tbase + kChSK, tbase + kChS0H, tbase + kChS0L, sbase + ChSmem::KQ,
                                 sbase + ChSmem::KQ + 32768, tc::idesc_bf16_f32(128, 128), false);
      tc::mma_commit(mbar + ChSmem::kSK);
      armed[ChSmem::kSK] = c;
      // T of the next chunk (its buffer's last reader, R T^T of chunk c - 1, is done)
      if (c + 1 < ce) load_t(c + 1);
    }
    if (worker) {
      // ---- (2) the previous chunk's outputs (its U^T P^T is done); v by the
      // conv, while S0 [K^; Q^]^T runs; then R_i = b_i (v_i - gam_i (S0 k^_i))
      // of state row `row`, rows [16 quarter, +16), into the tensor-memory
      // operand
      const float4 wv = VIMG ? make_float4(0.f, 0.f, 0.f, 0.f) : ldg_f4_fresh(vtaps);
      ok = work_wait(mbar + ChSmem::kPG + b, bpar, wlim) && ok;
      if (c > cb && (POST || !core)) {
        mma_wait(mbar + ChSmem::kUP, par ^ 1u, ok, wlim);
        if constexpr (POST) {
          outputs_f32(c - 1, sq);
        } else {
          outputs(c - 1, sq);
          tc::fence_async_smem();
        }
      }
      ok = work_wait(mbar + ChSmem::kVb, par, wlim) && ok;
      const float* gs = gates_of(c);
      const float* gam = gs + 64;
      const float* bv = gs + 192;
      const int i0 = 16 * quarter;
      // v of channel `row`, rows [16 quarter, +16): from its image, or the
      // conv + SiLU of the pre-conv rows in the chunk kernel's expression
      // (rows i and i + 8 as one packed pair), while S0 [K^; Q^]^T runs
      float vv[16];
      if (VIMG) {
        const float* vs = reinterpret_cast<const float*>(sm + ChSmem::XV) + i0 * D + row;
#pragma unroll
        for (int e = 0; e < 16; ++e) vv[e] = vs[e * D];
      } else {
        const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(sm + ChSmem::XV) + i0 * D + row;
        // row u of the 19 this thread convolves (a sequence's first three:
        // the carried window, or zeros); a sliding window of four rows for
        // each of the pair's outputs keeps few registers live
        const bool hist = c == 0 && quarter == 0;
        const __nv_bfloat16* wr = hist && V.win ? V.win + 2 * p.Hqk * D + h * D + row : nullptr;
        auto xrow = [&](int u) -> float {
          if (u < kWinRows && hist) return wr ? to_f32(wr[(int64_t)u * p.conv_dim]) : 0.f;
          return to_f32(xv[u * D]);
        };
        const f32x2 w0 = pack2(wv.x, wv.x), w1 = pack2(wv.y, wv.y), w2 = pack2(wv.z, wv.z), w3 = pack2(wv.w, wv.w);
        float a0 = xrow(0), a1 = xrow(1), a2 = xrow(2), b0 = xrow(8), b1 = xrow(9), b2 = xrow(10);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float a3 = xrow(i + 3), b3 = xrow(i + 11);
          f32x2 z = mul2(w0, pack2(a0, b0));
          z = fma2(w1, pack2(a1, b1), z);
          z = fma2(w2, pack2(a2, b2), z);
          z = fma2(w3, pack2(a3, b3), z);
          const float2 zz = unpack2(z);
          vv[i] = silu_fast(zz.x);
          vv[i + 8] = silu_fast(zz.y);
          a0 = a1; a1 = a2; a2 = a3;
          b0 = b1; b1 = b2; b2 = b3;
        }
      }
      mma_wait(mbar + ChSmem::kSK, par, ok, wlim);
      float a[16];
      if (core && !POST) tc::tmem_ld16(tbase + tlane + kChSK + i0, a);
      else tc::tmem_ld16x2(tbase + tlane + kChSK + i0, tbase + tlane + kChSQ + i0, a, sq);
#pragma unroll
      for (int e = 0; e < 16; ++e) a[e] = bv[i0 + e] * fmaf(-gam[i0 + e], a[e], vv[e]);
      split_to_tmem(a);
      if (core && !POST) {
        // the previous chunk's outputs after R (they use v's region), with its
        // S0 Q^T still in registers; then this chunk's
        if (c > cb) {
          mma_wait(mbar + ChSmem::kUP, par ^ 1u, ok, wlim);
          outputs_core(c - 1, sq, ok);
        }
        tc::tmem_ld16(tbase + tlane + kChSQ + i0, sq);
      }
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == kMma) {
      // U^T = R T^T (M 128, N 64, K 64)
      ok = work_wait(mbar + ChSmem::kTb + b, bpar, wlim) && ok;
      tc::mma3_ts<C / 16, 0>(tbase + kChU, tbase + kChUH, tbase + kChUL, sbase + ChSmem::TB + b * kImgT,
                             sbase + ChSmem::TB + b * kImgT + 8192, tc::idesc_bf16_f32(128, 64), false);
      tc::mma_commit(mbar + ChSmem::kU);
      armed[ChSmem::kU] = c;
    }
    if (tid == 0) {
      // (off the issuing thread's path, which goes on to R T^T) the previous
      // chunk's output tile; the next chunk's gates and P (their buffer's last
      // readers, the outputs and U^T P^T of chunk c - 1, are done), [K^; Q^]
      // (S0 [K^; Q^]^T is done) and the v rows (the conv has read them; the
      // packed core's outputs have left their region)
      if (c > cb && tma_out && full_chunk(c - 1)) {
        tc::tma_store_2d(&omap, h * D, (int)(row0 + (c - 1) * C), ot);
        tc::bulk_commit();
      }
      // packed core: this chunk's z rows (the tile region is free: the
      // previous chunk's outputs are done)
      if (core && !POST) load_z(c);
      if (c + 1 < ce) {
        load_pg(c + 1);
        load_kq(c + 1);
        load_v(c + 1);
      }
    }
    if (worker) {
      // ---- (3) gam_C S0 into the state's columns, which the state update
      // accumulates onto (S0 [K^; Q^]^T read only the hi / lo split), while
      // R T^T runs; then U (rows r, K = i) into the operand of the state
      // update and U^T P^T
      {
        const float gC = gates_of(c)[64 + C - 1];
        float v0[32];
        tc::tmem_ld32(tS, v0);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 gg = unpack2(mul2(pack2(v0[e], v0[e + 1]), pack2(gC, gC)));
          v0[e] = gg.x;
          v0[e + 1] = gg.y;
        }
        tc::tmem_st32(tS, v0);
        tc::tmem_st_wait();
      }
      mma_wait(mbar + ChSmem::kU, par, ok, wlim);
      float u[16];
      tc::tmem_ld16(tbase + tlane + kChU + 16 * quarter, u);
      split_to_tmem(u);
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == kMma) {
      // S += U^T (K^T diag(dec))^T (M 128, N 128, K 64) first, then U^T P^T (M 128, N 64, K 64)
      ok = work_wait(mbar + ChSmem::kKT, par, wlim) && ok;
      tc::mma3_ts<C / 16, 0>(tbase + kChS, tbase + kChUH, tbase + kChUL, sbase + ChSmem::KT,
                             sbase + ChSmem::KT + 16384, tc::idesc_bf16_f32(128, 128), true);
      tc::mma_commit(mbar + ChSmem::kS);
      ok = work_wait(mbar + ChSmem::kPG + b, bpar, wlim) && ok;
      tc::mma3_ts<C / 16, 0>(tbase + kChU, tbase + kChUH, tbase + kChUL, sbase + ChSmem::PB + b * kImgP,
                             sbase + ChSmem::PB + b * kImgP + 8192, tc::idesc_bf16_f32(128, 64), false);
      tc::mma_commit(mbar + ChSmem::kUP);
      armed[ChSmem::kS] = armed[ChSmem::kUP] = c;
      // K~ of the next chunk once the state update has read this chunk's
      if (c + 1 < ce) {
        if (work_wait(mbar + ChSmem::kS, par, wlim)) load_kt(c + 1);
        else ok = false;
      }
    }
  }

  // the last chunk's outputs (every thread takes these barriers: `ok` may
  // differ between threads until a barrier agrees on it)
  if (c > cb) {
    if (ok && worker) {   // (every worker: `ok` agreed at the loop's last barrier)
      mma_wait(mbar + ChSmem::kS, (uint32_t)((c - 1 - cb) & 1), ok, wlim);
      mma_wait(mbar + ChSmem::kUP, (uint32_t)((c - 1 - cb) & 1), ok, wlim);
      if (!core) {
        // the tile's previous store (issued in the last chunk's step 2) has
        // been read out before the last outputs rewrite it
        if (tid == 0) tc::bulk_wait_read();
        workers_sync();
      }
      if (core) {
        if constexpr (POST) outputs_f32(c - 1, sq);
        else outputs_core(c - 1, sq, ok);
      } else {
        outputs(c - 1, sq);
      }
      tc::fence_async_smem();
    }
    ok = cta_sync_ok(ok);
    if (ok && tid == 0 && tma_out && full_chunk(c - 1)) {
      tc::tma_store_2d(&omap, h * D, (int)(row0 + (c - 1) * C), ot);
      tc::bulk_commit();
    }
  }
  ok = cta_sync_ok(ok);
  if (ok) {
    if (worker) {
      // final state (and the checkpoint of a boundary at the piece's end)
      const int32_t ck = ce > cb ? boundary_page(start + (ce - 1) * C + (n - (ce - 1) * C < C ? n - (ce - 1) * C : C))
                                 : -1;
      float* dst = page_state(p.pool, final_page) + ((int64_t)h * D + row) * D + 32 * quarter;
      float* ckp = ck >= 0 ? page_state(p.pool, ck) + ((int64_t)h * D + row) * D + 32 * quarter : nullptr;
      float v0[32];
      tc::tmem_ld32(tS, v0);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 f0 = make_float4(v0[4 * c4], v0[4 * c4 + 1], v0[4 * c4 + 2], v0[4 * c4 + 3]);
        reinterpret_cast<float4*>(dst)[c4] = f0;
        if (ckp) reinterpret_cast<float4*>(ckp)[c4] = f0;
      }
    }
  } else {
    // a wait ran out: report it, give every copy and product armed so far one
    // more wait with the default bound (the last phase each mbarrier was armed
    // for; none is armed past it), release the tensor memory
    if (tid == 0) atomicExch(p.err, GDN_ERR_TIMEOUT);
    if (worker) {
#pragma unroll 1
      for (int k = 0; k < ChSmem::kBars; ++k) {
        const int64_t a = armed[k];
        if (a < cb) continue;
        const uint32_t ph = (uint32_t)((ChSmem::two_buffers(k) ? (a - cb) >> 1 : a - cb) & 1);
        tc::mbar_wait_bounded(mbar + k, ph, kWaitDefault);
      }
    }
  }
  if (tid == 0) tc::bulk_wait_all();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, kChCols);
}

// ============================================================================
// Packed core, overlapped levels: the gated RMS norm of the chain's fp32
// outputs.  One warp per (row, value head): lane l holds channels l, l + 32,
// l + 64, l + 96; the fused kernel's expression in its order (the sum of
// squares over the four, then the warp's butterfly; o * inv * w * silu(z)),
// so the paths give the same bits.  Memory-bound: 512 B of outputs and 256 B
// of z in, 256 B out.
// ============================================================================
__global__ void __launch_bounds__(256) core_gate_norm_kernel(const ScanParams p, const float* __restrict__ of) {
  using TOUT = __nv_bfloat16;
  constexpr int D = kD;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * 8;
  const int64_t total = p.total_rows * p.Hv;
  float nw[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) nw[m] = p.norm_w[lane + 32 * m];
  for (int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); w < total; w += nwarps) {
    const int64_t t = w / p.Hv;
    const int h = (int)(w - t * p.Hv);
    const float* orw = of + w * D;
    float v[4];
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      v[m] = orw[lane + 32 * m];
      ss = fmaf(v[m], v[m], ss);
    }
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss * (1.0f / D) + p.norm_eps2);
    const __nv_bfloat16* zrow = reinterpret_cast<const __nv_bfloat16*>(p.x) + t * p.x_ld + p.conv_dim + h * D;
    TOUT* orow = reinterpret_cast<TOUT*>(p.o) + w * D;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float z = to_f32(zrow[lane + 32 * m]);
      orow[lane + 32 * m] = from_f32<TOUT>(v[m] * inv * nw[m] * silu_fast(z));
    }
  }
}

// ============================================================================
// Host side
// ============================================================================
size_t tc_chain_workspace_bytes(int Hqk, int Hv, int32_t num_seqs, int64_t total_tokens, bool core) {
  const int64_t slots = total_tokens / kC + num_seqs + 1;
  const int64_t per_v = (int64_t)kImgT + kImgP + kImgK + kImgG + kImgV;
  const int64_t per_q = (int64_t)kImgKQ;
  const int64_t outs = core ? total_tokens * Hv * kD * (int64_t)sizeof(float) : 0;
  return (size_t)(slots * (Hv * per_v + Hqk * per_q) + outs) + 1024;
}

namespace {
ChunkWs bind_chunk_ws(void* ws, int Hqk, int Hv, int32_t num_seqs, int64_t total_tokens, bool core) {
  ChunkWs w;
  w.slots = total_tokens / kC + num_seqs + 1;
  uint8_t* b = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws) + 1023) & ~uintptr_t(1023));
  auto take = [&](int64_t bytes) {
    uint8_t* r = b;
    b += bytes;
    return r;
  };
  w.kq = take(w.slots * Hqk * (int64_t)kImgKQ);
  w.t = take(w.slots * Hv * (int64_t)kImgT);
  w.pm = take(w.slots * Hv * (int64_t)kImgP);
  w.k = take(w.slots * Hv * (int64_t)kImgK);
  w.v = reinterpret_cast<float*>(take(w.slots * Hv * (int64_t)kImgV));
  w.g = reinterpret_cast<float*>(take(w.slots * Hv * (int64_t)kImgG));
  w.core_o = core ? reinterpret_cast<float*>(take(total_tokens * Hv * kD * (int64_t)sizeof(float))) : nullptr;
  return w;
}
}  // namespace

// The chain kernel's per-chunk work is small beside a launch's fixed costs
// (state in and out, the first images' load, the slowest CTA, the gap between
// launches), so the pieces are longer than the fused kernel's: a launch
// counts as five chunk times.
constexpr double kChainLaunchCost = 5.0;
// Overlapped levels: an even number of chunks, at least 16, at most 64
// levels a call.
constexpr int64_t kSegMin = 16, kSegLevels = 64;

// A model of the paths in units of the fused kernel's chunk time (one chunk
// of one chain, ~13.7 us on a GB300), fitted to 17 measured calls of the
// 27B-shaped layer (1 to 64 sequences of 512 to 8,192 tokens, one of 65,536
// and of 229,376; within 6 % of each).  The fused kernel: each launch runs
// its chains a chunk at a time, ~3 for a launch and the window pass.  A chunk
// CTA costs ~0.4 + 0.4 G of one SM (G value heads a qk head: 21.9 us at
// G = 3), in whole waves over the SMs; a chain chunk ~0.32 (4.4 us), a chain
// launch ~1.6 more (the state in and out, the first images), and the call
// ~3 (its first launch and the window pass).
// Run one after the other, the two kernels take the chunk kernel's waves,
// then the chain launches.  Overlapped (one round of chains), the first
// level's chunk waves, then the longer of the chains' path and all the SM
// time spread over every SM, plus the restart of each level.
namespace {
constexpr double kChainChunk = 0.32, kChainLaunch = 1.6, kTwoFixed = 3.0, kFusedFixed = 3.0;

double chunk_cta_cost(int Hqk, int Hv) { return 0.4 + 0.4 * (double)Hv / Hqk; }

double waves(double ctas, int sms) { return std::ceil(ctas / sms); }

double chain_launches_cost(const PrefillSchedule& sc, int64_t maxc, int sms, double chunk, double launch) {
  if (sc.levels <= 1) return waves((double)sc.nchains, sms) * (double)maxc * chunk + launch;
  return (double)sc.launches * ((double)sc.piece * chunk + launch);
}

double two_kernel_cost(int Hqk, int Hv, int num_seqs, int64_t maxc, int sms, const PrefillSchedule& sc) {
  const double cta = chunk_cta_cost(Hqk, Hv);
  const double ctas = (double)num_seqs * maxc * Hqk;
  if (sc.chunk_launches <= 1)
    return waves(ctas, sms) * cta + kTwoFixed + chain_launches_cost(sc, maxc, sms, kChainChunk, kChainLaunch);
  const double all_sm = (ctas * cta + (double)sc.nchains * maxc * kChainChunk) / sms;
  const double path = (double)maxc * kChainChunk;
  const double first = waves((double)num_seqs * sc.piece * Hqk, sms) * cta;
  return first + (path > all_sm ? path : all_sm) + kChainLaunch * (double)sc.levels + kTwoFixed;
}
}  // namespace

PrefillSchedule tc_chain_schedule(int Hqk, int Hv, int num_seqs, int64_t max_len, int sms) {
  PrefillSchedule sc = tc_prefill_schedule_cost(Hv, num_seqs, max_len, sms, kChainLaunchCost);
  sc.chunk_launches = sc.nchains > 0 ? 1 : 0;
  const int64_t maxc = max_len > 0 ? (max_len + kC - 1) / kC : 0;
  if (sms <= 0 || Hqk <= 0 || sc.nchains <= 0 || sc.nchains > sms || maxc < 2 * kSegMin) return sc;
  // every chain has an SM of its own: the chains leave sms - nchains SMs to
  // the chunk kernel, which produces the next level's images meanwhile
  PrefillSchedule best = sc;
  double best_cost = two_kernel_cost(Hqk, Hv, num_seqs, maxc, sms, sc);
  const int64_t at_least = (maxc + kSegLevels - 1) / kSegLevels;
  for (int64_t P = at_least > kSegMin ? at_least + (at_least & 1) : kSegMin; 2 * P <= maxc; P += 2) {
    PrefillSchedule ov;
    ov.nchains = sc.nchains;
    ov.piece = P;
    ov.levels = (maxc + P - 1) / P;
    ov.width = sc.nchains;
    ov.launches = ov.levels;
    ov.chunk_launches = ov.levels;
    const double cost = two_kernel_cost(Hqk, Hv, num_seqs, maxc, sms, ov);
    if (cost < best_cost) {
      best_cost = cost;
      best = ov;
    }
  }
  return best;
}

bool tc_prefill_two_kernels_faster(int Hqk, int Hv, int num_seqs, int64_t max_len, int sms) {
  if (sms <= 0 || num_seqs <= 0 || max_len <= 0 || Hqk <= 0) return false;
  const int64_t maxc = (max_len + kC - 1) / kC;
  const PrefillSchedule fs = tc_prefill_schedule(Hv, num_seqs, max_len, sms);
  const double fused = chain_launches_cost(fs, maxc, sms, 1.0, kFusedFixed);
  const PrefillSchedule sc = tc_chain_schedule(Hqk, Hv, num_seqs, max_len, sms);
  return two_kernel_cost(Hqk, Hv, num_seqs, maxc, sms, sc) < 0.95 * fused;
}

namespace {

// The second stream of the overlapped levels (highest priority, so a level's
// chain CTAs take SMs before the chunk kernel's next launch) and the events
// of its fork and join, one set per device, made on first use.  The mutex
// keeps one call's enqueue of the fork, the levels and the join together.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t ready = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

// The stream of the current device, or nullptr when there is none to use:
// it does not exist yet and the caller's stream is capturing a graph (so
// that no stream or event is created inside a capture), the device index is
// past the table, or making it failed.  The call then runs its levels one
// after the other on the caller's stream (the same bits).
SideStream* side_stream(cudaStream_t caller) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream& ss = g_side[dev];
  if (!ss.stream) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(caller, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return nullptr;
    int least = 0, greatest = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e != cudaSuccess) return nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t r = nullptr, j = nullptr;
    e = cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, greatest);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&j, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      if (j) cudaEventDestroy(j);
      if (r) cudaEventDestroy(r);
      if (st) cudaStreamDestroy(st);
      return nullptr;
    }
    ss.stream = st;
    ss.ready = r;
    ss.join = j;
  }
  return &ss;
}

}  // namespace

cudaError_t launch_tc_prefill2(const ScanParams& p, void* workspace, int64_t max_len, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  if ((int64_t)p.Hv * p.num_seqs > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
  const ChunkWs ws = bind_chunk_ws(workspace, p.Hqk, p.Hv, p.num_seqs, p.total_rows, p.norm_w != nullptr);
  const int64_t maxc = max_len > 0 ? (max_len + kC - 1) / kC : 0;
  if (maxc > 65535) return cudaErrorInvalidValue;
  auto encode = tensor_map_encoder();
  if (p.total_rows > 0 && !encode) return cudaErrorNotSupported;
  const PrefillSchedule sc = tc_chain_schedule(p.Hqk, p.Hv, p.num_seqs, max_len, tc_prefill_sm_count());
  // With overlapped levels the chain is the call's critical path: the chunk
  // kernel convolves v and writes its image.  Otherwise the chain convolves v
  // from the rows itself (same arithmetic, same bits), which takes the
  // chunk kernel's largest task and 64 KB a chunk and head of image traffic
  // off the call.
  const bool vimg = sc.chunk_launches > 1;
  auto chunk_k = vimg ? tc_chunk_kernel<true> : tc_chunk_kernel<false>;
  // the packed core with overlapped levels: the gated norm in a pass of its
  // own after the chains, off the chain's critical path (the norm in the
  // chain would cost a chunk ~2.8 us)
  const bool post = vimg && p.norm_w != nullptr;
  auto chain_k = vimg ? (post ? tc_chain_kernel<true, true> : tc_chain_kernel<true, false>)
                      : tc_chain_kernel<false, false>;
  CUtensorMap xmap;
  memset(&xmap, 0, sizeof(xmap));
  const bool chunks = maxc > 0 && p.total_rows > 0;
  if (chunks) {
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {(cuuint64_t)p.x_ld, (cuuint64_t)p.total_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)p.x_ld * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kXRows};
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chunk_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CkSmem::ALLOC);
    if (e != cudaSuccess) return e;
  }
  // the chunk kernel over chunks [c0, c0 + cnt) of every sequence
  auto chunk_launch = [&](int64_t c0, int64_t cnt, cudaStream_t s) {
    if (!chunks || cnt <= 0) return cudaSuccess;
    chunk_k<<<dim3(p.Hqk, (unsigned)cnt, p.num_seqs), kThreads, CkSmem::ALLOC, s>>>(p, xmap, ws, c0);
    return cudaGetLastError();
  };
  // o as [rows][Hv * dv] bf16; a box is one head's 128 channels x 64 rows
  // (the chain's full chunks go out as one TMA store when o is 16-byte aligned)
  CUtensorMap omap;
  memset(&omap, 0, sizeof(omap));
  int tma_out = 0;
  if (p.total_rows > 0 && p.norm_w) {
    // packed core: the z columns of the rows, 128 x 64 boxes
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {(cuuint64_t)p.x_ld, (cuuint64_t)p.total_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)p.x_ld * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kC};
    if (encode(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else if (p.total_rows > 0 && (reinterpret_cast<uintptr_t>(p.o) & 15) == 0) {
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {(cuuint64_t)p.Hv * kD, (cuuint64_t)p.total_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)p.Hv * kD * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kC};
    if (encode(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.o, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      tma_out = 1;
  }
  cudaError_t e = cudaFuncSetAttribute(chain_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ChSmem::ALLOC);
  if (e != cudaSuccess) return e;
  PieceMap pm;
  pm.nseqs = p.num_seqs;
  pm.piece = (int32_t)sc.piece;
  pm.last_level = (int32_t)(sc.levels - 1);
  auto chain_launch = [&](int64_t level0, int32_t s0, int64_t cnt, cudaStream_t s) {
    pm.s0 = s0;
    pm.level0 = (int32_t)level0;
    chain_k<<<dim3(p.Hv, (unsigned)cnt), kThreads, ChSmem::ALLOC, s>>>(p, xmap, omap, tma_out, ws, pm, maxc);
    return cudaGetLastError();
  };
  if (sc.chunk_launches > 1) {
    // level l of every chain on the second stream once the chunk kernel's
    // launch l is done; its launch l + 1 meanwhile on the caller's stream
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream* ss = side_stream(st);
    if (!ss) {
      // no second stream to use: the levels one after the other
      for (int64_t l = 0; l < sc.levels && e == cudaSuccess; ++l) {
        const int64_t c0 = l * sc.piece;
        e = chunk_launch(c0, maxc - c0 < sc.piece ? maxc - c0 : sc.piece, st);
        if (e == cudaSuccess) e = chain_launch(l, 0, p.num_seqs, st);
      }
      if (e != cudaSuccess) return e;
    } else {
      for (int64_t l = 0; l < sc.levels && e == cudaSuccess; ++l) {
        const int64_t c0 = l * sc.piece;
        e = chunk_launch(c0, maxc - c0 < sc.piece ? maxc - c0 : sc.piece, st);
        if (e == cudaSuccess) e = cudaEventRecord(ss->ready, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->stream, ss->ready, 0);
        if (e == cudaSuccess) e = chain_launch(l, 0, p.num_seqs, ss->stream);
      }
      // the join, also after a failed launch (a capture needs its fork joined)
      const cudaError_t j = cudaEventRecord(ss->join, ss->stream);
      const cudaError_t w = j == cudaSuccess ? cudaStreamWaitEvent(st, ss->join, 0) : j;
      if (e != cudaSuccess) return e;
      if (w != cudaSuccess) return w;
    }
  } else {
    e = chunk_launch(0, maxc, st);
    if (e != cudaSuccess) return e;
    const int64_t pairs = sc.levels * p.num_seqs, per = sc.width / p.Hv;
    for (int64_t t = 0; t < sc.launches; ++t) {
      const int64_t base = t * per;
      const int64_t cnt = pairs - base < per ? pairs - base : per;
      e = chain_launch(base / p.num_seqs, (int32_t)(base % p.num_seqs), cnt, st);
      if (e != cudaSuccess) return e;
    }
  }
  if (post && p.total_rows > 0) {
    const int64_t warps = p.total_rows * p.Hv;
    const unsigned blocks = (unsigned)((warps + 7) / 8 < 65535 * 8 ? (warps + 7) / 8 : 65535 * 8);
    core_gate_norm_kernel<<<blocks, 256, 0, st>>>(p, ws.core_o);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  window_kernel<__nv_bfloat16, kPrefill><<<dim3((p.conv_dim + 255) / 256, p.num_seqs, window_slices(p, max_len)), 256, 0,
                                            st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
