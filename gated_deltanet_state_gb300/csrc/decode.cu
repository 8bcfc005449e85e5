// decode.cu — batched single-token step of the gated delta rule, fused with
// the one-row conv update ("Hybrid linear attention (gated DeltaNet)", section
// "The part that is easy to get wrong": gdn_conv_decode + gdn_decode).
//
// The step reads and writes every byte of the state once, so it is bound by
// HBM bandwidth.  One CTA owns one (sequence, qk head) pair: the value heads
// that share that qk head, and the conv-window channels of its q, k and v
// slices.  Owning all readers of those window channels lets the CTA shift the
// window in place after it has read it, with no cross-CTA ordering.
//
// In a mixed batch (prefill sequences and single decode tokens packed in one
// varlen batch: the pages' gdn_decode_mixed, same section) the kernel reads
// each decode sequence's token row through `row` and leaves the prefill
// sequences, marked in `decode`, to the prefill kernels.
//
// 256 threads stream the group's rows in passes of 64 rows (4 lanes per row,
// 128-bit loads); the next pass's rows are loaded while the current pass is
// computed, so every thread keeps two 512-byte row slices in flight.
#include "launch.h"

namespace gdn {

constexpr int kDecThreads = 256;
constexpr int kDecPassRows = kDecThreads / 4;

template <int DK, int DV, typename TIN, typename TOUT>
__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(const DecodeParams p) {
  constexpr int NCH = DK / 16;
  const int jq = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = tid & 3, rl = tid >> 2;
  const int G = p.Hv / p.Hqk;
  const int rows = G * DV;
  const int passes = (rows + kDecPassRows - 1) / kDecPassRows;

  if (p.decode && !p.decode[s]) return;   // a prefill sequence of a mixed batch
  const int64_t trow = p.row ? (int64_t)p.row[s] : (int64_t)s;   // token row in x, g, beta, o
  const int32_t slot = p.slot[s];
  if (!page_ok(p.pool, slot)) {
    if (jq == 0 && tid == 0) set_error(p.err, GDN_ERR_PAGE_RANGE);
    return;
  }
  const float* Sg = page_state(p.pool, slot) + (int64_t)jq * G * DV * DK;  // group's rows
  float* Sw = page_state(p.pool, slot) + (int64_t)jq * G * DV * DK;
  TIN* win = page_window<TIN>(p.pool, slot);

  extern __shared__ float4 dsm4[];
  float* y_s = reinterpret_cast<float*>(dsm4);     // [2*DK + G*DV] post-conv q | k | v
  float* a_s = y_s + 2 * DK + G * DV;              // [G]
  float* b_s = a_s + G;                            // [G]
  TIN* nw_s = reinterpret_cast<TIN*>(b_s + G);     // [3][2*DK + G*DV] shifted window
  float* o_s = reinterpret_cast<float*>(nw_s + 3 * (2 * DK + G * DV));   // [G*DV] packed core: outputs

  // ---- start streaming the first pass
  float4 cur[NCH], nxt[NCH];
  {
    const int row = rl;
#pragma unroll
    for (int m = 0; m < NCH; ++m)
      cur[m] = row < rows ? *reinterpret_cast<const float4*>(Sg + (int64_t)row * DK + 4 * (4 * m + cq))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---- conv + SiLU of this group's channels, and the shifted window
  const int NC = 2 * DK + G * DV;
  const TIN* xs = reinterpret_cast<const TIN*>(p.x) + trow * p.x_ld;
  for (int idx = tid; idx < NC; idx += kDecThreads) {
    const int c = idx < DK ? jq * DK + idx
                           : (idx < 2 * DK ? p.Hqk * DK + jq * DK + idx - DK
                                           : 2 * p.Hqk * DK + jq * G * DV + idx - 2 * DK);
    const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (int64_t)c * kConvK);
    const TIN r0 = win[c], r1 = win[p.conv_dim + c], r2 = win[2 * p.conv_dim + c], xv = xs[c];
    float z = w.x * to_f32(r0);
    z = fmaf(w.y, to_f32(r1), z);
    z = fmaf(w.z, to_f32(r2), z);
    z = fmaf(w.w, to_f32(xv), z);
    y_s[idx] = silu(z);
    nw_s[idx] = r1;
    nw_s[NC + idx] = r2;
    nw_s[2 * NC + idx] = xv;
  }
  if (tid < G) {
    const int h = jq * G + tid;
    if (p.ba) {   // packed core: g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)
      const TIN* ba = reinterpret_cast<const TIN*>(p.ba) + trow * 2 * p.Hv;
      const float b = to_f32(ba[h]), x = to_f32(ba[p.Hv + h]) + p.dt_bias[h];
      const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
      a_s[tid] = expf(-expf(p.A_log[h]) * sp);
      b_s[tid] = 1.0f / (1.0f + expf(-b));
    } else {
      a_s[tid] = expf(p.g[trow * p.Hv + h]);
      b_s[tid] = p.beta[trow * p.Hv + h];
    }
  }
  __syncthreads();
  if (warp < 2) {  // warp 0 normalises q, warp 1 normalises k
    float* vec = y_s + warp * DK;
    float ss = 0.f;
#pragma unroll
    for (int jj = 0; jj < DK / 32; ++jj) ss = fmaf(vec[lane + 32 * jj], vec[lane + 32 * jj], ss);
    ss = warp_sum(ss);
    const float f = (warp == 0 ? p.q_scale : 1.0f) / sqrtf(ss + p.eps);
#pragma unroll
    for (int jj = 0; jj < DK / 32; ++jj) vec[lane + 32 * jj] *= f;
  }
  __syncthreads();

  const float* q_s = y_s;
  const float* k_s = y_s + DK;
  const float* v_s = y_s + 2 * DK;
  TOUT* out = reinterpret_cast<TOUT*>(p.o);

  for (int pass = 0; pass < passes; ++pass) {
    const int row = pass * kDecPassRows + rl;
    const int nrow = row + kDecPassRows;
    if (pass + 1 < passes) {
#pragma unroll
      for (int m = 0; m < NCH; ++m)
        nxt[m] = nrow < rows ? *reinterpret_cast<const float4*>(Sg + (int64_t)nrow * DK + 4 * (4 * m + cq))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const bool valid = row < rows;
    const int hh = valid ? row / DV : 0;
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      const float4 k4 = *reinterpret_cast<const float4*>(k_s + 4 * (4 * m + cq));
      acc = fmaf(cur[m].x, k4.x, acc);
      acc = fmaf(cur[m].y, k4.y, acc);
      acc = fmaf(cur[m].z, k4.z, acc);
      acc = fmaf(cur[m].w, k4.w, acc);
    }
    const float u = quad_sum(acc);
    const float a = a_s[hh], b = b_s[hh];
    const float coef = b * fmaf(-a, u, valid ? v_s[row] : 0.f);
    float o = 0.f;
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      const float4 k4 = *reinterpret_cast<const float4*>(k_s + 4 * (4 * m + cq));
      const float4 q4 = *reinterpret_cast<const float4*>(q_s + 4 * (4 * m + cq));
      float4 sn;
      sn.x = fmaf(coef, k4.x, a * cur[m].x);
      sn.y = fmaf(coef, k4.y, a * cur[m].y);
      sn.z = fmaf(coef, k4.z, a * cur[m].z);
      sn.w = fmaf(coef, k4.w, a * cur[m].w);
      o = fmaf(sn.x, q4.x, o);
      o = fmaf(sn.y, q4.y, o);
      o = fmaf(sn.z, q4.z, o);
      o = fmaf(sn.w, q4.w, o);
      if (valid) *reinterpret_cast<float4*>(Sw + (int64_t)row * DK + 4 * (4 * m + cq)) = sn;
    }
    o = quad_sum(o);
    if (valid && cq == 0) {
      const int h = jq * G + hh, r = row - hh * DV;
      if (p.norm_w) o_s[row] = o;   // normalised per head below
      else out[(trow * p.Hv + h) * DV + r] = from_f32<TOUT>(o);
    }
#pragma unroll
    for (int m = 0; m < NCH; ++m) cur[m] = nxt[m];
  }

  // ---- packed core: gated RMS norm of each head's outputs (a warp per head),
  // gated by silu(z) from the packed row
  if (p.norm_w) {
    __syncthreads();
    constexpr int PER = DV / 32 > 0 ? DV / 32 : 1;
    for (int hh = warp; hh < G; hh += kDecThreads / 32) {
      float v[PER];
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < PER; ++m) {
        const int r = lane + 32 * m;
        v[m] = r < DV ? o_s[hh * DV + r] : 0.f;
        ss = fmaf(v[m], v[m], ss);
      }
      ss = warp_sum(ss);
      const float inv = 1.0f / sqrtf(ss / (float)DV + p.norm_eps2);
      const int h = jq * G + hh;
#pragma unroll
      for (int m = 0; m < PER; ++m) {
        const int r = lane + 32 * m;
        if (r < DV) {
          const float z = to_f32(xs[p.conv_dim + h * DV + r]);
          out[(trow * p.Hv + h) * DV + r] = from_f32<TOUT>(v[m] * inv * p.norm_w[r] * silu(z));
        }
      }
    }
  }

  // ---- shift the window of this group's channels (all reads happened above)
  for (int idx = tid; idx < NC; idx += kDecThreads) {
    const int c = idx < DK ? jq * DK + idx
                           : (idx < 2 * DK ? p.Hqk * DK + jq * DK + idx - DK
                                           : 2 * p.Hqk * DK + jq * G * DV + idx - 2 * DK);
    win[c] = nw_s[idx];
    win[p.conv_dim + c] = nw_s[NC + idx];
    win[2 * p.conv_dim + c] = nw_s[2 * NC + idx];
  }
}

template <int DK, int DV, typename TIN, typename TOUT>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t st) {
  const int G = p.Hv / p.Hqk;
  const int NC = 2 * DK + G * DV;
  const size_t smem = sizeof(float) * (NC + 2 * G) + sizeof(TIN) * 3 * NC + sizeof(float) * G * DV + 16;
  auto kern = decode_kernel<DK, DV, TIN, TOUT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.Hqk, p.num_seqs);
  kern<<<grid, kDecThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, int dk, int dv, int in_dtype, int out_dtype,
                          cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
#define GDN_DEC(D, TI, TO) \
  if (dk == D && dv == D) return launch_decode_t<D, D, TI, TO>(p, st);
  if (in_dtype == GDN_BF16 && out_dtype == GDN_BF16) {
    GDN_DEC(128, __nv_bfloat16, __nv_bfloat16)
    GDN_DEC(64, __nv_bfloat16, __nv_bfloat16)
    GDN_DEC(32, __nv_bfloat16, __nv_bfloat16)
  } else if (in_dtype == GDN_F32 && out_dtype == GDN_F32) {
    GDN_DEC(128, float, float)
    GDN_DEC(64, float, float)
    GDN_DEC(32, float, float)
  }
#undef GDN_DEC
  return cudaErrorInvalidValue;
}

}  // namespace gdn
