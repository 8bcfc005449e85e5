// scan_launch.cuh — host-side launch of the conv pre-pass, the scan and the
// window pass (shared by prefill and replay).
#pragma once

#include "launch.h"

namespace gdn {

// Workspace layout for `rows` token rows: y, norm factors, gates, each
// section 256-byte aligned.
struct WsLayout {
  size_t y, nrm, ab, bytes;
};
inline WsLayout ws_layout(int64_t rows, int conv_dim, int Hqk, int Hv) {
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  WsLayout L;
  L.y = 0;
  L.nrm = up(sizeof(float) * (size_t)rows * conv_dim);
  L.ab = L.nrm + up(sizeof(float) * (size_t)rows * 2 * Hqk);
  L.bytes = L.ab + up(sizeof(float) * (size_t)rows * Hv * 2);
  return L;
}
inline void ws_bind(ScanParams& p, void* ws, int64_t rows) {
  const WsLayout L = ws_layout(rows, p.conv_dim, p.Hqk, p.Hv);
  char* b = static_cast<char*>(ws);
  p.ws_y = reinterpret_cast<float*>(b + L.y);
  p.ws_nrm = reinterpret_cast<float*>(b + L.nrm);
  p.ws_ab = reinterpret_cast<float*>(b + L.ab);
}

template <int DK, int DV, int RPT, typename TIN, typename TOUT, int MODE>
cudaError_t launch_scan_t(const ScanParams& p, int64_t max_len, cudaStream_t st) {
  // 1. conv pre-pass: one CTA per (block of channels, 64-token tile, sequence)
  if (max_len > 0) {
    constexpr int per_cta = kConvThreads * Vec16<TIN>::N;
    const dim3 cgrid((p.conv_dim + per_cta - 1) / per_cta,
                     (unsigned)((max_len + kConvTokens - 1) / kConvTokens), p.num_seqs);
    conv_kernel<TIN, MODE, DK><<<cgrid, kConvThreads, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 2. the scan
  constexpr size_t smem = scan_smem_bytes<DK, DV, RPT>();
  auto kern = scan_kernel<DK, DV, RPT, TIN, TOUT, MODE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(DV / (32 * RPT), p.Hv, p.num_seqs);
  kern<<<grid, kScanThreads, smem, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // 3. windows: channel blocks x sequences (the append writes none)
  if (MODE != kAppend) {
    const unsigned zs = MODE == kPrefill ? window_slices(p, max_len) : 1u;
    window_kernel<TIN, MODE><<<dim3((p.conv_dim + 255) / 256, p.num_seqs, zs), 256, 0, st>>>(p);
    e = cudaGetLastError();
  }
  if (MODE == kFlush && e == cudaSuccess) {
    log_len_kernel<kFlush><<<(p.num_seqs + 255) / 256, 256, 0, st>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

// Rows per thread: two for dv >= 64 (fewer shared-memory loads per FMA), one
// for dv = 32.
#define GDN_SCAN_DISPATCH(MODE)                                                           \
  if (p.num_seqs == 0) return cudaSuccess;                                                \
  if (in_dtype == GDN_BF16 && out_dtype == GDN_BF16) {                                    \
    if (dk == 128 && dv == 128) return launch_scan_t<128, 128, 2, __nv_bfloat16, __nv_bfloat16, MODE>(p, max_len, st); \
    if (dk == 64 && dv == 64) return launch_scan_t<64, 64, 2, __nv_bfloat16, __nv_bfloat16, MODE>(p, max_len, st);    \
    if (dk == 32 && dv == 32) return launch_scan_t<32, 32, 1, __nv_bfloat16, __nv_bfloat16, MODE>(p, max_len, st);    \
  } else if (in_dtype == GDN_F32 && out_dtype == GDN_F32) {                               \
    if (dk == 128 && dv == 128) return launch_scan_t<128, 128, 2, float, float, MODE>(p, max_len, st); \
    if (dk == 64 && dv == 64) return launch_scan_t<64, 64, 2, float, float, MODE>(p, max_len, st);    \
    if (dk == 32 && dv == 32) return launch_scan_t<32, 32, 1, float, float, MODE>(p, max_len, st);    \
  }                                                                                       \
  return cudaErrorInvalidValue;

}  // namespace gdn
