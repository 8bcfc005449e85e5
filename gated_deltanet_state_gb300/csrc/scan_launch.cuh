// scan_launch.cuh — host-side launch of the scan kernel and its window pass.
#pragma once

#include "launch.h"

namespace gdn {

template <int DK, int DV, int RPT, typename TIN, typename TOUT, int MODE>
cudaError_t launch_scan_t(const ScanParams& p, cudaStream_t st) {
  constexpr size_t smem = scan_smem_bytes<DK, DV, RPT, TIN>();
  auto kern = scan_kernel<DK, DV, RPT, TIN, TOUT, MODE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(DV / (32 * RPT), p.Hv, p.num_seqs);
  kern<<<grid, kScanThreads, smem, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // Windows: channel blocks x sequences (the append writes none).
  if (MODE != kAppend) {
    window_kernel<TIN, MODE><<<dim3((p.conv_dim + 255) / 256, p.num_seqs), 256, 0, st>>>(p);
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
    if (dk == 128 && dv == 128) return launch_scan_t<128, 128, 2, __nv_bfloat16, __nv_bfloat16, MODE>(p, st); \
    if (dk == 64 && dv == 64) return launch_scan_t<64, 64, 2, __nv_bfloat16, __nv_bfloat16, MODE>(p, st);    \
    if (dk == 32 && dv == 32) return launch_scan_t<32, 32, 1, __nv_bfloat16, __nv_bfloat16, MODE>(p, st);    \
  } else if (in_dtype == GDN_F32 && out_dtype == GDN_F32) {                               \
    if (dk == 128 && dv == 128) return launch_scan_t<128, 128, 2, float, float, MODE>(p, st); \
    if (dk == 64 && dv == 64) return launch_scan_t<64, 64, 2, float, float, MODE>(p, st);    \
    if (dk == 32 && dv == 32) return launch_scan_t<32, 32, 1, float, float, MODE>(p, st);    \
  }                                                                                       \
  return cudaErrorInvalidValue;

}  // namespace gdn
