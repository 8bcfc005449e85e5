// prefill.cu — launcher of the prefill: on the tensor cores where the shape
// allows it (the chunk + chain kernels with a workspace, the fused kernel
// without), else the scan; then the window pass.
#include "scan_launch.cuh"

namespace gdn {

size_t scan_workspace_bytes(int64_t rows, int conv_dim, int Hqk, int Hv) {
  return ws_layout(rows, conv_dim, Hqk, Hv).bytes;
}

void bind_workspace(ScanParams& p, void* ws, int64_t rows) { ws_bind(p, ws, rows); }

cudaError_t launch_prefill(const ScanParams& p, void* workspace, int64_t max_len, int dk, int dv, int in_dtype,
                           int out_dtype, cudaStream_t st) {
  if (tc_prefill_supported(dk, dv, in_dtype, out_dtype, p.block_size))
    return workspace ? launch_tc_prefill2(p, workspace, max_len, st) : launch_tc_prefill(p, max_len, st);
  GDN_SCAN_DISPATCH(kPrefill)
}

// Packed core gates, one thread per (row, v head): g = -exp(A_log) softplus(a +
// dt_bias), beta = sigmoid(b) from the packed b | a rows ("Hybrid linear
// attention (gated DeltaNet)", "Packed-core traces"; the formulas are the
// library's reading, the pages name the weights only).
template <typename TIN>
__global__ void __launch_bounds__(256) core_gates_kernel(const TIN* ba, const float* A_log, const float* dt_bias,
                                                         int Hv, int64_t rows, float* g, float* beta) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * Hv) return;
  const int64_t t = i / Hv;
  const int h = (int)(i - t * Hv);
  const float b = to_f32(ba[t * 2 * Hv + h]);
  const float x = to_f32(ba[t * 2 * Hv + Hv + h]) + dt_bias[h];
  const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
  g[i] = -expf(A_log[h]) * sp;
  beta[i] = 1.0f / (1.0f + expf(-b));
}

cudaError_t launch_core_gates(const void* ba, int in_dtype, const float* A_log, const float* dt_bias, int Hv,
                              int64_t rows, float* g, float* beta, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((rows * Hv + 255) / 256);
  if (in_dtype == GDN_BF16)
    core_gates_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(ba), A_log,
                                                              dt_bias, Hv, rows, g, beta);
  else
    core_gates_kernel<float><<<blocks, 256, 0, st>>>(reinterpret_cast<const float*>(ba), A_log, dt_bias, Hv,
                                                     rows, g, beta);
  return cudaGetLastError();
}

}  // namespace gdn
