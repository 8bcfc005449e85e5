// replay.cu — replay verification on one checkpoint plus an input log
// ("Caching less to serve more requests", section "What we changed": one
// state and a buffer of the per-token inputs since it; outputs are computed
// from the two, a rollback removes buffer entries, and the state is rewritten
// only by the flush).
#include "scan_launch.cuh"

namespace gdn {

// Appends the m new rows (x, g, beta) after the n logged rows of request r and
// then publishes log_len[r] = n + m.  One CTA per request, launched after the
// append scan has read the old log_len.
template <typename TIN>
__global__ void __launch_bounds__(256) log_append_kernel(const ScanParams p) {
  const int r = blockIdx.x;
  const int32_t n = p.log_len[r];
  const int m = p.num_new;
  if (!page_ok(p.pool, p.ckpt_slot[r]) || n < 0 || n + m > GDN_REPLAY_LOG_SLOTS) return;
  const int64_t lrow = (int64_t)r * GDN_REPLAY_LOG_SLOTS + n;
  const int64_t nrow = (int64_t)r * m;
  TIN* lx = reinterpret_cast<TIN*>(const_cast<void*>(p.log_x)) + lrow * p.conv_dim;
  const TIN* xn = reinterpret_cast<const TIN*>(p.x_new) + nrow * p.conv_dim;
  const int64_t nx = (int64_t)m * p.conv_dim;
  for (int64_t i = threadIdx.x; i < nx; i += blockDim.x) lx[i] = xn[i];
  float* lg = const_cast<float*>(p.log_g) + lrow * p.Hv;
  float* lb = const_cast<float*>(p.log_beta) + lrow * p.Hv;
  for (int i = threadIdx.x; i < m * p.Hv; i += blockDim.x) {
    lg[i] = p.g_new[nrow * p.Hv + i];
    lb[i] = p.beta_new[nrow * p.Hv + i];
  }
  __syncthreads();
  if (threadIdx.x == 0) const_cast<int32_t*>(p.log_len)[r] = n + m;
}

cudaError_t launch_replay_append(const ScanParams& p, int dk, int dv, int in_dtype,
                                 int out_dtype, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  cudaError_t e = [&]() -> cudaError_t { GDN_SCAN_DISPATCH(kAppend) }();
  if (e != cudaSuccess) return e;
  if (p.num_new == 0) return cudaSuccess;
  if (in_dtype == GDN_BF16) log_append_kernel<__nv_bfloat16><<<p.num_seqs, 256, 0, st>>>(p);
  else log_append_kernel<float><<<p.num_seqs, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_replay_flush(const ScanParams& p, int dk, int dv, int in_dtype, int out_dtype,
                                cudaStream_t st) {
  GDN_SCAN_DISPATCH(kFlush)
}

__global__ void rollback_kernel(int32_t* log_len, const int32_t* accepted, int32_t num_appended,
                                int32_t n, int32_t* err) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n) return;
  const int32_t acc = accepted[r], len = log_len[r];
  const int32_t drop = num_appended - acc;
  if (acc < 0 || acc > num_appended || len - drop < 0) {
    set_error(err, GDN_ERR_ROLLBACK_RANGE);
    return;
  }
  log_len[r] = len - drop;
}

cudaError_t launch_replay_rollback(int32_t* log_len, const int32_t* accepted, int32_t num_appended,
                                   int32_t n, int32_t* err, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  rollback_kernel<<<(n + 255) / 256, 256, 0, st>>>(log_len, accepted, num_appended, n, err);
  return cudaGetLastError();
}

}  // namespace gdn
