// replay.cu — replay verification on one checkpoint plus an input log
// ("Caching less to serve more requests", section "What we changed": one
// state and a buffer of the per-token inputs since it; outputs are computed
// from the two, a rollback removes buffer entries, and the state is rewritten
// only by the flush).
#include "scan_launch.cuh"

namespace gdn {

// Copies the m new rows (x, g, beta) of request r after its n logged rows.
// Grid: (row chunks, requests).  log_len is published later by log_len_kernel.
template <typename TIN>
__global__ void __launch_bounds__(256) log_append_kernel(const ScanParams p) {
  const int r = blockIdx.y;
  const int32_t n = p.log_len[r];
  const int m = p.num_new;
  if (!page_ok(p.pool, p.ckpt_slot[r]) || n < 0 || n + m > GDN_REPLAY_LOG_SLOTS) return;
  const int64_t lrow = (int64_t)r * GDN_REPLAY_LOG_SLOTS + n;
  const int64_t nrow = (int64_t)r * m;
  // x rows as 16-byte words (conv_dim * sizeof(TIN) is a multiple of 16)
  uint4* lx = reinterpret_cast<uint4*>(reinterpret_cast<TIN*>(const_cast<void*>(p.log_x)) + lrow * p.conv_dim);
  const uint4* xn = reinterpret_cast<const uint4*>(reinterpret_cast<const TIN*>(p.x_new) + nrow * p.conv_dim);
  const int64_t nw = (int64_t)m * p.conv_dim * sizeof(TIN) / 16;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nw; i += (int64_t)gridDim.x * blockDim.x)
    lx[i] = xn[i];
  if (blockIdx.x == 0) {
    float* lg = const_cast<float*>(p.log_g) + lrow * p.Hv;
    float* lb = const_cast<float*>(p.log_beta) + lrow * p.Hv;
    for (int i = threadIdx.x; i < m * p.Hv; i += blockDim.x) {
      lg[i] = p.g_new[nrow * p.Hv + i];
      lb[i] = p.beta_new[nrow * p.Hv + i];
    }
  }
}

cudaError_t launch_replay_append(const ScanParams& p, int dk, int dv, int in_dtype,
                                 int out_dtype, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  // tensor-core outputs and log rows, then log_len
  if (tc_replay_supported(dk, dv, in_dtype)) return launch_tc_append(p, st);
  const int64_t max_len = GDN_REPLAY_LOG_SLOTS;
  cudaError_t e = [&]() -> cudaError_t { GDN_SCAN_DISPATCH(kAppend) }();
  if (e != cudaSuccess) return e;
  if (p.num_new == 0) return cudaSuccess;
  const int64_t words = (int64_t)p.num_new * p.conv_dim * (in_dtype == GDN_BF16 ? 2 : 4) / 16;
  const dim3 grid((unsigned)((words + 256 * 4 - 1) / (256 * 4)), p.num_seqs);
  if (in_dtype == GDN_BF16) log_append_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
  else log_append_kernel<float><<<grid, 256, 0, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  log_len_kernel<kAppend><<<(p.num_seqs + 255) / 256, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_replay_flush(const ScanParams& p, int dk, int dv, int in_dtype, int out_dtype,
                                cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  // tensor-core state update and v windows, then the q / k windows and the
  // log reset
  if (tc_replay_supported(dk, dv, in_dtype)) return launch_tc_flush(p, st);
  const int64_t max_len = GDN_REPLAY_LOG_SLOTS;
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
