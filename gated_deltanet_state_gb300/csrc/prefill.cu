// prefill.cu — launcher of the prefill: the tensor-core chunk kernel where the
// shape allows it, else the scan; then the window pass.
#include "scan_launch.cuh"

namespace gdn {

size_t scan_workspace_bytes(int64_t rows, int conv_dim, int Hqk, int Hv) {
  return ws_layout(rows, conv_dim, Hqk, Hv).bytes;
}

void bind_workspace(ScanParams& p, void* ws, int64_t rows) { ws_bind(p, ws, rows); }

cudaError_t launch_prefill(const ScanParams& p, int64_t max_len, int dk, int dv, int in_dtype,
                           int out_dtype, cudaStream_t st) {
  if (tc_prefill_supported(dk, dv, in_dtype, out_dtype, p.block_size)) return launch_tc_prefill(p, st);
  GDN_SCAN_DISPATCH(kPrefill)
}

}  // namespace gdn
