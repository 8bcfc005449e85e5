// prefill.cu — launcher of the prefill scan and its window pass.
#include "scan_launch.cuh"

namespace gdn {

cudaError_t launch_prefill(const ScanParams& p, int dk, int dv, int in_dtype, int out_dtype,
                           cudaStream_t st) {
  GDN_SCAN_DISPATCH(kPrefill)
}

}  // namespace gdn
