// checkpoint.cu — bit-exact page-to-page copies of a state payload ("Prefix
// caching on Gated DeltaNet hybrids", section "The in-page layout": save and
// restore copy the bytes, NaN encodings included).  The copy moves 16-byte
// words, so every bit pattern survives; it is HBM-bound (read + write once).
#include "launch.h"

namespace gdn {

__global__ void __launch_bounds__(256) copy_kernel(const CopyParams p) {
  const int i = blockIdx.y;
  const int32_t src = p.src[i], dst = p.dst[i];
  if (!page_ok(p.pool, src) || !page_ok(p.pool, dst)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(p.err, GDN_ERR_PAGE_RANGE);
    return;
  }
  if (src == dst) return;
  const uint4* s4 = reinterpret_cast<const uint4*>(p.pool.base + (int64_t)src * p.pool.page_bytes);
  uint4* d4 = reinterpret_cast<uint4*>(p.pool.base + (int64_t)dst * p.pool.page_bytes);
  const int64_t nv = p.payload_bytes / 16;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < nv;
       k += (int64_t)gridDim.x * blockDim.x)
    d4[k] = s4[k];
}

cudaError_t launch_copy(const CopyParams& p, cudaStream_t st) {
  if (p.n == 0) return cudaSuccess;
  const int64_t nv = p.payload_bytes / 16;
  int bx = (int)((nv + 256 * 8 - 1) / (256 * 8));  // ~8 words per thread
  if (bx < 1) bx = 1;
  copy_kernel<<<dim3(bx, p.n), 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
