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
  // two distinct pages never overlap
  const uint4* __restrict__ s4 = reinterpret_cast<const uint4*>(p.pool.base + (int64_t)src * p.pool.page_bytes);
  uint4* __restrict__ d4 = reinterpret_cast<uint4*>(p.pool.base + (int64_t)dst * p.pool.page_bytes);
  // 32-bit word indices: a payload is far below 2^31 words (checked at launch)
  const uint32_t nv = (uint32_t)(p.payload_bytes / 16);
  const uint32_t step = gridDim.x * blockDim.x;
  uint32_t k = blockIdx.x * blockDim.x + threadIdx.x;
  // four words in flight per thread (all four loads issue before the first
  // store): one word at a time leaves too few bytes in flight per SM to cover
  // the HBM latency
#pragma unroll 1
  for (; k + 3 * step < nv; k += 4 * step) {
    const uint4 w0 = s4[k], w1 = s4[k + step], w2 = s4[k + 2 * step], w3 = s4[k + 3 * step];
    d4[k] = w0;
    d4[k + step] = w1;
    d4[k + 2 * step] = w2;
    d4[k + 3 * step] = w3;
  }
#pragma unroll 1
  for (; k < nv; k += step) d4[k] = s4[k];
}

cudaError_t launch_copy(const CopyParams& p, cudaStream_t st) {
  if (p.n == 0) return cudaSuccess;
  const int64_t nv = p.payload_bytes / 16;
  if (nv >= (int64_t)1 << 30) return cudaErrorInvalidValue;
  int bx = (int)((nv + 256 * 8 - 1) / (256 * 8));  // ~8 words per thread
  if (bx < 1) bx = 1;
  copy_kernel<<<dim3(bx, p.n), 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
