// noalloc.cu — gdn_prefill_chunked_noalloc: the chunked prefill with its
// scratch in a fixed device array of this library instead of a caller buffer.
//
// Why: some callers cannot obtain device memory when they call the prefill.
// A serving runtime that reserved the GPU's free memory for its state and KV
// pools at start-up has nothing left for cudaMalloc (and a late cudaMalloc
// would fragment or evict those pools); a plain C caller embedded in another
// framework may not own an allocator at all.  This entry point lets them run
// the prefill without passing or allocating a workspace.
//
// The scratch lives in a file-scope __device__ array of
// GDN_NOALLOC_SCRATCH_BYTES; every GPU that loads the library holds it until
// the process exits.  Host code may not use the array's name as a device
// address (on the host it names a host-side stand-in), so the first call on
// each device that needs the scratch looks the device address up with
// cudaGetSymbolAddress while that device is current, and later calls reuse
// it; calls whose layer needs no scratch skip the array and the look-up.
#include <mutex>

#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch itself.  Its contents are whatever the last call left there.
__device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (set-up on first use).
gdn_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_prefill_chunked_noalloc(const gdn_layer_desc* desc, const gdn_pool* pool,
                                                  const gdn_prefill_args* args, void* stream) {
  if (!desc || !args) return GDN_ERR_INVALID_ARG;
  // a tensor-core layer takes the fused kernel, which needs no scratch: it
  // never touches the array (no set-up either)
  if (gdn::tc_prefill_supported(desc->head_dim_k, desc->head_dim_v, desc->in_dtype, desc->out_dtype,
                                desc->block_size))
    return gdn_prefill_chunked(desc, pool, args, nullptr, 0, stream);
  const size_t need = gdn_prefill_workspace_size(desc, args->num_seqs, args->total_tokens);
  if (need == 0) return gdn_prefill_chunked(desc, pool, args, nullptr, 0, stream);
  // Every workspace element the kernels read is written earlier in the same
  // call, so the scratch needs no clearing between calls.
  if (need > GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const gdn_status st = scratch_address(&scratch);
  if (st != GDN_OK) return st;
  return gdn_prefill_chunked(desc, pool, args, scratch, GDN_NOALLOC_SCRATCH_BYTES, stream);
}
