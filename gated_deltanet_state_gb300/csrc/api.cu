// api.cu — the exported C ABI (include/gdn.h): host-side validation, then the
// internal launchers.  Nothing here allocates memory or keeps state.
#include <cstring>

#include "launch.h"

using namespace gdn;

namespace {

constexpr int32_t kMaxGrid = 65535;  // grid y/z limit used for sequences / pages

bool shape_supported(const gdn_layer_desc* d) {
  if (d->conv_kernel != kConvK || d->reserved != 0) return false;
  const int dk = d->head_dim_k, dv = d->head_dim_v;
  if (dk != dv || (dk != 32 && dk != 64 && dk != 128)) return false;
  if (d->in_dtype != d->out_dtype) return false;
  if (d->num_v_heads % d->num_qk_heads != 0 || d->num_v_heads > kMaxGrid) return false;
  if (d->chunk_size != 16 && d->chunk_size != 32 && d->chunk_size != 64) return false;
  if (d->block_size <= 0 || d->block_size % d->chunk_size != 0) return false;
  return true;
}

gdn_status check_desc_pool(const gdn_layer_desc* d, const gdn_pool* pool) {
  if (!d || !pool) return GDN_ERR_INVALID_ARG;
  if (d->num_qk_heads <= 0 || d->num_v_heads <= 0 || d->head_dim_k <= 0 || d->head_dim_v <= 0)
    return GDN_ERR_INVALID_ARG;
  if (d->in_dtype != GDN_F32 && d->in_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (d->out_dtype != GDN_F32 && d->out_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (!(d->norm_eps >= 0.0f)) return GDN_ERR_INVALID_ARG;
  if (!shape_supported(d)) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (!pool->base || pool->num_pages <= 0) return GDN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(pool->base) % 256 != 0 || pool->page_bytes % 256 != 0)
    return GDN_ERR_INVALID_ARG;
  if (pool->page_bytes < gdn_mamba_page_bytes(d)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

Pool make_pool(const gdn_layer_desc* d, const gdn_pool* pool) {
  Pool p;
  p.base = static_cast<char*>(pool->base);
  p.page_bytes = pool->page_bytes;
  p.num_pages = pool->num_pages;
  p.state_bytes = (int64_t)d->num_v_heads * d->head_dim_v * d->head_dim_k * 4;
  return p;
}

ScanParams base_scan(const gdn_layer_desc* d, const gdn_pool* pool) {
  ScanParams p;
  memset(&p, 0, sizeof(p));
  p.pool = make_pool(d, pool);
  p.Hqk = d->num_qk_heads;
  p.Hv = d->num_v_heads;
  p.conv_dim = (int32_t)gdn_conv_dim(d);
  p.x_ld = p.conv_dim;
  p.block_size = d->block_size;
  p.q_scale = d->q_scale;
  p.eps = d->norm_eps;
  return p;
}

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// Pre-conv rows and conv taps are read in 16-byte words.
bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

extern "C" {

size_t gdn_prefill_workspace_size(const gdn_layer_desc* desc, int32_t num_seqs,
                                  int64_t total_tokens) {
  if (gdn_conv_dim(desc) <= 0 || total_tokens < 0) return 0;
  // the tensor-core shapes: the chunk kernel's operand images for the chain
  // kernel (without a workspace they take the fused kernel, which needs none)
  if (tc_prefill_supported(desc->head_dim_k, desc->head_dim_v, desc->in_dtype, desc->out_dtype,
                           desc->block_size))
    return tc_chain_workspace_bytes(desc->num_qk_heads, desc->num_v_heads, num_seqs < 0 ? 0 : num_seqs,
                                    total_tokens);
  return scan_workspace_bytes(total_tokens, (int)gdn_conv_dim(desc), desc->num_qk_heads,
                              desc->num_v_heads);
}

gdn_status gdn_prefill_plan_for(const gdn_layer_desc* desc, int32_t num_seqs, int64_t max_seq_len,
                                int32_t num_sms, int32_t path, gdn_prefill_plan* out) {
  if (!desc || !out || gdn_conv_dim(desc) <= 0 || num_seqs < 0 || num_seqs > kMaxGrid || max_seq_len < 0)
    return GDN_ERR_INVALID_ARG;
  if (!tc_prefill_supported(desc->head_dim_k, desc->head_dim_v, desc->in_dtype, desc->out_dtype,
                            desc->block_size))
    return GDN_ERR_UNSUPPORTED_SHAPE;
  if (path < GDN_PREFILL_AUTO || path > GDN_PREFILL_TWO_KERNELS) return GDN_ERR_INVALID_ARG;
  const int sms = num_sms > 0 ? num_sms : tc_prefill_sm_count();
  const bool two = path == GDN_PREFILL_TWO_KERNELS ||
                   (path == GDN_PREFILL_AUTO &&
                    tc_prefill_two_kernels_faster(desc->num_qk_heads, desc->num_v_heads, num_seqs, max_seq_len, sms));
  const PrefillSchedule sc = two ? tc_chain_schedule(desc->num_qk_heads, desc->num_v_heads, num_seqs, max_seq_len, sms)
                                 : tc_prefill_schedule(desc->num_v_heads, num_seqs, max_seq_len, sms);
  out->two_kernels = two ? 1 : 0;
  out->chains = sc.nchains;
  out->piece_chunks = sc.piece;
  out->levels = sc.levels;
  out->ctas_per_launch = sc.width;
  out->launches = sc.launches;
  out->chunk_launches = two ? sc.chunk_launches : 0;
  return GDN_OK;
}

size_t gdn_replay_workspace_size(const gdn_layer_desc* desc, int32_t num_reqs) {
  if (gdn_conv_dim(desc) <= 0 || num_reqs < 0) return 0;
  return scan_workspace_bytes((int64_t)num_reqs * GDN_REPLAY_LOG_SLOTS, (int)gdn_conv_dim(desc),
                              desc->num_qk_heads, desc->num_v_heads);
}

}  // extern "C"

namespace {

// The packed core's gates g, b of every row and value head (fp32), 256-byte
// rounded: the start of its workspace.
size_t core_gates_bytes(const gdn_layer_desc* desc, int64_t total_tokens) {
  const size_t b = 2 * sizeof(float) * (size_t)total_tokens * desc->num_v_heads;
  return (b + 255) / 256 * 256;
}

// The prefill, plain or on packed rows (core != nullptr).
gdn_status prefill_call(const gdn_layer_desc* desc, const gdn_pool* pool, const gdn_prefill_args* a,
                        const gdn_core_args* core, void* workspace, size_t workspace_bytes, void* stream) {
  gdn_status st = check_desc_pool(desc, pool);
  if (st != GDN_OK) return st;
  if (!a || a->num_seqs < 0 || a->num_seqs > kMaxGrid || a->total_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (a->num_seqs == 0) return GDN_OK;
  if (!a->cu_seqlens || !a->start_pos || !a->conv_w || !a->init_page || !a->out_slot ||
      !a->dev_error || a->max_blocks < 0 || (a->max_blocks > 0 && !a->block_table))
    return GDN_ERR_INVALID_ARG;
  if (a->total_tokens > 0 && (!a->x || (!core && (!a->g || !a->beta)) || !a->o)) return GDN_ERR_INVALID_ARG;
  if (core) {
    if (!tc_prefill_supported(desc->head_dim_k, desc->head_dim_v, desc->in_dtype, desc->out_dtype,
                              desc->block_size))
      return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!core->A_log || !core->dt_bias || !core->norm_w || (a->total_tokens > 0 && !core->ba))
      return GDN_ERR_INVALID_ARG;
  }
  if (!aligned16(a->x) || !aligned16(a->conv_w)) return GDN_ERR_INVALID_ARG;
  // Fail closed before launching anything when the host can see an
  // off-boundary resume or a cold start that does not begin at 0.
  if (a->start_pos_host) {
    for (int32_t s = 0; s < a->num_seqs; ++s) {
      const int64_t sp = a->start_pos_host[s];
      if (sp < 0) return GDN_ERR_INVALID_ARG;
      const bool cold = a->init_page_host ? a->init_page_host[s] == -1 : sp == 0;
      if (cold ? sp != 0 : (sp <= 0 || sp % desc->block_size != 0)) return GDN_ERR_NOT_BLOCK_ALIGNED;
    }
  }
  if (a->init_page_host)
    for (int32_t s = 0; s < a->num_seqs; ++s)
      if (a->init_page_host[s] < -1 || a->init_page_host[s] >= pool->num_pages) return GDN_ERR_PAGE_RANGE;
  if (a->max_seq_len < 0) return GDN_ERR_INVALID_ARG;
  const bool tc = tc_prefill_supported(desc->head_dim_k, desc->head_dim_v, desc->in_dtype, desc->out_dtype,
                                       desc->block_size);
  // the packed core: its rows' gates first in the workspace, then (two
  // kernels) the operand images; a workspace of the gates alone keeps the
  // fused kernel
  const size_t core_gates = core ? core_gates_bytes(desc, a->total_tokens) : 0;
  const size_t core_images =
      core && tc ? tc_chain_workspace_bytes(desc->num_qk_heads, desc->num_v_heads, a->num_seqs, a->total_tokens,
                                            true)
                 : 0;
  if (a->path < GDN_PREFILL_AUTO || a->path > GDN_PREFILL_TWO_KERNELS || a->reserved != 0)
    return GDN_ERR_INVALID_ARG;
  const int64_t max_len = a->max_seq_len > 0 ? a->max_seq_len : a->total_tokens;
  // a tensor-core layer: the two kernels when asked for, or (AUTO) when a
  // workspace is given and they are expected to be faster; else the fused one
  const bool has_ws = !(workspace == nullptr && workspace_bytes == 0);
  const bool core_fits_two = !core || workspace_bytes >= core_gates + core_images;
  const bool two_kernels =
      tc &&
      (a->path == GDN_PREFILL_TWO_KERNELS ||
       (a->path == GDN_PREFILL_AUTO && has_ws && core_fits_two &&
        tc_prefill_two_kernels_faster(desc->num_qk_heads, desc->num_v_heads, a->num_seqs, max_len,
                                      tc_prefill_sm_count())));
  const size_t need = core ? core_gates + (two_kernels ? core_images : 0)
                           : gdn_prefill_workspace_size(desc, a->num_seqs, a->total_tokens);
  const bool needs_ws = core || !tc || two_kernels || (a->path == GDN_PREFILL_AUTO && has_ws);
  if (need > 0 && needs_ws && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return GDN_ERR_WORKSPACE;
  ScanParams p = base_scan(desc, pool);
  p.num_seqs = a->num_seqs;
  p.conv_w = a->conv_w;
  p.o = a->o;
  p.err = a->dev_error;
  p.cu_seqlens = a->cu_seqlens;
  p.start_pos = a->start_pos;
  p.init_page = a->init_page;
  p.block_table = a->block_table;
  p.max_blocks = a->max_blocks;
  p.out_slot = a->out_slot;
  p.x = a->x;
  p.g = a->g;
  p.beta = a->beta;
  p.total_rows = a->total_tokens;
  p.wait_cycles = a->wait_cycles;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (core) {
    // packed rows q | k | v | z; the gates of every row into the workspace first
    p.x_ld = p.conv_dim + desc->num_v_heads * desc->head_dim_v;
    float* gw = static_cast<float*>(workspace);
    float* bw = gw + (size_t)a->total_tokens * desc->num_v_heads;
    p.g = gw;
    p.beta = bw;
    p.norm_w = core->norm_w;
    p.norm_eps2 = core->norm_eps;
    st = cuda_status(launch_core_gates(core->ba, desc->in_dtype, core->A_log, core->dt_bias, desc->num_v_heads,
                                       a->total_tokens, gw, bw, cs));
    if (st != GDN_OK) return st;
  } else if (need > 0 && !tc) {
    bind_workspace(p, workspace, a->total_tokens);
  }
  void* images = two_kernels ? static_cast<uint8_t*>(workspace) + core_gates : nullptr;
  return cuda_status(launch_prefill(p, images, max_len, desc->head_dim_k, desc->head_dim_v, desc->in_dtype,
                                    desc->out_dtype, cs));
}

}  // namespace

extern "C" {

gdn_status gdn_prefill_chunked(const gdn_layer_desc* desc, const gdn_pool* pool,
                               const gdn_prefill_args* a, void* workspace, size_t workspace_bytes,
                               void* stream) {
  return prefill_call(desc, pool, a, nullptr, workspace, workspace_bytes, stream);
}

size_t gdn_core_prefill_workspace_size(const gdn_layer_desc* desc, int32_t num_seqs, int64_t total_tokens) {
  if (gdn_conv_dim(desc) <= 0 || total_tokens < 0 || num_seqs < 0) return 0;
  const size_t gates = core_gates_bytes(desc, total_tokens);
  if (!tc_prefill_supported(desc->head_dim_k, desc->head_dim_v, desc->in_dtype, desc->out_dtype,
                            desc->block_size))
    return gates;
  return gates + tc_chain_workspace_bytes(desc->num_qk_heads, desc->num_v_heads, num_seqs, total_tokens, true);
}

gdn_status gdn_core_prefill(const gdn_layer_desc* desc, const gdn_pool* pool, const gdn_prefill_args* a,
                            const gdn_core_args* core, void* workspace, size_t workspace_bytes, void* stream) {
  if (!core) return GDN_ERR_INVALID_ARG;
  return prefill_call(desc, pool, a, core, workspace, workspace_bytes, stream);
}

gdn_status gdn_decode_step(const gdn_layer_desc* desc, const gdn_pool* pool,
                           const gdn_decode_args* a, void* stream) {
  gdn_status st = check_desc_pool(desc, pool);
  if (st != GDN_OK) return st;
  if (!a || a->num_seqs < 0 || a->num_seqs > kMaxGrid) return GDN_ERR_INVALID_ARG;
  if (a->num_seqs == 0) return GDN_OK;
  if (!a->x || !a->g || !a->beta || !a->conv_w || !a->slot || !a->o || !a->dev_error)
    return GDN_ERR_INVALID_ARG;
  if (!aligned16(a->conv_w)) return GDN_ERR_INVALID_ARG;
  DecodeParams p{};
  p.pool = make_pool(desc, pool);
  p.Hqk = desc->num_qk_heads;
  p.Hv = desc->num_v_heads;
  p.conv_dim = (int32_t)gdn_conv_dim(desc);
  p.x_ld = p.conv_dim;
  p.num_seqs = a->num_seqs;
  p.q_scale = desc->q_scale;
  p.eps = desc->norm_eps;
  p.x = a->x;
  p.g = a->g;
  p.beta = a->beta;
  p.conv_w = a->conv_w;
  p.slot = a->slot;
  p.o = a->o;
  p.err = a->dev_error;
  p.row = nullptr;
  p.decode = nullptr;
  return cuda_status(launch_decode(p, desc->head_dim_k, desc->head_dim_v, desc->in_dtype,
                                   desc->out_dtype, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_core_decode(const gdn_layer_desc* desc, const gdn_pool* pool, const gdn_decode_args* a,
                           const gdn_core_args* core, void* stream) {
  gdn_status st = check_desc_pool(desc, pool);
  if (st != GDN_OK) return st;
  if (!a || !core || a->num_seqs < 0 || a->num_seqs > kMaxGrid) return GDN_ERR_INVALID_ARG;
  if (a->num_seqs == 0) return GDN_OK;
  if (!a->x || !a->conv_w || !a->slot || !a->o || !a->dev_error || !core->ba || !core->A_log ||
      !core->dt_bias || !core->norm_w)
    return GDN_ERR_INVALID_ARG;
  if (!aligned16(a->conv_w)) return GDN_ERR_INVALID_ARG;
  DecodeParams p{};
  p.pool = make_pool(desc, pool);
  p.Hqk = desc->num_qk_heads;
  p.Hv = desc->num_v_heads;
  p.conv_dim = (int32_t)gdn_conv_dim(desc);
  p.x_ld = p.conv_dim + desc->num_v_heads * desc->head_dim_v;
  p.num_seqs = a->num_seqs;
  p.q_scale = desc->q_scale;
  p.eps = desc->norm_eps;
  p.x = a->x;
  p.conv_w = a->conv_w;
  p.slot = a->slot;
  p.o = a->o;
  p.err = a->dev_error;
  p.ba = core->ba;
  p.A_log = core->A_log;
  p.dt_bias = core->dt_bias;
  p.norm_w = core->norm_w;
  p.norm_eps2 = core->norm_eps;
  return cuda_status(launch_decode(p, desc->head_dim_k, desc->head_dim_v, desc->in_dtype,
                                   desc->out_dtype, static_cast<cudaStream_t>(stream)));
}

size_t gdn_mixed_workspace_size(const gdn_layer_desc* desc, int32_t num_seqs, int64_t total_tokens) {
  return gdn_prefill_workspace_size(desc, num_seqs, total_tokens);
}

gdn_status gdn_mixed_step(const gdn_layer_desc* desc, const gdn_pool* pool, const gdn_mixed_args* a,
                          void* workspace, size_t workspace_bytes, void* stream) {
  gdn_status st = check_desc_pool(desc, pool);
  if (st != GDN_OK) return st;
  if (!a || a->num_seqs < 0 || a->num_seqs > kMaxGrid || a->total_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (a->num_seqs == 0) return GDN_OK;
  if (!a->cu_seqlens || !a->cu_seqlens_host || !a->is_decode || !a->is_decode_host || !a->start_pos ||
      !a->init_page || !a->slot || !a->conv_w || !a->dev_error || a->max_blocks < 0 ||
      (a->max_blocks > 0 && !a->block_table))
    return GDN_ERR_INVALID_ARG;
  if (a->total_tokens > 0 && (!a->x || !a->g || !a->beta || !a->o)) return GDN_ERR_INVALID_ARG;
  if (!aligned16(a->x) || !aligned16(a->conv_w)) return GDN_ERR_INVALID_ARG;
  if (a->cu_seqlens_host[0] != 0 || a->cu_seqlens_host[a->num_seqs] != a->total_tokens)
    return GDN_ERR_INVALID_ARG;
  int32_t n_dec = 0;
  for (int32_t s = 0; s < a->num_seqs; ++s) {
    const int64_t len = (int64_t)a->cu_seqlens_host[s + 1] - a->cu_seqlens_host[s];
    if (len < 0) return GDN_ERR_INVALID_ARG;
    if (a->is_decode_host[s]) {
      if (len != 1) return GDN_ERR_INVALID_ARG;
      ++n_dec;
      continue;
    }
    if (a->start_pos_host) {
      const int64_t sp = a->start_pos_host[s];
      if (sp < 0) return GDN_ERR_INVALID_ARG;
      const bool cold = a->init_page_host ? a->init_page_host[s] == -1 : sp == 0;
      if (cold ? sp != 0 : (sp <= 0 || sp % desc->block_size != 0)) return GDN_ERR_NOT_BLOCK_ALIGNED;
    }
    if (a->init_page_host && (a->init_page_host[s] < -1 || a->init_page_host[s] >= pool->num_pages))
      return GDN_ERR_PAGE_RANGE;
  }
  if (a->max_seq_len < 0) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_mixed_workspace_size(desc, a->num_seqs, a->total_tokens);
  const bool tc = tc_prefill_supported(desc->head_dim_k, desc->head_dim_v, desc->in_dtype, desc->out_dtype,
                                       desc->block_size);
  // as gdn_prefill_chunked with GDN_PREFILL_AUTO
  const bool has_ws = !(workspace == nullptr && workspace_bytes == 0);
  const int64_t mixed_max_len = a->max_seq_len > 0 ? a->max_seq_len : a->total_tokens;
  const bool two_kernels = tc && has_ws &&
                           tc_prefill_two_kernels_faster(desc->num_qk_heads, desc->num_v_heads, a->num_seqs,
                                                         mixed_max_len, tc_prefill_sm_count());
  if (n_dec < a->num_seqs && need > 0 && (!tc || has_ws) &&
      (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return GDN_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // the prefill sequences (the decode ones are skipped by every prefill kernel)
  if (n_dec < a->num_seqs) {
    ScanParams p = base_scan(desc, pool);
    p.num_seqs = a->num_seqs;
    p.conv_w = a->conv_w;
    p.o = a->o;
    p.err = a->dev_error;
    p.cu_seqlens = a->cu_seqlens;
    p.start_pos = a->start_pos;
    p.init_page = a->init_page;
    p.block_table = a->block_table;
    p.max_blocks = a->max_blocks;
    p.out_slot = a->slot;
    p.x = a->x;
    p.g = a->g;
    p.beta = a->beta;
    p.total_rows = a->total_tokens;
    p.skip = a->is_decode;
    if (need > 0 && !tc) bind_workspace(p, workspace, a->total_tokens);
    const int64_t max_len = a->max_seq_len > 0 ? a->max_seq_len : a->total_tokens;
    st = cuda_status(launch_prefill(p, two_kernels ? workspace : nullptr, max_len, desc->head_dim_k,
                                    desc->head_dim_v, desc->in_dtype, desc->out_dtype, cs));
    if (st != GDN_OK) return st;
  }
  // the decode tokens (gdn_decode_mixed): row cu_seqlens[s] of the packed tensors
  if (n_dec > 0) {
    DecodeParams p{};
    p.pool = make_pool(desc, pool);
    p.Hqk = desc->num_qk_heads;
    p.Hv = desc->num_v_heads;
    p.conv_dim = (int32_t)gdn_conv_dim(desc);
    p.x_ld = p.conv_dim;
    p.num_seqs = a->num_seqs;
    p.q_scale = desc->q_scale;
    p.eps = desc->norm_eps;
    p.x = a->x;
    p.g = a->g;
    p.beta = a->beta;
    p.conv_w = a->conv_w;
    p.slot = a->slot;
    p.o = a->o;
    p.err = a->dev_error;
    p.row = a->cu_seqlens;
    p.decode = a->is_decode;
    st = cuda_status(launch_decode(p, desc->head_dim_k, desc->head_dim_v, desc->in_dtype, desc->out_dtype, cs));
  }
  return st;
}

static gdn_status checkpoint_copy(const gdn_layer_desc* desc, const gdn_pool* pool,
                                  const int32_t* src, const int32_t* dst,
                                  const int64_t* num_computed_host, int32_t n, int32_t* dev_error,
                                  void* stream) {
  gdn_status st = check_desc_pool(desc, pool);
  if (st != GDN_OK) return st;
  if (n < 0 || n > kMaxGrid) return GDN_ERR_INVALID_ARG;
  if (n == 0) return GDN_OK;
  if (!src || !dst || !num_computed_host || !dev_error) return GDN_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    if (num_computed_host[i] < 0) return GDN_ERR_INVALID_ARG;
    if (num_computed_host[i] % desc->block_size != 0) return GDN_ERR_NOT_BLOCK_ALIGNED;
  }
  CopyParams p;
  p.pool = make_pool(desc, pool);
  p.payload_bytes = gdn_mamba_page_bytes(desc);
  p.src = src;
  p.dst = dst;
  p.n = n;
  p.err = dev_error;
  return cuda_status(launch_copy(p, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_checkpoint_resume(const gdn_layer_desc* desc, const gdn_pool* pool,
                                 const int32_t* src_page, const int32_t* dst_page,
                                 const int64_t* num_computed_host, int32_t n, int32_t* dev_error,
                                 void* stream) {
  return checkpoint_copy(desc, pool, src_page, dst_page, num_computed_host, n, dev_error, stream);
}

gdn_status gdn_checkpoint_save(const gdn_layer_desc* desc, const gdn_pool* pool,
                               const int32_t* src_page, const int32_t* dst_page,
                               const int64_t* num_computed_host, int32_t n, int32_t* dev_error,
                               void* stream) {
  return checkpoint_copy(desc, pool, src_page, dst_page, num_computed_host, n, dev_error, stream);
}

static gdn_status replay_common(const gdn_layer_desc* desc, const gdn_pool* pool,
                                const gdn_replay_args* a, bool append, ScanParams* out) {
  gdn_status st = check_desc_pool(desc, pool);
  if (st != GDN_OK) return st;
  if (!a || a->num_reqs < 0 || a->num_reqs > kMaxGrid) return GDN_ERR_INVALID_ARG;
  if (!a->ckpt_slot || !a->log_x || !a->log_g || !a->log_beta || !a->log_len || !a->conv_w ||
      !a->dev_error)
    return a->num_reqs == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
  if (!aligned16(a->log_x) || !aligned16(a->conv_w) || (append && !aligned16(a->x_new)))
    return GDN_ERR_INVALID_ARG;
  if (append) {
    if (a->num_new < 0) return GDN_ERR_INVALID_ARG;
    if (a->num_new > GDN_REPLAY_LOG_SLOTS) return GDN_ERR_LOG_OVERFLOW;
    if (a->num_new > 0 && (!a->x_new || !a->g_new || !a->beta_new || !a->o)) return GDN_ERR_INVALID_ARG;
  }
  if (!append && a->boundary_rows) {
    // boundary checkpoints are written by the tensor-core flush only
    if (!a->boundary_page) return GDN_ERR_INVALID_ARG;
    if (!tc_replay_supported(desc->head_dim_k, desc->head_dim_v, desc->in_dtype)) return GDN_ERR_UNSUPPORTED_SHAPE;
  }
  const size_t need = gdn_replay_workspace_size(desc, a->num_reqs);
  if (!a->workspace || a->workspace_bytes < need || !aligned16(a->workspace)) return GDN_ERR_WORKSPACE;
  ScanParams p = base_scan(desc, pool);
  bind_workspace(p, a->workspace, (int64_t)a->num_reqs * GDN_REPLAY_LOG_SLOTS);
  p.num_seqs = a->num_reqs;
  p.conv_w = a->conv_w;
  p.o = a->o;
  p.err = a->dev_error;
  p.ckpt_slot = a->ckpt_slot;
  p.log_x = a->log_x;
  p.log_g = a->log_g;
  p.log_beta = a->log_beta;
  p.log_len = a->log_len;
  p.num_new = append ? a->num_new : 0;
  p.x_new = a->x_new;
  p.g_new = a->g_new;
  p.beta_new = a->beta_new;
  p.boundary_rows = append ? nullptr : a->boundary_rows;
  p.boundary_page = append ? nullptr : a->boundary_page;
  *out = p;
  return GDN_OK;
}

gdn_status gdn_replay_append(const gdn_layer_desc* desc, const gdn_pool* pool,
                             const gdn_replay_args* a, void* stream) {
  ScanParams p;
  gdn_status st = replay_common(desc, pool, a, true, &p);
  if (st != GDN_OK || a->num_reqs == 0) return st;
  return cuda_status(launch_replay_append(p, desc->head_dim_k, desc->head_dim_v, desc->in_dtype,
                                          desc->out_dtype, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_replay_flush(const gdn_layer_desc* desc, const gdn_pool* pool,
                            const gdn_replay_args* a, void* stream) {
  ScanParams p;
  gdn_status st = replay_common(desc, pool, a, false, &p);
  if (st != GDN_OK || a->num_reqs == 0) return st;
  return cuda_status(launch_replay_flush(p, desc->head_dim_k, desc->head_dim_v, desc->in_dtype,
                                         desc->out_dtype, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_replay_rollback(int32_t* log_len, const int32_t* accepted, int32_t num_appended,
                               int32_t n, int32_t* dev_error, void* stream) {
  if (n < 0 || num_appended < 0 || num_appended > GDN_REPLAY_LOG_SLOTS) return GDN_ERR_INVALID_ARG;
  if (n == 0) return GDN_OK;
  if (!log_len || !accepted || !dev_error) return GDN_ERR_INVALID_ARG;
  return cuda_status(launch_replay_rollback(log_len, accepted, num_appended, n, dev_error,
                                            static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
