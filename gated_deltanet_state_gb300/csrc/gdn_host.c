/*
 * gdn_host.c — exact host arithmetic of the block-aligned state cache and
 * the status strings.  Every function is a pure integer formula; the header
 * include/gdn.h cites the page and section each one restates.
 */
#include "gdn.h"

static int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED_SHAPE: return "unsupported layer shape";
    case GDN_ERR_NOT_BLOCK_ALIGNED: return "position is not on a block boundary";
    case GDN_ERR_PARTIAL_BLOCK: return "block is not full";
    case GDN_ERR_LOG_OVERFLOW: return "replay log overflow";
    case GDN_ERR_ROLLBACK_RANGE: return "rollback count out of range";
    case GDN_ERR_WORKSPACE: return "workspace missing or too small";
    case GDN_ERR_CUDA: return "CUDA runtime error";
    case GDN_ERR_PAGE_RANGE: return "page id outside the pool";
    case GDN_ERR_TIMEOUT: return "bounded device wait ran out";
    default: return "unknown status";
  }
}

int32_t gdn_version(void) { return 100; /* 0.1.0 */ }

static int desc_ok(const gdn_layer_desc* d) {
  if (!d) return 0;
  if (d->num_qk_heads <= 0 || d->num_v_heads <= 0) return 0;
  if (d->num_v_heads % d->num_qk_heads != 0) return 0;
  if (d->head_dim_k <= 0 || d->head_dim_v <= 0) return 0;
  if (d->conv_kernel < 1) return 0;
  if (d->in_dtype != GDN_F32 && d->in_dtype != GDN_BF16) return 0;
  if (d->out_dtype != GDN_F32 && d->out_dtype != GDN_BF16) return 0;
  return 1;
}

int64_t gdn_conv_dim(const gdn_layer_desc* d) {
  if (!desc_ok(d)) return -1;
  return 2 * (int64_t)d->num_qk_heads * d->head_dim_k +
         (int64_t)d->num_v_heads * d->head_dim_v;
}

int64_t gdn_mamba_page_bytes(const gdn_layer_desc* d) {
  if (!desc_ok(d)) return -1;
  int64_t state = (int64_t)d->num_v_heads * d->head_dim_v * d->head_dim_k * 4;
  int64_t elem = d->in_dtype == GDN_BF16 ? 2 : 4;
  int64_t window = (int64_t)(d->conv_kernel - 1) * gdn_conv_dim(d) * elem;
  return state + window;
}

int64_t gdn_block_size_for(int64_t mamba_page_bytes, int64_t attn_bytes_per_token,
                           int32_t alignment) {
  if (mamba_page_bytes <= 0 || attn_bytes_per_token <= 0 || alignment <= 0) return -1;
  return (int64_t)alignment *
         cdiv64(mamba_page_bytes, (int64_t)alignment * attn_bytes_per_token);
}

int64_t gdn_mamba_pages_per_request(int32_t num_gdn_layers, int32_t prefix_caching,
                                    int32_t num_spec_tokens) {
  if (num_gdn_layers < 0 || num_spec_tokens < 0) return -1;
  if (prefix_caching != 0 && prefix_caching != 1) return -1;
  return (int64_t)num_gdn_layers * (1 + prefix_caching + num_spec_tokens);
}

int64_t gdn_pool_blocks_for_pages(int64_t pages, int32_t layers_per_block) {
  if (pages < 0 || layers_per_block <= 0) return -1;
  return cdiv64(pages, layers_per_block);
}

int64_t gdn_chunk_end(int64_t num_computed, int64_t num_tokens, int64_t token_budget,
                      int32_t block_size) {
  if (num_computed < 0 || num_tokens < num_computed || token_budget < 0 || block_size <= 0)
    return -1;
  if (num_tokens - num_computed <= token_budget) return num_tokens;
  int64_t end = (num_computed + token_budget) / block_size * block_size;
  return end > num_computed ? end : num_computed;
}

int64_t gdn_cached_tokens(int64_t shared_tokens, int32_t block_size) {
  if (shared_tokens < 0 || block_size <= 0) return -1;
  int64_t full = shared_tokens / block_size;
  return full >= 2 ? (full - 1) * block_size : 0;
}

int32_t gdn_replay_boundary_rows(int64_t absorbed, int32_t kept, int32_t block_size) {
  if (absorbed < 0 || kept < 0 || block_size <= 0) return -1;
  /* first multiple of block_size above absorbed */
  const int64_t first = (absorbed / block_size + 1) * block_size;
  if (first > absorbed + kept) return 0;
  if (first + block_size <= absorbed + kept) return -1;   /* a second boundary */
  return (int32_t)(first - absorbed);
}

gdn_status gdn_resume_block(int64_t hit_tokens, int32_t block_size, int32_t* out_block) {
  if (!out_block || hit_tokens < 0 || block_size <= 0) return GDN_ERR_INVALID_ARG;
  if (hit_tokens % block_size != 0) return GDN_ERR_NOT_BLOCK_ALIGNED;
  int64_t k = hit_tokens / block_size;
  if (k - 1 > INT32_MAX) return GDN_ERR_INVALID_ARG;
  *out_block = (int32_t)(k - 1);
  return GDN_OK;
}

int64_t gdn_spec_copy_bytes(int32_t draft_tokens, int32_t num_gdn_layers, int64_t page_bytes) {
  if (draft_tokens < 0 || num_gdn_layers < 0 || page_bytes < 0) return -1;
  return (int64_t)(draft_tokens + 1) * num_gdn_layers * page_bytes;
}

int64_t gdn_replay_bytes_per_request(int32_t num_gdn_layers, int64_t page_bytes,
                                     int32_t log_slots, int64_t slot_bytes) {
  if (num_gdn_layers < 0 || page_bytes < 0 || log_slots < 0 || slot_bytes < 0) return -1;
  return (int64_t)num_gdn_layers * (page_bytes + (int64_t)log_slots * slot_bytes);
}
