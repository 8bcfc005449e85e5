// launch.h — internal launchers behind the C ABI (not exported).
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "scan.cuh"

namespace gdn {

struct DecodeParams {
  Pool pool;
  int32_t Hqk, Hv, conv_dim, num_seqs;
  float q_scale, eps;
  const void* x;
  const float* g;
  const float* beta;
  const float* conv_w;
  const int32_t* slot;
  void* o;
  int32_t* err;
  // mixed batches: the token row of sequence s in x, g, beta and o (nullptr:
  // row s), and the regime of each sequence (nullptr: every sequence
  // decodes; 0 = a prefill sequence, skipped here)
  const int32_t* row;
  const int8_t* decode;
  // packed core: x rows are q | k | v | z, x_ld elements apart; the gates come
  // from the b | a rows with A_log and dt_bias; the outputs are gated-normalised
  int32_t x_ld;
  const void* ba;        // nullptr: plain rows (g, beta given, outputs as they are)
  const float* A_log;
  const float* dt_bias;
  const float* norm_w;
  float norm_eps2;
};

struct CopyParams {
  Pool pool;
  int64_t payload_bytes;
  const int32_t* src;
  const int32_t* dst;
  int32_t n;
  int32_t* err;
};

// Workspace bytes of the conv pre-pass for `rows` token rows.
size_t scan_workspace_bytes(int64_t rows, int conv_dim, int Hqk, int Hv);
// p.ws_* must be bound (bind_workspace) before the launchers run.
void bind_workspace(ScanParams& p, void* ws, int64_t rows);

// workspace: the tensor-core shapes take the two-kernel prefill when it is
// given (nullptr: the fused kernel); the scan path reads p.ws_* (bound).
cudaError_t launch_prefill(const ScanParams& p, void* workspace, int64_t max_len, int dk, int dv, int in_dtype,
                           int out_dtype, cudaStream_t st);
cudaError_t launch_replay_append(const ScanParams& p, int dk, int dv, int in_dtype,
                                 int out_dtype, cudaStream_t st);
cudaError_t launch_replay_flush(const ScanParams& p, int dk, int dv, int in_dtype,
                                int out_dtype, cudaStream_t st);
cudaError_t launch_replay_rollback(int32_t* log_len, const int32_t* accepted, int32_t num_appended,
                                   int32_t n, int32_t* err, cudaStream_t st);
// Packed core: g and beta of `rows` rows from the b | a rows.
cudaError_t launch_core_gates(const void* ba, int in_dtype, const float* A_log, const float* dt_bias, int Hv,
                              int64_t rows, float* g, float* beta, cudaStream_t st);
cudaError_t launch_decode(const DecodeParams& p, int dk, int dv, int in_dtype, int out_dtype,
                          cudaStream_t st);
cudaError_t launch_copy(const CopyParams& p, cudaStream_t st);
// Tensor-core replay (dk = dv = 128, bf16 inputs).  Flush: the state update
// and the v windows, then a per-request pass for the q / k windows and
// log_len.  Append: outputs of the new rows and the log rows, then log_len.
bool tc_replay_supported(int dk, int dv, int in_dtype);
// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda); nullptr if the driver lacks it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
cudaError_t launch_tc_flush(const ScanParams& p, cudaStream_t st);
cudaError_t launch_tc_append(const ScanParams& p, cudaStream_t st);
// Tensor-core chunked prefill (dk = dv = 128, bf16 in and out, block size a
// multiple of 64), followed by the window pass; needs no workspace.  The
// (sequence, value head) chains run whole in one launch, or cut into pieces
// of `piece` chunks over several launches (tc_prefill_schedule).
struct PrefillSchedule {
  int64_t nchains;    // value heads x sequences
  int64_t piece;      // chunks per piece (the last level runs to the end)
  int64_t levels;     // pieces per chain of max_len tokens
  int64_t width;      // CTAs per launch
  int64_t launches;   // chain (or fused-kernel) launches
  // the two-kernel path: chunk-kernel launches.  Above 1, level l of every
  // chain runs on a second stream as soon as the chunk kernel's launch l
  // (that level's chunks) is done, while launch l + 1 takes the SMs the
  // chains leave idle.
  int64_t chunk_launches;
};
PrefillSchedule tc_prefill_schedule(int Hv, int num_seqs, int64_t max_len, int sms);
// The same plan with a launch's fixed cost given in chunk times.
PrefillSchedule tc_prefill_schedule_cost(int Hv, int num_seqs, int64_t max_len, int sms, double launch_cost);
int tc_prefill_sm_count();   // SMs of the current device (0 if unknown: one launch)
bool tc_prefill_supported(int dk, int dv, int in_dtype, int out_dtype, int block_size);
cudaError_t launch_tc_prefill(const ScanParams& p, int64_t max_len, cudaStream_t st);
// z CTAs of the prefill's window pass: one per block boundary a sequence of
// up to max_len tokens can cross (at least 1, at most 1,024; any count covers
// every boundary, the count sets how many are written at once)
inline unsigned window_slices(const ScanParams& p, int64_t max_len) {
  const int64_t b = p.block_size > 0 && max_len > 0 ? max_len / p.block_size + 1 : 1;
  return (unsigned)(b < 1 ? 1 : b > 1024 ? 1024 : b);
}
// The same prefill as two kernels (tc_chain.cu): the state-independent chunk
// kernel over every chunk of the call, writing operand images to the
// workspace, then the chain kernel (in pieces, as tc_chain_schedule plans),
// then the window pass.  The workspace holds tc_chain_workspace_bytes (with
// core: also the packed core's fp32 outputs before their gated norm).
size_t tc_chain_workspace_bytes(int Hqk, int Hv, int32_t num_seqs, int64_t total_tokens, bool core = false);
PrefillSchedule tc_chain_schedule(int Hqk, int Hv, int num_seqs, int64_t max_len, int sms);
cudaError_t launch_tc_prefill2(const ScanParams& p, void* workspace, int64_t max_len, cudaStream_t st);
// Whether the two kernels beat the fused one for a call of num_seqs sequences
// of at most max_len tokens on `sms` SMs (both give the same bits).
bool tc_prefill_two_kernels_faster(int Hqk, int Hv, int num_seqs, int64_t max_len, int sms);

}  // namespace gdn
