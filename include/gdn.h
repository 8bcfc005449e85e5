/*
 * gdn.h — C ABI of the Gated DeltaNet recurrent-state engine (sm_103a).
 *
 * What the engine computes
 * ------------------------
 * One Gated DeltaNet (GDN) layer keeps, per sequence and per value head h, a
 * fixed-size fp32 state S (dv rows x dk columns) and a rolling window of the
 * last three pre-convolution input rows.  Each token t runs
 *
 *   y      = SiLU( sum_{i=0..3} w[c][i] * x[t-3+i][c] )      per channel c
 *   q, k   = L2-normalised q and k slices of y (q also times q_scale)
 *   v      = v slice of y;  a = exp(g[t][h]);  b = beta[t][h]
 *   S_t    = a * S_{t-1} (I - b k k^T) + b v k^T
 *   o_t    = S_t q
 *
 * the gated delta rule (Yang, Kautz, Hatamizadeh, "Gated Delta Networks:
 * Improving Mamba2 with Delta Rule", 2024) preceded by the depthwise causal
 * convolution of kernel 4 whose three-row history is carried as conv state
 * ("Hybrid linear attention (gated DeltaNet)", section "Why this family is
 * different", item 1: a rolling convolution state plus a recurrent state of
 * fixed size).  Channels of y are ordered [q heads | k heads | v heads]; value
 * head h reads qk head floor(h / (Hv / Hqk)).
 *
 * Paged state pool
 * ----------------
 * A pool is a device array of equally sized pages.  A page holds one layer's
 * full GDN state ("mamba page"):
 *
 *   offset 0                     : S, fp32 [Hv][dv][dk]  (dk contiguous)
 *   offset Hv*dv*dk*4            : conv window, in_dtype [3][conv_dim]
 *                                  (row 0 = oldest of the three rows)
 *   rest up to page_bytes        : padding, never read or written
 *
 * with conv_dim = 2*Hqk*dk + Hv*dv.  Page p starts at base + p*page_bytes;
 * base and page_bytes must be multiples of 256 bytes.  A block table row maps
 * a sequence's logical block index j to the page holding the checkpoint taken
 * after (j+1)*block_size tokens ("Prefix caching on Gated DeltaNet hybrids",
 * section "Why hits were wrong": a full block keeps the state after its last
 * token, so a hit at k*block tokens resumes from block k-1).  Entry -1 means
 * "no page for this block": the checkpoint is skipped.
 *
 * Ownership, threading and errors
 * -------------------------------
 * The caller owns every buffer (pool, inputs, outputs, metadata, error word)
 * and every stream.  The library allocates no device or host memory and keeps
 * no global state, with one exception: gdn_prefill_chunked_noalloc's scratch,
 * a fixed device array of GDN_NOALLOC_SCRATCH_BYTES in the library's own
 * image (and the device addresses of it the library caches), held by every
 * GPU that loads the library.  All entry points are asynchronous and
 * stream-ordered, and may be called from several host threads on different
 * streams.
 * Host-detectable errors (bad shapes, null pointers, an off-boundary resume
 * visible in a host-side array) are returned before anything is launched.
 * Errors that only the device can see (a page id outside the pool, a log
 * overflow, a rollback out of range) are recorded with atomicCAS into the
 * caller's int32 error word (first error wins) and the offending sequence's
 * writes are skipped; kernels never trap.  The caller reads the word after
 * synchronising the stream.  Device pointers are plain CUDA device addresses;
 * every array is dense and row-major in the order its comment lists.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t gdn_status;

enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,       /* null pointer, negative count, bad enum   */
  GDN_ERR_UNSUPPORTED_SHAPE = 2, /* head dims / counts the kernels lack      */
  GDN_ERR_NOT_BLOCK_ALIGNED = 3, /* resume or save off a block boundary      */
  GDN_ERR_PARTIAL_BLOCK = 4,     /* copy of a block that is not yet full     */
  GDN_ERR_LOG_OVERFLOW = 5,      /* replay log would exceed its slots        */
  GDN_ERR_ROLLBACK_RANGE = 6,    /* accepted count outside [0, appended]     */
  GDN_ERR_WORKSPACE = 7,         /* workspace missing or too small           */
  GDN_ERR_CUDA = 8,              /* a CUDA runtime call failed               */
  GDN_ERR_PAGE_RANGE = 9,        /* page or slot id outside the pool         */
  GDN_ERR_TIMEOUT = 10           /* a bounded device-side wait ran out       */
};

enum { GDN_F32 = 0, GDN_BF16 = 1 };

/* Longest replay input log, in rows ("Caching less to serve more requests",
 * section "What we changed": one state plus a 32-slot input buffer). */
#define GDN_REPLAY_LOG_SLOTS 32

/* Shape of one GDN layer. */
typedef struct gdn_layer_desc {
  int32_t num_qk_heads;  /* Hqk                                              */
  int32_t num_v_heads;   /* Hv, a multiple of Hqk                            */
  int32_t head_dim_k;    /* dk: 32, 64 or 128                                */
  int32_t head_dim_v;    /* dv: 32, 64 or 128                                */
  int32_t conv_kernel;   /* must be 4                                        */
  int32_t block_size;    /* B: tokens per cache block (checkpoint spacing)   */
  int32_t chunk_size;    /* C: scan chunk; 16, 32 or 64 and divides B        */
  int32_t in_dtype;      /* GDN_F32 or GDN_BF16: x, conv window, replay log  */
  int32_t out_dtype;     /* GDN_F32 or GDN_BF16: o                           */
  float q_scale;         /* q is multiplied by this after L2 normalisation   */
  float norm_eps;        /* q <- q / sqrt(sum q^2 + norm_eps), same for k    */
  int32_t reserved;      /* must be 0                                        */
} gdn_layer_desc;

/* A pool of state pages in device memory (see the page layout above). */
typedef struct gdn_pool {
  void* base;            /* device, 256-byte aligned                         */
  int64_t page_bytes;    /* >= gdn_mamba_page_bytes(desc), multiple of 256   */
  int32_t num_pages;
  int32_t reserved;
} gdn_pool;

const char* gdn_status_string(gdn_status s);
/* Library version as major*10000 + minor*100 + patch. */
int32_t gdn_version(void);

/* ---------------------------------------------------------------------------
 * Host arithmetic: pure, exact integer functions (no device work).
 * ------------------------------------------------------------------------- */

/* conv_dim = 2*Hqk*dk + Hv*dv; -1 if desc is NULL or malformed. */
int64_t gdn_conv_dim(const gdn_layer_desc* desc);

/* Bytes of one layer's GDN state: Hv*dv*dk*4 (fp32 state) plus
 * (conv_kernel-1)*conv_dim*sizeof(in_dtype) (conv window).  27B-shaped layer
 * (Hqk 16, Hv 48, d 128, bf16 window): 3,207,168 B = 3.06 MiB
 * ("Hybrid linear attention (gated DeltaNet)", "Why this family is
 * different", items 1-2; "Prefix caching on Gated DeltaNet hybrids", "Why
 * hits were wrong").  -1 if desc is malformed. */
int64_t gdn_mamba_page_bytes(const gdn_layer_desc* desc);

/* Smallest block size, a multiple of `alignment`, whose attention page
 * (block * attn_bytes_per_token) covers one mamba page:
 *   alignment * ceil(mamba_page_bytes / (alignment * attn_bytes_per_token)).
 * ("Hybrid linear attention (gated DeltaNet)", "Why this family is
 * different", item 2: 16 * cdiv(3,207,168, 16 * 4,096) = 784.)  Returns -1
 * for non-positive arguments. */
int64_t gdn_block_size_for(int64_t mamba_page_bytes, int64_t attn_bytes_per_token,
                           int32_t alignment);

/* Pages one request holds per GDN layer in a shared pool: 1 + num_spec with
 * prefix caching off, 2 + num_spec with it on (the state being written plus
 * the last block-boundary checkpoint), times num_gdn_layers.  Same section,
 * item 2 (48 layers x 2 pages = 96 pages).  -1 for bad arguments. */
int64_t gdn_mamba_pages_per_request(int32_t num_gdn_layers, int32_t prefix_caching,
                                    int32_t num_spec_tokens);

/* Pool blocks those pages occupy when one block carries one page for each of
 * `layers_per_block` layers: ceil(pages / layers_per_block).  Reading of the
 * same item ("96 page(s) per request -> 6 block(s)" with 16-layer groups).
 * -1 for bad arguments. */
int64_t gdn_pool_blocks_for_pages(int64_t pages, int32_t layers_per_block);

/* End (exclusive token index) of the next prefill chunk under block-aligned
 * chunking: num_tokens if the rest fits in token_budget (the final chunk may
 * end inside a block); otherwise the largest multiple of block_size not above
 * num_computed + token_budget; num_computed itself (nothing schedulable) when
 * that multiple does not advance.  ("Hybrid linear attention (gated
 * DeltaNet)", item 3: 784 or 1568 of a 2048 budget, never 2048; "Prefix
 * caching on Gated DeltaNet hybrids", "Limits": 896 of a 1024 budget.)
 * -1 for bad arguments. */
int64_t gdn_chunk_end(int64_t num_computed, int64_t num_tokens, int64_t token_budget,
                      int32_t block_size);

/* Tokens a shared prefix returns from the cache when partial blocks are not
 * stored and the last full block stays open:
 *   max(0, floor(shared/block) - 1) * block
 * ("The cache block that is not a cache setting", "What that costs,
 * exactly"); below two blocks nothing caches.  -1 for bad arguments. */
int64_t gdn_cached_tokens(int64_t shared_tokens, int32_t block_size);

/* Block whose checkpoint a prefix hit of hit_tokens resumes from:
 * k*B -> k-1, 0 -> -1 (cold start); any other count -> GDN_ERR_NOT_BLOCK_ALIGNED
 * ("Prefix caching on Gated DeltaNet hybrids", "Why hits were wrong" and
 * "The in-page layout": fail closed on a resume off a block boundary). */
gdn_status gdn_resume_block(int64_t hit_tokens, int32_t block_size, int32_t* out_block);

/* Kept rows after which a replay flush crosses a block boundary: a request
 * whose checkpoint has absorbed `absorbed` tokens flushes `kept` logged rows,
 * and the state after the first j of them lies on a block boundary when
 * absorbed + j is a positive multiple of block_size.  Returns that j in
 * [1, kept], or 0 when no boundary is crossed; -1 for bad arguments or when
 * the rows cross more than one boundary (the flush writes one boundary
 * checkpoint; flush earlier).  ("Prefix caching on Gated DeltaNet hybrids",
 * "The in-page layout": a block's checkpoint is the state at its boundary;
 * "Caching less to serve more requests", "Other models": serving the replay
 * scheme with prefix caching.) */
int32_t gdn_replay_boundary_rows(int64_t absorbed, int32_t kept, int32_t block_size);

/* Bytes that per-position speculative state copies take for one request:
 * (draft_tokens + 1) * num_gdn_layers * page_bytes ("Caching less to serve
 * more requests", "Where the memory goes": (15+1) x 24 x 2.5 MiB = 960 MiB). */
int64_t gdn_spec_copy_bytes(int32_t draft_tokens, int32_t num_gdn_layers, int64_t page_bytes);

/* Bytes of the replay scheme for one request: one page plus log_slots input
 * rows of slot_bytes per layer: num_gdn_layers * (page_bytes + log_slots *
 * slot_bytes) (same page, "What we changed": 72 MiB over 24 layers). */
int64_t gdn_replay_bytes_per_request(int32_t num_gdn_layers, int64_t page_bytes,
                                     int32_t log_slots, int64_t slot_bytes);

/* ---------------------------------------------------------------------------
 * Device entry points.  All pointers are device pointers unless the field
 * name ends in _host.  `stream` is a cudaStream_t passed as void*.
 * ------------------------------------------------------------------------- */

/* Chunked prefill of N sequences, packed along the token axis.
 *
 * For sequence s the call consumes tokens [cu_seqlens[s], cu_seqlens[s+1])
 * of x/g/beta, which sit at absolute positions start_pos[s] ... of that
 * sequence.  The initial state and conv window come from page init_page[s]
 * (a resume: start_pos[s] must then be a positive multiple of block_size), or
 * are zero when init_page[s] == -1 (a cold start: start_pos[s] must be 0; the
 * pool is never read, so stale or NaN pages cannot leak in).  For every block
 * boundary P = (j+1)*block_size with start_pos < P <= start_pos + n_s the
 * state and conv window after token P are written to page block_table[s][j]
 * (skipped when that entry is -1): every crossed boundary is checkpointed,
 * also inside one call ("The prefix cache changed the answer", section "The
 * fix: one line").  The state after the last token goes to page out_slot[s],
 * which may equal init_page[s]; during the call the page may also hold the
 * state between launches (gdn_prefill_plan_for), so, as for any page
 * the call writes, no other sequence of the call may read or write it.  o
 * receives S_t q_t for every token.
 *
 * Determinism: results depend only on a sequence's own inputs, never on the
 * batch, the call's length or where earlier calls split the sequence; a
 * resume from a checkpoint reproduces the cold run bit for bit. */
typedef struct gdn_prefill_args {
  int32_t num_seqs;              /* N >= 0                                    */
  int32_t max_blocks;            /* row stride of block_table                 */
  int64_t total_tokens;          /* T = cu_seqlens[N]                         */
  int64_t max_seq_len;           /* host bound on any cu_seqlens[s+1] -
                                    cu_seqlens[s] (0: T); sizes the grid.  A
                                    longer sequence sets GDN_ERR_INVALID_ARG
                                    on the two-kernel path                    */
  const int32_t* cu_seqlens;     /* [N+1], non-decreasing, cu_seqlens[0] = 0  */
  const int64_t* start_pos;      /* [N] absolute position of the first token  */
  const int64_t* start_pos_host; /* optional host copy of start_pos ([N]) for
                                    pre-launch block-alignment checks         */
  const int32_t* init_page_host; /* optional host copy of init_page ([N])     */
  const void* x;                 /* [T][conv_dim] in_dtype, pre-conv rows     */
  const float* g;                /* [T][Hv] log decay (a = exp(g))            */
  const float* beta;             /* [T][Hv] write strength b                  */
  const float* conv_w;           /* [conv_dim][4]; tap 3 hits the current row */
  const int32_t* init_page;      /* [N] page id or -1 (cold)                  */
  const int32_t* block_table;    /* [N][max_blocks] page id or -1             */
  const int32_t* out_slot;       /* [N] page receiving the final state        */
  void* o;                       /* [T][Hv][dv] out_dtype                     */
  int32_t* dev_error;            /* one int32, set to a gdn_status on a fault */
  int64_t wait_cycles;           /* bound of each device-side wait of the
                                    tensor-core prefill in SM clocks; 0: the
                                    default (~2 s).  A wait that runs out sets
                                    GDN_ERR_TIMEOUT (over any earlier code);
                                    the call then writes no further states,
                                    checkpoints or windows.  < 0 makes every
                                    such wait report a timeout at once (a test
                                    of that path: nothing is written)         */
  int32_t path;                  /* GDN_PREFILL_AUTO (0), _FUSED or
                                    _TWO_KERNELS (tensor-core layers; see
                                    gdn_prefill_workspace_size)               */
  int32_t reserved;              /* 0                                         */
} gdn_prefill_args;

/* How a tensor-core layer's prefill runs (both give the same bits). */
enum { GDN_PREFILL_AUTO = 0, GDN_PREFILL_FUSED = 1, GDN_PREFILL_TWO_KERNELS = 2 };

/* Device workspace bytes gdn_prefill_chunked needs for a call of num_seqs
 * sequences with total_tokens tokens.
 *
 * Layers on the tensor cores (dk = dv = 128, bf16 in and out, block_size a
 * multiple of 64) run the prefill as two kernels when given this workspace:
 * a chunk kernel computes, for every 64-token chunk of the call at once,
 * everything that does not depend on the state (conv, norms, the chunk's
 * triangular solve and the products that fold it in) and leaves them here as
 * the fused kernel's own operand images (about 97 KB per chunk and value
 * head plus 64 KB per chunk and qk head; the 32 KB of v in that is written
 * only when the chains' levels overlap the chunk kernel, otherwise the chain
 * convolves v from the rows itself); a chain kernel then carries each
 * (sequence, value head) state through its chunks with the fused kernel's
 * state products.  The other path is one fused kernel that runs a chain's
 * chunks one after another on one SM and needs no scratch.  Both split and
 * multiply every operand alike and give the same bits, so the choice is
 * speed only: on a GB300 the two kernels win for long prompts (most for
 * one or two sequences, whose few chains leave SMs idle) and for batches of
 * 8,192-token sequences, the fused kernel for short calls of a few
 * sequences, where the second launch and the chunk kernel's fixed cost do
 * not pay.  With GDN_PREFILL_AUTO a call takes
 * the two kernels when it has a workspace and a model of both paths' times
 * (gdn_prefill_plan_for) favours them; a call without a workspace (NULL,
 * workspace_bytes 0) takes the fused kernel.
 *
 * Other layers run a conv pre-pass whose SiLU(conv) rows (fp32, computed
 * once and shared by every head that reads them), q / k norm factors and
 * gates live here; they need it.
 *
 * The caller allocates it (256-byte aligned); its contents are scratch,
 * overwritten by every call, so calls that share a workspace must not
 * overlap on the GPU.  0 for a malformed desc. */
size_t gdn_prefill_workspace_size(const gdn_layer_desc* desc, int32_t num_seqs,
                                  int64_t total_tokens);

/* How gdn_prefill_chunked runs a call of a layer on the tensor-core path:
 * the path (two_kernels; `path` GDN_PREFILL_AUTO resolves it as a call with
 * a workspace would) and the chain plan of that path.  Each (sequence, value
 * head) chain runs on one SM, its chunks in order.  With at least as many
 * chains as SMs and long chains, whole chains would leave SMs idle in the
 * last round, so the chains are cut
 * into pieces of piece_chunks chunks and run as `launches` launches of up to
 * ctas_per_launch CTAs: all chains' first pieces, then all second pieces, and
 * so on, ctas_per_launch at a time (a piece starts from the state the piece
 * before it left in page out_slot[s]; the last piece of a chain runs to its
 * end).  Every chunk's arithmetic is unchanged, so the results are bitwise
 * those of one launch.  One launch (levels = 1) is kept unless pieces save
 * an estimated 5 %.  The two-kernel path with no more chains than SMs and
 * chains of at least 32 chunks cuts every chain into levels of an even 16 to
 * 64 chunks (about 32 levels, at most 64) and overlaps them with the chunk
 * kernel (chunk_launches below).  The second stream and its two events are
 * made once per device, on the first such call, and kept for the process; a
 * first such call made while its stream captures a graph, or one for which
 * they cannot be made, runs its levels on its own stream alone instead (the
 * same bits), and later captures record the fork and the join. */
typedef struct gdn_prefill_plan {
  int64_t chains;           /* num_v_heads x num_seqs                        */
  int64_t piece_chunks;     /* chunks (64 tokens) per piece                  */
  int64_t levels;           /* pieces per chain of max_seq_len tokens        */
  int64_t ctas_per_launch;  /* CTAs of each launch (the last may have fewer) */
  int64_t launches;         /* chain launches (+1 window pass)              */
  int64_t two_kernels;      /* 1: the chunk + chain kernels, 0: the fused one */
  int64_t chunk_launches;   /* two-kernel path: chunk-kernel launches, 0 on
                               the fused path.  Above 1 the levels overlap:
                               level l of every chain runs on a second,
                               high-priority stream once the chunk kernel's
                               launch l (chunks [l x piece_chunks, +piece_chunks)
                               of every sequence) is done, while its launch
                               l + 1 runs on the SMs the chains leave idle;
                               the call's stream waits for the last level   */
} gdn_prefill_plan;

/* The plan of one gdn_prefill_chunked call with num_seqs sequences and the
 * call's max_seq_len (its total_tokens when max_seq_len is 0) on a GPU with
 * num_sms SMs (<= 0: the current device's count, as the call reads it).
 * Host-only; launches nothing.  GDN_ERR_UNSUPPORTED_SHAPE for a layer on the
 * conv pre-pass path, GDN_ERR_INVALID_ARG for a malformed argument. */
gdn_status gdn_prefill_plan_for(const gdn_layer_desc* desc, int32_t num_seqs, int64_t max_seq_len,
                                int32_t num_sms, int32_t path, gdn_prefill_plan* out);

gdn_status gdn_prefill_chunked(const gdn_layer_desc* desc, const gdn_pool* pool,
                               const gdn_prefill_args* args, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Allocation-free variant of gdn_prefill_chunked.  It has no counterpart on
 * the pages; it exists for callers that cannot provide device memory for the
 * workspace when they call the prefill: a serving runtime that reserved the
 * GPU's free memory for its state and KV pools at start-up (a later
 * cudaMalloc would fail or fragment those pools), or a C caller embedded in
 * another framework without an allocator of its own.
 *
 * Same arguments and results as gdn_prefill_chunked, minus the workspace: the
 * scratch is a fixed array of GDN_NOALLOC_SCRATCH_BYTES (64 MiB) in this
 * library's device memory, held by every GPU that loads the library until the
 * process exits.  Calls whose gdn_prefill_workspace_size exceeds it return
 * GDN_ERR_WORKSPACE and launch nothing (layers on the conv pre-pass path:
 * about 3,200 tokens per call at d = 64 with 16 / 48 heads; split longer
 * prefills at block boundaries, gdn_chunk_end).  Layers on the tensor-core
 * path need no scratch and have no limit.
 * The entry point calls no cudaMalloc, cudaFree or other allocating routine.
 * A call whose layer needs no scratch (gdn_prefill_workspace_size 0) goes
 * straight to gdn_prefill_chunked and never touches the array.  The first
 * call on a device that does need it looks up the array's device address
 * with cudaGetSymbolAddress (that device current); make that first call
 * before any stream capture.  Every call shares the one array and it keeps the last
 * call's contents (the kernels write every element they read, so nothing is
 * cleared): calls that overlap on the GPU, on any streams, race. */
#define GDN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
gdn_status gdn_prefill_chunked_noalloc(const gdn_layer_desc* desc, const gdn_pool* pool,
                                       const gdn_prefill_args* args, void* stream);

/* Batched single-token decode: for each sequence s the state and conv window
 * in page slot[s] advance by one token in place and o[s] = S_t q_t
 * ("Hybrid linear attention (gated DeltaNet)", "The part that is easy to get
 * wrong": the gdn_conv_decode + gdn_decode pair, fused here). */
typedef struct gdn_decode_args {
  int32_t num_seqs;              /* N >= 0; slots must be distinct            */
  int32_t reserved;
  const void* x;                 /* [N][conv_dim] in_dtype                    */
  const float* g;                /* [N][Hv]                                   */
  const float* beta;             /* [N][Hv]                                   */
  const float* conv_w;           /* [conv_dim][4]                             */
  const int32_t* slot;           /* [N] page ids                              */
  void* o;                       /* [N][Hv][dv] out_dtype                     */
  int32_t* dev_error;
} gdn_decode_args;

gdn_status gdn_decode_step(const gdn_layer_desc* desc, const gdn_pool* pool,
                           const gdn_decode_args* args, void* stream);

/* Packed core ("Hybrid linear attention (gated DeltaNet)", "Packed-core
 * traces"): the input rows are packed q | k | v | z and b | a, the output
 * rows are gated-normalised values; the core owns the conv taps, dt_bias,
 * A_log (float32) and the norm scale.  The pages name the weights only; the
 * library reads them as
 *   g    = -exp(A_log[h]) * softplus(a[h] + dt_bias[h])    (the decay is exp(g))
 *   beta = sigmoid(b[h])
 *   y    = o / sqrt(mean_dv(o^2) + norm_eps) * norm_w * silu(z)   per token and v head,
 * with o the output of the plain step. */
typedef struct gdn_core_args {
  const void* ba;                /* [rows][2*Hv] in_dtype: b | a per v head   */
  const float* A_log;            /* [Hv]                                      */
  const float* dt_bias;          /* [Hv]                                      */
  const float* norm_w;           /* [dv], shared by the heads                 */
  float norm_eps;
  int32_t reserved;
} gdn_core_args;

/* Device workspace of gdn_core_prefill: the gates of every row (fp32,
 * 2 x 4 x T x Hv bytes rounded up to 256), then, on the tensor-core path,
 * the two kernels' operand images (as gdn_prefill_workspace_size) and a
 * T x Hv x dv fp32 buffer where the chains leave the outputs before the
 * gated norm when the chain levels overlap the chunk launches.  A
 * workspace of the gates alone (at least that many bytes, less than this
 * size) runs the fused kernel; with this size, GDN_PREFILL_AUTO chooses as
 * gdn_prefill_chunked does.  Both paths give the same bits. */
size_t gdn_core_prefill_workspace_size(const gdn_layer_desc* desc, int32_t num_seqs, int64_t total_tokens);

/* gdn_prefill_chunked on packed rows: args->x is [T][conv_dim + Hv*dv]
 * in_dtype (q | k | v | z; the conv and the windows use the first conv_dim
 * channels), args->g and args->beta are ignored (may be NULL), args->o
 * receives y.  States, checkpoints and windows are those of the plain
 * prefill on the same q | k | v rows and gates.  args->path chooses between
 * the fused kernel and the two kernels as for gdn_prefill_chunked
 * (GDN_PREFILL_TWO_KERNELS needs the full gdn_core_prefill_workspace_size,
 * else GDN_ERR_WORKSPACE).  Layers on the tensor-core path only (dk = dv =
 * 128, bf16, block a multiple of 64), else GDN_ERR_UNSUPPORTED_SHAPE. */
gdn_status gdn_core_prefill(const gdn_layer_desc* desc, const gdn_pool* pool, const gdn_prefill_args* args,
                            const gdn_core_args* core, void* workspace, size_t workspace_bytes, void* stream);

/* gdn_decode_step on packed rows: args->x is [N][conv_dim + Hv*dv]
 * (q | k | v | z), args->g / args->beta are ignored, args->o receives y. */
gdn_status gdn_core_decode(const gdn_layer_desc* desc, const gdn_pool* pool, const gdn_decode_args* args,
                           const gdn_core_args* core, void* stream);

/* Mixed batch: prefill sequences and single decode tokens packed in one
 * varlen batch, in one call ("Hybrid linear attention (gated DeltaNet)", "The
 * part that is easy to get wrong": in the mixed regime the prefill kernels
 * run on the prefill sequences and gdn_decode_mixed on the decode tokens).
 * Sequence s owns rows [cu_seqlens[s], cu_seqlens[s+1]) of x, g, beta and o.
 * is_decode[s] = 1: exactly one row; the state and window in page slot[s]
 * advance by that token in place (gdn_decode_step's step; start_pos,
 * init_page and its block_table row are ignored).  is_decode[s] = 0: the
 * sequence is prefilled as by gdn_prefill_chunked, with slot[s] as out_slot.
 * Both parts run on `stream`, the prefill kernels first; every sequence gets
 * exactly the bits of the corresponding separate call.
 *
 * Host checks (GDN_ERR_INVALID_ARG unless noted, nothing launched): the host
 * copies of cu_seqlens and is_decode are required; a decode entry must have
 * exactly one row; prefill entries are checked as in gdn_prefill_chunked
 * (GDN_ERR_NOT_BLOCK_ALIGNED, GDN_ERR_PAGE_RANGE), and the workspace is
 * gdn_mixed_workspace_size bytes (0 on the tensor-core path). */
typedef struct gdn_mixed_args {
  int32_t num_seqs;              /* N >= 0                                    */
  int32_t max_blocks;            /* columns of block_table                    */
  int64_t total_tokens;          /* rows of x, g, beta, o                     */
  int64_t max_seq_len;           /* longest sequence, or 0 (= total_tokens)   */
  const int32_t* cu_seqlens;     /* [N+1] device                              */
  const int32_t* cu_seqlens_host;/* [N+1] host                                */
  const int8_t* is_decode;       /* [N] device: 1 decode token, 0 prefill     */
  const int8_t* is_decode_host;  /* [N] host copy                             */
  const int64_t* start_pos;      /* [N] device (prefill entries)              */
  const int64_t* start_pos_host; /* [N] host copy or NULL                     */
  const int32_t* init_page;      /* [N] device (prefill entries), -1 = cold   */
  const int32_t* init_page_host; /* [N] host copy or NULL                     */
  const int32_t* block_table;    /* [N][max_blocks] (prefill entries)         */
  const int32_t* slot;           /* [N] prefill: out_slot; decode: its page   */
  const void* x;                 /* [T][conv_dim] in_dtype                    */
  const float* g;                /* [T][Hv]                                   */
  const float* beta;             /* [T][Hv]                                   */
  const float* conv_w;           /* [conv_dim][4]                             */
  void* o;                       /* [T][Hv][dv] out_dtype                     */
  int32_t* dev_error;
} gdn_mixed_args;

size_t gdn_mixed_workspace_size(const gdn_layer_desc* desc, int32_t num_seqs, int64_t total_tokens);
gdn_status gdn_mixed_step(const gdn_layer_desc* desc, const gdn_pool* pool, const gdn_mixed_args* args,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Bit-exact copies of whole state payloads (S and conv window, NaN encodings
 * included) between pages: dst_page[i] <- src_page[i] for i < n.  A page may
 * only be copied at a block boundary: num_computed_host[i] (tokens the state
 * has absorbed) must be a multiple of block_size, otherwise
 * GDN_ERR_NOT_BLOCK_ALIGNED is returned and nothing is launched ("Prefix
 * caching on Gated DeltaNet hybrids", "The in-page layout": save and restore
 * through bit-exact copies; fail closed on a partial block or an off-boundary
 * resume).  resume = block page -> working slot; save = slot -> block page. */
gdn_status gdn_checkpoint_resume(const gdn_layer_desc* desc, const gdn_pool* pool,
                                 const int32_t* src_page, const int32_t* dst_page,
                                 const int64_t* num_computed_host, int32_t n,
                                 int32_t* dev_error, void* stream);
gdn_status gdn_checkpoint_save(const gdn_layer_desc* desc, const gdn_pool* pool,
                               const int32_t* src_page, const int32_t* dst_page,
                               const int64_t* num_computed_host, int32_t n,
                               int32_t* dev_error, void* stream);

/* Replay verification ("Caching less to serve more requests", "What we
 * changed"): each request keeps one checkpoint page (state and conv window
 * before its logged rows) and a log of up to 32 pre-conv input rows since.
 *
 * append: for request r with n = log_len[r] logged rows, runs the recurrence
 *   from the checkpoint over the n logged rows and the m = num_new new rows,
 *   writes the outputs of the m new rows to o and appends the rows to the log
 *   (log_len[r] += m).  The checkpoint page is not written.  n + m > 32 sets
 *   GDN_ERR_LOG_OVERFLOW and skips the request.
 * rollback: log_len[r] -= num_appended - accepted[r]; accepted[r] outside
 *   [0, num_appended] or beyond the log sets GDN_ERR_ROLLBACK_RANGE and leaves
 *   log_len[r] unchanged.
 * flush: applies the log_len[r] logged rows to the checkpoint page (state and
 *   conv window, in place) as one block and sets log_len[r] = 0.  With
 *   boundary_rows given (prefix caching), a request with j = boundary_rows[r]
 *   in [1, log_len[r]] also gets the state and conv window after its first j
 *   kept rows written to page boundary_page[r] (a block-boundary checkpoint,
 *   see gdn_replay_boundary_rows); j <= 0 writes none.  j > log_len[r] or a
 *   boundary page equal to the checkpoint page sets GDN_ERR_INVALID_ARG, a
 *   boundary page outside the pool GDN_ERR_PAGE_RANGE; such a request is left
 *   unchanged.  Boundary checkpoints need the tensor-core path (dk = dv = 128,
 *   bf16): other shapes return GDN_ERR_UNSUPPORTED_SHAPE before any launch. */
typedef struct gdn_replay_args {
  int32_t num_reqs;              /* N >= 0; ckpt slots must be distinct       */
  int32_t num_new;               /* m, append only: 0 <= m <= 32              */
  const int32_t* ckpt_slot;      /* [N] page ids                              */
  void* log_x;                   /* [N][32][conv_dim] in_dtype                */
  float* log_g;                  /* [N][32][Hv]                               */
  float* log_beta;               /* [N][32][Hv]                               */
  int32_t* log_len;              /* [N] rows in the log                       */
  const void* x_new;             /* [N][m][conv_dim] in_dtype (append)        */
  const float* g_new;            /* [N][m][Hv] (append)                       */
  const float* beta_new;         /* [N][m][Hv] (append)                       */
  const float* conv_w;           /* [conv_dim][4]                             */
  void* o;                       /* [N][m][Hv][dv] out_dtype (append)         */
  int32_t* dev_error;
  void* workspace;               /* device scratch, >= gdn_replay_workspace_size */
  size_t workspace_bytes;
  const int32_t* boundary_rows;  /* [N] flush only, optional (NULL: none)     */
  const int32_t* boundary_page;  /* [N] page ids, required with boundary_rows */
} gdn_replay_args;

/* Device workspace bytes of gdn_replay_append / gdn_replay_flush for
 * num_reqs requests (32 log rows each); same contract as the prefill's. */
size_t gdn_replay_workspace_size(const gdn_layer_desc* desc, int32_t num_reqs);

gdn_status gdn_replay_append(const gdn_layer_desc* desc, const gdn_pool* pool,
                             const gdn_replay_args* args, void* stream);
gdn_status gdn_replay_rollback(int32_t* log_len, const int32_t* accepted,
                               int32_t num_appended, int32_t n, int32_t* dev_error,
                               void* stream);
gdn_status gdn_replay_flush(const gdn_layer_desc* desc, const gdn_pool* pool,
                            const gdn_replay_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
