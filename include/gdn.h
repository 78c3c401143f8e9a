/*
 * gdn.h — C ABI of the GB300 (sm_103a) Gated DeltaNet recurrence library.
 *
 * The operation.  The page "Optimizing on-device inference for Apple Silicon"
 * (section "Qwen creates three distinct workload shapes") describes the Gated
 * DeltaNet layer: a fixed-size recurrent matrix state per head, a learned gate
 * that keeps part of the old state, and a delta update that writes the current
 * token; each token depends on the state the previous token produced.  The
 * equation the library evaluates, per value head h and token t, is the gated
 * delta rule:
 *
 *     alpha_t = exp(g_t)
 *     S_t     = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t     = S_t (scale * q_t)
 *
 * The same section says a prefill may either scan tokens directly while
 * carrying the state or regroup the updates into blocks that expose matrix
 * work, and that which is faster depends on model dimensions, workload and
 * hardware: gdn_prefill offers both (GDN_ALGO_SCAN, GDN_ALGO_CHUNKED) and picks
 * by a measured crossover (GDN_ALGO_AUTO).  Section "Keep the recurrent state
 * on-chip" fixes the state and its gate to fp32 while q and k may be bf16.
 * Section "Reduce intermediate and state traffic" fuses the decode-time
 * recurrent update into one kernel: gdn_decode_step.
 *
 * Shapes and layouts (all tensors dense, contiguous, row-major):
 *   q, k      [T][h_k][d_k]           dtype        (decode: [B][h_k][d_k])
 *   v, o      [T][h_v][d_v]           dtype        (decode: [B][h_v][d_v])
 *   g, beta   [T][h_v]                fp32         (decode: [B][h_v])
 *   state     [N][h_v][d_v][d_k]      fp32         row i = value dim, col j = key dim
 *   cu_seqlens[N+1]                   int32, device memory
 * Value head h reads key/query head h / (h_v / h_k): consecutive value heads
 * share a key head.  d_k and d_v are each one of 16, 32, 64, 128; h_v must be
 * a multiple of h_k.  g must be finite (alpha = exp(g) may underflow to 0).
 *
 * Ownership.  The caller owns every buffer; the library allocates no device
 * memory in any call below.  Scratch space for gdn_prefill is the caller's
 * `workspace` (size from gdn_prefill_workspace_size); gdn_prefill_noalloc
 * uses a fixed array the library holds instead.
 *
 * Asynchrony.  Calls are ordered on the caller's `stream` and return after
 * the launches are enqueued.  Errors that the host can see (NULL pointers,
 * shapes, dtypes, 16-byte alignment, workspace size) return synchronously and
 * launch nothing.  Errors only the device can see (inconsistent cu_seqlens)
 * are recorded in a per-device error word owned by the library; the affected
 * sequences are skipped, and gdn_stream_status reports and clears the word.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gdn_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  GDN_OK = 0,
  GDN_ERR_NULL_POINTER = 1,      /* a required pointer is NULL */
  GDN_ERR_INVALID_ARG = 2,       /* negative size, bad enum, partial state overlap */
  GDN_ERR_UNSUPPORTED_SHAPE = 3, /* d_k/d_v not in {16,32,64,128}, h_v % h_k != 0, T >= 2^31 */
  GDN_ERR_UNSUPPORTED_DTYPE = 4, /* dtype not supported by the requested algorithm */
  GDN_ERR_MISALIGNED = 5,        /* a tensor pointer is not 16-byte aligned */
  GDN_ERR_BAD_CU_SEQLENS = 6,    /* device-detected: cu[0] != 0, decreasing, or cu[N] != T */
  GDN_ERR_WORKSPACE_TOO_SMALL = 7,
  GDN_ERR_DEVICE_TIMEOUT = 8,    /* device-detected: a bounded wait expired */
  GDN_ERR_CUDA = 9,              /* a CUDA runtime call failed */
  GDN_ERR_BAD_CACHE_LEN = 10     /* device-detected: a cache_len outside 0 .. capacity */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype; /* dtype of q, k, v and o */

/*
 * Options of the *_ex entry points, gdn_decode_multi and gdn_prefill_streamed
 * (bitwise OR; 0 = the plain recurrence).
 *
 * GDN_OPT_QK_L2NORM: divide q and k of every (token, key head) by
 * sqrt(sum of squares + 1e-6) before the recurrence (q is then multiplied by
 * `scale`).  Page "Optimizing on-device inference for Apple Silicon", section
 * "Reduce intermediate and state traffic": the decode path fuses the recurrent
 * update with its normalization; per-head L2 normalisation of q and k is the
 * reading taken here, done inside the kernels instead of as a separate pass.
 */
#define GDN_OPT_QK_L2NORM 1u

typedef enum {
  GDN_ALGO_AUTO = 0,          /* by a table measured per shape: scan for short sequences, else
                                 the fastest chunked form the call can run (see gdn_prefill) */
  GDN_ALGO_SCAN = 1,          /* token scan, state rows resident in registers (fp32 and bf16) */
  GDN_ALGO_CHUNKED = 2,       /* chunks of 64 tokens on tcgen05 tensor cores (bf16); the library
                                 picks the fused or the two-kernel form (see gdn_prefill) */
  GDN_ALGO_CHUNKED_FUSED = 3, /* chunked, one fused kernel, no workspace */
  GDN_ALGO_CHUNKED_SPLIT = 4, /* chunked, two kernels through the workspace (required) */
  GDN_ALGO_CHUNKED_COOP = 5   /* chunked, one cooperative kernel through the workspace (required;
                                 d_v a multiple of 64, num_seqs x h_v x d_v / 64 at most two
                                 thirds of the SMs, else GDN_ERR_UNSUPPORTED_SHAPE) */
} gdn_algo;

/*
 * gdn_prefill — evaluate the recurrence over N packed sequences.
 *
 * Sequence n owns tokens cu_seqlens[n] .. cu_seqlens[n+1]-1.  Its state starts
 * from state_in[n] (all zeros when state_in is NULL) and its final state is
 * written to state_out[n]; o[t] = S_t q_t for each of its tokens.  An empty
 * sequence copies its initial state and writes no output.  state_in may equal
 * state_out (in-place carry); any other overlap is GDN_ERR_INVALID_ARG.
 * Output rows of tokens outside every sequence are not written.
 *
 * Arguments: q, k, v, o in `dtype`; g, beta, state_in, state_out fp32;
 * cu_seqlens int32 device pointer of num_seqs+1 entries with cu[0] = 0,
 * non-decreasing, cu[num_seqs] = total_tokens; scale multiplies q (1 for the
 * plain reading o_t = S_t q_t).  algo selects the evaluation (see gdn_algo);
 * the chunked algorithms with GDN_F32 return GDN_ERR_UNSUPPORTED_DTYPE.
 * workspace: scratch, 16-byte aligned, or NULL.  The chunked evaluation
 * (bf16; d_k 128, or 64 with the two-kernel and cooperative forms, which pad
 * each key head to 128 columns with zeros; d_v a multiple of 32) runs either
 * as one fused kernel that needs no workspace (d_k 128 only), or as two
 * kernels (the per-chunk state-independent work spread over all SMs, then the
 * sequential state pass) that meet in the workspace, or as one cooperative
 * kernel whose prepare CTAs and state-pass CTAs overlap (GDN_ALGO_CHUNKED_COOP;
 * its results equal the two kernels' bit for bit).  GDN_ALGO_SCAN and the
 * forced chunked forms run what they name; GDN_ALGO_CHUNKED_SPLIT and
 * GDN_ALGO_CHUNKED_COOP return GDN_ERR_NULL_POINTER or
 * GDN_ERR_WORKSPACE_TOO_SMALL without the workspace they need.
 * GDN_ALGO_AUTO and GDN_ALGO_CHUNKED choose by a table measured on GB300 per
 * (d_k, d_v, h_v, num_seqs) (the nearest measured shape): sequences shorter
 * than its scan threshold take the token scan (the whole batch when the
 * sequences average less; AUTO only); the others the fused kernel, or the two
 * kernels from the table's average length when workspace_bytes is at least
 * gdn_prefill_workspace_size(...) (always, when the fused kernel does not
 * cover the call; with too little workspace AUTO then scans and CHUNKED
 * returns GDN_ERR_WORKSPACE_TOO_SMALL), or the cooperative form from its
 * average length when its state passes fit and the workspace holds its ready
 * flags.  gdn_prefill_form reports the choice for given sizes.  Results agree
 * within rounding; the workspace is not used after the launches complete.
 */
gdn_status gdn_prefill(const void* q, const void* k, const void* v, const float* g,
                       const float* beta, const float* state_in, float* state_out, void* o,
                       const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                       int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype,
                       float scale, gdn_algo algo, void* workspace, size_t workspace_bytes,
                       gdn_stream_t stream);

/* gdn_prefill with `options` (see GDN_OPT_QK_L2NORM); other bits return
 * GDN_ERR_INVALID_ARG.  gdn_prefill is gdn_prefill_ex with options = 0.
 * With GDN_OPT_QK_L2NORM the chunked evaluation is the two-kernel form only:
 * GDN_ALGO_CHUNKED_FUSED returns GDN_ERR_INVALID_ARG, GDN_ALGO_CHUNKED needs a
 * workspace of gdn_prefill_workspace_size(..., GDN_ALGO_CHUNKED_SPLIT) bytes
 * (else GDN_ERR_WORKSPACE_TOO_SMALL), and GDN_ALGO_AUTO without such a
 * workspace runs the token scan for every sequence. */
gdn_status gdn_prefill_ex(const void* q, const void* k, const void* v, const float* g,
                          const float* beta, const float* state_in, float* state_out, void* o,
                          const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                          int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype,
                          float scale, gdn_algo algo, void* workspace, size_t workspace_bytes,
                          uint32_t options, gdn_stream_t stream);

/* Bytes of workspace for the fastest gdn_prefill path with these arguments
 * (0 when that path uses none); for GDN_ALGO_CHUNKED_SPLIT and
 * GDN_ALGO_CHUNKED_COOP, the bytes each needs.  An upper bound computed from the
 * host arguments: the 1 KB-rounded (2N+1) int32 header + I * 57 KB with
 * I = (T/64 + N + 1) * h_v items, plus (I + 1) int32 ready flags (1 KB-rounded)
 * except for GDN_ALGO_CHUNKED_SPLIT. */
size_t gdn_prefill_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t h_k,
                                  int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype,
                                  gdn_algo algo);

/*
 * gdn_prefill_streamed — one sequence of total_tokens tokens prefilled as
 * consecutive pieces of piece_tokens tokens (a positive multiple of 64; the
 * last piece may be shorter), the state carried from piece to piece in
 * state_out.  Page "Optimizing on-device inference for Apple Silicon", section
 * "Limit scratch memory by splitting prompts into chunks": a long prompt runs
 * as bounded pieces whose recurrent state carries the context, so the scratch
 * memory is bounded by the piece, not the prompt.
 *
 * Same tensors as gdn_prefill for one sequence (no cu_seqlens: the sequence is
 * tokens 0 .. total_tokens-1); state_in may be NULL (zeros) or equal state_out.
 * Every piece runs the two-kernel chunked evaluation (bf16, d_k 128 or 64,
 * d_v a multiple of 32), else the token scan, so the result equals bit for bit
 * gdn_prefill with GDN_ALGO_CHUNKED_SPLIT (resp. GDN_ALGO_SCAN) on the whole
 * sequence.  workspace: required, 16-byte aligned, at least
 * gdn_prefill_streamed_workspace_size(piece_tokens, ...) bytes, which does not
 * depend on total_tokens.  Errors: GDN_ERR_INVALID_ARG for a bad piece size,
 * GDN_ERR_WORKSPACE_TOO_SMALL, and those of gdn_prefill.  `options` as for
 * gdn_prefill_ex.
 */
gdn_status gdn_prefill_streamed(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* state_in, float* state_out,
                                void* o, int64_t total_tokens, int32_t h_k, int32_t h_v,
                                int32_t d_k, int32_t d_v, gdn_dtype dtype, float scale,
                                int64_t piece_tokens, void* workspace, size_t workspace_bytes,
                                uint32_t options, gdn_stream_t stream);

/* Workspace bytes for gdn_prefill_streamed with pieces of piece_tokens tokens
 * (0 for an invalid piece size or head shape). */
size_t gdn_prefill_streamed_workspace_size(int64_t piece_tokens, int32_t h_k, int32_t h_v,
                                           int32_t d_k, int32_t d_v, gdn_dtype dtype);

/*
 * gdn_prefill_host — gdn_prefill_streamed for a sequence whose tensors live in
 * HOST memory: q, k, v, g, beta, state_in (or NULL: zeros), state_out and o are
 * host pointers with the layouts of gdn_prefill_streamed; workspace is DEVICE
 * memory of at least gdn_prefill_host_workspace_size(piece_tokens, ...) bytes,
 * 16-byte aligned.  The prompt is cut into pieces of piece_tokens tokens (a
 * positive multiple of 64) and the copy of one piece's inputs to the device,
 * the prefill of the previous piece and the copy of the piece before that back
 * to the host overlap: the library orders them with two copy streams of its
 * own and events, joined back into `stream` (graph capture works as for one
 * stream).  The source pages have no host-side counterpart; it serves callers
 * whose data is on the host, where copies, not the prefill, set the time.
 * Host memory should be page-locked (cudaHostAlloc / cudaHostRegister): from
 * pageable memory the driver stages each copy and nothing overlaps.
 *
 * Results equal gdn_prefill_streamed with the same piece size bit for bit and
 * are complete in host memory when `stream` reaches the point after this call
 * (synchronise it before reading them).  Calls on one device are serialised
 * while they enqueue work.  Errors: those of gdn_prefill_streamed; host
 * pointers are not checked beyond NULL.
 */
gdn_status gdn_prefill_host(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* state_in, float* state_out, void* o,
                            int64_t total_tokens, int32_t h_k, int32_t h_v, int32_t d_k,
                            int32_t d_v, gdn_dtype dtype, float scale, int64_t piece_tokens,
                            void* workspace, size_t workspace_bytes, uint32_t options,
                            gdn_stream_t stream);

/* Device workspace bytes for gdn_prefill_host with pieces of piece_tokens
 * tokens: two buffers of one piece's inputs and outputs, the state, and one
 * piece's prefill workspace (0 for invalid arguments). */
size_t gdn_prefill_host_workspace_size(int64_t piece_tokens, int32_t h_k, int32_t h_v,
                                       int32_t d_k, int32_t d_v, gdn_dtype dtype);

/*
 * gdn_prefill_noalloc — gdn_prefill with GDN_ALGO_CHUNKED_SPLIT (the
 * two-kernel chunked evaluation), taking its scratch from a fixed array of
 * GDN_NOALLOC_SCRATCH_BYTES that the library holds in device memory instead of
 * a caller workspace.  The source pages have no counterpart: it exists for
 * callers that cannot allocate device memory when they call in, such as a host
 * framework whose memory pool owns the device and hands its plugins no
 * scratch buffer, or a serving loop that must not call cudaMalloc / cudaFree
 * (they can synchronise the device and stall every stream in flight).  It
 * allocates nothing and calls no allocating routine.
 *
 * Arguments, layouts, ownership of the caller's buffers and asynchronous
 * errors are those of gdn_prefill; dtype must be GDN_BF16, d_k 128 or 64 and d_v
 * a multiple of 32 (else GDN_ERR_UNSUPPORTED_*).  Limit: returns
 * GDN_ERR_WORKSPACE_TOO_SMALL, touching no device, when
 * gdn_prefill_workspace_size(..., GDN_ALGO_CHUNKED_SPLIT) for these arguments
 * exceeds GDN_NOALLOC_SCRATCH_BYTES (128 MiB: e.g. one 4,096-token sequence at
 * 32 value heads needs 123.3 MB); larger problems go through gdn_prefill with a
 * workspace.
 *
 * Set-up: the first call with a given device current looks up that device's
 * copy of the array (cudaGetSymbolAddress); make that first call before any
 * stream capture.  The address is kept for the life of the process, so
 * destroying the device's primary context after that first call (for example
 * with cudaDeviceReset) is not supported: the kept address would be stale.
 * The device error word that every entry point reports through
 * gdn_stream_status is located the same way, once per device.
 * Sharing: every call on a device uses the same array.
 * Nothing in it has to start at zero (each call writes what it later reads),
 * but calls whose kernels overlap on the GPU (other streams, other host
 * threads) race on it: order them, e.g. on one stream.  The array takes
 * GDN_NOALLOC_SCRATCH_BYTES of each device where the library's code is loaded.
 */
#define GDN_NOALLOC_SCRATCH_BYTES ((size_t)128 << 20)

gdn_status gdn_prefill_noalloc(const void* q, const void* k, const void* v, const float* g,
                               const float* beta, const float* state_in, float* state_out,
                               void* o, const int32_t* cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, int32_t h_k, int32_t h_v, int32_t d_k,
                               int32_t d_v, gdn_dtype dtype, float scale, gdn_stream_t stream);

/*
 * gdn_decode_step — one token for each of `batch` independent sequences,
 * state updated in place (one read and one write of every state element).
 * Same equation and head mapping as gdn_prefill with one token per sequence:
 * q, k [batch][h_k][d_k], v, o [batch][h_v][d_v] in `dtype`; g, beta
 * [batch][h_v] fp32; state [batch][h_v][d_v][d_k] fp32.
 */
gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float* state, void* o, int32_t batch, int32_t h_k,
                           int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype, float scale,
                           gdn_stream_t stream);

/* gdn_decode_step with `options` (see GDN_OPT_QK_L2NORM). */
gdn_status gdn_decode_step_ex(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* state, void* o, int32_t batch,
                              int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype,
                              float scale, uint32_t options, gdn_stream_t stream);

/*
 * gdn_decode_step_rmsnorm — gdn_decode_step_ex with the layer's output
 * normalised inside the same kernel.  Page "Optimizing on-device inference for
 * Apple Silicon", section "Reduce intermediate and state traffic": the decode
 * path fuses the recurrent update with its normalization; the page does not
 * give the normalisation's form, and this entry point takes the plainest one
 * for an output: a root-mean-square normalisation of each (sequence, value
 * head)'s d_v outputs with a per-channel weight shared by the heads,
 *
 *     o[b,h,i] = w_i * y_i / sqrt( (1 / d_v) sum_j y_j^2 + norm_eps )
 *
 * where y is the step's output in fp32 (before rounding to `dtype`).
 * norm_weight: [d_v] fp32, 16-byte aligned, or NULL for w = 1; norm_eps >= 0
 * (else GDN_ERR_INVALID_ARG).  The state update is exactly gdn_decode_step_ex's
 * (bit for bit).  The CTAs that share a (sequence, head) form one thread-block
 * cluster and exchange their partial sums of squares through distributed
 * shared memory, so o is written once, already normalised.
 */
gdn_status gdn_decode_step_rmsnorm(const void* q, const void* k, const void* v, const float* g,
                                   const float* beta, float* state, void* o,
                                   const float* norm_weight, float norm_eps, int32_t batch,
                                   int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v,
                                   gdn_dtype dtype, float scale, uint32_t options,
                                   gdn_stream_t stream);

/*
 * gdn_output_rmsnorm — the same normalisation as a pass of its own, in place,
 * over o [rows][h_v][d_v] in `dtype` (for example a gdn_prefill output; the
 * values are those stored in o, already rounded to `dtype`).  norm_weight and
 * norm_eps as for gdn_decode_step_rmsnorm; d_v one of 16, 32, 64, 128.
 * Reads and writes o once.
 */
gdn_status gdn_output_rmsnorm(void* o, const float* norm_weight, int64_t rows, int32_t h_v,
                              int32_t d_v, gdn_dtype dtype, float norm_eps, gdn_stream_t stream);

/*
 * gdn_decode_multi — n_tokens (1 .. 1024) consecutive tokens for each of
 * `batch` sequences in one launch: the state is read once, carried through the
 * tokens and written once.  Page "Optimizing on-device inference for Apple
 * Silicon", section "Limits of further optimization": speculative decoding
 * verifies groups of two to five rows per step; after a rejected draft token
 * the caller goes back to the state after the last accepted one, which
 * `snapshots` provides.  The results equal n_tokens successive gdn_decode_step
 * calls bit for bit.
 *
 * q, k [batch][n_tokens][h_k][d_k] and v, o [batch][n_tokens][h_v][d_v] in
 * `dtype`; g, beta [batch][n_tokens][h_v] fp32; state [batch][h_v][d_v][d_k]
 * fp32, updated in place to the state after the last token; snapshots NULL or
 * [batch][n_tokens][h_v][d_v][d_k] fp32 receiving the state after each token
 * (must not overlap the state).  Same head mapping and scale as
 * gdn_decode_step; `options` as for gdn_decode_step_ex.
 */
gdn_status gdn_decode_multi(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float* state, void* o, float* snapshots,
                            int32_t batch, int32_t n_tokens, int32_t h_k, int32_t h_v,
                            int32_t d_k, int32_t d_v, gdn_dtype dtype, float scale,
                            uint32_t options, gdn_stream_t stream);

/*
 * gdn_attn_decode — grouped-query attention for one new token of each of
 * `batch` sequences over its KV cache (the full-attention layers that sit
 * between the recurrent layers of the same hybrid model).  Page "Optimizing
 * on-device inference for Apple Silicon", section "Read the attention cache
 * efficiently": the decode step reads the whole cache, so the kernel is bound
 * by the bytes it reads; the query heads that share a KV head are served
 * together so each cached row is read once ("Group query heads to reuse KV
 * rows"); and at long context the cache is split into equal fixed blocks
 * processed in parallel whose partial softmax results are then merged
 * ("Switch attention layouts at long context", for heads of 256 values with
 * eight query heads per KV head).
 *
 * For sequence b, query head h and its KV head j = h / (h_q / h_kv), over the
 * L_b = cache_len[b] cached keys:
 *     s_i = scale * (q_{b,h} . k_{b,j,i}),   o_{b,h} = sum_i softmax(s)_i v_{b,j,i}
 * and o_{b,h} = 0 when L_b = 0.  Cache slots at or past L_b are never read into
 * a result (they may hold anything, NaN included).
 *
 * Arguments: q [batch][h_q][head_dim], o [batch][h_q][head_dim], k_cache and
 * v_cache [batch][h_kv][capacity][head_dim], all GDN_BF16 (else
 * GDN_ERR_UNSUPPORTED_DTYPE); cache_len [batch] int32 device pointer with
 * 0 <= cache_len[b] <= capacity (a value outside sets GDN_ERR_BAD_CACHE_LEN in
 * the error word and that sequence gets o = 0).  head_dim must be 256 and
 * h_q / h_kv an integer from 1 to 8, batch x h_kv x capacity below 2^31 (else
 * GDN_ERR_UNSUPPORTED_SHAPE).  Pointers 16-byte aligned; k_cache and v_cache
 * may be NULL only when capacity is 0.
 *
 * layout and block_keys: GDN_ATTN_GENERAL gives each (sequence, KV head) one
 * CTA over its whole cache and writes o directly.  GDN_ATTN_FIXED_BLOCK splits
 * the cache into blocks of block_keys keys (a positive multiple of 64, or 0 for
 * a size the library picks from the SM count so that the blocks fill the GPU
 * about once) processed by separate CTAs, then a combine pass merges their
 * partial results through `workspace`; it needs workspace_bytes >=
 * gdn_attn_decode_workspace_size(...) (else GDN_ERR_NULL_POINTER or
 * GDN_ERR_WORKSPACE_TOO_SMALL).  GDN_ATTN_AUTO takes the fixed blocks when the
 * (sequence, KV head) pairs are too few to fill the GPU and the workspace is
 * large enough, else the general layout.  block_keys other than 0 or a
 * positive multiple of 64 is GDN_ERR_INVALID_ARG.  The layouts agree within
 * fp32 rounding of the softmax sums and the bf16 rounding of o.
 */
typedef enum {
  GDN_ATTN_AUTO = 0,
  GDN_ATTN_GENERAL = 1,
  GDN_ATTN_FIXED_BLOCK = 2
} gdn_attn_layout;

gdn_status gdn_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* cache_len, void* o, int32_t batch, int32_t h_q,
                           int32_t h_kv, int32_t head_dim, int32_t capacity, gdn_dtype dtype,
                           float scale, gdn_attn_layout layout, int32_t block_keys,
                           void* workspace, size_t workspace_bytes, gdn_stream_t stream);

/* Workspace bytes sufficient for gdn_attn_decode with these arguments, computed
 * on the host: 0 for GDN_ATTN_GENERAL, else batch x h_q x n x (head_dim + 2) x
 * 4 with n = ceil(capacity / block_keys), block_keys taken as 128 when 0 (the
 * smallest block the library picks).  0 for invalid arguments. */
size_t gdn_attn_decode_workspace_size(int32_t batch, int32_t h_q, int32_t h_kv,
                                      int32_t head_dim, int32_t capacity,
                                      gdn_attn_layout layout, int32_t block_keys);

/* The block of keys each CTA takes in gdn_attn_decode with these arguments on
 * the current device, given a large enough workspace (capacity, or at least 1,
 * for the general layout); -1 for invalid arguments or when the device cannot
 * be queried.  The call launches ceil(capacity / result) CTAs per (sequence,
 * KV head). */
int32_t gdn_attn_decode_block_keys(int32_t batch, int32_t h_q, int32_t h_kv, int32_t head_dim,
                                   int32_t capacity, gdn_attn_layout layout,
                                   int32_t block_keys);

/*
 * gdn_stream_status — synchronise `stream`, then report (and clear) the
 * current device's error word: GDN_OK, GDN_ERR_BAD_CU_SEQLENS,
 * GDN_ERR_BAD_CACHE_LEN, GDN_ERR_DEVICE_TIMEOUT, or GDN_ERR_CUDA if the
 * stream reported a CUDA error.
 */
gdn_status gdn_stream_status(gdn_stream_t stream);

/*
 * gdn_selftest_wait_timeout — a check of the library's failure path that
 * needs no fault: one CTA on `stream` waits, with the bounded mbarrier wait
 * every tensor-core kernel here uses for its hand-offs, on a barrier that
 * nothing completes.  The wait gives up after timeout_us microseconds
 * (1 .. 1,000,000), the kernel records GDN_ERR_DEVICE_TIMEOUT in the device
 * error word and returns; the next gdn_stream_status on the stream reports
 * and clears it, and the context stays usable.  Returns GDN_ERR_INVALID_ARG
 * for a timeout outside the range, GDN_ERR_CUDA if the launch fails.
 */
gdn_status gdn_selftest_wait_timeout(int32_t timeout_us, gdn_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* gdn_status_string(gdn_status status);

/*
 * gdn_prefill_form — which evaluation gdn_prefill / gdn_prefill_ex would run
 * for these sizes, algorithm, workspace size (0: no workspace) and options,
 * without launching anything: GDN_ALGO_SCAN when only the token scan runs, else
 * the form of the chunked evaluation of the sequences at or above the
 * crossover (GDN_ALGO_CHUNKED_FUSED, GDN_ALGO_CHUNKED_SPLIT or
 * GDN_ALGO_CHUNKED_COOP; with more than one sequence the shorter ones still
 * take the scan).  sm_count is the device's SM count (0: query the current
 * device).  On arguments the call would refuse it returns the negated status
 * (-GDN_ERR_...).  The cooperative form is reported when the call would try
 * it; if the device then refuses the cooperative launch (other work holds
 * SMs), AUTO and CHUNKED run the two kernels instead.
 */
int32_t gdn_prefill_form(int32_t num_seqs, int64_t total_tokens, int32_t h_k, int32_t h_v,
                         int32_t d_k, int32_t d_v, gdn_dtype dtype, gdn_algo algo,
                         size_t workspace_bytes, uint32_t options, int32_t sm_count);

/*
 * gdn_prefill_crossover_tokens — the sequence length at and above which
 * GDN_ALGO_AUTO uses the chunked evaluation for these head dimensions and
 * dtype, for a single sequence (the table measured on GB300; a batch of N
 * sequences may take another threshold, which gdn_prefill_form applies);
 * shorter sequences use the token scan.  Returns INT32_MAX when the chunked
 * evaluation does not support the case.
 */
int32_t gdn_prefill_crossover_tokens(int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v,
                                     gdn_dtype dtype);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
