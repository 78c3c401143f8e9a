// params.h — launch arguments passed from the C ABI layer to the kernels.
// Plain structs of pointers and sizes; no torch types.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

enum Dtype : int { kF32 = 0, kBF16 = 1 };

// Device error codes written to the library's error word (same values as
// gdn_status in include/gdn.h).
enum DeviceError : int { kErrBadCuSeqlens = 6, kErrDeviceTimeout = 8, kErrBadCacheLen = 10 };

struct DecodeArgs {
  const void* q;       // [B][h_k][d_k] dtype
  const void* k;       // [B][h_k][d_k] dtype
  const void* v;       // [B][h_v][d_v] dtype
  const float* g;      // [B][h_v]
  const float* beta;   // [B][h_v]
  float* state;        // [B][h_v][d_v][d_k], in place
  void* o;             // [B][h_v][d_v] dtype
  int32_t batch, h_k, h_v, d_k, d_v;
  int dtype;
  float scale;
  int qk_norm;  // divide q and k by their L2 norm (+1e-6 under the root) first
  // Output RMS normalisation in the same kernel (out_norm != 0): o[b,h,:] scaled
  // by w / sqrt(mean of its squares + norm_eps); norm_weight [d_v] or NULL (ones).
  int out_norm;
  const float* norm_weight;
  float norm_eps;
};

// Several tokens per sequence: q, k [B][n][h_k][d_k], v, o [B][n][h_v][d_v],
// g, beta [B][n][h_v]; state [B][h_v][d_v][d_k] in place; snapshots
// [B][n][h_v][d_v][d_k] (the state after each token) or nullptr.
struct DecodeMultiArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  float* state;
  void* o;
  float* snapshots;
  int32_t batch, n_tokens, h_k, h_v, d_k, d_v;
  int dtype;
  float scale;
  int qk_norm;
};

struct PrefillArgs {
  const void* q;            // [T][h_k][d_k] dtype
  const void* k;            // [T][h_k][d_k] dtype
  const void* v;            // [T][h_v][d_v] dtype
  const float* g;           // [T][h_v]
  const float* beta;        // [T][h_v]
  const float* state_in;    // [N][h_v][d_v][d_k] or nullptr (zeros)
  float* state_out;         // [N][h_v][d_v][d_k]
  void* o;                  // [T][h_v][d_v] dtype
  const int32_t* cu_seqlens;  // [N+1], device
  int32_t num_seqs;
  int64_t total_tokens;
  int32_t h_k, h_v, d_k, d_v;
  int dtype;
  float scale;
  int qk_norm;  // divide q and k by their L2 norm (+1e-6 under the root) first
  // Per-sequence split between the two evaluations: a sequence of length L
  // is handled by the scan when L < min_chunk_len and by the chunked kernel
  // otherwise.  (0 = chunked takes every sequence; INT32_MAX = scan takes all.)
  int32_t min_chunk_len;
  void* workspace;
  size_t workspace_bytes;
  int* err;                 // library error word on this device
};

// Grouped-query decode attention: q [B][h_q][D]; k_cache, v_cache
// [B][h_kv][capacity][D]; cache_len [B] (device); o [B][h_q][D]; all bf16
// except cache_len.  Each CTA takes block_keys cached keys of one (sequence,
// KV head); with n_split > 1 it writes an unnormalised partial [acc[D], m, l]
// per query head to `partial` [B][h_q][n_split][D + 2] and a combine pass
// produces o.
struct AttnArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* cache_len;
  void* o;
  float* partial;
  int32_t batch, h_q, h_kv, head_dim, capacity;
  int32_t block_keys, n_split;
  float scale;
  int* err;
};

// Decode-attention layouts (values of gdn_attn_layout) and the block plan:
// general = one block spanning the cache; fixed-block = n_split equal blocks of
// block_keys keys whose partial results a combine pass merges.
enum AttnLayout : int { kAttnAuto = 0, kAttnGeneral = 1, kAttnFixedBlock = 2 };
struct AttnPlan {
  int32_t block_keys, n_split;
};
AttnPlan attn_plan(int32_t batch, int32_t h_kv, int32_t capacity, int layout, int32_t block_keys,
                   int sm_count);
size_t attn_partial_bytes(int32_t batch, int32_t h_q, const AttnPlan& plan);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
// The output RMS normalisation in place over n_vec vectors of d_v values (output_norm.cu).
cudaError_t launch_output_rmsnorm(void* o, const float* weight, int64_t n_vec, int32_t d_v,
                                  int dtype, float eps, cudaStream_t stream);
cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_decode_multi(const DecodeMultiArgs& a, cudaStream_t stream);
cudaError_t launch_scan(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_chunked(const PrefillArgs& a, cudaStream_t stream);
size_t chunked_workspace_bytes(int32_t num_seqs, int64_t total_tokens, int32_t h_k, int32_t h_v,
                               int32_t d_k, int32_t d_v);
bool chunked_supports(int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, int dtype);
bool fused_supports(int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, int dtype);
// Two-kernel chunked prefill (prepare + chain) through a caller workspace.
size_t split_workspace_bytes(int32_t num_seqs, int64_t total_tokens, int32_t h_v);
cudaError_t launch_chunked_split(const PrefillArgs& a, void* workspace, cudaStream_t stream);
// One cooperative kernel (prepare slots and 64-row chains in one resident grid,
// chained by per-item ready flags) through a caller workspace: the two-kernel
// workspace plus one int per item.  Supported when d_v is a multiple of 64 and
// the chains take at most two thirds of the SMs.
size_t coop_workspace_bytes(int32_t num_seqs, int64_t total_tokens, int32_t h_v);
bool coop_supported(int32_t num_seqs, int32_t h_v, int32_t d_v, int sm_count);
cudaError_t launch_chunked_coop(const PrefillArgs& a, void* workspace, cudaStream_t stream);
// One CTA whose bounded mbarrier wait expires (selftest.cu).
cudaError_t launch_selftest_wait(uint64_t timeout_ns, int* err, cudaStream_t stream);

}  // namespace gdn
