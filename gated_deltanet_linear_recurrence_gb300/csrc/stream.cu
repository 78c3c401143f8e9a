// stream.cu — gdn_prefill_streamed: one long prompt prefilled as consecutive
// pieces of a fixed number of tokens, the state carried from piece to piece in
// state_out, with a workspace bounded by the piece size instead of the prompt
// length (contract in include/gdn.h).
//
// The page "Optimizing on-device inference for Apple Silicon" (section "Limit
// scratch memory by splitting prompts into chunks") processes a long prompt as a
// series of bounded pieces, the recurrent state carrying the context from one
// piece to the next, so that temporary storage stops growing with the whole
// prompt.  Here each piece is one gdn_prefill call with an explicit evaluation,
// so the result does not depend on the piece size when pieces are whole chunks.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"
#include "params.h"

namespace {

// Workspace head: two single-sequence cu_seqlens arrays, {0, piece} at byte 0
// and {0, last piece} at byte 16; the rest serves every piece's gdn_prefill.
constexpr size_t kHeadBytes = 256;
constexpr int64_t kPieceQuantum = 64;  // pieces are whole chunks of the chunked evaluation

__global__ void piece_cu_kernel(int32_t* cu, int32_t piece, int32_t last) {
  cu[0] = 0;
  cu[1] = piece;
  cu[4] = 0;
  cu[5] = last;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool head_dim_ok(int32_t d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// The host checks gdn_prefill makes, made here before anything is launched.
gdn_status host_checks(const void* q, const void* k, const void* v, const float* g,
                       const float* beta, const float* state_in, const float* state_out,
                       const void* o, int64_t total_tokens, int32_t h_k, int32_t h_v,
                       int32_t d_k, int32_t d_v) {
  if (h_k <= 0 || h_v <= 0 || d_k <= 0 || d_v <= 0) return GDN_ERR_INVALID_ARG;
  if (h_v % h_k != 0 || !head_dim_ok(d_k) || !head_dim_ok(d_v) || h_v > 65535)
    return GDN_ERR_UNSUPPORTED_SHAPE;
  if (total_tokens > INT32_MAX) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (!state_out) return GDN_ERR_NULL_POINTER;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_NULL_POINTER;
  const void* ptrs[] = {q, k, v, g, beta, state_in, state_out, o};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
  const size_t state_bytes = (size_t)h_v * d_v * d_k * sizeof(float);
  if (state_in && state_in != state_out) {
    const char* a = reinterpret_cast<const char*>(state_in);
    const char* b = reinterpret_cast<const char*>(state_out);
    if (a < b + state_bytes && b < a + state_bytes) return GDN_ERR_INVALID_ARG;
  }
  return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_prefill_streamed_workspace_size(int64_t piece_tokens, int32_t h_k, int32_t h_v,
                                           int32_t d_k, int32_t d_v, gdn_dtype dtype) {
  if (piece_tokens <= 0 || piece_tokens % kPieceQuantum || piece_tokens > INT32_MAX) return 0;
  if (h_k <= 0 || h_v <= 0 || d_k <= 0 || d_v <= 0) return 0;
  return kHeadBytes + gdn_prefill_workspace_size(1, piece_tokens, h_k, h_v, d_k, d_v, dtype,
                                                 GDN_ALGO_CHUNKED_SPLIT);
}

gdn_status gdn_prefill_streamed(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* state_in, float* state_out,
                                void* o, int64_t total_tokens, int32_t h_k, int32_t h_v,
                                int32_t d_k, int32_t d_v, gdn_dtype dtype, float scale,
                                int64_t piece_tokens, void* workspace, size_t workspace_bytes,
                                uint32_t options, gdn_stream_t stream) {
  if (total_tokens < 0 || piece_tokens <= 0 || piece_tokens % kPieceQuantum ||
      piece_tokens > INT32_MAX)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED_DTYPE;
  const gdn_status chk = host_checks(q, k, v, g, beta, state_in, state_out, o, total_tokens, h_k,
                                     h_v, d_k, d_v);
  if (chk != GDN_OK) return chk;
  if (!workspace) return GDN_ERR_NULL_POINTER;
  if (!aligned16(workspace)) return GDN_ERR_MISALIGNED;
  const size_t need =
      gdn_prefill_streamed_workspace_size(piece_tokens, h_k, h_v, d_k, d_v, dtype);
  if (need == 0) return GDN_ERR_INVALID_ARG;
  if (workspace_bytes < need) return GDN_ERR_WORKSPACE_TOO_SMALL;
  // The two-kernel chunked evaluation where it applies (bf16, d_k 128, d_v a
  // multiple of 32), the token scan otherwise; the same for every piece.
  const gdn_algo algo = gdn::chunked_supports(h_k, h_v, d_k, d_v, dtype) ? GDN_ALGO_CHUNKED_SPLIT
                                                                          : GDN_ALGO_SCAN;
  const int64_t n_pieces = total_tokens == 0 ? 1 : (total_tokens + piece_tokens - 1) / piece_tokens;
  const int64_t last = total_tokens - (n_pieces - 1) * piece_tokens;
  int32_t* cu = static_cast<int32_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  piece_cu_kernel<<<1, 1, 0, s>>>(cu, static_cast<int32_t>(piece_tokens),
                                  static_cast<int32_t>(last));
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  const size_t es = dtype == GDN_BF16 ? 2 : 4;
  const size_t qk_row = static_cast<size_t>(h_k) * d_k * es;  // bytes per token
  const size_t vo_row = static_cast<size_t>(h_v) * d_v * es;
  uint8_t* piece_ws = static_cast<uint8_t*>(workspace) + kHeadBytes;
  for (int64_t i = 0; i < n_pieces; ++i) {
    const int64_t t0 = i * piece_tokens;
    const int64_t len = i == n_pieces - 1 ? last : piece_tokens;
    const int32_t* cu_i = i == n_pieces - 1 ? cu + 4 : cu;
    const gdn_status st = gdn_prefill_ex(
        q ? static_cast<const char*>(q) + t0 * qk_row : nullptr,
        k ? static_cast<const char*>(k) + t0 * qk_row : nullptr,
        v ? static_cast<const char*>(v) + t0 * vo_row : nullptr, g ? g + t0 * h_v : nullptr,
        beta ? beta + t0 * h_v : nullptr, i == 0 ? state_in : state_out, state_out,
        o ? static_cast<char*>(o) + t0 * vo_row : nullptr, cu_i, 1, len, h_k, h_v, d_k, d_v,
        dtype, scale, algo, piece_ws, workspace_bytes - kHeadBytes, options, stream);
    if (st != GDN_OK) return st;
  }
  return GDN_OK;
}

}  // extern "C"
