// host_prefill.cu — gdn_prefill_host: one sequence prefilled from and to HOST
// memory, with the host-to-device copies, the prefill and the device-to-host
// copies of consecutive pieces overlapped (contract in include/gdn.h).
//
// Copies between host and device run at a few hundred GB/s, several times
// slower than the prefill reads HBM, so a call that copies everything in, then
// computes, then copies everything out spends most of its time in copies that
// leave the GPU idle.  Here the sequence is cut into pieces of piece_tokens
// tokens (a multiple of 64) and three queues work on different pieces at once:
//   copy-in   (library stream): inputs of piece i into device buffer i % 2
//   compute   (caller's stream): prefill of piece i, the state carried in the
//             workspace exactly as gdn_prefill_streamed carries it
//   copy-out  (library stream): output of piece i back to the host
// ordered by events, so that a buffer is refilled only after the prefill (for
// inputs) or the copy-out (for outputs) of the piece two steps earlier is done.
// The result equals gdn_prefill_streamed with the same piece size bit for bit.
// Host memory should be page-locked: copies from pageable memory are staged by
// the driver and do not overlap.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdn.h"
#include "params.h"

namespace {

constexpr int64_t kPieceQuantum = 64;  // pieces are whole chunks of the chunked evaluation
constexpr size_t kAlign = 256;
constexpr int kRing = 3;  // event ring: waits reach back two pieces

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool head_dim_ok(int32_t d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// Byte sizes of one piece's device buffers.
struct PieceBytes {
  size_t q, v, g;  // q and k; v and o; g and beta
};
PieceBytes piece_bytes(int64_t piece, int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v,
                       size_t es) {
  return {round_up((size_t)piece * h_k * d_k * es), round_up((size_t)piece * h_v * d_v * es),
          round_up((size_t)piece * h_v * sizeof(float))};
}

// Workspace: [cu arrays | state | 2 x (q, k, v, g, beta) | 2 x o | one piece's prefill workspace]
struct Layout {
  size_t cu, state, in[2], out[2], prefill, total, prefill_bytes;
  PieceBytes pb;
};
Layout layout(int64_t piece, int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype) {
  Layout L{};
  const size_t es = dtype == GDN_BF16 ? 2 : 4;
  L.pb = piece_bytes(piece, h_k, h_v, d_k, d_v, es);
  const size_t in_bytes = 2 * L.pb.q + L.pb.v + 2 * L.pb.g;
  L.cu = 0;
  L.state = kAlign;
  L.in[0] = L.state + round_up((size_t)h_v * d_v * d_k * sizeof(float));
  L.in[1] = L.in[0] + in_bytes;
  L.out[0] = L.in[1] + in_bytes;
  L.out[1] = L.out[0] + L.pb.v;
  L.prefill = L.out[1] + L.pb.v;
  L.prefill_bytes =
      gdn_prefill_workspace_size(1, piece, h_k, h_v, d_k, d_v, dtype, GDN_ALGO_CHUNKED_SPLIT);
  L.total = L.prefill + round_up(L.prefill_bytes);
  return L;
}

__global__ void host_cu_kernel(int32_t* cu, int32_t piece, int32_t last) {
  cu[0] = 0;
  cu[1] = piece;
  cu[4] = 0;
  cu[5] = last;
}

// The library's copy streams and events, one set per device, created on the
// first call made with that device current.  A call enqueues its whole
// schedule under the mutex: a wait captures the event's latest record when it
// is enqueued, so a later call re-recording the ring cannot disturb it.
struct Pipe {
  bool ready = false;
  cudaStream_t in_stream = nullptr, out_stream = nullptr;
  cudaEvent_t start = nullptr, in_done[kRing] = {}, comp_done[kRing] = {}, out_done[kRing] = {};
  cudaEvent_t state_done = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
Pipe g_pipes[kMaxDevices];

cudaError_t make_pipe(Pipe& P) {
  if (P.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&P.in_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&P.out_stream, cudaStreamNonBlocking);
  cudaEvent_t* evs[] = {&P.start, &P.state_done};
  for (cudaEvent_t* ev : evs)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  for (int i = 0; i < kRing && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&P.in_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&P.comp_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&P.out_done[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) P.ready = true;
  return e;
}

}  // namespace

extern "C" {

size_t gdn_prefill_host_workspace_size(int64_t piece_tokens, int32_t h_k, int32_t h_v,
                                       int32_t d_k, int32_t d_v, gdn_dtype dtype) {
  if (piece_tokens <= 0 || piece_tokens % kPieceQuantum || piece_tokens > INT32_MAX) return 0;
  if (h_k <= 0 || h_v <= 0 || d_k <= 0 || d_v <= 0) return 0;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return 0;
  return layout(piece_tokens, h_k, h_v, d_k, d_v, dtype).total;
}

gdn_status gdn_prefill_host(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* state_in, float* state_out, void* o,
                            int64_t total_tokens, int32_t h_k, int32_t h_v, int32_t d_k,
                            int32_t d_v, gdn_dtype dtype, float scale, int64_t piece_tokens,
                            void* workspace, size_t workspace_bytes, uint32_t options,
                            gdn_stream_t stream) {
  if (total_tokens < 0 || piece_tokens <= 0 || piece_tokens % kPieceQuantum ||
      piece_tokens > INT32_MAX)
    return GDN_ERR_INVALID_ARG;
  if (options & ~static_cast<uint32_t>(GDN_OPT_QK_L2NORM)) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED_DTYPE;
  if (h_k <= 0 || h_v <= 0 || d_k <= 0 || d_v <= 0) return GDN_ERR_INVALID_ARG;
  if (h_v % h_k != 0 || !head_dim_ok(d_k) || !head_dim_ok(d_v) || h_v > 65535)
    return GDN_ERR_UNSUPPORTED_SHAPE;
  if (total_tokens > INT32_MAX) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (!state_out || !workspace) return GDN_ERR_NULL_POINTER;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_NULL_POINTER;
  if (!aligned16(workspace)) return GDN_ERR_MISALIGNED;
  const Layout L = layout(piece_tokens, h_k, h_v, d_k, d_v, dtype);
  if (workspace_bytes < L.total) return GDN_ERR_WORKSPACE_TOO_SMALL;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  Pipe& P = g_pipes[dev];
  if (make_pipe(P) != cudaSuccess) return GDN_ERR_CUDA;

  const gdn_algo algo = gdn::chunked_supports(h_k, h_v, d_k, d_v, dtype) ? GDN_ALGO_CHUNKED_SPLIT
                                                                          : GDN_ALGO_SCAN;
  const size_t es = dtype == GDN_BF16 ? 2 : 4;
  const size_t qk_row = (size_t)h_k * d_k * es, vo_row = (size_t)h_v * d_v * es;
  const size_t gb_row = (size_t)h_v * sizeof(float);
  const size_t state_bytes = (size_t)h_v * d_v * d_k * sizeof(float);
  const int64_t n_pieces =
      total_tokens == 0 ? 1 : (total_tokens + piece_tokens - 1) / piece_tokens;
  const int64_t last = total_tokens - (n_pieces - 1) * piece_tokens;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* cu = reinterpret_cast<int32_t*>(ws + L.cu);
  float* dstate = reinterpret_cast<float*>(ws + L.state);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
#define GDN_TRY(x) \
  if ((x) != cudaSuccess) return GDN_ERR_CUDA

  host_cu_kernel<<<1, 1, 0, s>>>(cu, static_cast<int32_t>(piece_tokens),
                                 static_cast<int32_t>(last));
  GDN_TRY(cudaGetLastError());
  GDN_TRY(cudaEventRecord(P.start, s));
  GDN_TRY(cudaStreamWaitEvent(P.in_stream, P.start, 0));
  GDN_TRY(cudaStreamWaitEvent(P.out_stream, P.start, 0));
  if (state_in) GDN_TRY(cudaMemcpyAsync(dstate, state_in, state_bytes, h2d, P.in_stream));
  for (int64_t i = 0; i < n_pieces; ++i) {
    const int r = (int)(i % kRing), b = (int)(i & 1);
    const int64_t t0 = i * piece_tokens;
    const int64_t len = i == n_pieces - 1 ? last : piece_tokens;
    uint8_t* in = ws + L.in[b];
    uint8_t *dq = in, *dk = in + L.pb.q, *dv = in + 2 * L.pb.q;
    float* dg = reinterpret_cast<float*>(in + 2 * L.pb.q + L.pb.v);
    float* dbeta = reinterpret_cast<float*>(in + 2 * L.pb.q + L.pb.v + L.pb.g);
    uint8_t* dout = ws + L.out[b];
    // copy-in: the buffer's previous piece (i - 2) has been consumed by its prefill
    if (i >= 2) GDN_TRY(cudaStreamWaitEvent(P.in_stream, P.comp_done[(i - 2) % kRing], 0));
    if (len > 0) {
      GDN_TRY(cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + t0 * qk_row, len * qk_row, h2d,
                              P.in_stream));
      GDN_TRY(cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + t0 * qk_row, len * qk_row, h2d,
                              P.in_stream));
      GDN_TRY(cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + t0 * vo_row, len * vo_row, h2d,
                              P.in_stream));
      GDN_TRY(cudaMemcpyAsync(dg, g + t0 * h_v, len * gb_row, h2d, P.in_stream));
      GDN_TRY(cudaMemcpyAsync(dbeta, beta + t0 * h_v, len * gb_row, h2d, P.in_stream));
    }
    GDN_TRY(cudaEventRecord(P.in_done[r], P.in_stream));
    // compute: inputs landed, and the output buffer's previous piece has been copied out
    GDN_TRY(cudaStreamWaitEvent(s, P.in_done[r], 0));
    if (i >= 2) GDN_TRY(cudaStreamWaitEvent(s, P.out_done[(i - 2) % kRing], 0));
    const gdn_status st = gdn_prefill_ex(
        dq, dk, dv, dg, dbeta, (i == 0 && !state_in) ? nullptr : dstate, dstate, dout,
        i == n_pieces - 1 ? cu + 4 : cu, 1, len, h_k, h_v, d_k, d_v, dtype, scale, algo,
        ws + L.prefill, L.prefill_bytes, options, stream);
    if (st != GDN_OK) return st;
    GDN_TRY(cudaEventRecord(P.comp_done[r], s));
    // copy-out
    GDN_TRY(cudaStreamWaitEvent(P.out_stream, P.comp_done[r], 0));
    if (len > 0)
      GDN_TRY(cudaMemcpyAsync(static_cast<uint8_t*>(o) + t0 * vo_row, dout, len * vo_row, d2h,
                              P.out_stream));
    GDN_TRY(cudaEventRecord(P.out_done[r], P.out_stream));
  }
  // the final state after the last piece, then join both library streams into the caller's
  GDN_TRY(cudaMemcpyAsync(state_out, dstate, state_bytes, d2h, P.out_stream));
  GDN_TRY(cudaEventRecord(P.state_done, P.out_stream));
  GDN_TRY(cudaStreamWaitEvent(s, P.state_done, 0));
#undef GDN_TRY
  return GDN_OK;
}

}  // extern "C"
