// noalloc.cu — gdn_prefill_noalloc: the two-kernel chunked prefill with its
// scratch in a fixed array of library-owned device memory, for callers that
// cannot allocate device memory when they call in (contract in include/gdn.h).
//
// Who cannot allocate, and why: a host framework whose memory pool owns the
// device's memory and hands its plugins no scratch buffer, or a serving loop
// that must not call cudaMalloc / cudaFree on its hot path, because those calls
// can synchronise the device and stall every stream in flight.  This entry
// point needs no buffer beyond its inputs and outputs: the scratch that
// gdn_prefill takes as `workspace` is g_noalloc_scratch below.
//
// The array is shared by every call on a device (each device has its own
// copy of a __device__ variable).  Nothing in it has to start at zero: each
// call's first kernel writes the chunk table the later ones read, and the
// prepare kernel writes every package before the chain kernel reads it.
// Calls whose kernels overlap on one GPU therefore race on it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdn.h"

namespace {

constexpr size_t kScratchBytes = GDN_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the current device's copy of the array, looked up on the
// first call made with that device current.
gdn_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return GDN_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_prefill_noalloc(const void* q, const void* k, const void* v,
                                          const float* g, const float* beta,
                                          const float* state_in, float* state_out, void* o,
                                          const int32_t* cu_seqlens, int32_t num_seqs,
                                          int64_t total_tokens, int32_t h_k, int32_t h_v,
                                          int32_t d_k, int32_t d_v, gdn_dtype dtype, float scale,
                                          gdn_stream_t stream) {
  // Size check first, on the host arguments alone: a problem whose scratch
  // would not fit is refused before anything touches the device.
  const size_t need = gdn_prefill_workspace_size(num_seqs, total_tokens, h_k, h_v, d_k, d_v, dtype,
                                                 GDN_ALGO_CHUNKED_SPLIT);
  if (need > kScratchBytes) return GDN_ERR_WORKSPACE_TOO_SMALL;
  // need == 0 only for arguments that gdn_prefill refuses before it touches
  // the device (bad sizes, shapes or dtype): no set-up for those.
  void* scratch = nullptr;
  if (need > 0) {
    const gdn_status st = scratch_for_current_device(&scratch);
    if (st != GDN_OK) return st;
  }
  return gdn_prefill(q, k, v, g, beta, state_in, state_out, o, cu_seqlens, num_seqs, total_tokens,
                     h_k, h_v, d_k, d_v, dtype, scale, GDN_ALGO_CHUNKED_SPLIT, scratch,
                     scratch ? kScratchBytes : 0, stream);
}
