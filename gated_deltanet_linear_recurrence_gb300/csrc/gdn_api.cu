// gdn_api.cu — the C ABI: argument validation, algorithm choice, launches,
// and the per-device error word.  Declarations and contracts: include/gdn.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <cstdlib>
#include <mutex>

#include "gdn.h"
#include "params.h"

namespace {

// Device-side error word (one per device that loads the library).  Kernels
// receive its address as an argument; gdn_stream_status reads and clears it.
__device__ int g_gdn_error_word = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};

gdn_status error_word(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gdn_error_word) != cudaSuccess) return GDN_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_err_ptr[dev];
  return GDN_OK;
}

bool head_dim_ok(int32_t d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_heads(int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v) {
  if (h_k <= 0 || h_v <= 0 || d_k <= 0 || d_v <= 0) return GDN_ERR_INVALID_ARG;
  if (h_v % h_k != 0 || !head_dim_ok(d_k) || !head_dim_ok(d_v) || h_v > 65535)
    return GDN_ERR_UNSUPPORTED_SHAPE;
  return GDN_OK;
}

// Which evaluation is fastest, by shape: a table measured on GB300 with
// bench.py --sweep (N sequences of equal length L = 8 ... 8192, at most 65,536
// tokens a call, bf16, L2 flushed before each call, every form timed at every
// L; a threshold is the smallest swept L from which the faster form stays
// faster, so it is known to a factor of two and flips between neighbouring
// lengths where two forms time within noise of each other).  Per entry:
//   scan_below      sequences shorter than this take the token scan (per
//                   sequence, so one call can mix the two);
//   split_from_avg  the two-kernel form instead of the fused kernel from this
//                   average length (when the caller's workspace holds it);
//   coop_from_avg   the cooperative form instead of the two kernels from this
//                   average length (when its chains fit: coop_supported).
// A shape takes the entry with the same d_k that is nearest in d_v, then in
// log2(h_v), then in log2(N).  fp32 inputs, and shapes no chunked form covers,
// always scan.
struct FormThresholds {
  int32_t scan_below;
  int64_t split_from_avg, coop_from_avg;
};
struct CrossoverEntry {
  int32_t d_k, d_v, h_v, n;
  FormThresholds t;
};
constexpr int64_t kNever = INT64_MAX;
constexpr CrossoverEntry kCrossover[] = {
    // d_k, d_v, h_v, N: {scan below, two kernels from, cooperative from}
    {128, 128, 32, 1, {8, 256, 4096}},
    {128, 128, 32, 4, {16, 8, kNever}},
    {128, 128, 32, 16, {8, 8, kNever}},
    {128, 128, 4, 1, {16, 256, kNever}},
    {128, 128, 4, 4, {16, 512, kNever}},
    {128, 128, 4, 16, {32, 128, kNever}},
    {128, 64, 32, 1, {16, 256, 4096}},
    {128, 64, 32, 4, {16, 128, kNever}},
    {128, 64, 32, 16, {16, 8, kNever}},
    {128, 64, 4, 1, {16, 256, kNever}},
    {128, 64, 4, 4, {8, 256, kNever}},
    {128, 64, 4, 16, {16, 512, kNever}},
    {128, 32, 32, 1, {16, 256, kNever}},
    {128, 32, 32, 4, {16, 4096, kNever}},
    {128, 32, 32, 16, {32, 1024, kNever}},
    {128, 32, 4, 1, {16, 256, kNever}},
    {128, 32, 4, 4, {16, 512, kNever}},
    {128, 32, 4, 16, {16, 512, kNever}},
    {64, 128, 32, 1, {16, 0, 4096}},
    {64, 128, 32, 4, {32, 0, kNever}},
    {64, 128, 32, 16, {16, 0, kNever}},
    {64, 128, 4, 1, {16, 0, kNever}},
    {64, 128, 4, 4, {32, 0, kNever}},
    {64, 128, 4, 16, {32, 0, kNever}},
    {64, 64, 32, 1, {16, 0, 4096}},
    {64, 64, 32, 4, {32, 0, kNever}},
    {64, 64, 32, 16, {32, 0, kNever}},
    {64, 64, 4, 1, {16, 0, kNever}},
    {64, 64, 4, 4, {32, 0, kNever}},
    {64, 64, 4, 16, {32, 0, kNever}},
    {64, 32, 32, 1, {16, 0, kNever}},
    {64, 32, 32, 4, {32, 0, kNever}},
    {64, 32, 32, 16, {64, 0, kNever}},
    {64, 32, 4, 1, {16, 0, kNever}},
    {64, 32, 4, 4, {32, 0, kNever}},
    {64, 32, 4, 16, {32, 0, kNever}},
};

// The sequences average at least `threshold` tokens (no overflow for kNever).
bool avg_at_least(int64_t total_tokens, int32_t num_seqs, int64_t threshold) {
  return num_seqs > 0 && total_tokens / num_seqs >= threshold;
}

int log2_floor(int64_t x) {
  int r = 0;
  while (x > 1) {
    x >>= 1;
    ++r;
  }
  return r;
}

FormThresholds thresholds_for(int32_t h_v, int32_t d_k, int32_t d_v, int32_t num_seqs) {
  const CrossoverEntry* best = nullptr;
  int64_t best_key = INT64_MAX;
  for (const CrossoverEntry& e : kCrossover) {
    const int64_t dk = e.d_k == d_k ? 0 : 1;
    const int64_t dv = e.d_v > d_v ? e.d_v - d_v : d_v - e.d_v;
    const int64_t dh = std::abs(log2_floor(e.h_v) - log2_floor(h_v));
    const int64_t dn = std::abs(log2_floor(e.n) - log2_floor(num_seqs > 0 ? num_seqs : 1));
    const int64_t key = ((dk * 1024 + dv) * 64 + dh) * 64 + dn;
    if (key < best_key) {
      best_key = key;
      best = &e;
    }
  }
  return best->t;
}

int32_t crossover_for(int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, int dtype,
                      int32_t num_seqs = 1) {
  if (!gdn::chunked_supports(h_k, h_v, d_k, d_v, dtype)) return INT32_MAX;
  return thresholds_for(h_v, d_k, d_v, num_seqs).scan_below;
}

constexpr int32_t kAttnHeadDim = 256;
constexpr int32_t kAttnMaxGroup = 8;
constexpr int32_t kAttnMinBlock = 128;  // the smallest block the library picks

gdn_status attn_shape(int32_t batch, int32_t h_q, int32_t h_kv, int32_t head_dim,
                      int32_t capacity, int layout, int32_t block_keys) {
  if (batch < 0 || capacity < 0 || h_q <= 0 || h_kv <= 0 || head_dim <= 0)
    return GDN_ERR_INVALID_ARG;
  if (layout < GDN_ATTN_AUTO || layout > GDN_ATTN_FIXED_BLOCK) return GDN_ERR_INVALID_ARG;
  if (block_keys < 0 || block_keys % 64 != 0) return GDN_ERR_INVALID_ARG;
  if (head_dim != kAttnHeadDim || h_q % h_kv != 0 || h_q / h_kv > kAttnMaxGroup)
    return GDN_ERR_UNSUPPORTED_SHAPE;
  if (batch > 65535 || h_kv > 65535 || (int64_t)batch * h_kv * capacity > INT32_MAX)
    return GDN_ERR_UNSUPPORTED_SHAPE;
  return GDN_OK;
}

// Checks of a prefill call's sizes, enums and options (no pointers).  With the
// normalisation option the chunked evaluation is the two-kernel one (the fused
// kernel does not implement the option).
gdn_status prefill_sizes(int32_t num_seqs, int64_t total_tokens, int32_t h_k, int32_t h_v,
                         int32_t d_k, int32_t d_v, gdn_dtype dtype, gdn_algo algo,
                         uint32_t options) {
  if (num_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (options & ~static_cast<uint32_t>(GDN_OPT_QK_L2NORM)) return GDN_ERR_INVALID_ARG;
  if (algo != GDN_ALGO_AUTO && algo != GDN_ALGO_SCAN && algo != GDN_ALGO_CHUNKED &&
      algo != GDN_ALGO_CHUNKED_FUSED && algo != GDN_ALGO_CHUNKED_SPLIT &&
      algo != GDN_ALGO_CHUNKED_COOP)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED_DTYPE;
  const gdn_status st = check_heads(h_k, h_v, d_k, d_v);
  if (st != GDN_OK) return st;
  if (total_tokens > INT32_MAX) return GDN_ERR_UNSUPPORTED_SHAPE;  // cu_seqlens is int32
  if ((options & GDN_OPT_QK_L2NORM) && algo == GDN_ALGO_CHUNKED_FUSED) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

// The current device's SM count, or -1 if the query fails.
int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return sms;
}

// Which kernels a prefill call runs, from its sizes alone (shared by
// gdn_prefill_ex and gdn_prefill_form).  have_ws / ws_aligned: a workspace
// pointer is given / it is 16-byte aligned; sms: the device's SM count (< 0:
// the query failed).  Errors are those gdn_prefill returns for these sizes.
struct Route {
  gdn_status st = GDN_OK;
  bool run_scan = true, run_chunk = false, split = false, coop = false;
  int32_t min_chunk_len = INT32_MAX;
};
Route route_prefill(gdn_algo algo, int32_t num_seqs, int64_t total_tokens, int32_t h_k,
                    int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype, bool qk_norm,
                    bool have_ws, bool ws_aligned, size_t workspace_bytes, int sms) {
  Route r;
  auto fail = [&r](gdn_status st) {
    r.st = st;
    return r;
  };
  const bool chunk_ok = gdn::chunked_supports(h_k, h_v, d_k, d_v, dtype);
  // the fused kernel covers d_k = 128 without the normalisation option
  const bool fused_ok = gdn::fused_supports(h_k, h_v, d_k, d_v, dtype) && !qk_norm;
  const bool chunk_only = algo == GDN_ALGO_CHUNKED || algo == GDN_ALGO_CHUNKED_FUSED ||
                          algo == GDN_ALGO_CHUNKED_SPLIT || algo == GDN_ALGO_CHUNKED_COOP;
  if (chunk_only && !chunk_ok)
    return fail(dtype == GDN_F32 ? GDN_ERR_UNSUPPORTED_DTYPE : GDN_ERR_UNSUPPORTED_SHAPE);
  if (algo == GDN_ALGO_CHUNKED_FUSED && !gdn::fused_supports(h_k, h_v, d_k, d_v, dtype))
    return fail(GDN_ERR_UNSUPPORTED_SHAPE);
  const FormThresholds th = thresholds_for(h_v, d_k, d_v, num_seqs);
  // Scan for sequences shorter than min_chunk_len, chunked for the rest.  With
  // one sequence its length is total_tokens, so only the kernel with work runs.
  if (algo == GDN_ALGO_SCAN) {
    r.min_chunk_len = INT32_MAX;
  } else if (chunk_only) {
    r.min_chunk_len = 0;
    r.run_scan = false;
    r.run_chunk = true;
  } else {
    // The table was measured on batches of equal lengths, so a batch whose
    // sequences average fewer than scan_below tokens goes to the scan whole
    // (no chunked launch with nothing to do); otherwise sequences shorter than
    // scan_below still take the scan, beside the chunked kernels.
    r.run_chunk = chunk_ok && avg_at_least(total_tokens, num_seqs, th.scan_below);
    r.min_chunk_len = r.run_chunk ? th.scan_below : INT32_MAX;
    r.run_scan = !(num_seqs == 1 && r.run_chunk);
  }
  // The chunked evaluation runs as one fused kernel, as two kernels meeting in
  // the caller's workspace (forced by GDN_ALGO_CHUNKED_SPLIT; otherwise when the
  // sequences are long enough, or the fused kernel does not cover the call, and
  // the workspace is large enough), or as one cooperative kernel through it.
  if (r.run_chunk && algo == GDN_ALGO_CHUNKED_COOP) {
    if (!have_ws) return fail(GDN_ERR_NULL_POINTER);
    if (!ws_aligned) return fail(GDN_ERR_MISALIGNED);
    if (workspace_bytes < gdn::coop_workspace_bytes(num_seqs, total_tokens, h_v))
      return fail(GDN_ERR_WORKSPACE_TOO_SMALL);
    if (sms < 0) return fail(GDN_ERR_CUDA);
    if (!gdn::coop_supported(num_seqs, h_v, d_v, sms)) return fail(GDN_ERR_UNSUPPORTED_SHAPE);
    r.coop = true;
  } else if (r.run_chunk && algo != GDN_ALGO_CHUNKED_FUSED) {
    const size_t need = gdn::split_workspace_bytes(num_seqs, total_tokens, h_v);
    if (algo == GDN_ALGO_CHUNKED_SPLIT) {
      if (!have_ws) return fail(GDN_ERR_NULL_POINTER);
      if (workspace_bytes < need) return fail(GDN_ERR_WORKSPACE_TOO_SMALL);
    }
    if (have_ws && !ws_aligned) return fail(GDN_ERR_MISALIGNED);
    r.split = have_ws && workspace_bytes >= need &&
              (algo == GDN_ALGO_CHUNKED_SPLIT || !fused_ok ||
               avg_at_least(total_tokens, num_seqs, th.split_from_avg));
    if (!fused_ok && !r.split) {  // no room for the two kernels: the token scan takes everything
      if (algo == GDN_ALGO_CHUNKED) return fail(GDN_ERR_WORKSPACE_TOO_SMALL);
      r.run_chunk = false;
      r.run_scan = true;
      r.min_chunk_len = INT32_MAX;
    }
  }
  if (r.split && algo != GDN_ALGO_CHUNKED_SPLIT &&
      avg_at_least(total_tokens, num_seqs, th.coop_from_avg) &&
      workspace_bytes >= gdn::coop_workspace_bytes(num_seqs, total_tokens, h_v) && sms > 0 &&
      gdn::coop_supported(num_seqs, h_v, d_v, sms)) {
    r.coop = true;
    r.split = false;
  }
  return r;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_NULL_POINTER: return "GDN_ERR_NULL_POINTER";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED_SHAPE: return "GDN_ERR_UNSUPPORTED_SHAPE";
    case GDN_ERR_UNSUPPORTED_DTYPE: return "GDN_ERR_UNSUPPORTED_DTYPE";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
    case GDN_ERR_BAD_CU_SEQLENS: return "GDN_ERR_BAD_CU_SEQLENS";
    case GDN_ERR_WORKSPACE_TOO_SMALL: return "GDN_ERR_WORKSPACE_TOO_SMALL";
    case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_BAD_CACHE_LEN: return "GDN_ERR_BAD_CACHE_LEN";
  }
  return "GDN_ERR_UNKNOWN";
}

int32_t gdn_prefill_crossover_tokens(int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v,
                                     gdn_dtype dtype) {
  if (check_heads(h_k, h_v, d_k, d_v) != GDN_OK) return INT32_MAX;
  return crossover_for(h_k, h_v, d_k, d_v, dtype);
}

size_t gdn_prefill_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t h_k,
                                  int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype,
                                  gdn_algo algo) {
  if (num_seqs < 0 || total_tokens < 0 || check_heads(h_k, h_v, d_k, d_v) != GDN_OK) return 0;
  if (algo == GDN_ALGO_SCAN || algo == GDN_ALGO_CHUNKED_FUSED) return 0;
  if (!gdn::chunked_supports(h_k, h_v, d_k, d_v, dtype)) return 0;
  if (algo == GDN_ALGO_CHUNKED_SPLIT) return gdn::split_workspace_bytes(num_seqs, total_tokens, h_v);
  // AUTO and CHUNKED: none while the fused kernel is the faster form (and covers
  // the shape), else room for the cooperative form (the two-kernel form plus flags)
  const FormThresholds th = thresholds_for(h_v, d_k, d_v, num_seqs);
  if (algo != GDN_ALGO_CHUNKED_COOP && gdn::fused_supports(h_k, h_v, d_k, d_v, dtype) &&
      !avg_at_least(total_tokens, num_seqs, th.split_from_avg))
    return 0;
  return gdn::coop_workspace_bytes(num_seqs, total_tokens, h_v);
}

int32_t gdn_prefill_form(int32_t num_seqs, int64_t total_tokens, int32_t h_k, int32_t h_v,
                         int32_t d_k, int32_t d_v, gdn_dtype dtype, gdn_algo algo,
                         size_t workspace_bytes, uint32_t options, int32_t sm_count) {
  const gdn_status st =
      prefill_sizes(num_seqs, total_tokens, h_k, h_v, d_k, d_v, dtype, algo, options);
  if (st != GDN_OK) return -static_cast<int32_t>(st);
  if (num_seqs == 0) return GDN_ALGO_SCAN;  // nothing runs
  const int sms = sm_count > 0 ? sm_count : device_sm_count();
  const Route r = route_prefill(algo, num_seqs, total_tokens, h_k, h_v, d_k, d_v, dtype,
                                (options & GDN_OPT_QK_L2NORM) != 0, workspace_bytes > 0, true,
                                workspace_bytes, sms);
  if (r.st != GDN_OK) return -static_cast<int32_t>(r.st);
  if (!r.run_chunk) return GDN_ALGO_SCAN;
  return r.coop ? GDN_ALGO_CHUNKED_COOP : r.split ? GDN_ALGO_CHUNKED_SPLIT : GDN_ALGO_CHUNKED_FUSED;
}

gdn_status gdn_prefill(const void* q, const void* k, const void* v, const float* g,
                       const float* beta, const float* state_in, float* state_out, void* o,
                       const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                       int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype,
                       float scale, gdn_algo algo, void* workspace, size_t workspace_bytes,
                       gdn_stream_t stream) {
  return gdn_prefill_ex(q, k, v, g, beta, state_in, state_out, o, cu_seqlens, num_seqs,
                        total_tokens, h_k, h_v, d_k, d_v, dtype, scale, algo, workspace,
                        workspace_bytes, 0u, stream);
}

gdn_status gdn_prefill_ex(const void* q, const void* k, const void* v, const float* g,
                          const float* beta, const float* state_in, float* state_out, void* o,
                          const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                          int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype,
                          float scale, gdn_algo algo, void* workspace, size_t workspace_bytes,
                          uint32_t options, gdn_stream_t stream) {
  gdn_status st = prefill_sizes(num_seqs, total_tokens, h_k, h_v, d_k, d_v, dtype, algo, options);
  if (st != GDN_OK) return st;
  if (num_seqs == 0) return GDN_OK;
  if (!cu_seqlens || !state_out) return GDN_ERR_NULL_POINTER;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_NULL_POINTER;
  const void* ptrs[] = {q, k, v, g, beta, state_in, state_out, o, cu_seqlens};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
  // state_in may be state_out exactly; any partial overlap is refused
  const size_t state_bytes = (size_t)num_seqs * h_v * d_v * d_k * sizeof(float);
  if (state_in && state_in != state_out) {
    const char* a = reinterpret_cast<const char*>(state_in);
    const char* b = reinterpret_cast<const char*>(state_out);
    if (a < b + state_bytes && b < a + state_bytes) return GDN_ERR_INVALID_ARG;
  }
  const bool qk_norm = (options & GDN_OPT_QK_L2NORM) != 0;
  const int sms = device_sm_count();
  const Route r = route_prefill(algo, num_seqs, total_tokens, h_k, h_v, d_k, d_v, dtype, qk_norm,
                                workspace != nullptr, !workspace || aligned16(workspace),
                                workspace_bytes, sms);
  if (r.st != GDN_OK) return r.st;

  gdn::PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.state_in = state_in; a.state_out = state_out; a.o = o; a.cu_seqlens = cu_seqlens;
  a.num_seqs = num_seqs; a.total_tokens = total_tokens;
  a.h_k = h_k; a.h_v = h_v; a.d_k = d_k; a.d_v = d_v;
  a.dtype = dtype; a.scale = scale;
  a.qk_norm = qk_norm ? 1 : 0;
  a.workspace = workspace; a.workspace_bytes = workspace_bytes;
  a.min_chunk_len = r.min_chunk_len;
  const bool run_scan = r.run_scan, run_chunk = r.run_chunk, split = r.split, coop = r.coop;
  st = error_word(&a.err);
  if (st != GDN_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (run_chunk) {
    cudaError_t e = coop    ? gdn::launch_chunked_coop(a, workspace, s)
                    : split ? gdn::launch_chunked_split(a, workspace, s)
                            : gdn::launch_chunked(a, s);
    // The cooperative grid needs every SM free for it; when AUTO or CHUNKED chose
    // it and the launch is refused (other work holds SMs), the two kernels run.
    if (coop && algo != GDN_ALGO_CHUNKED_COOP &&
        (e == cudaErrorNotSupported || e == cudaErrorCooperativeLaunchTooLarge)) {
      (void)cudaGetLastError();  // a refused launch configuration, not a sticky error
      e = gdn::launch_chunked_split(a, workspace, s);
    }
    if (e == cudaErrorNotSupported || e == cudaErrorCooperativeLaunchTooLarge)
      return GDN_ERR_UNSUPPORTED_SHAPE;
    if (e != cudaSuccess) return GDN_ERR_CUDA;
  }
  if (run_scan && gdn::launch_scan(a, s) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float* state, void* o, int32_t batch, int32_t h_k,
                           int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype, float scale,
                           gdn_stream_t stream) {
  return gdn_decode_step_ex(q, k, v, g, beta, state, o, batch, h_k, h_v, d_k, d_v, dtype, scale,
                            0u, stream);
}

gdn_status gdn_decode_step_ex(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* state, void* o, int32_t batch,
                              int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, gdn_dtype dtype,
                              float scale, uint32_t options, gdn_stream_t stream) {
  if (batch < 0) return GDN_ERR_INVALID_ARG;
  if (options & ~static_cast<uint32_t>(GDN_OPT_QK_L2NORM)) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED_DTYPE;
  gdn_status st = check_heads(h_k, h_v, d_k, d_v);
  if (st != GDN_OK) return st;
  if (batch == 0) return GDN_OK;
  if (!q || !k || !v || !g || !beta || !state || !o) return GDN_ERR_NULL_POINTER;
  const void* ptrs[] = {q, k, v, g, beta, state, o};
  for (const void* p : ptrs)
    if (!aligned16(p)) return GDN_ERR_MISALIGNED;
  gdn::DecodeArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.state = state; a.o = o;
  a.batch = batch; a.h_k = h_k; a.h_v = h_v; a.d_k = d_k; a.d_v = d_v;
  a.dtype = dtype; a.scale = scale;
  a.qk_norm = (options & GDN_OPT_QK_L2NORM) ? 1 : 0;
  if (gdn::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_decode_step_rmsnorm(const void* q, const void* k, const void* v, const float* g,
                                   const float* beta, float* state, void* o,
                                   const float* norm_weight, float norm_eps, int32_t batch,
                                   int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v,
                                   gdn_dtype dtype, float scale, uint32_t options,
                                   gdn_stream_t stream) {
  if (batch < 0) return GDN_ERR_INVALID_ARG;
  if (options & ~static_cast<uint32_t>(GDN_OPT_QK_L2NORM)) return GDN_ERR_INVALID_ARG;
  if (!(norm_eps >= 0.f) || norm_eps > 3.0e38f) return GDN_ERR_INVALID_ARG;  // NaN too
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED_DTYPE;
  gdn_status st = check_heads(h_k, h_v, d_k, d_v);
  if (st != GDN_OK) return st;
  if (batch == 0) return GDN_OK;
  if (!q || !k || !v || !g || !beta || !state || !o) return GDN_ERR_NULL_POINTER;
  const void* ptrs[] = {q, k, v, g, beta, state, o, norm_weight};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
  gdn::DecodeArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.state = state; a.o = o;
  a.batch = batch; a.h_k = h_k; a.h_v = h_v; a.d_k = d_k; a.d_v = d_v;
  a.dtype = dtype; a.scale = scale;
  a.qk_norm = (options & GDN_OPT_QK_L2NORM) ? 1 : 0;
  a.out_norm = 1;
  a.norm_weight = norm_weight;
  a.norm_eps = norm_eps;
  if (gdn::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_output_rmsnorm(void* o, const float* norm_weight, int64_t rows, int32_t h_v,
                              int32_t d_v, gdn_dtype dtype, float norm_eps, gdn_stream_t stream) {
  if (rows < 0 || h_v <= 0 || d_v <= 0) return GDN_ERR_INVALID_ARG;
  if (!(norm_eps >= 0.f) || norm_eps > 3.0e38f) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED_DTYPE;
  if (!head_dim_ok(d_v) || h_v > 65535) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return GDN_OK;
  if (!o) return GDN_ERR_NULL_POINTER;
  if (!aligned16(o) || (norm_weight && !aligned16(norm_weight))) return GDN_ERR_MISALIGNED;
  if (gdn::launch_output_rmsnorm(o, norm_weight, rows * h_v, d_v, dtype, norm_eps,
                                 reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_decode_multi(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float* state, void* o, float* snapshots,
                            int32_t batch, int32_t n_tokens, int32_t h_k, int32_t h_v,
                            int32_t d_k, int32_t d_v, gdn_dtype dtype, float scale,
                            uint32_t options, gdn_stream_t stream) {
  if (batch < 0 || n_tokens < 1 || n_tokens > 1024) return GDN_ERR_INVALID_ARG;
  if (options & ~static_cast<uint32_t>(GDN_OPT_QK_L2NORM)) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED_DTYPE;
  gdn_status st = check_heads(h_k, h_v, d_k, d_v);
  if (st != GDN_OK) return st;
  if (batch == 0) return GDN_OK;
  if (!q || !k || !v || !g || !beta || !state || !o) return GDN_ERR_NULL_POINTER;
  const void* ptrs[] = {q, k, v, g, beta, state, o, snapshots};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
  if (snapshots) {  // the snapshots must not overlap the state
    const size_t state_bytes = (size_t)batch * h_v * d_v * d_k * sizeof(float);
    const char* a = reinterpret_cast<const char*>(state);
    const char* b = reinterpret_cast<const char*>(snapshots);
    if (a < b + state_bytes * n_tokens && b < a + state_bytes) return GDN_ERR_INVALID_ARG;
  }
  gdn::DecodeMultiArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.state = state; a.o = o;
  a.snapshots = snapshots;
  a.batch = batch; a.n_tokens = n_tokens; a.h_k = h_k; a.h_v = h_v; a.d_k = d_k; a.d_v = d_v;
  a.dtype = dtype; a.scale = scale;
  a.qk_norm = (options & GDN_OPT_QK_L2NORM) ? 1 : 0;
  if (gdn::launch_decode_multi(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

size_t gdn_attn_decode_workspace_size(int32_t batch, int32_t h_q, int32_t h_kv,
                                      int32_t head_dim, int32_t capacity,
                                      gdn_attn_layout layout, int32_t block_keys) {
  if (attn_shape(batch, h_q, h_kv, head_dim, capacity, layout, block_keys) != GDN_OK) return 0;
  if (layout == GDN_ATTN_GENERAL) return 0;
  const int64_t bk = block_keys > 0 ? block_keys : kAttnMinBlock;
  const int64_t n = capacity > 0 ? (capacity + bk - 1) / bk : 1;
  if (n <= 1) return 0;
  return (size_t)batch * h_q * n * (head_dim + 2) * sizeof(float);
}

int32_t gdn_attn_decode_block_keys(int32_t batch, int32_t h_q, int32_t h_kv, int32_t head_dim,
                                   int32_t capacity, gdn_attn_layout layout,
                                   int32_t block_keys) {
  if (attn_shape(batch, h_q, h_kv, head_dim, capacity, layout, block_keys) != GDN_OK) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return gdn::attn_plan(batch, h_kv, capacity, layout, block_keys, sms).block_keys;
}

gdn_status gdn_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* cache_len, void* o, int32_t batch, int32_t h_q,
                           int32_t h_kv, int32_t head_dim, int32_t capacity, gdn_dtype dtype,
                           float scale, gdn_attn_layout layout, int32_t block_keys,
                           void* workspace, size_t workspace_bytes, gdn_stream_t stream) {
  gdn_status st = attn_shape(batch, h_q, h_kv, head_dim, capacity, layout, block_keys);
  if (st != GDN_OK) return st;
  if (dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED_DTYPE;
  if (batch == 0) return GDN_OK;
  if (!q || !o || !cache_len) return GDN_ERR_NULL_POINTER;
  if (capacity > 0 && (!k_cache || !v_cache)) return GDN_ERR_NULL_POINTER;
  const void* ptrs[] = {q, o, k_cache, v_cache, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(cache_len) & 3u) != 0) return GDN_ERR_MISALIGNED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GDN_ERR_CUDA;
  gdn::AttnPlan plan = gdn::attn_plan(batch, h_kv, capacity, layout, block_keys, sms);
  size_t need = gdn::attn_partial_bytes(batch, h_q, plan);
  if (need > 0 && (!workspace || workspace_bytes < need)) {
    if (layout == GDN_ATTN_FIXED_BLOCK)
      return workspace ? GDN_ERR_WORKSPACE_TOO_SMALL : GDN_ERR_NULL_POINTER;
    plan = gdn::attn_plan(batch, h_kv, capacity, gdn::kAttnGeneral, 0, sms);  // AUTO: one block
    need = 0;
  }
  gdn::AttnArgs a{};
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.cache_len = cache_len; a.o = o;
  a.partial = need > 0 ? static_cast<float*>(workspace) : nullptr;
  a.batch = batch; a.h_q = h_q; a.h_kv = h_kv; a.head_dim = head_dim; a.capacity = capacity;
  a.block_keys = plan.block_keys; a.n_split = plan.n_split; a.scale = scale;
  st = error_word(&a.err);
  if (st != GDN_OK) return st;
  if (gdn::launch_attn_decode(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_selftest_wait_timeout(int32_t timeout_us, gdn_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return GDN_ERR_INVALID_ARG;
  int* err = nullptr;
  const gdn_status st = error_word(&err);
  if (st != GDN_OK) return st;
  if (gdn::launch_selftest_wait((uint64_t)timeout_us * 1000u, err,
                                reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_stream_status(gdn_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  int* err = nullptr;
  gdn_status st = error_word(&err);
  if (st != GDN_OK) return st;
  int word = 0;
  if (cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return GDN_ERR_CUDA;
  }
  return static_cast<gdn_status>(word);
}

}  // extern "C"
