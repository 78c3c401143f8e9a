// scan_prefill.cu — token-scan prefill: every state row stays in registers
// from the first token of its sequence to the last.
//
// Page "Optimizing on-device inference for Apple Silicon", section "Keep the
// recurrent state on-chip": each slice of the state matrix is loaded into the
// registers of one SIMD group once, carried across the whole scan, partial
// results are exchanged with SIMD-group operations instead of threadgroup
// memory, and the state is written back only after the scan.  Section "Qwen
// creates three distinct workload shapes": the scan is one of the two ways to
// evaluate a prefill; the chunked kernel is the other.
//
// Work split: one warp per (sequence, value head, kRowsPerWarp rows); the
// per-token arithmetic is the row identity of rows.cuh.  The loads for token
// t+1 are issued before the arithmetic of token t.
//
// cu_seqlens is read on the device.  Each CTA checks its own sequence's bounds
// (0 <= cu[n] <= cu[n+1] <= T, cu[0] = 0, cu[N] = T); on a violation it records
// GDN_ERR_BAD_CU_SEQLENS in the error word and touches no memory.
#include <cuda_bf16.h>

#include "params.h"
#include "rows.cuh"

namespace gdn {
namespace {

constexpr int kScanWarps = 4;

template <int DK, int M, typename T>
struct TokenIn {
  float4 k4[M], q4[M];
  float g, beta, v;
};

template <int DK, int L, int M, typename T>
__device__ __forceinline__ void load_token(TokenIn<DK, M, T>& x, const T* __restrict__ q,
                                           const T* __restrict__ k, const T* __restrict__ v,
                                           const float* __restrict__ g,
                                           const float* __restrict__ beta, int64_t t,
                                           int32_t h_k, int32_t h_v, int32_t d_v, int hk, int h,
                                           int lam, int row_mine) {
  const int64_t qk = (t * h_k + hk) * DK + 4 * lam;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    x.k4[m] = load4(k + qk + 4 * L * m);
    x.q4[m] = load4(q + qk + 4 * L * m);
  }
  const int64_t tv = t * h_v + h;
  x.g = __ldg(g + tv);
  x.beta = __ldg(beta + tv);
  x.v = load1(v + tv * d_v + row_mine);
}

template <int DK, int L, int R, typename T>
__global__ void __launch_bounds__(kScanWarps * 32)
    scan_prefill_kernel(const T* __restrict__ q, const T* __restrict__ k,
                        const T* __restrict__ v, const float* __restrict__ g,
                        const float* __restrict__ beta, const float* state_in, float* state_out,
                        T* __restrict__ o, const int32_t* __restrict__ cu, int32_t num_seqs,
                        int64_t total_tokens, int32_t h_k, int32_t h_v, int32_t d_v,
                        int32_t blocks_per_head, float scale, int32_t max_len, int qk_norm,
                        int* err) {
  using LY = RowLayout<DK, L, R>;
  constexpr int M = LY::M;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int n = blockIdx.x / blocks_per_head;
  const int rb = blockIdx.x - n * blocks_per_head;
  const int h = blockIdx.y;

  const int64_t t0 = cu[n], t1 = cu[n + 1];
  const bool bad = t0 < 0 || t1 < t0 || t1 > total_tokens || (n == 0 && t0 != 0) ||
                   (n == num_seqs - 1 && t1 != total_tokens);
  if (bad) {
    if (threadIdx.x == 0 && rb == 0 && h == 0) raise_error(err, kErrBadCuSeqlens);
    return;
  }
  if (t1 - t0 >= (int64_t)max_len) return;  // this sequence belongs to the chunked kernel

  const int row0 = (rb * kScanWarps + warp) * LY::kRowsPerWarp;
  if (row0 >= d_v) return;
  const int grp = lane / L;
  const int lam = lane % L;
  const int hk = h / (h_v / h_k);
  const int64_t nh = (int64_t)n * h_v + h;
  const int idx = lam / LY::Q;
  const int r_mine = idx >> 1;
  const int row_mine = row0 + r_mine * LY::G + grp;
  const int64_t s_base = (nh * d_v + row0 + grp) * (int64_t)DK + 4 * lam;

  float4 s[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      if (state_in)
        s[r][m] = load4(state_in + s_base + (int64_t)r * LY::G * DK + 4 * L * m);
      else
        s[r][m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

  TokenIn<DK, M, T> cur, nxt;
  if (t0 < t1)
    load_token<DK, L, M, T>(cur, q, k, v, g, beta, t0, h_k, h_v, d_v, hk, h, lam, row_mine);
  for (int64_t t = t0; t < t1; ++t) {
    if (t + 1 < t1)
      load_token<DK, L, M, T>(nxt, q, k, v, g, beta, t + 1, h_k, h_v, d_v, hk, h, lam,
                              row_mine);
    if (qk_norm) {
      l2_normalize<L, M>(cur.k4);
      l2_normalize<L, M>(cur.q4);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      cur.q4[m].x *= scale;
      cur.q4[m].y *= scale;
      cur.q4[m].z *= scale;
      cur.q4[m].w *= scale;
    }
    float kq = 0.f;
#pragma unroll
    for (int m = 0; m < M; ++m) kq = dot4(cur.k4[m], cur.q4[m], kq);
    kq = group_sum<L>(kq);
    const float alpha = expf(cur.g);
    const float out =
        row_token_update<DK, L, R>(s, cur.k4, cur.q4, kq, alpha, cur.beta, cur.v, lane);
    if ((idx & 1) && (lam % LY::Q) == 0) store1(o + (t * h_v + h) * d_v + row_mine, out);
    cur = nxt;
  }

#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m)
      *reinterpret_cast<float4*>(state_out + s_base + (int64_t)r * LY::G * DK + 4 * L * m) =
          s[r][m];
}

template <int DK, int L, int R, typename T>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t stream) {
  constexpr int rows_per_block = kScanWarps * RowLayout<DK, L, R>::kRowsPerWarp;
  const int blocks_per_head = (a.d_v + rows_per_block - 1) / rows_per_block;
  const int64_t gx = (int64_t)a.num_seqs * blocks_per_head;
  if (gx > 0x7fffffffLL || a.h_v > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)gx, (unsigned)a.h_v);
  scan_prefill_kernel<DK, L, R, T><<<grid, kScanWarps * 32, 0, stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v), a.g,
      a.beta, a.state_in, a.state_out, static_cast<T*>(a.o), a.cu_seqlens, a.num_seqs,
      a.total_tokens, a.h_k, a.h_v, a.d_v, blocks_per_head, a.scale, a.min_chunk_len, a.qk_norm,
      a.err);
  return cudaGetLastError();
}

// One float4 per lane per row (L = d_k / 4) and two rows per lane group: the
// per-token chain is one 5-level butterfly, and B=1 with 32 heads of 128 rows
// still yields 2048 warps.
template <typename T>
cudaError_t launch_typed(const PrefillArgs& a, cudaStream_t stream) {
  switch (a.d_k) {
    case 16: return launch_t<16, 4, 1, T>(a, stream);
    case 32: return launch_t<32, 8, 2, T>(a, stream);
    case 64: return launch_t<64, 16, 2, T>(a, stream);
    case 128: return launch_t<128, 32, 2, T>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_scan(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  if (a.dtype == kBF16) return launch_typed<__nv_bfloat16>(a, stream);
  return launch_typed<float>(a, stream);
}

}  // namespace gdn
