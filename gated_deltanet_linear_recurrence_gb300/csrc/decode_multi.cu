// decode_multi.cu — several tokens per sequence in one launch (a verification
// group), the state read once, carried in registers through the tokens, and
// written once, optionally with the state after every token.
//
// Page "Optimizing on-device inference for Apple Silicon", section "Limits of
// further optimization": speculative decoding verifies groups of two to five
// rows per step, and a rejected draft token means going back to the state
// after the last accepted one — hence the per-token state snapshots.  The
// per-row arithmetic is the decode step's (rows.cuh, row identity), so n
// tokens here equal n successive gdn_decode_step calls bit for bit.
//
// Work split as in decode_step.cu: one CTA of 4 warps per block of rows of one
// (sequence, value head), each warp kRowsPerWarp rows of d_k floats spread over
// L lanes.  Bytes: the state once in and once out (plus one state per token
// when snapshots are written); q, k, v, o, g, beta per token are small.
#include <cuda_bf16.h>

#include "params.h"
#include "rows.cuh"

namespace gdn {
namespace {

constexpr int kMultiWarps = 4;

template <int DK, int R, typename T>
__global__ void __launch_bounds__(kMultiWarps * 32)
    decode_multi_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                        const float* __restrict__ g, const float* __restrict__ beta,
                        float* __restrict__ state, T* __restrict__ o, float* __restrict__ snap,
                        int32_t n_tok, int32_t h_k, int32_t h_v, int32_t d_v,
                        int32_t blocks_per_head, float scale, int qk_norm) {
  constexpr int L = DK / 4;
  using LY = RowLayout<DK, L, R>;
  constexpr int M = LY::M;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x / blocks_per_head;
  const int rb = blockIdx.x - b * blocks_per_head;
  const int h = blockIdx.y;
  const int row0 = (rb * kMultiWarps + warp) * LY::kRowsPerWarp;
  if (row0 >= d_v) return;
  const int grp = lane / L;
  const int lam = lane % L;
  const int hk = h / (h_v / h_k);
  const int64_t bh = (int64_t)b * h_v + h;
  const int64_t row_off = (int64_t)(row0 + grp) * DK + 4 * lam;  // within one head's state

  float* srow = state + bh * d_v * (int64_t)DK + row_off;
  float4 s[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m)
      s[r][m] = __ldcs(reinterpret_cast<const float4*>(srow + (int64_t)r * LY::G * DK + 4 * L * m));

  const int idx = lam / LY::Q;
  const int r_mine = idx >> 1;
  const int row_mine = row0 + r_mine * LY::G + grp;
  for (int t = 0; t < n_tok; ++t) {
    const int64_t bt_tok = (int64_t)b * n_tok + t;  // token row of (sequence b, token t)
    const T* kp = k + (bt_tok * h_k + hk) * DK + 4 * lam;
    const T* qp = q + (bt_tok * h_k + hk) * DK + 4 * lam;
    float4 k4[M], q4[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      k4[m] = load4(kp + 4 * L * m);
      q4[m] = load4(qp + 4 * L * m);
    }
    if (qk_norm) {
      l2_normalize<L, M>(k4);
      l2_normalize<L, M>(q4);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      q4[m].x *= scale;
      q4[m].y *= scale;
      q4[m].z *= scale;
      q4[m].w *= scale;
    }
    const int64_t th = bt_tok * h_v + h;
    const float v_mine = load1(v + th * d_v + row_mine);
    const float alpha = expf(__ldg(g + th));
    const float bt = __ldg(beta + th);
    float kq = 0.f;
#pragma unroll
    for (int m = 0; m < M; ++m) kq = dot4(k4[m], q4[m], kq);
    kq = group_sum<L>(kq);
    const float out = row_token_update<DK, L, R>(s, k4, q4, kq, alpha, bt, v_mine, lane);
    if ((idx & 1) && (lam % LY::Q) == 0) store1(o + th * d_v + row_mine, out);
    if (snap) {
      float* prow = snap + th * d_v * (int64_t)DK + row_off;
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m)
          __stcs(reinterpret_cast<float4*>(prow + (int64_t)r * LY::G * DK + 4 * L * m), s[r][m]);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m)
      __stcs(reinterpret_cast<float4*>(srow + (int64_t)r * LY::G * DK + 4 * L * m), s[r][m]);
}

template <int DK, int R, typename T>
cudaError_t launch_t(const DecodeMultiArgs& a, cudaStream_t stream) {
  constexpr int L = DK / 4;
  constexpr int rows_per_block = kMultiWarps * RowLayout<DK, L, R>::kRowsPerWarp;
  const int blocks_per_head = (a.d_v + rows_per_block - 1) / rows_per_block;
  const int64_t gx = (int64_t)a.batch * blocks_per_head;
  if (gx > 0x7fffffffLL || a.h_v > 65535) return cudaErrorInvalidConfiguration;
  // Plain launch: with programmatic stream serialization (as the single-token
  // step uses) back-to-back calls measured 6 % slower (212 vs 199 us at 256
  // sequences x 4 tokens), the next grid's early CTAs competing with this one's.
  dim3 grid((unsigned)gx, (unsigned)a.h_v);
  decode_multi_kernel<DK, R, T><<<grid, kMultiWarps * 32, 0, stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v), a.g,
      a.beta, a.state, static_cast<T*>(a.o), a.snapshots, a.n_tokens, a.h_k, a.h_v, a.d_v,
      blocks_per_head, a.scale, a.qk_norm);
  return cudaGetLastError();
}

// The decode step's choice of rows per lane group (same rows, same reduction
// order, hence the same results as successive single steps).
template <int DK, typename T>
cudaError_t launch_dk(const DecodeMultiArgs& a, cudaStream_t stream) {
  constexpr int L = DK / 4;
  constexpr int R_BIG = L / 2;
  constexpr int R_SMALL = (L / 8) > 0 ? (L / 8) : 1;
  const int64_t rows = (int64_t)a.batch * a.h_v * a.d_v;
  if (rows >= (int64_t)16 * 4 * 152 * kMultiWarps) return launch_t<DK, R_BIG, T>(a, stream);
  return launch_t<DK, R_SMALL, T>(a, stream);
}

template <typename T>
cudaError_t launch_typed(const DecodeMultiArgs& a, cudaStream_t stream) {
  switch (a.d_k) {
    case 16: return launch_dk<16, T>(a, stream);
    case 32: return launch_dk<32, T>(a, stream);
    case 64: return launch_dk<64, T>(a, stream);
    case 128: return launch_dk<128, T>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_multi(const DecodeMultiArgs& a, cudaStream_t stream) {
  if (a.batch == 0 || a.n_tokens == 0) return cudaSuccess;
  if (a.dtype == kBF16) return launch_typed<__nv_bfloat16>(a, stream);
  return launch_typed<float>(a, stream);
}

}  // namespace gdn
