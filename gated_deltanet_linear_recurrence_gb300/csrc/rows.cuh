// rows.cuh — per-row arithmetic of the gated delta rule, shared by the decode
// step and the token-scan prefill.
//
// Row identity.  Right-multiplying S by (I - beta k k^T) acts on each row of S
// separately, so row i (a value dimension) evolves on its own given k, q,
// alpha and beta.  With s = S_{t-1,i} . k and p = S_{t-1,i} . q, both read
// before the update:
//     u       = beta (v_i - alpha s)
//     S_t,i   = alpha S_{t-1,i} + u k^T
//     o_t,i   = S_t,i . q = alpha p + u (k . q)
// so one fused pass over the row produces both dot products, and the readout
// needs no second pass over the updated row.  (Page "Optimizing on-device
// inference for Apple Silicon": "Keep the recurrent state on-chip" keeps each
// state slice in registers for the whole scan and exchanges partial results
// with SIMD-group operations; "Reduce intermediate and state traffic" fuses the
// decode-time update into one kernel.  Warp shuffles play the SIMD-group role.)
//
// Register layout.  A row of d_k fp32 values is spread over L lanes; lane l of
// a lane group holds float4 chunks l, l+L, l+2L, ... (M = d_k / (4L) chunks),
// so one warp-wide 128-bit load covers 32 consecutive chunks.  A warp holds
// G = 32 / L lane groups and each group R rows: row (r, grp) = row0 + r*G + grp.
//
// Reductions.  The 2R partial dot products of a lane group (s and p of R rows)
// are summed with a transposing butterfly: at each step a lane keeps half of
// its values and receives the partner's other half, so 2R sums over L lanes
// cost 2R-1 + log2(L/2R) shuffles instead of 2R*log2(L).  Afterwards lane l of
// the group holds the sum of value index l / (L / 2R): index 2r is s of row r,
// index 2r+1 is p of row r.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {

constexpr unsigned kFullMask = 0xffffffffu;

__device__ __forceinline__ float4 load4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  float4 f;
  f.x = __uint_as_float(u.x << 16);
  f.y = __uint_as_float(u.x & 0xffff0000u);
  f.z = __uint_as_float(u.y << 16);
  f.w = __uint_as_float(u.y & 0xffff0000u);
  return f;
}
__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store1(float* p, float x) { *p = x; }
__device__ __forceinline__ void store1(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  acc = fmaf(a.w, b.w, acc);
  return acc;
}

// Sum V values per lane over lane groups of L lanes; lane l (in its group)
// receives the group sum of value index l / (L / V).
template <int L, int V>
__device__ __forceinline__ float transpose_reduce(float (&x)[V], int lane) {
  static_assert((L & (L - 1)) == 0 && L >= 1 && L <= 32, "L must be a power of two <= 32");
  static_assert((V & (V - 1)) == 0 && V >= 1 && V <= L, "V must be a power of two <= L");
#pragma unroll
  for (int step = 0; (V >> step) > 1; ++step) {
    const int n = V >> step;
    const int off = L >> (step + 1);
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? x[i] : x[i + n / 2];
      const float keep = upper ? x[i + n / 2] : x[i];
      x[i] = keep + __shfl_xor_sync(kFullMask, send, off);
    }
  }
  float r = x[0];
#pragma unroll
  for (int off = L / V / 2; off >= 1; off >>= 1) r += __shfl_xor_sync(kFullMask, r, off);
  return r;
}

// Sum one value over the lane group (every lane receives the sum).
template <int L>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int off = L / 2; off >= 1; off >>= 1) x += __shfl_xor_sync(kFullMask, x, off);
  return x;
}

// x <- x / sqrt(|x|^2 + 1e-6) for a vector of d_k values spread over the L
// lanes of a lane group (M float4 chunks per lane): the optional per-head L2
// normalisation of q and k.
template <int L, int M>
__device__ __forceinline__ void l2_normalize(float4 (&x)[M]) {
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < M; ++m) ss = dot4(x[m], x[m], ss);
  ss = group_sum<L>(ss);
  const float r = rsqrtf(ss + 1e-6f);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    x[m].x *= r;
    x[m].y *= r;
    x[m].z *= r;
    x[m].w *= r;
  }
}

template <int DK, int L, int R>
struct RowLayout {
  static constexpr int M = DK / (4 * L);  // float4 chunks per lane per row
  static constexpr int G = 32 / L;        // lane groups per warp
  static constexpr int V = 2 * R;         // reduced values per lane group
  static constexpr int Q = L / V;         // lanes that share one reduced value
  static constexpr int kRowsPerWarp = G * R;
  static_assert(DK % (4 * L) == 0, "d_k must split into float4 chunks over L lanes");
  static_assert(V <= L, "2R must not exceed L");
};

// One token of the row identity for the R rows a lane group holds.
//   s[r][m]  : state chunks (updated in place)
//   k4, q4   : this lane's chunks of k and (scaled) q
//   kq       : k . q over the full d_k (same on every lane)
//   v_mine   : v of the row whose s this lane holds after the reduction
// Returns o of the row whose p this lane holds (valid on lanes with odd
// reduced index, see RowLayout::Q).
template <int DK, int L, int R>
__device__ __forceinline__ float row_token_update(float4 (&s)[R][DK / (4 * L)],
                                                  const float4 (&k4)[DK / (4 * L)],
                                                  const float4 (&q4)[DK / (4 * L)], float kq,
                                                  float alpha, float beta, float v_mine,
                                                  int lane) {
  using LY = RowLayout<DK, L, R>;
  float x[LY::V];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int m = 0; m < LY::M; ++m) {
      sk = dot4(s[r][m], k4[m], sk);
      sq = dot4(s[r][m], q4[m], sq);
    }
    x[2 * r] = sk;
    x[2 * r + 1] = sq;
  }
  const float red = transpose_reduce<L, LY::V>(x, lane);
  // lanes holding s of row r compute u_r; lanes holding p fetch it from the
  // lane Q below (same row, even index).
  const float u = beta * (v_mine - alpha * red);
  const float u_left = __shfl_sync(kFullMask, u, (lane - LY::Q) & 31);
  const float o = fmaf(alpha, red, u_left * kq);
  const int grp_base = lane & ~(L - 1);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float ur = __shfl_sync(kFullMask, u, grp_base + 2 * r * LY::Q);
#pragma unroll
    for (int m = 0; m < LY::M; ++m) {
      s[r][m].x = fmaf(alpha, s[r][m].x, ur * k4[m].x);
      s[r][m].y = fmaf(alpha, s[r][m].y, ur * k4[m].y);
      s[r][m].z = fmaf(alpha, s[r][m].z, ur * k4[m].z);
      s[r][m].w = fmaf(alpha, s[r][m].w, ur * k4[m].w);
    }
  }
  return o;
}

// Record the first device-side error in the library's error word.
__device__ __forceinline__ void raise_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

}  // namespace gdn
