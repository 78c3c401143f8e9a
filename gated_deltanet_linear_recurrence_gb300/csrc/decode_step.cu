// decode_step.cu — fused single-token update of the gated delta rule for a
// batch of independent sequences, state updated in place.
//
// Page "Optimizing on-device inference for Apple Silicon", section "Reduce
// intermediate and state traffic": the decode-time recurrent update runs as one
// fused kernel whose temporaries stay in registers.  Section "Decode: minimize
// bytes moved per token": decode throughput is set by the bytes moved, so the
// kernel reads every state element once and writes it once (128-bit coalesced
// accesses: a warp-wide load covers 512 contiguous bytes, as in the page's
// "Coalesce attention-cache reads") and does all arithmetic on the way through.
//
// Work split.  One CTA of 4 warps owns a block of rows of one (sequence, value
// head); each warp holds kRowsPerWarp rows (see rows.cuh) and issues all of its
// state loads before any arithmetic so that many bytes are in flight per SM.
// k and q are read once per warp, v once per row.  The state is HBM traffic
// (1 GiB per step at 256 sequences x 32 heads x 128 x 128 fp32, read + write);
// everything else is under 1% of the bytes.
#include <cuda_bf16.h>

#include "params.h"
#include "rows.cuh"
#include "tc.cuh"

namespace gdn {
namespace {

constexpr int kDecodeWarps = 4;  // warps per CTA of the large-batch and normalising steps

// The step for the warp's rows row0 ..: loads, update and in-place store of the
// state rows; returns this lane's output value, and whether the lane holds one
// (mine) for row row_mine.
template <int DK, int R, bool kPrefetch, typename T>
__device__ __forceinline__ float step_rows(const T* __restrict__ q, const T* __restrict__ k,
                                           const T* __restrict__ v, const float* __restrict__ g,
                                           const float* __restrict__ beta,
                                           float* __restrict__ state, int32_t h_k, int32_t h_v,
                                           int32_t d_v, float scale, int qk_norm, int b, int h,
                                           int row0, int lane, int& row_mine, bool& mine) {
  constexpr int L = DK / 4;  // one float4 per lane per row
  using LY = RowLayout<DK, L, R>;
  constexpr int M = LY::M;
  const int grp = lane / L;
  const int lam = lane % L;
  const int hk = h / (h_v / h_k);
  const int64_t bh = (int64_t)b * h_v + h;
  // Launched with programmatic stream serialization: the next kernel in the
  // stream may be scheduled now, and every input is read only once the kernel
  // before this one has completed.  The warp's state rows (contiguous) are
  // prefetched into L2 before that wait (small batches, kPrefetch): a prefetch
  // changes no value a load returns, and in a chain of decode calls (one per
  // layer) each call's state then streams in while the call before it still
  // runs.
  tc::allow_dependents();
  if (kPrefetch && lane == 0) {
    const int rows = d_v - row0 < LY::kRowsPerWarp ? d_v - row0 : LY::kRowsPerWarp;
    tc::prefetch_l2(state + (bh * d_v + row0) * (int64_t)DK, (uint32_t)rows * DK * 4u);
  }
  tc::wait_prerequisites();

  // state rows first: they are the bytes that matter
  float* srow = state + (bh * d_v + row0 + grp) * (int64_t)DK + 4 * lam;
  float4 s[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m)
      s[r][m] = __ldcs(reinterpret_cast<const float4*>(srow + (int64_t)r * LY::G * DK + 4 * L * m));

  const T* kp = k + ((int64_t)b * h_k + hk) * DK + 4 * lam;
  const T* qp = q + ((int64_t)b * h_k + hk) * DK + 4 * lam;
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
  const int idx = lam / LY::Q;  // reduced value index this lane will hold
  const int r_mine = idx >> 1;
  row_mine = row0 + r_mine * LY::G + grp;
  const float v_mine = load1(v + bh * d_v + row_mine);
  const float alpha = expf(__ldg(g + bh));
  const float bt = __ldg(beta + bh);

  float kq = 0.f;
#pragma unroll
  for (int m = 0; m < M; ++m) kq = dot4(k4[m], q4[m], kq);
  kq = group_sum<L>(kq);

  const float out = row_token_update<DK, L, R>(s, k4, q4, kq, alpha, bt, v_mine, lane);
  mine = (idx & 1) && (lam % LY::Q) == 0;

#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m)
      __stcs(reinterpret_cast<float4*>(srow + (int64_t)r * LY::G * DK + 4 * L * m), s[r][m]);
  return out;
}

// Output RMS normalisation fused into the step (kNorm): the CTAs of one
// (sequence, value head) form a thread-block cluster; each sums the squares of
// its rows' outputs, the partial sums are exchanged through distributed shared
// memory, and every CTA scales its own outputs before storing them.
struct OutNorm {
  const float* weight;  // [d_v] or NULL (ones)
  float eps;
};

template <int DK, int R, int W, bool kPrefetch, bool kNorm, typename T>
__global__ void __launch_bounds__(W * 32)
    decode_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                       const float* __restrict__ g, const float* __restrict__ beta,
                       float* __restrict__ state, T* __restrict__ o, int32_t h_k, int32_t h_v,
                       int32_t d_v, int32_t blocks_per_head, float scale, int qk_norm,
                       OutNorm nrm) {
  constexpr int L = DK / 4;  // one float4 per lane per row
  using LY = RowLayout<DK, L, R>;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x / blocks_per_head;
  const int rb = blockIdx.x - b * blocks_per_head;
  const int h = blockIdx.y;
  const int row0 = (rb * W + warp) * LY::kRowsPerWarp;
  if constexpr (kNorm) {
    // every warp takes part in the cluster's reduction, idle ones with nothing
    __shared__ float part[W + 1];
    float sq = 0.f, out = 0.f;
    int row_mine = 0;
    bool mine = false;
    if (row0 < d_v)
      out = step_rows<DK, R, kPrefetch>(q, k, v, g, beta, state, h_k, h_v, d_v, scale, qk_norm,
                                        b, h, row0, lane, row_mine, mine);
    if (mine) sq = out * out;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sq += __shfl_xor_sync(kFullMask, sq, off);
    if (lane == 0) part[warp] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) t += part[w];
      part[W] = t;
    }
    tc::cluster_sync();  // every CTA's partial sum is written
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int r = 0; r < blocks_per_head; ++r) t += tc::ld_cluster_f32(&part[W], r);
      part[0] = rsqrtf(t / (float)d_v + nrm.eps);  // own slot 0 is read by no other CTA
    }
    tc::cluster_sync();  // the partial sums have been read: no CTA leaves before that
    if (mine) {
      const float wgt = nrm.weight ? __ldg(nrm.weight + row_mine) : 1.f;
      store1(o + ((int64_t)b * h_v + h) * d_v + row_mine, out * part[0] * wgt);
    }
  } else {
    if (row0 >= d_v) return;  // whole warp idle (d_v is a multiple of 16)
    int row_mine;
    bool mine;
    const float out = step_rows<DK, R, kPrefetch>(q, k, v, g, beta, state, h_k, h_v, d_v, scale,
                                                  qk_norm, b, h, row0, lane, row_mine, mine);
    if (mine) store1(o + ((int64_t)b * h_v + h) * d_v + row_mine, out);
  }
}

template <int DK, int R, int W, bool kPrefetch, bool kNorm, typename T>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int L = DK / 4;
  constexpr int rows_per_block = W * RowLayout<DK, L, R>::kRowsPerWarp;
  const int blocks_per_head = (a.d_v + rows_per_block - 1) / rows_per_block;
  const int64_t gx = (int64_t)a.batch * blocks_per_head;
  if (gx > 0x7fffffffLL || a.h_v > 65535) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // the CTAs of one (sequence, head)
  attr[1].val.clusterDim.x = (unsigned)blocks_per_head;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  if (kNorm && blocks_per_head > 8) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)gx, (unsigned)a.h_v);
  cfg.blockDim = dim3(W * 32);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = kNorm ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, decode_step_kernel<DK, R, W, kPrefetch, kNorm, T>,
                            static_cast<const T*>(a.q), static_cast<const T*>(a.k),
                            static_cast<const T*>(a.v), a.g, a.beta, a.state, static_cast<T*>(a.o),
                            a.h_k, a.h_v, a.d_v, blocks_per_head, a.scale, a.qk_norm,
                            OutNorm{a.norm_weight, a.norm_eps});
}

// Rows per lane group: R = L/2 gives 16 rows per warp (most bytes in flight
// per warp) in CTAs of four warps.  With few rows in total the state is
// prefetched into L2 ahead of the dependency wait, and the CTAs are single
// warps of L/4 x (32/L) rows (8 rows at d_k = 128), so that more SMs stream at
// once and the next call's CTAs find room early.  Measured on GB300, batch 1
// through 30 layers in one CUDA graph (us per step): 78.3 without the prefetch
// in four-warp CTAs of 4 rows per warp, 70.1 with it; then with the prefetch,
// by warps per CTA x rows per warp: 8 x 4 78.3, 4 x 4 69.1, 2 x 4 66.0, 1 x 4
// 59.9, 1 x 8 57.8, 1 x 1 145.9, and 1 x 4 without the prefetch 68.1.  With
// the output normalisation a head's CTAs (at most 8) form one cluster, so that
// step keeps four-warp CTAs.
template <int DK, typename T>
cudaError_t launch_dk(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int L = DK / 4;
  constexpr int R_BIG = L / 2;
  constexpr int R_SMALL = (L / 8) > 0 ? (L / 8) : 1;   // normalising step, four warps
  constexpr int R_ONE = (L / 4) > 0 ? (L / 4) : 1;     // single-warp CTAs
  const int64_t rows = (int64_t)a.batch * a.h_v * a.d_v;
  // 16 rows per warp still gives >= 4 warps on every one of 152 SMs
  const bool big = rows >= (int64_t)16 * 4 * 152 * kDecodeWarps;
  if (a.out_norm)
    return big ? launch_t<DK, R_BIG, kDecodeWarps, false, true, T>(a, stream)
               : launch_t<DK, R_SMALL, kDecodeWarps, true, true, T>(a, stream);
  return big ? launch_t<DK, R_BIG, kDecodeWarps, false, false, T>(a, stream)
             : launch_t<DK, R_ONE, 1, true, false, T>(a, stream);
}

template <typename T>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.d_k) {
    case 16: return launch_dk<16, T>(a, stream);
    case 32: return launch_dk<32, T>(a, stream);
    case 64: return launch_dk<64, T>(a, stream);
    case 128: return launch_dk<128, T>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  if (a.dtype == kBF16) return launch_typed<__nv_bfloat16>(a, stream);
  return launch_typed<float>(a, stream);
}

}  // namespace gdn
