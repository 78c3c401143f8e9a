// output_norm.cu — the output RMS normalisation as a pass of its own, in place
// over o [rows][h_v][d_v] (the normalisation the decode step can also fuse;
// contract in include/gdn.h, gdn_output_rmsnorm):
//
//     o[r,h,i] <- w_i o[r,h,i] / sqrt( (1 / d_v) sum_j o[r,h,j]^2 + eps )
//
// One warp per (row, value head) vector; a lane holds d_v / 32 consecutive
// values (one 16-byte or 8-byte access per lane for d_v = 128), the sum of
// squares is a warp-shuffle reduction in fp32, and the scaled values are
// stored back rounded to nearest even.  HBM-bound: o is read and written once.
#include <cuda_bf16.h>

#include "params.h"
#include "rows.cuh"

namespace gdn {
namespace {

constexpr int kNormWarps = 8;

template <int DV, typename T>
__global__ void __launch_bounds__(kNormWarps * 32)
    output_rmsnorm_kernel(T* __restrict__ o, const float* __restrict__ weight, int64_t n_vec,
                          float eps) {
  constexpr int P = DV >= 32 ? DV / 32 : 1;  // values per lane
  constexpr int kLanes = DV >= 32 ? 32 : DV;  // lanes holding values
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kNormWarps;
  for (int64_t vi = (int64_t)blockIdx.x * kNormWarps + (threadIdx.x >> 5); vi < n_vec;
       vi += stride) {
    T* base = o + vi * DV + lane * P;
    float x[P];
    if (lane < kLanes) {
#pragma unroll
      for (int e = 0; e < P; ++e) x[e] = load1(base + e);
    } else {
#pragma unroll
      for (int e = 0; e < P; ++e) x[e] = 0.f;
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < P; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(kFullMask, ss, off);
    const float r = rsqrtf(ss / (float)DV + eps);
    if (lane < kLanes) {
#pragma unroll
      for (int e = 0; e < P; ++e) {
        const float w = weight ? __ldg(weight + lane * P + e) : 1.f;
        store1(base + e, x[e] * r * w);
      }
    }
  }
}

template <int DV, typename T>
cudaError_t launch_norm_t(void* o, const float* weight, int64_t n_vec, float eps,
                          cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t want = (n_vec + kNormWarps - 1) / kNormWarps;
  const int64_t cap = (int64_t)sms * 16;  // a few resident waves, then grid-stride
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  output_rmsnorm_kernel<DV, T><<<grid, kNormWarps * 32, 0, stream>>>(static_cast<T*>(o), weight,
                                                                     n_vec, eps);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_norm(void* o, const float* weight, int64_t n_vec, int32_t d_v, float eps,
                        cudaStream_t stream) {
  switch (d_v) {
    case 16: return launch_norm_t<16, T>(o, weight, n_vec, eps, stream);
    case 32: return launch_norm_t<32, T>(o, weight, n_vec, eps, stream);
    case 64: return launch_norm_t<64, T>(o, weight, n_vec, eps, stream);
    case 128: return launch_norm_t<128, T>(o, weight, n_vec, eps, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_output_rmsnorm(void* o, const float* weight, int64_t n_vec, int32_t d_v,
                                  int dtype, float eps, cudaStream_t stream) {
  if (n_vec == 0) return cudaSuccess;
  if (dtype == kBF16) return launch_norm<__nv_bfloat16>(o, weight, n_vec, d_v, eps, stream);
  return launch_norm<float>(o, weight, n_vec, d_v, eps, stream);
}

}  // namespace gdn
