// chunk_common.cuh — device helpers shared by the chunked-prefill kernels:
// bf16 packing into swizzled shared-memory operands, group barriers, and the
// 64x64 unit-lower-triangular inverse T = (I + A)^{-1} of the WY/UT form.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "tc.cuh"

namespace gdn {
namespace chunk {

constexpr int kC = 64;      // chunk length
constexpr int kDK = 128;    // key dimension handled by the chunked kernels
constexpr int kDVS = 32;    // value rows per chain CTA
constexpr int kLdM = 68;    // row stride (floats) of the fp32 A / T buffer (16-byte rows)
constexpr int kLdY = 40;    // row stride of the solve scratch [32][40]

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Store 8 consecutive bf16 values (16 bytes) at a swizzled offset.
template <int kBits>
__device__ __forceinline__ void st_chunk(uint8_t* base, uint32_t off, const float* x) {
  uint4 u;
  u.x = pack_bf16(x[0], x[1]);
  u.y = pack_bf16(x[2], x[3]);
  u.z = pack_bf16(x[4], x[5]);
  u.w = pack_bf16(x[6], x[7]);
  *reinterpret_cast<uint4*>(base + tc::swizzle<kBits>(off)) = u;
}

// Wait on an mbarrier phase; the outcome is made uniform over a named-barrier group.
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, uint32_t id,
                                           uint32_t count) {
  const bool ok = tc::mbar_wait(bar, parity);
  tc::fence_after_sync();
  return tc::named_sync_and(id, count, ok);
}

__device__ __forceinline__ void group_sync(uint32_t id, uint32_t count) {
  tc::fence_before_sync();
  tc::named_sync(id, count);
  tc::fence_after_sync();
}

// Warp-level tf32 tensor-core product for the small block products of the
// triangular solve: C (16 x 8) = A (16 x K) B (K x 8), fp32 accumulation.
// Fragment layout of mma.m16n8k8 (PTX ISA): g = lane / 4, t = lane % 4;
// A: (g, t), (g+8, t), (g, t+4), (g+8, t+4); B: (t, g), (t+4, g);
// C: (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1).
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
template <int K>
__device__ __forceinline__ void warp_mma_16x8(float (&c)[4], const float* A, int lda,
                                              const float* B, int ldb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  c[0] = c[1] = c[2] = c[3] = 0.f;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 8) {
    const uint32_t a0 = to_tf32(A[g * lda + k0 + t]);
    const uint32_t a1 = to_tf32(A[(g + 8) * lda + k0 + t]);
    const uint32_t a2 = to_tf32(A[g * lda + k0 + t + 4]);
    const uint32_t a3 = to_tf32(A[(g + 8) * lda + k0 + t + 4]);
    const uint32_t b0 = to_tf32(B[(k0 + t) * ldb + g]);
    const uint32_t b1 = to_tf32(B[(k0 + t + 4) * ldb + g]);
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}
// Store a C fragment (scaled by s) into a row-major fp32 block.
__device__ __forceinline__ void store_16x8(float* C, int ldc, const float (&c)[4], float s,
                                           int lane) {
  const int g = lane >> 2, t = lane & 3;
  C[g * ldc + 2 * t] = s * c[0];
  C[g * ldc + 2 * t + 1] = s * c[1];
  C[(g + 8) * ldc + 2 * t] = s * c[2];
  C[(g + 8) * ldc + 2 * t + 1] = s * c[3];
}

// T = (I + A)^{-1}, in place, for the strictly lower 64x64 A held row-major in
// MF (row stride kLdM; its strictly upper part is zero).  Three levels:
// 16x16 diagonal blocks by forward substitution (fp32 FFMA), then 32x32 blocks
// as [[T0, 0], [-T1 A10 T0, T1]], then the 64x64 matrix the same way; the block
// products of the last two levels run on the warp tensor cores in tf32.  Each
// level only overwrites blocks that later levels read as T.
template <uint32_t kCount>
__device__ __forceinline__ void unit_lower_inverse(float* MF, float* YF, int pt, int lane,
                                                   uint32_t bar) {
  const int pw = pt >> 5;
  if (pw < 2) {  // level 1: warp pw handles diagonal blocks 2pw, 2pw+1; lane = column
    const int blk = 2 * pw + (lane >> 4), cc = lane & 15, o = 16 * blk;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float av[16];
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        if (4 * i4 < r) {
          const float4 v4 = *reinterpret_cast<const float4*>(MF + (o + r) * kLdM + o + 4 * i4);
          av[4 * i4] = v4.x; av[4 * i4 + 1] = v4.y; av[4 * i4 + 2] = v4.z; av[4 * i4 + 3] = v4.w;
        }
      }
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int i = 0; i < r; ++i) {
        if (i & 1) a1 = fmaf(av[i], x[i], a1); else a0 = fmaf(av[i], x[i], a0);
      }
      x[r] = (r == cc) ? 1.f : ((r > cc) ? -(a0 + a1) : 0.f);
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 16; ++r) MF[(o + r) * kLdM + o + cc] = x[r];
  }
  tc::named_sync(bar, kCount);
  // level 2: pairs (0,1) and (2,3): Y = A10 T0 (warps 0-3: pair, 8-column tile)
  if (pw < 4) {
    const int pr = pw >> 1, nt = pw & 1, o0 = 32 * pr, o1 = o0 + 16;
    float c[4];
    warp_mma_16x8<16>(c, MF + o1 * kLdM + o0, kLdM, MF + o0 * kLdM + o0 + 8 * nt, kLdM, lane);
    store_16x8(YF + (16 * pr) * kLdY + 8 * nt, kLdY, c, 1.f, lane);
  }
  tc::named_sync(bar, kCount);
  if (pw < 4) {  // T10 = -T1 Y
    const int pr = pw >> 1, nt = pw & 1, o0 = 32 * pr, o1 = o0 + 16;
    float c[4];
    warp_mma_16x8<16>(c, MF + o1 * kLdM + o1, kLdM, YF + (16 * pr) * kLdY + 8 * nt, kLdY, lane);
    store_16x8(MF + o1 * kLdM + o0 + 8 * nt, kLdM, c, -1.f, lane);
  }
  tc::named_sync(bar, kCount);
  // level 3, eight 16x8 tiles (rows 16 (tile >> 2), columns 8 (tile & 3)) over the warps
  constexpr int kWarps = (int)(kCount / 32);
  static_assert(kWarps >= 4 && 8 % kWarps == 0, "the solve runs on 4 or 8 warps");
  for (int tile = pw; tile < 8; tile += kWarps) {  // Y = A_BL T_TL (32x32x32)
    const int mt = tile >> 2, nt = tile & 3;
    float c[4];
    warp_mma_16x8<32>(c, MF + (32 + 16 * mt) * kLdM, kLdM, MF + 8 * nt, kLdM, lane);
    store_16x8(YF + (16 * mt) * kLdY + 8 * nt, kLdY, c, 1.f, lane);
  }
  tc::named_sync(bar, kCount);
  for (int tile = pw; tile < 8; tile += kWarps) {  // T_BL = -T_BR Y
    const int mt = tile >> 2, nt = tile & 3;
    float c[4];
    warp_mma_16x8<32>(c, MF + (32 + 16 * mt) * kLdM + 32, kLdM, YF + 8 * nt, kLdY, lane);
    store_16x8(MF + (32 + 16 * mt) * kLdM + 8 * nt, kLdM, c, -1.f, lane);
  }
  tc::named_sync(bar, kCount);
}


}  // namespace chunk
}  // namespace gdn
