// attn_decode.cu — grouped-query decode attention on tcgen05: one new query
// token per sequence attends over the sequence's KV cache.
//
// Page "Optimizing on-device inference for Apple Silicon", section "Read the
// attention cache efficiently": every decode step of a full-attention layer
// reads the whole KV cache, so the step is bound by the bytes it moves.  Three
// of its points shape this kernel:
//   * "Coalesce attention-cache reads": the cache is read in whole 64-key tiles
//     by TMA (each row of a head is 512 contiguous bytes);
//   * "Group query heads to reuse KV rows": the (up to) eight query heads that
//     share a KV head are served by one CTA, which loads each K and V row once;
//   * "Switch attention layouts at long context": the general layout gives one
//     CTA a whole (sequence, KV head); the fixed-block layout splits the cache
//     into equal blocks of keys processed in parallel and combines their
//     partial softmax results afterwards.
//
// Per 64-key tile (head dimension 256, G <= 8 query heads, zero-padded to 8):
//   S^T = K Q^T      tcgen05, M = 64 keys,  N = 8 heads, K = 256 dims
//   online softmax   four epilogue warps, from TMEM; P (bf16) to shared memory
//   O^T += V^T P^T   tcgen05, M = 64 dims (x4), N = 8 heads, K = 64 keys,
//                    accumulated in TMEM and rescaled there when a head's
//                    running maximum grows
// Warp roles: a producer warp (TMA, 3-stage ring of K and V tiles), an MMA warp
// (whole warp converged, one elected lane issues) and four epilogue warps.
// Cache slots past a sequence's length are never read into a result: their
// scores are masked and their V rows zeroed in shared memory first.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "params.h"
#include "per_device.h"
#include "rows.cuh"
#include "tc.cuh"

namespace gdn {
namespace {

constexpr int kD = 256;     // head dimension
constexpr int kG = 8;       // query heads per CTA (MMA N)
constexpr int kTile = 64;   // keys per tile
constexpr int kAStages = 3;
constexpr int kEpiThreads = 128;
constexpr int kAProducerWarp = 4, kAMmaWarp = 5;
constexpr int kAThreads = kEpiThreads + 64;
constexpr uint32_t kABarEpi = 1;  // named barrier of the epilogue warps
// Shared memory: stage s holds the K tile (4 boxes [64 keys][64 dims], SW128)
// then the V tile (same); then Q^T (4 boxes [8 heads][64 dims]), two P buffers
// ([8 heads][64 keys], SW128), the softmax reduction scratch and the barriers.
constexpr uint32_t AS_STAGE = 65536, AS_V = 32768;
constexpr uint32_t AS_Q = kAStages * AS_STAGE;
constexpr uint32_t AS_P = AS_Q + 4096;
constexpr uint32_t AS_RED = AS_P + 2048;  // tile maxima [2][4 warps][8 heads] fp32
constexpr uint32_t AS_BAR = AS_RED + 2 * 4 * kG * 4;
constexpr uint32_t kAttnSmem = AS_BAR + 256 + 1024;  // + barriers, TMEM slot, alignment
static_assert(kAttnSmem <= 227 * 1024, "shared memory budget");
// TMEM: S^T in two buffers of 8 columns, O^T in four blocks of 64 dimensions x
// 8 columns.  Both products are M = 64 (the only M that allows N = 8), whose
// accumulator row m sits in TMEM lane 32 (m / 16) + m % 16.
constexpr uint32_t kAttnTmemCols = 64;
constexpr uint32_t TA_S = 0, TA_O = 16;
constexpr uint32_t IDA_S = tc::idesc_bf16_f32(64, kG, false, false);  // K Q^T
constexpr uint32_t IDA_O = tc::idesc_bf16_f32(64, kG, true, false);   // V^T P^T
constexpr float kLog2e = 1.4426950408889634f;
constexpr int64_t kMinBlockKeys = 128;
constexpr float kRescaleSlack = 8.f;  // e^8: largest softmax weight before a rescale

__device__ __forceinline__ float exp_f(float x) { return exp2f(x * kLog2e); }

__global__ void __launch_bounds__(kAThreads, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  tc::allow_dependents();    // the combine pass may be scheduled; it waits for this grid
  tc::wait_prerequisites();  // q, the caches and the lengths come from earlier kernels
  const int G = p.h_q / p.h_kv;
  const int64_t head0 = (int64_t)b * p.h_q + (int64_t)kvh * G;  // first query head
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o);
  const int64_t part_stride = (int64_t)p.n_split * (kD + 2);  // between query heads
  int len = p.cache_len[b];
  if (len < 0 || len > p.capacity) {  // recorded, and the sequence gets no keys
    if (tid == 0 && split == 0 && kvh == 0) raise_error(p.err, kErrBadCacheLen);
    len = 0;
  }
  const int start = split * p.block_keys;
  const int end = min(len, start + p.block_keys);
  const int nt = end > start ? (end - start + kTile - 1) / kTile : 0;

  if (nt == 0) {  // no cached key in this block: o = 0, or an empty partial
    if (tid < kEpiThreads) {
      for (int h = 0; h < G; ++h)
        for (int d = tid; d < kD; d += kEpiThreads) {
          if (p.n_split == 1) {
            o[(head0 + h) * kD + d] = __float2bfloat16_rn(0.f);
          } else {
            float* part = p.partial + (head0 + h) * part_stride + (int64_t)split * (kD + 2);
            part[d] = 0.f;
            if (d == 0) {
              part[kD] = -INFINITY;
              part[kD + 1] = 0.f;
            }
          }
        }
    }
    return;
  }

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + AS_BAR);
  uint64_t* empty = full + kAStages;
  uint64_t* bar_s = empty + kAStages;  // [2] S^T of a tile in TMEM
  uint64_t* p_ready = bar_s + 2;       // [2] P of a tile staged (128 epilogue arrivals)
  uint64_t* bar_o = p_ready + 2;       // [2] P V of a tile accumulated
  uint64_t* q_ready = bar_o + 2;       // Q^T staged (128 arrivals)
  uint64_t* drained = q_ready + 1;     // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drained + 1);
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kAttnTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kAStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bar_s[i], 1);
      tc::mbar_init(&p_ready[i], kEpiThreads);
      tc::mbar_init(&bar_o[i], 1);
    }
    tc::mbar_init(q_ready, kEpiThreads);
    tc::mbar_init(drained, 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = tc::smem_u32(smem);
  bool ok = true;

  if (warp == kAProducerWarp) {
    if (lane == 0) {
      tc::prefetch_tmap(&tm_k);
      tc::prefetch_tmap(&tm_v);
      const int64_t row0 = ((int64_t)b * p.h_kv + kvh) * p.capacity + start;
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int st = i % kAStages;
        if (i >= kAStages && !(ok = tc::mbar_wait(&empty[st], ((i / kAStages) - 1) & 1))) break;
        uint8_t* dst = smem + st * AS_STAGE;
        const int32_t y = static_cast<int32_t>(row0 + (int64_t)i * kTile);
        tc::mbar_arrive_expect_tx(&full[st], AS_STAGE);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          tc::tma_load_2d(dst + kb * 8192, &tm_k, 64 * kb, y, &full[st]);
          tc::tma_load_2d(dst + AS_V + kb * 8192, &tm_v, 64 * kb, y, &full[st]);
        }
        issued = i + 1;
      }
      // copies still in flight land before the CTA exits (already so unless a wait expired)
      for (int j = max(0, issued - kAStages); j < issued; ++j)
        if (!tc::mbar_wait(&full[j % kAStages], (j / kAStages) & 1)) ok = false;
    }
  } else if (warp == kAMmaWarp) {
    // the whole warp runs the loop; one elected lane issues
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      const bool w = tc::mbar_wait(bar, parity);
      tc::fence_after_sync();
      return __all_sync(kFullMask, w) != 0;
    };
    const uint64_t dQ = tc::smem_desc(sbase + AS_Q, 16, 1024, tc::kLayoutSw128);
    const uint64_t dK0 = tc::smem_desc(sbase, 16, 1024, tc::kLayoutSw128);
    const uint64_t dV0 = tc::smem_desc(sbase + AS_V, 8192, 1024, tc::kLayoutSw128);
    const uint64_t dP0 = tc::smem_desc(sbase + AS_P, 16, 1024, tc::kLayoutSw128);
    const bool leader = tc::elect_one();  // issues every product and commit of this warp
    auto issue_s = [&](int i) {  // S^T = K Q^T into S buffer i & 1
      const uint64_t so = (uint64_t)(((i % kAStages) * AS_STAGE) >> 4);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          tc::mma_bf16(tmem + TA_S + 8 * (i & 1),
                       dK0 + so + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
                       dQ + (((kk >> 2) * 1024 + (kk & 3) * 32) >> 4), IDA_S, kk > 0);
        tc::mma_commit(&bar_s[i & 1]);
      }
      __syncwarp();
    };
    ok = warp_wait(q_ready, 0) && warp_wait(&full[0], 0);
    if (ok) issue_s(0);
    for (int i = 0; i < nt && ok; ++i) {
      if (i + 1 < nt) {
        if (!(ok = warp_wait(&full[(i + 1) % kAStages], ((i + 1) / kAStages) & 1))) break;
        issue_s(i + 1);
      }
      if (!(ok = warp_wait(&p_ready[i & 1], (i >> 1) & 1))) break;
      const uint64_t so = (uint64_t)(((i % kAStages) * AS_STAGE) >> 4);
      if (leader) {
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)    // dims 64 kb .. 64 kb + 63
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // keys 16 kk .. 16 kk + 15
            tc::mma_bf16(tmem + TA_O + 8 * kb, dV0 + so + ((kb * 8192 + kk * 2048) >> 4),
                         dP0 + (((i & 1) * 1024 + kk * 32) >> 4), IDA_O, (i > 0) || (kk > 0));
        tc::mma_commit(&bar_o[i & 1]);
        tc::mma_commit(&empty[i % kAStages]);  // K and V of the tile consumed
      }
      __syncwarp();
    }
    // every MMA this warp issued has finished before TMEM is released
    if (leader) tc::mma_commit(drained);
    __syncwarp();
    if (!warp_wait(drained, 0)) ok = false;
  } else {
    // ---------------------------------------------------------- epilogue warps
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    {  // Q^T: row hh of the B operand = query head kvh G + hh (zeros past G)
      const int hh = tid >> 4, part = tid & 15;  // 16 threads per head, 16 dims each
      uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
      if (hh < G) {
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(p.q) + (head0 + hh) * kD + 16 * part);
        u0 = src[0];
        u1 = src[1];
      }
      uint8_t* box = smem + AS_Q + (part >> 2) * 1024;
      const uint32_t off = hh * 128 + 32 * (part & 3);
      *reinterpret_cast<uint4*>(box + tc::swizzle<3>(off)) = u0;
      *reinterpret_cast<uint4*>(box + tc::swizzle<3>(off + 16)) = u1;
      tc::fence_proxy_async();
      tc::mbar_arrive(q_ready);
    }
    // Online softmax with a lazy rescale: each head keeps a reference maximum m
    // and moves it only when a tile's maximum exceeds it by more than
    // kRescaleSlack, so the weights exp(s - m) stay below e^kRescaleSlack and O
    // is rescaled in TMEM only a few times per sequence; the result is the same
    // softmax.  Each thread sums its own keys' weights; the sums are reduced once
    // at the end.  Only the tile maxima cross warps (double-buffered by tile).
    float* red = reinterpret_cast<float*>(smem + AS_RED);  // [2][4 warps][8 heads]
    float m[kG], l[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    const int kloc = 16 * warp + lane;  // this thread's key in a tile (lanes 0-15 hold keys)
    bool carried = true;                // a wait that expired after the last barrier
    for (int i = 0; i < nt && ok; ++i) {
      const int st = i % kAStages;
      const int tile_valid = min(kTile, end - (start + i * kTile));
      bool mine = carried && tc::mbar_wait(&bar_s[i & 1], (i >> 1) & 1);
      tc::fence_after_sync();
      if (tile_valid < kTile && mine) {  // V rows past the end: zero them (they may hold anything)
        mine = tc::mbar_wait(&full[st], (i / kAStages) & 1);
        if (mine) {
          uint8_t* vt = smem + st * AS_STAGE + AS_V;
          const int n16 = (kTile - tile_valid) * 4 * 8;  // 16-byte chunks
          for (int c = tid; c < n16; c += kEpiThreads) {
            const int row = tile_valid + c / 32, rem = c % 32;
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * 8192 + row * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
      }
      // P buffer i & 1 is free once P V of tile i - 2 has completed
      if (i >= 2 && mine) mine = tc::mbar_wait(&bar_o[i & 1], ((i - 2) >> 1) & 1);
      float s[kG];
      tc::tmem_ld8(tmem + lane_base + TA_S + 8 * (i & 1), s);
      const bool valid = lane < 16 && kloc < tile_valid;
      float* rmax = red + (i & 1) * 4 * kG;
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        s[h] = (valid && h < G) ? s[h] * p.scale : -INFINITY;
        float x = s[h];
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kFullMask, x, off));
        if (lane == 0) rmax[warp * kG + h] = x;
      }
      if (!(ok = tc::named_sync_and(kABarEpi, kEpiThreads, mine))) break;  // uniform exit
      float alpha[kG];
      bool grow = false;
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        const float mt = fmaxf(fmaxf(rmax[h], rmax[kG + h]), fmaxf(rmax[2 * kG + h], rmax[3 * kG + h]));
        const float mn = mt > m[h] + kRescaleSlack ? mt : m[h];
        alpha[h] = mn == m[h] ? 1.f : exp_f(m[h] - mn);
        grow = grow || (mn != m[h]);
        m[h] = mn;
        s[h] = s[h] == -INFINITY ? 0.f : exp_f(s[h] - mn);
        l[h] = fmaf(l[h], alpha[h], s[h]);
      }
      if (lane < 16) {  // P (bf16): row h, column kloc of the K-major B operand
        uint8_t* pb = smem + AS_P + (i & 1) * 1024;
#pragma unroll
        for (int h = 0; h < kG; ++h)
          *reinterpret_cast<__nv_bfloat16*>(pb + tc::swizzle<3>(h * 128 + kloc * 2)) =
              __float2bfloat16_rn(s[h]);
      }
      if (i > 0 && grow) {  // O holds P V up to tile i - 1: rescale it (grow is CTA-uniform)
        const bool w = __all_sync(kFullMask, tc::mbar_wait(&bar_o[(i - 1) & 1], ((i - 1) >> 1) & 1));
        tc::fence_after_sync();
        if (w) {  // warp-uniform: the TMEM accesses below are warp-collective
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            float ov[kG];
            tc::tmem_ld8(tmem + lane_base + TA_O + 8 * kb, ov);
#pragma unroll
            for (int h = 0; h < kG; ++h) ov[h] *= alpha[h];
            tc::tmem_st8(tmem + lane_base + TA_O + 8 * kb, ov);
          }
        }
        carried = w;
      }
      tc::fence_proxy_async();  // P and the zeroed V rows -> the tensor core
      tc::fence_before_sync();
      tc::mbar_arrive(&p_ready[i & 1]);
    }
    if (ok) {  // the loop ran to its end in every epilogue warp
      const bool fin = carried && tc::mbar_wait(&bar_o[(nt - 1) & 1], ((nt - 1) >> 1) & 1);
      tc::fence_after_sync();
      float* rsum = red + (nt & 1) * 4 * kG;  // last read before the final tile's barrier
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        float x = l[h];
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) x += __shfl_xor_sync(kFullMask, x, off);
        if (lane == 0) rsum[warp * kG + h] = x;
      }
      ok = tc::named_sync_and(kABarEpi, kEpiThreads, fin);
      if (ok) {
#pragma unroll
        for (int h = 0; h < kG; ++h) l[h] = (rsum[h] + rsum[kG + h]) + (rsum[2 * kG + h] + rsum[3 * kG + h]);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          float ov[kG];
          tc::tmem_ld8(tmem + lane_base + TA_O + 8 * kb, ov);
          const int d = 64 * kb + 16 * warp + lane;  // valid for lanes 0-15
          if (lane < 16) {
#pragma unroll
            for (int h = 0; h < kG; ++h) {
              if (h >= G) break;
              if (p.n_split == 1) {
                o[(head0 + h) * kD + d] = __float2bfloat16_rn(l[h] > 0.f ? ov[h] / l[h] : 0.f);
              } else {
                float* part = p.partial + (head0 + h) * part_stride + (int64_t)split * (kD + 2);
                part[d] = ov[h];
                if (d == 0) {
                  part[kD] = m[h];
                  part[kD + 1] = l[h];
                }
              }
            }
          }
        }
      }
    }
  }
  if (!ok) raise_error(p.err, kErrDeviceTimeout);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, kAttnTmemCols);
}

// Merge the fixed-block partials of one (sequence, query head):
// o = sum_s e^{m_s - M} acc_s / sum_s e^{m_s - M} l_s with M = max_s m_s.  A block
// takes 64 of the 256 dimensions with four groups of threads, each summing every
// fourth split, so that many independent loads are in flight; the maximum, the
// weights and the normaliser are computed across the block (one split per thread).
constexpr int kCombineDims = 64, kCombineGroups = 4;
constexpr int kCombineThreads = kCombineDims * kCombineGroups;
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const AttnArgs p) {
  tc::wait_prerequisites();  // the partials of the attention kernel
  __shared__ float wsm[kCombineThreads], rsm[kCombineThreads / 32],
      part[kCombineGroups][kCombineDims];
  const int64_t bh = blockIdx.x;
  const int d0 = blockIdx.y * kCombineDims;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int dl = t % kCombineDims, grp = t / kCombineDims;
  const int64_t stride = kD + 2;
  const float* base = p.partial + bh * (int64_t)p.n_split * stride;
  float mx = -INFINITY;
  for (int s = t; s < p.n_split; s += kCombineThreads) mx = fmaxf(mx, base[s * stride + kD]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));
  if (lane == 0) rsm[warp] = mx;
  __syncthreads();
  float M = rsm[0];
#pragma unroll
  for (int w = 1; w < kCombineThreads / 32; ++w) M = fmaxf(M, rsm[w]);
  __syncthreads();  // rsm is reused for the normaliser below
  float num = 0.f, den = 0.f;
  for (int c0 = 0; c0 < p.n_split; c0 += kCombineThreads) {
    const int n = min(kCombineThreads, p.n_split - c0);
    if (t < n) {
      const float ms = base[(c0 + t) * stride + kD];
      const float w = (ms == -INFINITY || M == -INFINITY) ? 0.f : exp_f(ms - M);
      wsm[t] = w;
      den = fmaf(w, base[(c0 + t) * stride + kD + 1], den);
    }
    __syncthreads();
    const float* col = base + (int64_t)c0 * stride + d0 + dl;
#pragma unroll 8
    for (int j = grp; j < n; j += kCombineGroups) num = fmaf(wsm[j], col[j * stride], num);
    __syncthreads();
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(kFullMask, den, off);
  if (lane == 0) rsm[warp] = den;
  part[grp][dl] = num;
  __syncthreads();
  if (grp == 0) {
    float tot = 0.f, l = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < kCombineGroups; ++g2) tot += part[g2][dl];
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) l += rsm[w];
    static_cast<__nv_bfloat16*>(p.o)[bh * kD + d0 + dl] =
        __float2bfloat16_rn(l > 0.f ? tot / l : 0.f);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [rows][256] bf16 viewed as a 2-D tensor, 64 x 64 boxes with the 128-byte swizzle
bool encode_cache(CUtensorMap* map, const void* base, uint64_t rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {kD, rows};
  const cuuint64_t strides[1] = {kD * 2};
  const cuuint32_t box[2] = {64, kTile};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

AttnPlan attn_plan(int32_t batch, int32_t h_kv, int32_t capacity, int layout, int32_t block_keys,
                   int sm_count) {
  AttnPlan pl{};
  const int64_t cap = capacity > 0 ? capacity : 1;
  int64_t bk = block_keys;
  if (layout == kAttnGeneral) {
    bk = cap;
  } else if (bk <= 0) {
    // Fixed blocks sized so the CTAs (one resident per SM) fill the GPU about
    // once: (sequence, KV head) pairs x blocks ~ SM count, each block at least
    // kMinBlockKeys keys (measured at batch 1: 128-key blocks are fastest at 4K
    // and 8K keys; larger caches get larger blocks from the SM count anyway).
    const int64_t pairs = (int64_t)batch * h_kv;
    const int64_t want = pairs >= sm_count ? 1 : sm_count / (pairs > 0 ? pairs : 1);
    bk = (cap + want - 1) / want;
    bk = (bk + kTile - 1) / kTile * kTile;
    if (bk < kMinBlockKeys) bk = kMinBlockKeys;
    if (layout == kAttnAuto && bk >= cap) bk = cap;
  }
  if (bk > cap) bk = cap;
  pl.block_keys = static_cast<int32_t>(bk);
  pl.n_split = static_cast<int32_t>((cap + bk - 1) / bk);
  return pl;
}

size_t attn_partial_bytes(int32_t batch, int32_t h_q, const AttnPlan& pl) {
  if (pl.n_split <= 1) return 0;
  return (size_t)batch * h_q * pl.n_split * (kD + 2) * sizeof(float);
}

cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  const uint64_t rows = (uint64_t)a.batch * a.h_kv * a.capacity;
  if (rows > 0x7fffffffULL || a.h_kv > 65535 || a.batch > 65535 || a.n_split < 1)
    return cudaErrorInvalidValue;
  // With an empty cache (capacity 0) no block has a key and no copy is ever
  // issued; the maps then describe one row of q, which is never read through them.
  const void* kb = rows > 0 ? a.k_cache : a.q;
  const void* vb = rows > 0 ? a.v_cache : a.q;
  CUtensorMap mk, mv;
  if (!encode_cache(&mk, kb, rows > 0 ? rows : 1) || !encode_cache(&mv, vb, rows > 0 ? rows : 1))
    return cudaErrorInvalidValue;
  static PerDeviceOnce attrs;
  const cudaError_t attr_err = attrs.run([] {
    return cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kAttnSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  // Both kernels launch with programmatic stream serialization: each may be
  // scheduled while the kernel before it drains, and waits for that kernel's
  // results with griddepcontrol.wait before reading its inputs.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)a.n_split, (unsigned)a.h_kv, (unsigned)a.batch);
  cfg.blockDim = dim3(kAThreads);
  cfg.dynamicSmemBytes = kAttnSmem;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_decode_kernel, mk, mv, a);
  if (e != cudaSuccess || a.n_split == 1) return e;
  cfg.gridDim = dim3((unsigned)((int64_t)a.batch * a.h_q), kD / kCombineDims);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, a);
}

}  // namespace gdn
