// chunk_split.cu — chunked (WY/UT) prefill as two kernels that meet in a
// caller-provided workspace.
//
// The block form of the recurrence (page "Optimizing on-device inference for
// Apple Silicon", section "Qwen creates three distinct workload shapes") splits
// into work that does not depend on the state — per chunk of 64 tokens and
// value head: gates, the Q K^T / K K^T masks, the triangular solve
// T = (I + A)^{-1}, W = T diag(b Gamma) K, U~ = T diag(b) V — and the
// sequential state pass.
// chunk_prepare_kernel does the first part once per (chunk, value head), spread
// over every SM, and writes a "package" per item to the workspace, already in
// the swizzled shared-memory layout the tensor cores read:
//
//   [ -W half 0 | -W half 1 ]  bf16 [r][j], K-major SWIZZLE_128B, 2 x 8 KB
//   [ P ]                      bf16 [r][i], 8 KB   (e^{gamma_r - gamma_i} q_r.k_i, i <= r)
//   [ U~ slices 0..3 ]         bf16 [r][32 values of d_v], 64-byte rows with the
//                              SW64 XOR pattern, 4 x 4 KB  (U~ = T diag(beta) V)
//   [ gates ]                  fp32 Gamma_r / |q_r| [64], decay_r / |k_r| [64]
//                              (decay_r = e^{gamma_n - gamma_r}; |.| = 1 without the
//                              normalisation option), Gamma_n
//
// chunk_chain_kernel walks each (sequence, value head, 32-row slice of d_v) in
// chunk order with the fp32 state in TMEM, bulk-copying the packages into a
// 3-stage ring next to the TMA'd Q and K:
//   D = [U~; 0] + [-W; Q] S^T  (the product accumulates onto a buffer preloaded
//                               with U~, so D_top is U itself),
//   S^T <- Gamma_n S^T + K^T (decay U),  O = Gamma D_bottom + P U.
// Warp roles: a producer warp (copies), an MMA warp (one thread issues every
// product; an issue blocks while the tensor pipe is busy, so it gets a warp of
// its own) and four epilogue warps, handing over through mbarriers.  Only D,
// U, the state update and the state's staging are on the chunk-to-chunk
// critical path: P U of chunk c runs while chunk c's state is staged, and
// chunk c's output is written once chunk c+2's state is staged (D and P U are
// triple-buffered in TMEM), away from the U epilogue and the state staging.
// chunk_plan_kernel computes each sequence's first package index (an exclusive
// prefix sum of its chunk count) into the workspace header and records an
// inconsistent cu_seqlens in the error word.
//
// Compared with the single fused kernel (chunk_prefill.cu) the key-side work is
// done once per head instead of once per slice, and the chain's SM no longer
// shares its tensor pipe and shared memory with it.
//
// chunk_coop_kernel runs the same two parts in one cooperative grid, every CTA
// resident: prepare slots publish a ready flag per package and the state passes
// (64 rows of a head per CTA) follow them chunk by chunk, so the two overlap
// instead of running one after the other (the faster form from 4,096 tokens).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "chunk_common.cuh"
#include "params.h"
#include "per_device.h"
#include "rows.cuh"
#include "tc.cuh"

namespace gdn {

// Workspace layout (shared with the host-side size computation).
constexpr uint32_t kPkgW = 0, kPkgP = 16384, kPkgU = 24576, kPkgDK = 40960, kPkgGates = 57344;
constexpr uint32_t kPkgUSlice = 4096;  // U~ of one 32-wide slice of d_v
constexpr uint32_t kPkgBytes = 58368;  // 57 KB, a multiple of 1024 (swizzle phase)

size_t split_header_bytes(int32_t num_seqs) {
  // chunk_base [N+1] and the state passes' sequence order [N]
  return ((size_t)(2 * num_seqs + 1) * sizeof(int32_t) + 1023) / 1024 * 1024;
}
size_t split_max_items(int32_t num_seqs, int64_t total_tokens, int32_t h_v) {
  // sum_n ceil(L_n / 64) <= T / 64 + N
  return ((size_t)(total_tokens / chunk::kC) + (size_t)num_seqs + 1) * (size_t)h_v;
}

namespace {

using namespace chunk;

struct SplitParams {
  const float* g;
  const float* beta;
  const float* state_in;
  float* state_out;
  __nv_bfloat16* o;
  const int32_t* cu;
  int32_t num_seqs;
  int64_t total_tokens;
  int32_t h_k, h_v, d_v;  // (d_k: the kernels' template parameter DKP)
  float scale;
  int32_t min_len;
  int qk_norm;          // q and k divided by their L2 norm (+1e-6 under the root)
  int32_t* chunk_base;  // [N+1] in the workspace header (unused when single)
  int32_t* order;       // [N] after it: sequences by chunk count, longest first
  int single;           // one sequence: chunk c is item c * h_v + h, no plan kernel ran
  uint8_t* packages;    // items x kPkgBytes
  int64_t max_items;
  int* err;
};

__device__ __forceinline__ bool seq_range(const SplitParams& p, int n, int64_t& t0, int64_t& t1) {
  t0 = p.cu[n];
  t1 = p.cu[n + 1];
  return !(t0 < 0 || t1 < t0 || t1 > p.total_tokens || (n == 0 && t0 != 0) ||
           (n == p.num_seqs - 1 && t1 != p.total_tokens));
}

using tc::allow_dependents;
using tc::wait_prerequisites;

// ------------------------------------------------------------------ plan
__global__ void __launch_bounds__(256) chunk_plan_kernel(const SplitParams p) {
  allow_dependents();  // the prepare kernel's CTAs wait for this table themselves
  __shared__ int32_t warp_sums[8];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < p.num_seqs; base += 256) {
    const int n = base + threadIdx.x;
    int32_t cnt = 0;
    if (n < p.num_seqs) {
      int64_t t0, t1;
      if (seq_range(p, n, t0, t1)) {
        const int64_t L = t1 - t0;
        if (L >= p.min_len) cnt = (int32_t)((L + kC - 1) / kC);
      } else {
        raise_error(p.err, kErrBadCuSeqlens);
      }
    }
    // block-wide exclusive scan of cnt
    int32_t x = cnt;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(kFullMask, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    int32_t wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += warp_sums[w];
    const int32_t incl = carry + wbase + x;
    if (n < p.num_seqs) p.chunk_base[n] = incl - cnt;
    __syncthreads();
    if (threadIdx.x == 255) carry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) p.chunk_base[p.num_seqs] = carry;
  // The order in which the two-kernel form's state passes take sequences:
  // longest first, so that the longest chains start in the first wave (a
  // counting sort on floor(log2(chunks)), descending; the order within a
  // bucket is whatever the atomics give, which changes no result).
  __shared__ int32_t bucket[33];
  if (threadIdx.x < 33) bucket[threadIdx.x] = 0;
  __syncthreads();
  auto key = [&](int n) {  // 32 - floor(log2(chunks)) - 1 for chunks >= 1, else 32
    const int32_t cnt = p.chunk_base[n + 1] - p.chunk_base[n];
    return cnt > 0 ? __clz(cnt) : 32;
  };
  for (int n = threadIdx.x; n < p.num_seqs; n += 256) atomicAdd(&bucket[key(n)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t run = 0;
    for (int b = 0; b < 33; ++b) {
      const int32_t c = bucket[b];
      bucket[b] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int n = threadIdx.x; n < p.num_seqs; n += 256) p.order[atomicAdd(&bucket[key(n)], 1)] = n;
}

// ------------------------------------------------------------------ bulk copies
// global -> shared, completing on an mbarrier
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}
// shared -> global, in the issuing thread's bulk group
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(tc::smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The thread's committed bulk stores have read their shared memory ...
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... or have completed.
__device__ __forceinline__ void bulk_wait_done() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------ prepare
constexpr int kPrepThreads = 128;  // 4 warps; 4 CTAs per SM (TMEM, registers, shared memory)
constexpr uint32_t kBarAll = 1, kBarGateP = 2;
constexpr float kFactorRange = 80.f;  // |gamma| bound for Gamma_r / Gamma_i (e^80 < 2^127)
// Shared memory of the prepare kernel, reused as the item advances:
//   [0, 32K)     per d_k half kb: [Q 8K][K 8K] (TMA).  After G: Q0 stages P for
//                its bulk store, then holds V's first 64 columns (TMA); Q1 holds
//                the solve scratch, then T diag(b Gamma).  After W: K0 and Q1
//                stage the two halves of -W.  After U~: K1 and Q0 stage U~.
//   [32K, 49K)   A, then T: fp32 [64][kLdM]; then T diag(b) (bf16) at its start
//                and V's last 64 columns (TMA) 8K further on
//   gates        Gamma[64], decay[64], the mask column factors |k_i|^-1 / Gamma_i [64],
//                gamma[64], beta[64], the reciprocal L2 norms of the chunk's k rows
//                and q rows (1 without the normalisation option), and a flag: the
//                chunk's gamma range allows the factorised masks
constexpr uint32_t PP_KQ = 0;
constexpr uint32_t PP_Q1 = 16384;                  // solve scratch, then T diag(b Gamma)
constexpr uint32_t PP_Q0 = 0, PP_K0 = 8192, PP_K1 = 24576;
constexpr uint32_t PP_MF = 32768;
constexpr uint32_t PP_TA = PP_MF;                  // T diag(b), once T is in registers
constexpr uint32_t PP_V1 = PP_MF + 8192;           // V's columns 64-127 (V's 0-63 at Q0)
static_assert(PP_V1 + 8192 <= PP_MF + 64 * kLdM * 4, "V's second half inside the solve buffer");
constexpr uint32_t PP_GATE = PP_MF + 64 * kLdM * 4;
constexpr uint32_t PP_MISC = PP_GATE + 7 * 64 * 4 + 16;  // + the factorisation flag
constexpr uint32_t kPrepSmem = PP_MISC + 64 + 1024;
static_assert(4 * (kPrepSmem + 1024) <= 233472, "four prepare CTAs per SM");
constexpr uint32_t kPrepTmemCols = 128;  // G (cols 0-63), then W, then U~ (0-127)
constexpr uint32_t IDP_G = tc::idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDP_W = tc::idesc_bf16_f32(64, 128, false, true);

// The sequence n and chunk c of package item `item` (chunk-major: item = chunk
// id * h_v + value head); false past the last chunk.
__device__ __forceinline__ bool item_chunk(const SplitParams& p, int64_t item, int& n, int& c) {
  const int64_t cid = item / p.h_v;
  if (p.single) {  // no chunk table: the sequence's range is checked here instead
    int64_t t0, t1;
    if (!seq_range(p, 0, t0, t1)) {
      if (item == 0) raise_error(p.err, kErrBadCuSeqlens);
      return false;
    }
    const int64_t L = t1 - t0;
    if (L < p.min_len || cid >= (L + kC - 1) / kC) return false;
    n = 0;
    c = (int)cid;
    return true;
  }
  if (cid >= p.chunk_base[p.num_seqs]) return false;
  // the sequence owning chunk cid: last n with chunk_base[n] <= cid (skipping empty ones)
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.chunk_base[mid] <= cid) lo = mid; else hi = mid - 1;
  }
  n = lo;
  c = (int)(cid - p.chunk_base[n]);
  return true;
}

// Copy the 64-column half kb of key head hk's Q or K rows y .. y + 63.  The
// kernels below are compiled once per key dimension DKP: for DKP = 128 the map
// is 2-D ([rows][h_k * 128]); for DKP = 64 it is 3-D ([rows][h_k][64]) and the
// half at column 64 lies past the head's columns, so it arrives as zeros: the
// kernels see every key head zero-padded to 128 columns.  (A single build with
// a run-time choice measured ~5 % slower at 4,096 tokens than the 128-only code.)
template <int DKP>
__device__ __forceinline__ void kq_load(void* dst, const CUtensorMap* map, int hk, int kb,
                                        int32_t y, uint64_t* bar) {
  static_assert(DKP == kDK || DKP == kDK / 2, "key dimension 128 or 64");
  if constexpr (DKP == kDK)
    tc::tma_load_2d(dst, map, hk * kDK + 64 * kb, y, bar);
  else
    tc::tma_load_3d(dst, map, 64 * kb, hk, y, bar);
}

// Thread 0 of a prepare item issues the copies of its chunk's Q and K rows
// (key head of value head h) into the item's shared memory; bars[0] counts them.
template <int DKP>
__device__ __forceinline__ void prepare_loads(const SplitParams& p, const CUtensorMap* tm_q,
                                              const CUtensorMap* tm_k, uint8_t* smem,
                                              uint64_t* bars, int64_t item, int n, int c) {
  const int h = (int)(item % p.h_v);
  const int hk = h / (p.h_v / p.h_k);
  const int32_t y = static_cast<int32_t>(p.cu[n] + (int64_t)c * kC);
  tc::mbar_arrive_expect_tx(bars, 32768);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    kq_load<DKP>(smem + PP_KQ + kb * 16384, tm_q, hk, kb, y, bars);
    kq_load<DKP>(smem + PP_KQ + kb * 16384 + 8192, tm_k, hk, kb, y, bars);
  }
}

// One prepare item (chunk, value head) on 128 threads (pt = 0..127) with the
// shared-memory layout above at `smem`, 128 TMEM columns at `tmem`, three
// mbarriers `bars` (Q/K landed, an MMA done, V landed; initialised with count 1)
// that have seen k earlier items, and the named barriers bA (128 threads) and
// bG (threads 0-63); prepare_loads has been issued for it.  Writes the item's
// package: the gates with plain stores, P, -W and U~ staged in shared memory
// and written by bulk copies that thread 96 issues, and has seen complete when
// the item returns; false if a wait expired.
// The barrier ids are run-time values so that the cooperative form's four
// slots run one copy of this code (instruction-cache footprint).
__device__ __forceinline__ bool prepare_item(const SplitParams& p, const CUtensorMap* tm_v,
                                             uint8_t* smem, uint32_t tmem, uint64_t* bars,
                                             uint32_t k, int pt, int64_t item, int n, int c,
                                             uint32_t bA, uint32_t bG) {
  const int pw = pt >> 5, lane = pt & 31;
  const int h = (int)(item % p.h_v);
  const int64_t t_beg = p.cu[n], t_end = p.cu[n + 1];
  const int64_t t0 = t_beg + (int64_t)c * kC;
  uint8_t* pkg = p.packages + item * (int64_t)kPkgBytes;
  float* MF = reinterpret_cast<float*>(smem + PP_MF);
  float* YF = reinterpret_cast<float*>(smem + PP_Q1);
  float* gsm = reinterpret_cast<float*>(smem + PP_GATE);
  float *Gam = gsm, *dec = gsm + 64, *cf = gsm + 128, *gam = gsm + 192, *bet = gsm + 256;
  float *rk = gsm + 320, *rq = gsm + 384, *fact_flag = gsm + 448;
  uint64_t* bar_tma = bars;      // Q, K
  uint64_t* bar_mma = bars + 1;
  uint64_t* bar_v = bars + 2;    // V (needed only for U~)
  const uint32_t sbase = tc::smem_u32(smem);
  const int32_t y = static_cast<int32_t>(t0);
  float gr = 0.f, br = 0.f;
  if (pt < kC && t0 + pt < t_end) {
    gr = p.g[(t0 + pt) * p.h_v + h];
    br = p.beta[(t0 + pt) * p.h_v + h];
  }
  const uint32_t lane_base = static_cast<uint32_t>(pw * 32) << 16;
  bool ok = tc::mbar_wait(bar_tma, k & 1);
  tc::fence_after_sync();
  ok = tc::named_sync_and(bA, kPrepThreads, ok);
  if (ok) {
    if (pt == 64) {  // G = [Q;K] K^T: rows 0-63 Q K^T, rows 64-127 K K^T
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
        tc::mma_bf16(tmem, tc::smem_desc(sbase + PP_KQ + ko, 16, 1024, tc::kLayoutSw128),
                     tc::smem_desc(sbase + PP_KQ + ko + 8192, 16, 1024, tc::kLayoutSw128), IDP_G,
                     kk > 0);
      }
      tc::mma_commit(bar_mma);
    }
    {  // 1 / |row| of K (threads 0-63) and Q (64-127) with the normalisation option, else 1
      float r = 1.f;
      if (p.qk_norm) {
        const int t = pt & 63;
        const uint8_t* base = smem + PP_KQ + (pt < 64 ? 8192 : 0);
        float ss = 0.f;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const uint4 u = *reinterpret_cast<const uint4*>(
                base + kb * 16384 + tc::swizzle<3>(t * 128 + c8 * 16));
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
              ss = fmaf(lo, lo, ss);
              ss = fmaf(hi, hi, ss);
            }
          }
        r = rsqrtf(ss + 1e-6f);
      }
      (pt < 64 ? rk : rq)[pt & 63] = r;
    }
    if (pt < 64) {  // gates: inclusive scan of g over the chunk
      float x = gr;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float yv = __shfl_up_sync(kFullMask, x, off);
        if (lane >= off) x += yv;
      }
      if (pt == 31) MF[0] = x;
      tc::named_sync(bG, 64);
      if (pw == 1) x += MF[0];
      gam[pt] = x;
      const float Gx = tc::fast_exp(x);
      Gam[pt] = Gx;
      bet[pt] = br;
      float lo = x, hi = x;  // range of gamma over the chunk
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(kFullMask, lo, off));
        hi = fmaxf(hi, __shfl_xor_sync(kFullMask, hi, off));
      }
      if (lane == 0) {
        MF[2 + pw] = lo;
        MF[4 + pw] = hi;
      }
      tc::named_sync(bG, 64);
      dec[pt] = tc::fast_exp(gam[kC - 1] - x);
      // exp(gamma_r - gamma_i) = Gamma_r / Gamma_i without overflow or underflow
      // while every gamma of the chunk lies in [-kFactorRange, kFactorRange]
      const bool fact = fminf(MF[2], MF[3]) >= -kFactorRange && fmaxf(MF[4], MF[5]) <= kFactorRange;
      cf[pt] = fact ? rk[pt] / Gx : 0.f;
      if (pt == 0) *fact_flag = fact ? 1.f : 0.f;
    }
    ok = tc::mbar_wait(bar_mma, (3 * k) & 1);
    tc::fence_after_sync();
    ok = tc::named_sync_and(bA, kPrepThreads, ok);
    if (pt < 64) {  // the chain's per-row factors: Gamma_r / |q_r| for the output, decay_r / |k_r|
      float* gout = reinterpret_cast<float*>(pkg + kPkgGates);
      gout[pt] = Gam[pt] * rq[pt];
      gout[64 + pt] = dec[pt] * rk[pt];
      if (pt == 0) gout[128] = Gam[kC - 1];
    }
  }
  if (ok) {
    // masks, one G row per thread (TMEM lane pt): P rows (warps 0, 1) to the
    // package, A rows (warps 2, 3) to MF; 32 columns at a time.  Rows 0-31 have
    // no entry in columns 32-63 (above the diagonal).  The decay factor
    // exp(gamma_r - gamma_i) is the product of a row and a column factor when
    // the chunk's gamma range allows it (one exponential per element otherwise).
    const int r = 32 * (pw & 1) + lane;
    const float g_r = gam[r], b_r = bet[r];
    const float n_r = pw < 2 ? rq[r] : rk[r];  // q_r for P rows, k_r for A rows
    const bool fact = *fact_flag != 0.f;
    const float rowf = (pw < 2 ? 1.f : b_r) * Gam[r] * n_r;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      const int i0 = 32 * half;
      float a[32];
      const bool above = (pw & 1) == 0 && half == 1;  // warp-uniform
      if (above) {
#pragma unroll
        for (int e = 0; e < 32; ++e) a[e] = 0.f;
      } else {
        tc::tmem_ld32(tmem + lane_base + i0, a);
        const int lim = pw < 2 ? r : r - 1;  // P keeps i <= r, A keeps i < r
        if (fact) {
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 c4 = *reinterpret_cast<const float4*>(cf + i0 + 4 * e4);
            const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int e = 4 * e4 + q;
              a[e] = (i0 + e <= lim) ? (a[e] * cv[q]) * rowf : 0.f;
            }
          }
        } else {
          const float bf = pw < 2 ? 1.f : b_r;
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 gi = *reinterpret_cast<const float4*>(gam + i0 + 4 * e4);
            const float4 ki = *reinterpret_cast<const float4*>(rk + i0 + 4 * e4);
            const float gv[4] = {gi.x, gi.y, gi.z, gi.w}, kv[4] = {ki.x, ki.y, ki.z, ki.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int e = 4 * e4 + q;
              a[e] = (i0 + e <= lim) ? bf * tc::fast_exp(g_r - gv[q]) * a[e] * (n_r * kv[q]) : 0.f;
            }
          }
        }
      }
      if (pw < 2) {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8)
          st_chunk<3>(smem + PP_Q0, r * 128 + (4 * half + c8) * 16, a + 8 * c8);
      } else {
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4)
          *reinterpret_cast<float4*>(MF + r * kLdM + i0 + 4 * e4) =
              make_float4(a[4 * e4], a[4 * e4 + 1], a[4 * e4 + 2], a[4 * e4 + 3]);
      }
    }
    tc::fence_proxy_async();  // P's staging before its bulk store
    tc::fence_before_sync();
    tc::named_sync(bA, kPrepThreads);
    tc::fence_after_sync();
    if (pw >= 2) {  // warps 2-3 have no part in the solve's first level
      if (pt == 96) {
        bulk_s2g(pkg + kPkgP, smem + PP_Q0, 8192);
        bulk_commit();
        bulk_wait_read();  // then V's first 64 columns over the staged P
        tc::mbar_arrive_expect_tx(bar_v, 16384);
        tc::tma_load_2d(smem + PP_Q0, tm_v, h * p.d_v, y, bar_v);
      }
      // The state update's decayed K, diag(decay_r / |k_r|) K, into the package
      // as an image of K's two swizzled 64-column halves: a row's 16-byte pieces
      // move within its 128 bytes only, so piece o of the image is piece o of K
      // scaled by its row's factor; consecutive threads take consecutive pieces
      // (coalesced stores, conflict-free loads).
      const int u = pt - 64;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const uint32_t o = (uint32_t)(u + 64 * i) * 16;  // byte offset in the 16 KB image
        const uint32_t kb = o >> 13, ob = o & 8191;
        const float f = dec[ob >> 7] * rk[ob >> 7];
        const uint4 v = *reinterpret_cast<const uint4*>(smem + PP_KQ + kb * 16384 + 8192 + ob);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o4[e] = pack_bf16(__uint_as_float(w4[e] << 16) * f,
                            __uint_as_float(w4[e] & 0xffff0000u) * f);
        *reinterpret_cast<uint4*>(pkg + kPkgDK + o) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    }

    unit_lower_inverse<kPrepThreads>(MF, YF, pt, lane, bA);

    {  // T diag(b Gamma) over Q1 (W operand), T diag(b) over the start of MF (U~ operand)
      const int rr = pt >> 1, q = pt & 1;  // row rr, columns 32 q .. 32 q + 31
      float t[32];
      // the two threads of a row read their halves in orders 16 banks apart
      // (the halves start 32 floats apart: the same banks)
      float4 m[8];  // m[j]: columns 4 ((j + 4 q) mod 8) .. of the half
#pragma unroll
      for (int j = 0; j < 8; ++j)
        m[j] = *reinterpret_cast<const float4*>(MF + rr * kLdM + 32 * q + 4 * ((j + 4 * q) & 7));
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 v = q ? m[(e4 + 4) & 7] : m[e4];
        t[4 * e4] = v.x; t[4 * e4 + 1] = v.y; t[4 * e4 + 2] = v.z; t[4 * e4 + 3] = v.w;
      }
      tc::named_sync(bA, kPrepThreads);  // every row of T is read before TA overwrites MF
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const int ii = 32 * q + 8 * c8;
        float xa[8], xb[8], bv[8], gv[8], kv[8];
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4) {
          const float4 b4 = *reinterpret_cast<const float4*>(bet + ii + 4 * h4);
          const float4 g4 = *reinterpret_cast<const float4*>(Gam + ii + 4 * h4);
          const float4 k4 = *reinterpret_cast<const float4*>(rk + ii + 4 * h4);
          bv[4 * h4] = b4.x; bv[4 * h4 + 1] = b4.y; bv[4 * h4 + 2] = b4.z; bv[4 * h4 + 3] = b4.w;
          gv[4 * h4] = g4.x; gv[4 * h4 + 1] = g4.y; gv[4 * h4 + 2] = g4.z; gv[4 * h4 + 3] = g4.w;
          kv[4 * h4] = k4.x; kv[4 * h4 + 1] = k4.y; kv[4 * h4 + 2] = k4.z; kv[4 * h4 + 3] = k4.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          xa[e] = t[8 * c8 + e] * bv[e];
          xb[e] = xa[e] * gv[e] * kv[e];  // W = T diag(b Gamma / |k|) K
        }
        st_chunk<3>(smem + PP_TA, rr * 128 + (4 * q + c8) * 16, xa);
        st_chunk<3>(smem + PP_Q1, rr * 128 + (4 * q + c8) * 16, xb);
      }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    tc::named_sync(bA, kPrepThreads);
    tc::fence_after_sync();
    // V's columns 64-127 over the part of MF past T diag(b); columns past this
    // head's d_v (d_v < 128) belong to the next head or lie outside the tensor
    // (zero fill), and the slices built from them are never written
    if (pt == 96) tc::tma_load_2d(smem + PP_V1, tm_v, h * p.d_v + 64, y, bar_v);
    if (pt == 64) {  // W = (T b Gamma) K: M=64 N=128 K=64 (over G's columns)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16(tmem, tc::smem_desc(sbase + PP_Q1 + kk * 32, 16, 1024, tc::kLayoutSw128),
                     tc::smem_desc(sbase + PP_KQ + 8192 + kk * 2048, 16384, 1024, tc::kLayoutSw128),
                     IDP_W, kk > 0);
      tc::mma_commit(bar_mma);
    }
    ok = tc::mbar_wait(bar_mma, (3 * k + 1) & 1);
    tc::fence_after_sync();
    ok = tc::named_sync_and(bA, kPrepThreads, ok);
  }
  if (ok) {
    // -W (M=64 accumulator: row 16 w + l on lanes l = 0-15 of warp w's quarter),
    // staged in K0 (columns 0-63) and Q1 (64-127); thread l < 16 takes columns
    // 32 q .., thread l + 16 the same row's columns 64 + 32 q ..
    const int r = 16 * pw + (lane & 15), hi = lane >> 4;
    float w[32];
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {
      tc::tmem_ld16x2<64>(tmem + lane_base + 32 * q, w);
#pragma unroll
      for (int e = 0; e < 32; ++e) w[e] = -w[e];
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8)
        st_chunk<3>(smem + (hi ? PP_Q1 : PP_K0), r * 128 + (4 * q + c8) * 16, w + 8 * c8);
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    tc::named_sync(bA, kPrepThreads);  // W's columns are read before U~ overwrites them
    tc::fence_after_sync();
    if (pt == 96) {
      bulk_s2g(pkg + kPkgW, smem + PP_K0, 8192);
      bulk_s2g(pkg + kPkgW + 8192, smem + PP_Q1, 8192);
      bulk_commit();
    }
    if (pt == 64 && tc::mbar_wait(bar_v, k & 1)) {  // (on a timeout nothing commits: all time out)
      tc::fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // U~ = (T b) V: M=64 N=128 K=64
        tc::mma_bf16(tmem, tc::smem_desc(sbase + PP_TA + kk * 32, 16, 1024, tc::kLayoutSw128),
                     tc::smem_desc(sbase + PP_Q0 + kk * 2048, PP_V1 - PP_Q0, 1024,
                                   tc::kLayoutSw128),
                     IDP_W,
                     kk > 0);
      tc::mma_commit(bar_mma);
    }
    ok = tc::mbar_wait(bar_mma, (3 * k + 2) & 1);
    tc::fence_after_sync();
    ok = tc::named_sync_and(bA, kPrepThreads, ok);
    if (ok) {  // U~ slices (bf16, 64-byte rows with the SW64 XOR pattern): 0-1 in K1, 2-3 in Q0
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        tc::tmem_ld16x2<64>(tmem + lane_base + 32 * q, w);
        const int sl = q + 2 * hi;
        if (sl * kDVS < p.d_v) {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8)
            st_chunk<2>(smem + (hi ? PP_Q0 : PP_K1) + q * kPkgUSlice, r * 64 + c8 * 16,
                        w + 8 * c8);
        }
      }
    }
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  tc::named_sync(bA, kPrepThreads);
  tc::fence_after_sync();
  if (pt == 96) {  // U~'s bulk stores; every store of the item complete before it returns
    if (ok) {
#pragma unroll
      for (int sl = 0; sl < 4; ++sl)
        if (sl * kDVS < p.d_v)
          bulk_s2g(pkg + kPkgU + sl * kPkgUSlice,
                   smem + ((sl >> 1) ? PP_Q0 : PP_K1) + (sl & 1) * kPkgUSlice, kPkgUSlice);
      bulk_commit();
    }
    bulk_wait_done();
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  return ok;
}

template <int DKP>
__global__ void __launch_bounds__(kPrepThreads, 4)
    chunk_prepare_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int pt = threadIdx.x;
  const int64_t item = blockIdx.x;
  // The chain kernel may launch once every CTA of this grid has started; its
  // CTAs need an SM with room, so they start as this grid drains.
  allow_dependents();
  wait_prerequisites();  // the chunk table of the plan kernel
  int n, c;
  if (!item_chunk(p, item, n, c)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PP_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3);
  if (pt < 32) {
    tc::tmem_alloc(tmem_slot, kPrepTmemCols);
    tc::tmem_relinquish();
  }
  if (pt == 0) {
    for (int i = 0; i < 3; ++i) tc::mbar_init(&bars[i], 1);
    tc::fence_mbar_init();
    prepare_loads<DKP>(p, &tm_q, &tm_k, smem, bars, item, n, c);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool ok = prepare_item(p, &tm_v, smem, *tmem_slot, bars, 0, pt, item, n, c, kBarAll,
                               kBarGateP);
  if (!ok && pt == 0) raise_error(p.err, kErrDeviceTimeout);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (pt < 32) tc::tmem_dealloc(*tmem_slot, kPrepTmemCols);
}

// ------------------------------------------------------------------ chain
constexpr uint32_t kBarChainCta = 3;                     // named barrier of a chain's threads
// Main stage: per d_k half kb [-W | Q | K] (8 KB each; [-W; Q] is one 128-row
// operand), then the CTA's U~ slices (4 KB per 32 values); released once the
// chunk's state update is done.  Tail stage: P (8 KB) and, in a ring of their
// own after the other buffers, the chunk's gates; released after the chunk's
// output (one chunk later).  The 64 rows before each P are valid shared
// memory, as an M=128 operand whose other half is never read.
constexpr uint32_t kHalf = 24576;
constexpr uint32_t SC_W = 0, SC_Q = 8192, SC_K = 16384, SC_U = 2 * kHalf;
constexpr uint32_t kTail = 8192;      // P
constexpr uint32_t kGateBytes = 528;  // the package's gates: Gamma q[64], decay k[64], Gamma_n
constexpr uint32_t kTailTx = kTail + kGateBytes;

// A chain CTA that owns DVS (32 or 64) rows of a head's state (value dims),
// runs NSTG pipeline stages and EW epilogue warps (4, or 8 for DVS = 64: warps w
// and w + 4 share TMEM lanes 32 (w % 4) .. and take one 32-value block each).
// Operands of 32 values per row are SW64 blocks; DVS = 64 uses two blocks side
// by side (the MMA descriptors' leading offset).
template <int DVS, int NSTG, int EW = 4>
struct ChainCfg {
  static constexpr int NB = DVS / 32;
  static constexpr int BPW = NB * 4 / EW;  // 32-value blocks per epilogue warp
  static constexpr int kThreads = 32 * EW + 64;
  static constexpr int kProducerWarp = EW, kMmaWarp = EW + 1;
  static constexpr int kStages = NSTG, kEW = EW;
  static constexpr uint32_t kMain = SC_U + NB * kPkgUSlice;
  static constexpr uint32_t kMainTx = 4 * 8192 + 2 * 8192 + NB * kPkgUSlice;
  static constexpr uint32_t CC_TAIL = NSTG * kMain;
  static constexpr uint32_t CC_SS = CC_TAIL + NSTG * kTail;  // S^T bf16 [j][i]: NB x [128][32]
  // U bf16 [r][i]: NB x [64][32], two buffers (chunk parity), so that U of a
  // chunk is staged while P U of the previous one may still be reading its own
  static constexpr uint32_t CC_UB = CC_SS + NB * 8192;
  static constexpr uint32_t kUB = NB * 4096;
  static constexpr uint32_t CC_GATE = CC_UB + 2 * kUB;       // NSTG x kGateBytes
  static constexpr uint32_t CC_MISC = CC_GATE + NSTG * kGateBytes;
  static constexpr uint32_t kSmem = CC_MISC + 256 + 1024;
  static constexpr uint32_t kTmemCols = DVS == 32 ? 256 : 512;
  static constexpr uint32_t TC_D0 = 0, TC_O0 = 3 * DVS, TC_S = 6 * DVS;  // D, P U triple-buffered
  static constexpr uint32_t IDC_WQ = tc::idesc_bf16_f32(128, DVS, false, true);  // [-W; Q] S^T
  static constexpr uint32_t IDC_SU = tc::idesc_bf16_f32(128, DVS, true, true);   // (decay K)^T U
  static constexpr uint32_t IDC_PU = tc::idesc_bf16_f32(128, DVS, false, true);  // [.; P] U
  static_assert(DVS == 32 || DVS == 64, "32 or 64 state rows per CTA");
  static_assert((EW == 4 || EW == 8) && BPW >= 1, "4 or 8 epilogue warps, at most one per block");
  static_assert(kMainTx == kMain, "every main-stage byte arrives by TMA or bulk copy");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kMain % 1024 == 0 && kTail % 1024 == 0 && CC_TAIL % 1024 == 0 &&
                    CC_SS % 1024 == 0 && SC_U % 512 == 0,
                "swizzled operands need 1024 / 512 byte alignment");
  static_assert(7 * DVS <= (int)kTmemCols, "TMEM columns");
};

// Bounded wait for a prepare item's ready flag (stored with release semantics
// by the CTA that wrote the package), then order it before this thread's bulk
// copies of the package (async proxy).
__device__ __forceinline__ bool wait_item_flag(const int* flag,
                                               uint64_t timeout_ns = 200000000ull) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  if (v == 0) {
    const uint64_t t0 = tc::globaltimer_ns();
    do {
      __nanosleep(100);
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      if (v == 0 && tc::globaltimer_ns() - t0 > timeout_ns) return false;
    } while (v == 0);
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// The sequential state pass of one (sequence n, value head h, DVS-row slice s)
// on ChainCfg::kThreads threads: EW epilogue warps, a producer warp and an MMA
// warp.  With item_flags, a chunk's package is copied only once its flag is
// set (its prepare item runs in another CTA of the same cooperative grid).
template <int DVS, int NSTG, int EW, int DKP>
__device__ __forceinline__ void chain_run(const SplitParams& p, const CUtensorMap* tm_q,
                                          const CUtensorMap* tm_k, uint8_t* smem, int n, int h,
                                          int s, int tid, const int* item_flags) {
  using CF = ChainCfg<DVS, NSTG, EW>;
  constexpr int BPW = CF::BPW;
  constexpr int kEpiThreads = 32 * EW;
  const int warp = tid >> 5, lane = tid & 31;
  const int b0 = (warp >> 2) * BPW;      // first 32-value block of an epilogue warp
  const int jrow = 32 * (warp & 3) + lane;  // its TMEM lane: row of S^T (key dim)
  const int hk = h / (p.h_v / p.h_k);
  int64_t t_beg, t_end;
  if (!seq_range(p, n, t_beg, t_end)) {  // reported by the plan kernel, or here for one sequence
    if (p.single && tid == 0) raise_error(p.err, kErrBadCuSeqlens);
    return;
  }
  const int64_t L = t_end - t_beg;
  if (L < p.min_len) return;  // the token scan owns this sequence
  const int nchunks = (int)((L + kC - 1) / kC);
  const int64_t srow0 = ((int64_t)n * p.h_v + h) * p.d_v + s * DVS;

  // mbarriers.  full/tfull: TMA and bulk copies landed; empty: the stage's MMAs
  // are done (tcgen05.commit); tempty: the output warps took the chunk's gates.
  // bar_d, bar_s, bar_o: D, the state update, P U complete (tcgen05.commit;
  // bar_o one per chunk modulo 3); bar_u: the U warps staged U; bar_ss: every
  // epilogue warp staged the state.
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + CF::CC_MISC);
  uint64_t* empty = full + NSTG;
  uint64_t* tfull = empty + NSTG;
  uint64_t* tempty = tfull + NSTG;
  uint64_t* bar_d = tempty + NSTG;
  uint64_t* bar_s = bar_d + 1;
  uint64_t* bar_u = bar_s + 1;
  uint64_t* bar_ss = bar_u + 1;
  uint64_t* bar_o = bar_ss + 1;  // one per chunk modulo 3
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_o + 3);
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, CF::kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NSTG; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 2);  // after D and after the state update
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], 2 * kEpiThreads / 4);
    }
    tc::mbar_init(bar_d, 1);
    tc::mbar_init(bar_s, 1);
    tc::mbar_init(bar_u, 2 * kEpiThreads / 4);
    tc::mbar_init(bar_ss, kEpiThreads);
    for (int i = 0; i < 3; ++i) tc::mbar_init(&bar_o[i], 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  tc::named_sync(kBarChainCta, CF::kThreads);
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  bool ok = true;
  wait_prerequisites();  // the packages and chunk table (set-up above overlapped the prepare)
  const int64_t first_item = p.single ? h : (int64_t)p.chunk_base[n] * p.h_v + h;

  if (warp == CF::kProducerWarp) {
    if (lane == 0) {
      tc::prefetch_tmap(tm_q);
      tc::prefetch_tmap(tm_k);
      for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c % NSTG;
        const int64_t item = first_item + (int64_t)c * p.h_v;
        const uint8_t* pkg = p.packages + item * kPkgBytes;
        if (c >= NSTG) ok = tc::mbar_wait(&empty[st], ((c / NSTG) - 1) & 1);
        if (ok && item_flags) ok = wait_item_flag(item_flags + item);
        if (!ok) break;
        uint8_t* dst = smem + st * CF::kMain;
        const int32_t y = static_cast<int32_t>(t_beg + (int64_t)c * kC);
        uint64_t* fb = &full[st];
        tc::mbar_arrive_expect_tx(fb, CF::kMainTx);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          kq_load<DKP>(dst + kb * kHalf + SC_Q, tm_q, hk, kb, y, fb);
          bulk_g2s(dst + kb * kHalf + SC_K, pkg + kPkgDK + kb * 8192, 8192, fb);
          bulk_g2s(dst + kb * kHalf + SC_W, pkg + kPkgW + kb * 8192, 8192, fb);
        }
        bulk_g2s(dst + SC_U, pkg + kPkgU + s * CF::NB * kPkgUSlice, CF::NB * kPkgUSlice, fb);
        if (c >= NSTG) ok = tc::mbar_wait(&tempty[st], ((c / NSTG) - 1) & 1);
        if (!ok) break;
        tc::mbar_arrive_expect_tx(&tfull[st], kTailTx);
        bulk_g2s(smem + CF::CC_TAIL + st * kTail, pkg + kPkgP, 8192, &tfull[st]);
        bulk_g2s(smem + CF::CC_GATE + st * kGateBytes, pkg + kPkgGates, kGateBytes, &tfull[st]);
      }
    }
  } else if (warp == CF::kMmaWarp) {
    // Issues every tensor-core product, in the order the chain needs them.  The
    // whole warp runs the loop converged: every lane waits on the barrier
    // itself, and one elected lane issues the MMAs and commits.  (Measured on
    // GB300, this issues ~10 % faster per call than a loop that only lane 0
    // runs, and much faster than lane 0 waiting and broadcasting by shuffle.)
    // Per chunk c:  [stage landed, state staged] D(c) -> [U staged] S update(c) -> P U(c)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      const bool w = tc::mbar_wait(bar, parity);
      tc::fence_after_sync();
      return __all_sync(kFullMask, w) != 0;
    };
    // Operand descriptors built once; a stage or K step only adds its byte
    // offset / 16 to the start-address field (every address is below 256 KB).
    // The leading byte offset steps between the 32-value blocks (DVS = 64).
    const uint64_t dSS = tc::smem_desc(sbase + CF::CC_SS, 8192, 512, tc::kLayoutSw64);
    const uint64_t dUB = tc::smem_desc(sbase + CF::CC_UB, 4096, 512, tc::kLayoutSw64);
    const uint64_t dW0 = tc::smem_desc(sbase + SC_W, 16, 1024, tc::kLayoutSw128);
    const uint64_t dK0 = tc::smem_desc(sbase + SC_K, kHalf, 1024, tc::kLayoutSw128);
    const uint64_t dP0 =
        tc::smem_desc(sbase + CF::CC_TAIL - 8192, 16, 1024, tc::kLayoutSw128);
    const bool leader = tc::elect_one();  // issues every product and commit of this warp
    for (int c = 0; c < nchunks && ok; ++c) {
      const int st = c % NSTG;
      const uint64_t so = (uint64_t)((st * CF::kMain) >> 4), to = (uint64_t)((st * kTail) >> 4);
      const uint64_t dW = dW0 + so, dK = dK0 + so, dP = dP0 + to;
      const uint64_t dU = dUB + (uint64_t)(((c & 1) * CF::kUB) >> 4);
      const uint32_t td = tmem + CF::TC_D0 + DVS * (c % 3), to2 = tmem + CF::TC_O0 + DVS * (c % 3);
      if (!(ok = warp_wait(&full[st], (c / NSTG) & 1) && warp_wait(bar_ss, c & 1))) break;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // D = [U~; 0] + [-W; Q] S_s^T (preloaded buffer)
          tc::mma_bf16(td, dW + (((kk >> 2) * kHalf + (kk & 3) * 32) >> 4),
                       dSS + ((kk * 1024) >> 4), CF::IDC_WQ, 1);
        tc::mma_commit(bar_d);
        tc::mma_commit(&empty[st]);  // D has read -W and Q of the stage
      }
      __syncwarp();
      if (!(ok = warp_wait(bar_u, c & 1))) break;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // S^T += (decayed K)^T U, onto Gamma_n S^T
          tc::mma_bf16(tmem + CF::TC_S, dK + ((kk * 2048) >> 4), dU + ((kk * 1024) >> 4),
                       CF::IDC_SU, 1);
        tc::mma_commit(bar_s);
        tc::mma_commit(&empty[st]);  // the update has read K of the stage
      }
      __syncwarp();
      if (!(ok = warp_wait(&tfull[st], (c / NSTG) & 1))) break;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // O2 = P U (rows 64-127)
          tc::mma_bf16(to2, dP + ((kk * 32) >> 4), dU + ((kk * 1024) >> 4), CF::IDC_PU, kk > 0);
        tc::mma_commit(&bar_o[c % 3]);
      }
      __syncwarp();
    }
  } else if (warp < EW) {
    // Epilogue warps.  Those on TMEM lanes 0-63 form U (staged once: the update
    // takes the package's decayed K, so no per-row scaling is left on this
    // critical step) and preload the next chunk's U~; those on lanes 64-127
    // take the previous chunk's gates, clear rows 64-127 of the next D buffer
    // and, once the state is staged, store the previous chunk's output; all
    // stage the state.  Every hand-off is an mbarrier with a bounded wait.
    const int rl = 32 * (warp & 1) + lane;  // accumulator row of this thread within its half
    // Output of chunk cp (the warps on lanes 64-127): O = Gamma Q S^T + P U, in
    // two parts.  take_gates(cp) waits for P U, reads the rows' output factors
    // and releases the chunk's tail stage early, so that the next tail copy has
    // time to land; write_output(cp) forms and stores the rows after the next
    // state has been staged, so that its global stores neither compete with the
    // U warps' shared-memory stores nor delay the state (D and P U are
    // triple-buffered in TMEM for that).
    auto take_gates = [&](int cp) {
      const int stp = cp % NSTG;
      // P U of chunk cp + 3 is issued only after these warps stage chunk cp + 3's
      // state, later than this wait, so the phase parity is unambiguous
      ok = tc::mbar_wait(&bar_o[cp % 3], (cp / 3) & 1) && ok;
      tc::fence_after_sync();
      const float gr =
          reinterpret_cast<const float*>(smem + CF::CC_GATE + stp * kGateBytes)[rl];
      tc::fence_before_sync();
      tc::mbar_arrive(&tempty[stp]);
      return gr;
    };
    auto write_output = [&](int cp, float Gam_r) {
      const int64_t t0p = t_beg + (int64_t)cp * kC;
      const int nvp = (int)((L - (int64_t)cp * kC) < kC ? (L - (int64_t)cp * kC) : kC);
#pragma unroll
      for (int b = b0; b < b0 + BPW; ++b) {
        float o1[32], o2[32];
        tc::tmem_ld32(tmem + lane_base + CF::TC_D0 + DVS * (cp % 3) + 32 * b, o1);
        tc::tmem_ld32(tmem + lane_base + CF::TC_O0 + DVS * (cp % 3) + 32 * b, o2);
        if (rl < nvp) {
#pragma unroll
          for (int i = 0; i < 32; ++i) o1[i] = p.scale * fmaf(Gam_r, o1[i], o2[i]);
          uint4* dst = reinterpret_cast<uint4*>(p.o + ((t0p + rl) * p.h_v + h) * (int64_t)p.d_v +
                                                s * DVS + 32 * b);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint4 q4;
            q4.x = pack_bf16(o1[8 * c4 + 0], o1[8 * c4 + 1]);
            q4.y = pack_bf16(o1[8 * c4 + 2], o1[8 * c4 + 3]);
            q4.z = pack_bf16(o1[8 * c4 + 4], o1[8 * c4 + 5]);
            q4.w = pack_bf16(o1[8 * c4 + 6], o1[8 * c4 + 7]);
            dst[c4] = q4;
          }
        }
      }
    };
    // S (fp32, thread j holds column j of the slice) -> bf16 operand copy for
    // chunk cn's D, then Gamma_n of chunk cn applied in TMEM (the update MMA
    // accumulates onto it); then tell the MMA warp.
    auto stage_state = [&](float (&sc)[32 * BPW], int cn) {
#pragma unroll
      for (int b = 0; b < BPW; ++b)
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          st_chunk<2>(smem + CF::CC_SS + (b0 + b) * 8192, jrow * 64 + c4 * 16, sc + 32 * b + 8 * c4);
      const int stn = cn % NSTG;
      ok = tc::mbar_wait(&tfull[stn], (cn / NSTG) & 1) && ok;
      const float Gam_n =
          reinterpret_cast<const float*>(smem + CF::CC_GATE + stn * kGateBytes)[128];
#pragma unroll
      for (int i = 0; i < 32 * BPW; ++i) sc[i] *= Gam_n;
#pragma unroll
      for (int b = 0; b < BPW; ++b)
        tc::tmem_st32(tmem + lane_base + CF::TC_S + 32 * (b0 + b),
                      *reinterpret_cast<const float(*)[32]>(sc + 32 * b));
      tc::fence_proxy_async();
      tc::fence_before_sync();
      tc::mbar_arrive(bar_ss);
    };
    // D of chunk cn accumulates onto its TMEM buffer, preloaded with U~ in rows
    // 0-63 (by the warps on those lanes) and zeros in rows 64-127 (the output
    // warps), so that U = U~ - W S^T comes out of the product itself.  Written
    // before the warps stage the state that D waits for; off the critical path.
    auto preload = [&](int cn) {
      const int stn = cn % NSTG;
      const uint32_t td = tmem + lane_base + CF::TC_D0 + DVS * (cn % 3);
      float u[32];
      if ((warp & 3) < 2) {
        ok = tc::mbar_wait(&full[stn], (cn / NSTG) & 1) && ok;  // U~ arrived by bulk copy
#pragma unroll
        for (int b = b0; b < b0 + BPW; ++b) {
          const uint8_t* ut = smem + stn * CF::kMain + SC_U + b * kPkgUSlice;  // row of U~, bf16
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 q4 =
                *reinterpret_cast<const uint4*>(ut + tc::swizzle<2>(rl * 64 + j * 16));
            const uint32_t w4[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              u[8 * j + 2 * e] = __uint_as_float(w4[e] << 16);
              u[8 * j + 2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
            }
          }
          tc::tmem_st32(td + 32 * b, u);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] = 0.f;
#pragma unroll
        for (int b = b0; b < b0 + BPW; ++b) tc::tmem_st32(td + 32 * b, u);
      }
    };
    {  // initial state: rows 32 b0 .. of the slice, column jrow
      float sc[32 * BPW];
#pragma unroll
      for (int i = 0; i < 32 * BPW; ++i)
        sc[i] = p.state_in && jrow < DKP ? p.state_in[(srow0 + 32 * b0 + i) * DKP + jrow]
                                         : 0.f;  // key columns past d_k stay zero
      if (nchunks == 0) {
        if (jrow < DKP)
#pragma unroll
          for (int i = 0; i < 32 * BPW; ++i)
            p.state_out[(srow0 + 32 * b0 + i) * DKP + jrow] = sc[i];
      } else {
        preload(0);
        stage_state(sc, 0);
      }
    }
    float gam_prev = 0.f;  // output factor of the previous chunk's rows (output warps)
    for (int c = 0; c < nchunks && ok; ++c) {
      if ((warp & 3) < 2) {  // U = U~ - W S^T for rows r = lanes 0-63
        // D(c) completes after P U(c - 2), the last reader of the U buffer about
        // to be rewritten: one thread issued both and committed bar_d after D(c),
        // and a commit covers every earlier product of its thread.  (Waiting on
        // P U(c - 2)'s own barrier here measured ~2 % slower per call.)
        ok = tc::mbar_wait(bar_d, c & 1) && ok;
        tc::fence_after_sync();
#pragma unroll
        for (int b = b0; b < b0 + BPW; ++b) {
          float u[32];
          tc::tmem_ld32(tmem + lane_base + CF::TC_D0 + DVS * (c % 3) + 32 * b, u);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            st_chunk<2>(smem + CF::CC_UB + (c & 1) * CF::kUB + b * 4096, rl * 64 + c4 * 16,
                        u + 8 * c4);
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        tc::mbar_arrive(bar_u);
        if (c + 1 < nchunks) preload(c + 1);  // while the state update runs
      } else {
        if (c > 0) gam_prev = take_gates(c - 1);
        if (c + 1 < nchunks) preload(c + 1);  // the buffer's rows were read by output c - 2
        ok = tc::mbar_wait(bar_d, c & 1) && ok;  // D has read the staged state rewritten below
      }
      ok = tc::mbar_wait(bar_s, c & 1) && ok;
      tc::fence_after_sync();
      float sc[32 * BPW];
#pragma unroll
      for (int b = 0; b < BPW; ++b)
        tc::tmem_ld32(tmem + lane_base + CF::TC_S + 32 * (b0 + b),
                      *reinterpret_cast<float(*)[32]>(sc + 32 * b));
      if (c == nchunks - 1) {
        if (jrow < DKP)
#pragma unroll
          for (int i = 0; i < 32 * BPW; ++i)
            p.state_out[(srow0 + 32 * b0 + i) * DKP + jrow] = sc[i];
      } else {
        stage_state(sc, c + 1);
      }
      if ((warp & 3) >= 2 && c > 0) write_output(c - 1, gam_prev);  // after the staging
    }
    if (ok && nchunks > 0 && (warp & 3) >= 2)  // the last output
      write_output(nchunks - 1, take_gates(nchunks - 1));
  }
  if (!ok) raise_error(p.err, kErrDeviceTimeout);
  tc::fence_before_sync();
  tc::named_sync(kBarChainCta, CF::kThreads);
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, CF::kTmemCols);
}

// The chain of the two-kernel form: 32 state rows per CTA, 3 stages, 4
// epilogue warps; or, when the batch's chains fill more than one wave of SMs,
// 64 rows per CTA (N = 64 products, 8 epilogue warps), which costs less SM
// time per row.  With more than one sequence, CTAs take sequences in the plan
// kernel's order (longest first).
using SplitChain = ChainCfg<kDVS, 3, 4>;
using SplitChain64 = ChainCfg<64, 3, 8>;

template <class CF, int DKP>
__global__ void __launch_bounds__(CF::kThreads, 1)
    chunk_chain_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kRows = CF::NB * 32;
  const int ns = p.d_v / kRows;
  const int s = blockIdx.x % ns;
  const int h = (blockIdx.x / ns) % p.h_v;
  int n = 0;
  if (!p.single) {
    wait_prerequisites();  // the plan kernel's order
    n = p.order[blockIdx.x / (ns * p.h_v)];
  }
  chain_run<kRows, CF::kStages, CF::kEW, DKP>(p, &tm_q, &tm_k, smem, n, h, s, threadIdx.x,
                                              nullptr);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// Q or K for d_k < 128 as a 3-D tensor [rows][heads][d] (d innermost) read in
// boxes of 64 columns x 1 head x 64 tokens (see kq_load).
bool encode_heads_map(CUtensorMap* map, const void* base, uint64_t d, uint64_t heads,
                      uint64_t rows) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d, heads, rows};
  const cuuint64_t strides[2] = {d * 2, heads * d * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kC};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ cooperative form
// One grid with every CTA resident (cooperative launch, one CTA per SM).  The
// first n_chain CTAs each run the chain of one (sequence, value head, 64-row
// slice); the others run prepare items in four slots of 128 threads, in chunk
// order, and store a ready flag per item once its package is written.  A
// chain's producer waits for the flag before copying the package, so the
// chain follows the prepare chunk by chunk instead of starting after all of it.
// Waits go one way only (chain on prepare), and every CTA is resident, so the
// grid cannot deadlock; each wait is bounded as well.
using CoopChain = ChainCfg<64, 3, 8>;
constexpr int kCoopSlots = 4;
constexpr int kCoopThreads = kCoopSlots * kPrepThreads;
constexpr uint32_t kPrepSlotBytes = (kPrepSmem - 1024 + 1023) / 1024 * 1024;
constexpr uint32_t kCoopSmem = CoopChain::kSmem > kCoopSlots * kPrepSlotBytes + 1024
                                   ? CoopChain::kSmem
                                   : kCoopSlots * kPrepSlotBytes + 1024;
static_assert(CoopChain::kThreads <= kCoopThreads, "the chain fits in the grid's CTAs");
static_assert(kCoopSmem <= 227 * 1024, "shared memory budget");
static_assert(kCoopSlots * kPrepTmemCols <= 512, "TMEM of the prepare slots");

// Slot s of a CTA starts kSlotStaggerNs x s after slot 0: the first items
// (the first chunks, which every state pass waits for) then do not all pass
// through the same phases on an SM at once.
constexpr uint32_t kSlotStaggerNs = 2000;

// One prepare slot: 128 threads with their own shared memory, TMEM, mbarriers
// and named barriers bA, bG.  Its first item is `first` (slot s of prepare CTA
// r takes s x n_prep + r, so the first chunks spread over the SMs); later items
// come from a counter shared by all n_slots slots (flags[max_items], zero at
// launch), in increasing order, i.e. chunk by chunk.
template <int DKP>
__device__ __forceinline__ void coop_prepare_slot(const SplitParams& p, const CUtensorMap* tm_q,
                                                  const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                                  uint8_t* smem, int pt, int* flags, uint32_t bA,
                                                  uint32_t bG, int slot, int first, int n_slots) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PP_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3);
  int* next = reinterpret_cast<int*>(bars + 4);  // the slot's item, from the shared counter
  if (pt < 32) tc::tmem_alloc(tmem_slot, kPrepTmemCols);
  if (pt == 0) {
    for (int i = 0; i < 3; ++i) tc::mbar_init(&bars[i], 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  tc::named_sync(bA, kPrepThreads);
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (pt == 0 && slot > 0) {  // a fixed delay (a sleep, not a wait on anything)
    const uint64_t t0 = tc::globaltimer_ns();
    while (tc::globaltimer_ns() - t0 < (uint64_t)slot * kSlotStaggerNs) __nanosleep(256);
  }
  bool ok = true;
  uint32_t k = 0;
  for (;; ++k) {
    if (pt == 0) *next = k == 0 ? first : n_slots + atomicAdd(flags + p.max_items, 1);
    tc::named_sync(bA, kPrepThreads);
    const int64_t item = *next;
    int n, c;
    if (!ok || item >= p.max_items || !item_chunk(p, item, n, c)) break;  // past the last chunk
    if (pt == 0) prepare_loads<DKP>(p, tm_q, tm_k, smem, bars, item, n, c);
    ok = prepare_item(p, tm_v, smem, tmem, bars, k, pt, item, n, c, bA, bG);
    // Every thread's package stores are visible device-wide before the flag;
    // the slot's shared memory and TMEM are free for the next item.
    __threadfence();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    tc::fence_proxy_async();
    tc::fence_before_sync();
    tc::named_sync(bA, kPrepThreads);
    tc::fence_after_sync();
    if (pt == 96 && ok)  // the thread that saw the package's bulk stores complete
      asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flags + item), "r"(1) : "memory");
  }
  if (!ok && pt == 0) raise_error(p.err, kErrDeviceTimeout);
  tc::fence_before_sync();
  tc::named_sync(bA, kPrepThreads);
  tc::fence_after_sync();
  if (pt < 32) tc::tmem_dealloc(tmem, kPrepTmemCols);
}

template <int DKP>
__global__ void __launch_bounds__(kCoopThreads, 1)
    chunk_coop_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const SplitParams p, int n_chain,
                      int* flags) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  if ((int)blockIdx.x < n_chain) {
    if ((int)threadIdx.x >= CoopChain::kThreads) return;
    constexpr int kRows = CoopChain::NB * 32;
    const int ns = p.d_v / kRows;
    const int s = blockIdx.x % ns;
    const int h = (blockIdx.x / ns) % p.h_v;
    const int n = blockIdx.x / (ns * p.h_v);
    chain_run<kRows, CoopChain::kStages, CoopChain::kEW, DKP>(p, &tm_q, &tm_k, smem, n, h, s,
                                                         threadIdx.x, flags);
    return;
  }
  wait_prerequisites();  // the chunk table of the plan kernel
  const int slot = threadIdx.x / kPrepThreads, pt = threadIdx.x % kPrepThreads;
  uint8_t* sm = smem + slot * kPrepSlotBytes;
  // named barriers 1 + 2 slot (the slot's 128 threads) and 2 + 2 slot (its first 64)
  const int n_prep = (int)gridDim.x - n_chain;
  coop_prepare_slot<DKP>(p, &tm_q, &tm_k, &tm_v, sm, pt, flags, 1u + 2u * slot, 2u + 2u * slot,
                         slot,
                    slot * n_prep + ((int)blockIdx.x - n_chain), n_prep * kCoopSlots);
}

}  // namespace

size_t split_workspace_bytes(int32_t num_seqs, int64_t total_tokens, int32_t h_v) {
  return split_header_bytes(num_seqs) + split_max_items(num_seqs, total_tokens, h_v) * kPkgBytes;
}

size_t coop_workspace_bytes(int32_t num_seqs, int64_t total_tokens, int32_t h_v) {
  // one ready flag per item and the item counter of the prepare slots
  const size_t flags =
      ((split_max_items(num_seqs, total_tokens, h_v) + 1) * sizeof(int) + 1023) / 1024 * 1024;
  return split_workspace_bytes(num_seqs, total_tokens, h_v) + flags;
}

bool coop_supported(int32_t num_seqs, int32_t h_v, int32_t d_v, int sm_count) {
  // 64-row chain slices; at least a third of the SMs left for the prepare slots
  if (d_v % 64 != 0) return false;
  const int64_t n_chain = (int64_t)num_seqs * h_v * (d_v / 64);
  return n_chain >= 1 && n_chain <= (int64_t)sm_count * 2 / 3;
}

// Tensor maps (Q, K, V in 64-column boxes) and kernel parameters shared by the
// two-kernel and the cooperative forms.
bool split_setup(const PrefillArgs& a, void* workspace, CUtensorMap& mq, CUtensorMap& mk,
                 CUtensorMap& mv, SplitParams& p) {
  const uint64_t rows = a.total_tokens > 0 ? (uint64_t)a.total_tokens : 1;
  const void* qp = a.total_tokens > 0 ? a.q : a.state_out;
  const void* kp = a.total_tokens > 0 ? a.k : a.state_out;
  const void* vp = a.total_tokens > 0 ? a.v : a.state_out;
  const bool kq_ok =
      a.d_k == kDK
          ? encode_map(&mq, qp, (uint64_t)a.h_k * kDK, rows, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
                encode_map(&mk, kp, (uint64_t)a.h_k * kDK, rows, 64, kC,
                           CU_TENSOR_MAP_SWIZZLE_128B)
          : encode_heads_map(&mq, qp, (uint64_t)a.d_k, (uint64_t)a.h_k, rows) &&
                encode_heads_map(&mk, kp, (uint64_t)a.d_k, (uint64_t)a.h_k, rows);
  if (!kq_ok ||
      !encode_map(&mv, vp, (uint64_t)a.h_v * a.d_v, rows, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  p.g = a.g;
  p.beta = a.beta;
  p.state_in = a.state_in;
  p.state_out = a.state_out;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.cu = a.cu_seqlens;
  p.num_seqs = a.num_seqs;
  p.total_tokens = a.total_tokens;
  p.h_k = a.h_k;
  p.h_v = a.h_v;
  p.d_v = a.d_v;
  p.scale = a.scale;
  p.min_len = a.min_chunk_len;
  p.qk_norm = a.qk_norm;
  p.chunk_base = static_cast<int32_t*>(workspace);
  p.order = p.chunk_base + (a.num_seqs + 1);
  p.packages = static_cast<uint8_t*>(workspace) + split_header_bytes(a.num_seqs);
  p.max_items = (int64_t)split_max_items(a.num_seqs, a.total_tokens, a.h_v);
  p.err = a.err;
  p.single = a.num_seqs == 1 ? 1 : 0;
  return true;
}

namespace {

template <int DKP>
cudaError_t launch_coop_dk(const PrefillArgs& a, void* workspace, cudaStream_t stream, int sms) {
  CUtensorMap mq, mk, mv;
  SplitParams p;
  if (!split_setup(a, workspace, mq, mk, mv, p)) return cudaErrorInvalidValue;
  if (p.max_items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.run([] {
    return cudaFuncSetAttribute(chunk_coop_kernel<DKP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kCoopSmem);
  });
  if (e != cudaSuccess) return e;
  int resident = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, chunk_coop_kernel<DKP>,
                                                    kCoopThreads, kCoopSmem);
  if (e != cudaSuccess) return e;
  if (resident < 1) return cudaErrorNotSupported;
  int* flags = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) +
                                      split_workspace_bytes(a.num_seqs, a.total_tokens, a.h_v));
  if (!p.single) {  // one sequence needs no chunk table
    chunk_plan_kernel<<<1, 256, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess)
    e = cudaMemsetAsync(flags, 0, (size_t)(p.max_items + 1) * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  const int n_chain = a.num_seqs * a.h_v * (a.d_v / 64);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(kCoopThreads);
  cfg.dynamicSmemBytes = kCoopSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_coop_kernel<DKP>, mq, mk, mv, p, n_chain, flags);
}

template <int DKP>
cudaError_t launch_split_dk(const PrefillArgs& a, void* workspace, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;  // mv: V in 64-column boxes for the prepare kernel's U~
  SplitParams p;
  if (!split_setup(a, workspace, mq, mk, mv, p)) return cudaErrorInvalidValue;
  static PerDeviceOnce attrs;
  const cudaError_t attr_err = attrs.run([] {
    cudaError_t e = cudaFuncSetAttribute(chunk_prepare_kernel<DKP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(chunk_chain_kernel<SplitChain, DKP>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, SplitChain::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(chunk_chain_kernel<SplitChain64, DKP>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, SplitChain64::kSmem);
    return e;
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaError_t e = cudaSuccess;
  if (!p.single) {  // one sequence needs no chunk table
    chunk_plan_kernel<<<1, 256, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  // prepare and chain launch with programmatic stream serialization: each may
  // start its set-up before the kernel before it has finished (the kernels
  // wait for that kernel's results with griddepcontrol.wait)
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (e != cudaSuccess) return e;
  if (p.max_items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3((unsigned)p.max_items);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.dynamicSmemBytes = kPrepSmem;
  e = cudaLaunchKernelEx(&cfg, chunk_prepare_kernel<DKP>, mq, mk, mv, p);
  if (e != cudaSuccess) return e;
  // 64-row chain CTAs once the 32-row ones would need more than one wave
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t narrow = (int64_t)a.num_seqs * a.h_v * (a.d_v / 32);
  const bool wide = a.d_v % 64 == 0 && narrow > sms;
  const int64_t grid = wide ? narrow / 2 : narrow;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3((unsigned)grid);
  if (wide) {
    cfg.blockDim = dim3(SplitChain64::kThreads);
    cfg.dynamicSmemBytes = SplitChain64::kSmem;
    return cudaLaunchKernelEx(&cfg, chunk_chain_kernel<SplitChain64, DKP>, mq, mk, p);
  }
  cfg.blockDim = dim3(SplitChain::kThreads);
  cfg.dynamicSmemBytes = SplitChain::kSmem;
  return cudaLaunchKernelEx(&cfg, chunk_chain_kernel<SplitChain, DKP>, mq, mk, p);
}

}  // namespace

cudaError_t launch_chunked_coop(const PrefillArgs& a, void* workspace, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (!coop_supported(a.num_seqs, a.h_v, a.d_v, sms)) return cudaErrorNotSupported;
  if (a.d_k == kDK) return launch_coop_dk<kDK>(a, workspace, stream, sms);
  if (a.d_k == kDK / 2) return launch_coop_dk<kDK / 2>(a, workspace, stream, sms);
  return cudaErrorNotSupported;
}

cudaError_t launch_chunked_split(const PrefillArgs& a, void* workspace, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  if (a.d_k == kDK) return launch_split_dk<kDK>(a, workspace, stream);
  if (a.d_k == kDK / 2) return launch_split_dk<kDK / 2>(a, workspace, stream);
  return cudaErrorNotSupported;
}

}  // namespace gdn
