// chunk_prefill.cu — chunked (WY/UT) prefill on tcgen05 tensor cores.
//
// Page "Optimizing on-device inference for Apple Silicon", section "Qwen
// creates three distinct workload shapes": besides scanning tokens while
// carrying the state, a prefill can regroup the updates into blocks that
// expose matrix operations and token-level parallelism.  This file is that
// block form, with blocks (chunks) of C = 64 tokens.  Per chunk of n <= 64
// tokens, with S the d_v x d_k state at the chunk start, gamma the in-chunk
// cumulative sum of the log-gates g and Gamma = exp(gamma):
//
//   A_ri = beta_r e^{gamma_r - gamma_i} (k_r . k_i)   (i < r)     strictly lower
//   P_ri =        e^{gamma_r - gamma_i} (q_r . k_i)   (i <= r)
//   T    = (I + A)^{-1}                               (unit lower triangular)
//   W    = T diag(beta Gamma) K,   U~ = T diag(beta) V,   U = U~ - W S^T
//   O    = diag(Gamma) Q S^T + P U
//   S'   = Gamma_n S + U^T diag(e^{gamma_n - gamma}) K
//
// which follows from the row identity u_r = beta_r (v_r - alpha_r S_{r-1} k_r),
// S_r = alpha_r S_{r-1} + u_r k_r^T unrolled over the chunk; the sequential
// recurrence and this form agree up to rounding.  The state and the gates stay
// fp32 ("Keep the recurrent state on-chip"): the state of the CTA's slice
// lives in TMEM as an fp32 accumulator for the whole sequence and only a bf16
// copy of it is staged in shared memory as an MMA operand.
//
// Work split: one CTA per (sequence, value head, slice of 32 value rows); the
// CTA walks its sequence's chunks in order.  Inside the CTA three roles run
// concurrently, handing buffers over through mbarriers:
//   * producer warp: TMA of the chunk's Q, K (two 64-column boxes each) and
//     V slice into a ring of 3 stages;
//   * 8 "prep" warps: everything that does not depend on the state, one chunk
//     ahead of the chain: gates, Q K^T / K K^T masks, the triangular solve,
//     W (written next to Q in the stage) and U~ (into double-buffered TMEM);
//   * 4 "chain" warps: the state-dependent steps of the current chunk.
// Measured on GB300, a dependent K=16 step of tcgen05.mma costs about 60-70
// cycles whatever N (up to 128) and the tensor pipe runs MMAs one at a time,
// so the kernel is organised to issue few, wide MMAs: [-W; Q] share one M=128
// operand, and the state update (on the critical path) is issued before the
// P U product.  The key-only work is recomputed by the 4 slices of a head,
// which keeps slices independent and puts 4x more CTAs on the chain at batch 1.
//
// Tensor-core products (bf16 operands, fp32 TMEM accumulators; an operand
// written [X; Y] is an M=128 operand whose X rows are don't-care):
//   prep:  G  = [Q;K] K^T          M=128 N=64  K=128  (rows 0-63: Q K^T, 64-127: K K^T)
//          W  = (T b Gamma) K      M=64  N=128 K=64
//          U~ = [T b; .] V_s       M=128 N=32  K=64
//   chain: D  = [-W; Q] S_s^T      M=128 N=32  K=128  (rows 0-63: -W S^T, 64-127: Q S^T)
//          S^T += K^T (e^{..} U)   M=128 N=32  K=64   (onto Gamma_n S^T)
//          O2 = [.; P] U           M=128 N=32  K=64
// then U = U~ + D_top and O = Gamma D_bottom + O2.  The triangular solve runs
// in place: 16x16 diagonal blocks by fp32 forward substitution, then 32x32 and
// 64x64 block combinations whose 16-32 wide products use warp-level tf32
// tensor-core instructions (too small for the 64-row tcgen05 shapes, and on
// the prep warps' critical path).
//
// Partial last chunk: rows n..63 get g = 0 and beta = 0, which makes them an
// exact no-op (A, W, U~ and U rows vanish, Gamma stays at Gamma_{n-1}); their
// outputs are not stored.  Inputs must be finite.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "params.h"
#include "per_device.h"
#include "rows.cuh"
#include "tc.cuh"
#include "chunk_common.cuh"

namespace gdn {
namespace {

using namespace chunk;

constexpr int kChainWarps = 4, kPrepWarps = 8;
constexpr int kChainThreads = 32 * kChainWarps;   // 128
constexpr int kPrepThreads = 32 * kPrepWarps;     // 256
constexpr int kThreads = kChainThreads + kPrepThreads + 32;  // + producer warp = 416
constexpr int kProducerWarp = kChainWarps + kPrepWarps;      // warp 12
constexpr uint32_t kBarChain = 1, kBarPrep = 2, kBarGate = 3;  // named barrier ids
constexpr int kStages = 3;

// Shared-memory layout (byte offsets from a 1024-aligned base).
// A stage holds, per 64-wide half kb of d_k, [ -W | Q | K ] (8 KB each, K-major
// SW128 rows of 128 B): Q and K come from TMA, -W is written by the prep warps,
// so [-W; Q] and [Q; K] are both contiguous 128-row MMA operands.  Then the
// V slice [64 tokens][32] (SW64).
constexpr uint32_t kHalfBytes = 3 * 8192;
constexpr uint32_t kStageBytes = 2 * kHalfBytes + 4096;
constexpr uint32_t ST_W = 0, ST_Q = 8192, ST_K = 16384, ST_V = 2 * kHalfBytes;
constexpr uint32_t kTmaBytes = 4 * 8192 + 4096;
constexpr uint32_t OFF_STAGE = 0;
// TB, TA, P0, P1 are contiguous: the 64 rows after TB / TA / P0 are valid
// smem, so each can be the upper half of an M=128 operand whose lower half is
// never read back.
constexpr uint32_t OFF_TB = kStages * kStageBytes;  // T diag(b Gamma) bf16 [r][i], SW128
constexpr uint32_t OFF_TA = OFF_TB + 8192;          // T diag(b) bf16 [r][i], SW128
constexpr uint32_t OFF_PP = OFF_TA + 8192;          // 2 x P bf16 [r][i], SW128
constexpr uint32_t OFF_SS = OFF_PP + 2 * 8192;      // S slice bf16 [j][i], SW64, 8 KB
constexpr uint32_t OFF_UB = OFF_SS + 8192;          // U bf16 [r][i], SW64, 4 KB
constexpr uint32_t OFF_UK = OFF_UB + 4096;          // decayed U bf16 [r][i], SW64, 4 KB
constexpr uint32_t OFF_MF = OFF_UK + 4096;
constexpr uint32_t OFF_YF = OFF_TB;
constexpr uint32_t OFF_GATE = OFF_MF + 64 * kLdM * 4;  // 2 x {gamma, Gamma, beta, decay}[64]
constexpr uint32_t kGateFloats = 4 * 64;
constexpr uint32_t OFF_MISC = OFF_GATE + 2 * kGateFloats * 4;
constexpr uint32_t kSmemUsed = OFF_MISC + 256;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(OFF_TB % 1024 == 0 && OFF_PP % 1024 == 0 && OFF_SS % 512 == 0 &&
                  OFF_UB % 512 == 0 && OFF_UK % 512 == 0 && kStageBytes % 1024 == 0 &&
                  32 * kLdY * 4 <= 8192 && (kLdM * 4) % 16 == 0,
              "swizzled operands need 1024 (SW128) / 512 (SW64) byte alignment");

// TMEM columns (fp32, 128 lanes each).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_G = 0, TM_W = 64, TM_U0 = 192, TM_D0 = 256, TM_O2 = 320, TM_S = 352;

// Instruction descriptors.
constexpr uint32_t ID_G = tc::idesc_bf16_f32(128, 64, false, false);   // [Q;K] K^T
constexpr uint32_t ID_W = tc::idesc_bf16_f32(64, 128, false, true);    // TB K
constexpr uint32_t ID_UT = tc::idesc_bf16_f32(128, 32, false, true);   // [TA;.] V_s
constexpr uint32_t ID_WQ = tc::idesc_bf16_f32(128, 32, false, true);   // [-W;Q] S_s^T
constexpr uint32_t ID_SU = tc::idesc_bf16_f32(128, 32, true, true);    // K^T (decay U)
constexpr uint32_t ID_PU = tc::idesc_bf16_f32(128, 32, false, true);   // [.;P] U

struct ChunkParams {
  const float* g;
  const float* beta;
  const float* state_in;
  float* state_out;
  __nv_bfloat16* o;
  const int32_t* cu;
  int32_t num_seqs;
  int64_t total_tokens;
  int32_t h_k, h_v, d_v;
  float scale;
  int32_t min_len;
  int* err;
};

// mbarriers in the MISC area
struct Bars {
  uint64_t tma_full[kStages];    // producer -> consumers (transaction bytes)
  uint64_t stage_free[kStages];  // prep + chain -> producer (2 arrivals)
  uint64_t prep_ready[2];        // prep -> chain: -W, P, U~, gates of a chunk ready
  uint64_t chain_free[2];        // chain -> prep: that buffer set consumed
  uint64_t mma_prep;             // prep MMA completion
  uint64_t mma_chain;            // chain MMA completion ([-W;Q] S^T, then the S update)
  uint64_t mma_out;              // chain MMA completion (P U)
  uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 256, "misc area");

__global__ void __launch_bounds__(kThreads, 1)
    chunk_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const ChunkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ns = p.d_v / kDVS;
  const int s = blockIdx.x % ns;
  const int h = (blockIdx.x / ns) % p.h_v;
  const int n = blockIdx.x / (ns * p.h_v);
  const int hk = h / (p.h_v / p.h_k);

  const int64_t t_beg = p.cu[n], t_end = p.cu[n + 1];
  const bool bad = t_beg < 0 || t_end < t_beg || t_end > p.total_tokens ||
                   (n == 0 && t_beg != 0) || (n == p.num_seqs - 1 && t_end != p.total_tokens);
  if (bad) {
    if (tid == 0 && h == 0 && s == 0) raise_error(p.err, kErrBadCuSeqlens);
    return;
  }
  const int64_t L = t_end - t_beg;
  if (L < p.min_len) return;  // the token scan owns this sequence

  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_MISC);
  float* MF = reinterpret_cast<float*>(smem + OFF_MF);
  float* YF = reinterpret_cast<float*>(smem + OFF_YF);
  const int64_t srow0 = ((int64_t)n * p.h_v + h) * p.d_v + s * kDVS;  // first state row
  const int nchunks = (int)((L + kC - 1) / kC);

  if (warp == 0) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&bars->tma_full[i], 1);
      tc::mbar_init(&bars->stage_free[i], 2);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars->prep_ready[i], 1);
      tc::mbar_init(&bars->chain_free[i], 1);
    }
    tc::mbar_init(&bars->mma_prep, 1);
    tc::mbar_init(&bars->mma_chain, 1);
    tc::mbar_init(&bars->mma_out, 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  bool ok = true;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      tc::prefetch_tmap(&tm_v);
      for (int c = 0; c < nchunks; ++c) {
        const int st = c % kStages;
        if (c >= kStages && !tc::mbar_wait(&bars->stage_free[st], ((c / kStages) - 1) & 1)) {
          raise_error(p.err, kErrDeviceTimeout);
          break;
        }
        uint8_t* dst = smem + OFF_STAGE + st * kStageBytes;
        const int32_t y = static_cast<int32_t>(t_beg + (int64_t)c * kC);
        uint64_t* fb = &bars->tma_full[st];
        tc::mbar_arrive_expect_tx(fb, kTmaBytes);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          tc::tma_load_2d(dst + kb * kHalfBytes + ST_Q, &tm_q, hk * kDK + 64 * kb, y, fb);
          tc::tma_load_2d(dst + kb * kHalfBytes + ST_K, &tm_k, hk * kDK + 64 * kb, y, fb);
        }
        tc::tma_load_2d(dst + ST_V, &tm_v, h * p.d_v + s * kDVS, y, fb);
      }
    }
  } else if (warp >= kChainWarps) {
    // ------------------------------------------------------------ prep
    const int pt = tid - kChainThreads;  // 0..255
    const int pw = pt >> 5;              // prep warp 0..7
    const int sp = pw & 3;               // TMEM subpartition of this warp
    const bool leader = pt == 0;         // arrives on the hand-off barriers
    const bool issuer = pt == 64;        // issues the prep MMAs (not a gate warp)
    uint32_t mma_phase = 0;
    // gates of the next chunk are loaded one iteration ahead (global latency)
    auto load_gates = [&](int c, float& gv, float& bv) {
      const int64_t tt = t_beg + (int64_t)c * kC + pt;
      gv = 0.f;
      bv = 0.f;
      if (c < nchunks && pt < kC && tt < t_end) {
        gv = p.g[tt * p.h_v + h];
        bv = p.beta[tt * p.h_v + h];
      }
    };
    float g_next, b_next;
    load_gates(0, g_next, b_next);
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1, st = c % kStages;
      const uint32_t stg = sbase + OFF_STAGE + st * kStageBytes;
      uint8_t* stg_ptr = smem + OFF_STAGE + st * kStageBytes;
      float* gate = reinterpret_cast<float*>(smem + OFF_GATE) + b * kGateFloats;
      float *gam = gate, *Gam = gate + 64, *bet = gate + 128, *dec = gate + 192;

      float gr = g_next, br = b_next;
      load_gates(c + 1, g_next, b_next);
      // buffers b were last used by the chain for chunk c-2
      if (c >= 2) {
        ok = group_wait(&bars->chain_free[b], ((c >> 1) - 1) & 1, kBarPrep, kPrepThreads);
        if (!ok) break;
      }
      ok = group_wait(&bars->tma_full[st], (c / kStages) & 1, kBarPrep, kPrepThreads);
      if (!ok) break;
      if (issuer) {  // G = [Q;K] K^T: rows 0-63 Q K^T, rows 64-127 K K^T
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ko = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          tc::mma_bf16(tmem + TM_G, tc::smem_desc(stg + ko + ST_Q, 16, 1024, tc::kLayoutSw128),
                       tc::smem_desc(stg + ko + ST_K, 16, 1024, tc::kLayoutSw128), ID_G, kk > 0);
        }
        tc::mma_commit(&bars->mma_prep);
      }
      // gates: inclusive scan of g over the chunk (prep warps 0 and 1)
      if (pt < 64) {
        float x = gr;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(kFullMask, x, off);
          if (lane >= off) x += y;
        }
        if (pt == 31) MF[0] = x;  // scratch is free until the masks
        gr = x;
        tc::named_sync(kBarGate, 64);
        if (pw == 1) gr += MF[0];
        gam[pt] = gr;
        Gam[pt] = tc::fast_exp(gr);
        bet[pt] = br;
        tc::named_sync(kBarGate, 64);
        dec[pt] = tc::fast_exp(gam[kC - 1] - gr);
      }

      // masks: P (bf16 operand) from rows 0-63, A (fp32, solve input) from rows 64-127
      ok = group_wait(&bars->mma_prep, mma_phase & 1, kBarPrep, kPrepThreads);
      ++mma_phase;
      if (!ok) break;
      {
        const int half = pw >> 2;  // column half
        float a[32];
        tc::tmem_ld32(tmem + lane_base + TM_G + 32 * half, a);
        const int i0 = 32 * half;
        if (sp < 2) {
          const int r = 32 * sp + lane;
          const float g_r = gam[r];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 gi = *reinterpret_cast<const float4*>(gam + i0 + 4 * e4);
            const float gv[4] = {gi.x, gi.y, gi.z, gi.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int e = 4 * e4 + q, i = i0 + e;
              a[e] = (i <= r) ? tc::fast_exp(g_r - gv[q]) * a[e] : 0.f;
            }
          }
          uint8_t* pp = smem + OFF_PP + b * 8192;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8)
            st_chunk<3>(pp, r * 128 + (4 * half + c8) * 16, a + 8 * c8);
        } else {
          const int r = 32 * (sp - 2) + lane;
          const float g_r = gam[r], b_r = bet[r];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 gi = *reinterpret_cast<const float4*>(gam + i0 + 4 * e4);
            const float gv[4] = {gi.x, gi.y, gi.z, gi.w};
            float o4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = i0 + 4 * e4 + q;
              o4[q] = (i < r) ? b_r * tc::fast_exp(g_r - gv[q]) * a[4 * e4 + q] : 0.f;
            }
            *reinterpret_cast<float4*>(MF + r * kLdM + i0 + 4 * e4) =
                make_float4(o4[0], o4[1], o4[2], o4[3]);
          }
        }
      }
      group_sync(kBarPrep, kPrepThreads);

      unit_lower_inverse<kPrepThreads>(MF, YF, pt, lane, kBarPrep);

      {  // operands T diag(b Gamma) and T diag(b): thread = (row r, 16-column quarter)
        const int r = pt >> 2, q = pt & 3;
#pragma unroll
        for (int c8 = 0; c8 < 2; ++c8) {
          const int i0 = 16 * q + 8 * c8;
          const float4 m0 = *reinterpret_cast<const float4*>(MF + r * kLdM + i0);
          const float4 m1 = *reinterpret_cast<const float4*>(MF + r * kLdM + i0 + 4);
          const float4 b0 = *reinterpret_cast<const float4*>(bet + i0);
          const float4 b1 = *reinterpret_cast<const float4*>(bet + i0 + 4);
          const float4 G0 = *reinterpret_cast<const float4*>(Gam + i0);
          const float4 G1 = *reinterpret_cast<const float4*>(Gam + i0 + 4);
          float xa[8] = {m0.x * b0.x, m0.y * b0.y, m0.z * b0.z, m0.w * b0.w,
                         m1.x * b1.x, m1.y * b1.y, m1.z * b1.z, m1.w * b1.w};
          float xb[8] = {xa[0] * G0.x, xa[1] * G0.y, xa[2] * G0.z, xa[3] * G0.w,
                         xa[4] * G1.x, xa[5] * G1.y, xa[6] * G1.z, xa[7] * G1.w};
          st_chunk<3>(smem + OFF_TA, r * 128 + (2 * q + c8) * 16, xa);
          st_chunk<3>(smem + OFF_TB, r * 128 + (2 * q + c8) * 16, xb);
        }
      }
      tc::fence_proxy_async();
      group_sync(kBarPrep, kPrepThreads);

      // W = T b Gamma K and U~ = T b V on the tensor cores
      if (issuer) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tmem + TM_W, tc::smem_desc(sbase + OFF_TB + kk * 32, 16, 1024, tc::kLayoutSw128),
                       tc::smem_desc(stg + ST_K + kk * 2048, kHalfBytes, 1024, tc::kLayoutSw128),
                       ID_W, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tmem + TM_U0 + 32 * b,
                       tc::smem_desc(sbase + OFF_TA + kk * 32, 16, 1024, tc::kLayoutSw128),
                       tc::smem_desc(stg + ST_V + kk * 1024, 4096, 512, tc::kLayoutSw64), ID_UT,
                       kk > 0);
        tc::mma_commit(&bars->mma_prep);
      }
      ok = group_wait(&bars->mma_prep, mma_phase & 1, kBarPrep, kPrepThreads);
      ++mma_phase;
      if (!ok) break;
      {  // -W into the stage's W slots (K-major); M=64 accumulator: row 16 sp + lane, lane < 16
        const int half = pw >> 2, r = 16 * sp + lane;
        float w[32];
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          tc::tmem_ld32(tmem + lane_base + TM_W + 64 * half + 32 * q2, w);
          if (lane < 16) {
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = -w[e];
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
              st_chunk<3>(stg_ptr + half * kHalfBytes + ST_W, r * 128 + (4 * q2 + c8) * 16,
                          w + 8 * c8);
          }
        }
      }
      tc::fence_proxy_async();
      group_sync(kBarPrep, kPrepThreads);
      if (leader) {
        tc::mbar_arrive(&bars->prep_ready[b]);
        tc::mbar_arrive(&bars->stage_free[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ chain
    const bool leader = tid == 0;
    uint32_t chain_phase = 0, out_phase = 0;
    const uint32_t ss = sbase + OFF_SS;
    {  // initial state: thread j holds column j of the slice (rows i = 0..31)
      float sc[32];
#pragma unroll
      for (int i = 0; i < kDVS; ++i)
        sc[i] = p.state_in ? p.state_in[(srow0 + i) * kDK + tid] : 0.f;
      if (nchunks == 0) {
#pragma unroll
        for (int i = 0; i < kDVS; ++i) p.state_out[(srow0 + i) * kDK + tid] = sc[i];
      } else {
        tc::tmem_st32(tmem + lane_base + TM_S, sc);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) st_chunk<2>(smem + OFF_SS, tid * 64 + c4 * 16, sc + 8 * c4);
      }
      tc::fence_proxy_async();
      group_sync(kBarChain, kChainThreads);
    }
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1, st = c % kStages;
      const uint32_t stg = sbase + OFF_STAGE + st * kStageBytes;
      const float* gate = reinterpret_cast<const float*>(smem + OFF_GATE) + b * kGateFloats;
      const int64_t t0 = t_beg + (int64_t)c * kC;
      const int nv = (int)((L - (int64_t)c * kC) < kC ? (L - (int64_t)c * kC) : kC);

      ok = group_wait(&bars->prep_ready[b], (c >> 1) & 1, kBarChain, kChainThreads);
      if (!ok) break;
      if (leader) {  // D = [-W; Q] S_s^T: rows 0-63 -W S^T, rows 64-127 Q S^T
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ko = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          tc::mma_bf16(tmem + TM_D0 + 32 * b,
                       tc::smem_desc(stg + ko + ST_W, 16, 1024, tc::kLayoutSw128),
                       tc::smem_desc(ss + kk * 1024, 4096, 512, tc::kLayoutSw64), ID_WQ, kk > 0);
        }
        tc::mma_commit(&bars->mma_chain);
      }
      // gates this thread needs, read before the buffer set is released
      const int rl = 32 * (warp & 1) + lane;  // accumulator row of this thread within its half
      const float Gam_n = gate[64 + kC - 1];
      const float dec_r = gate[192 + rl];
      const float Gam_r = gate[64 + rl];
      {  // S <- Gamma_n S (the update MMA accumulates onto it)
        float sc[32];
        tc::tmem_ld32(tmem + lane_base + TM_S, sc);
#pragma unroll
        for (int i = 0; i < 32; ++i) sc[i] *= Gam_n;
        tc::tmem_st32(tmem + lane_base + TM_S, sc);
      }
      ok = group_wait(&bars->mma_chain, chain_phase & 1, kBarChain, kChainThreads);
      ++chain_phase;
      if (!ok) break;
      if (warp < 2) {  // U = U~ - W S^T for rows r = lanes 0-63
        float u[32], d[32];
        tc::tmem_ld32(tmem + lane_base + TM_U0 + 32 * b, u);
        tc::tmem_ld32(tmem + lane_base + TM_D0 + 32 * b, d);
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] += d[i];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) st_chunk<2>(smem + OFF_UB, rl * 64 + c4 * 16, u + 8 * c4);
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] *= dec_r;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) st_chunk<2>(smem + OFF_UK, rl * 64 + c4 * 16, u + 8 * c4);
      }
      tc::fence_proxy_async();
      group_sync(kBarChain, kChainThreads);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // S^T += K^T (decayed U): the next chunk waits on this
          tc::mma_bf16(tmem + TM_S, tc::smem_desc(stg + ST_K + kk * 2048, kHalfBytes, 1024, tc::kLayoutSw128),
                       tc::smem_desc(sbase + OFF_UK + kk * 1024, 4096, 512, tc::kLayoutSw64), ID_SU,
                       1);
        tc::mma_commit(&bars->mma_chain);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // O2 = P U in rows 64-127
          tc::mma_bf16(tmem + TM_O2,
                       tc::smem_desc(sbase + OFF_PP + b * 8192 - 8192 + kk * 32, 16, 1024,
                                     tc::kLayoutSw128),
                       tc::smem_desc(sbase + OFF_UB + kk * 1024, 4096, 512, tc::kLayoutSw64), ID_PU,
                       kk > 0);
        tc::mma_commit(&bars->mma_out);
      }
      ok = group_wait(&bars->mma_chain, chain_phase & 1, kBarChain, kChainThreads);
      ++chain_phase;
      if (!ok) break;
      if (leader) tc::mbar_arrive(&bars->stage_free[st]);  // K, Q, -W of the stage consumed
      {
        float sc[32];
        tc::tmem_ld32(tmem + lane_base + TM_S, sc);
        if (c == nchunks - 1) {
#pragma unroll
          for (int i = 0; i < kDVS; ++i) p.state_out[(srow0 + i) * kDK + tid] = sc[i];
        } else {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            st_chunk<2>(smem + OFF_SS, tid * 64 + c4 * 16, sc + 8 * c4);
        }
      }
      tc::fence_proxy_async();
      group_sync(kBarChain, kChainThreads);
      ok = group_wait(&bars->mma_out, out_phase & 1, kBarChain, kChainThreads);
      ++out_phase;
      if (!ok) break;
      if (leader) tc::mbar_arrive(&bars->chain_free[b]);  // P, U~, gates of buffer b consumed
      if (warp >= 2) {  // O = Gamma Q S^T + P U for rows r = lanes 64-127
        float o1[32], o2[32];
        tc::tmem_ld32(tmem + lane_base + TM_D0 + 32 * b, o1);
        tc::tmem_ld32(tmem + lane_base + TM_O2, o2);
        if (rl < nv) {
#pragma unroll
          for (int i = 0; i < 32; ++i) o1[i] = p.scale * fmaf(Gam_r, o1[i], o2[i]);
          uint4* dst = reinterpret_cast<uint4*>(p.o + ((t0 + rl) * p.h_v + h) * (int64_t)p.d_v +
                                                s * kDVS);
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
    }
  }
  if (!ok && (tid == 0 || tid == kChainThreads)) raise_error(p.err, kErrDeviceTimeout);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

bool encode_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Shapes the chunked evaluation covers: bf16 operands, d_v a multiple of 32,
// d_k 128 or 64 (the two-kernel and cooperative forms read Q and K as 3-D
// tiles whose columns past d_k arrive as zeros, so d_k = 64 runs as 128 with
// zero padding); the fused kernel needs d_k = 128.
bool chunked_supports(int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, int dtype) {
  return dtype == kBF16 && (d_k == kDK || d_k == kDK / 2) && d_v >= kDVS && d_v % kDVS == 0 &&
         h_k > 0 && h_v % h_k == 0;
}

bool fused_supports(int32_t h_k, int32_t h_v, int32_t d_k, int32_t d_v, int dtype) {
  return chunked_supports(h_k, h_v, d_k, d_v, dtype) && d_k == kDK;
}

size_t chunked_workspace_bytes(int32_t, int64_t, int32_t, int32_t, int32_t, int32_t) { return 0; }

cudaError_t launch_chunked(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  if (!fused_supports(a.h_k, a.h_v, a.d_k, a.d_v, a.dtype)) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  const uint64_t rows = a.total_tokens > 0 ? (uint64_t)a.total_tokens : 1;
  // With no tokens every sequence is empty and no TMA is issued; the maps still
  // need a valid (non-null) address, so point them at the state buffer.
  const void* qp = a.total_tokens > 0 ? a.q : a.state_out;
  const void* kp = a.total_tokens > 0 ? a.k : a.state_out;
  const void* vp = a.total_tokens > 0 ? a.v : a.state_out;
  if (!encode_2d(&mq, qp, (uint64_t)a.h_k * a.d_k, rows, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&mk, kp, (uint64_t)a.h_k * a.d_k, rows, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&mv, vp, (uint64_t)a.h_v * a.d_v, rows, kDVS, kC, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  static PerDeviceOnce attrs;
  const cudaError_t attr_err = attrs.run([] {
    return cudaFuncSetAttribute(chunk_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  ChunkParams p;
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
  p.err = a.err;
  const int64_t grid = (int64_t)a.num_seqs * a.h_v * (a.d_v / kDVS);
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  chunk_prefill_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace gdn
