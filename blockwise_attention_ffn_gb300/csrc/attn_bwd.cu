// attn_bwd.cu -- attention backward with the probabilities rebuilt tile by
// tile from Q, K and the saved log-sum-exp (nothing of size s x s is stored).
//
// Gradient rules ("Training memory: model states, activations and
// checkpointing", section 2, the softmax and product rows): with
// S = Q K^T / sqrt(d), P = softmax(S) = exp(S - LSE), O = P V,
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D) with D = rowsum(dO * O)
//   (= rowsum(P * dP)),  dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d).
// The rebuild is the backward-pass remat of every key/value block step that
// "Blockwise Parallel Transformer for Long Context Large Models", section
// 3.4, "Implementation Details (Figure 3)" describes.
//
// Two kernels, neither with atomics:
//  * dK/dV: one CTA per 128-row key/value tile j of one key/value head; it
//    loops over the G query heads of the group and their query tiles i >= j
//    (causal), accumulating dK and dV in TMEM.  It works in 64-query
//    sub-tiles with double-buffered S^T and dP^T, taken alternately by two
//    groups of compute warps with their own MMA-issuing warps.  K and V are
//    TMEM operands for head dims 64 and 80; for 96 to 128, whose
//    accumulators leave no TMEM for them, they stay in shared memory.
//  * dQ: one CTA per 128-row query tile i of one query head; it loops over
//    the key/value tiles j <= i in 64-key sub-tiles the same way,
//    accumulating dQ in TMEM, and writes it once.
// Both rebuild S and dP (the dQ kernel for its own tile order), so a pair of
// tiles costs 7 tensor-core products instead of 5; in exchange no partial dQ
// tile is ever reduced through L2 (in a one-kernel design that traffic is
// tens of GB per step at s = 32K and bounds the whole backward pass).
#include <math.h>
#include <string.h>

#include <algorithm>

#include "../../include/bpt.h"
#include "attn_common.cuh"
#include "internal.h"

namespace bpt {

namespace {

struct AttnBwdParams {
  CUtensorMap map_qkv;  // 3-D {ld_qkv, s, b}, box {CW, 128, 1}
  CUtensorMap map_do;   // 3-D {ld_do, s, b}, box {CW, 128, 1}
  CUtensorMap map_aux;  // 2-D {8, b*H*s_pad} bf16, box {8, 128}, no swizzle
  int s, s_pad, H, Hkv, G, causal, b;
  int q_col, k_col, v_col, do_col;
  const float* lse;     // [b, H_total, s_pad] at head offset lse_head0
  const float* Dsum;    // [b, H, s_pad]
  const float* nl2;     // [b, H, s_pad]: -LSE * log2(e)
  const __nv_bfloat16* qkv;  // the packed projection (rows copied into TMEM directly)
  long long ld_qkv;
  const __nv_bfloat16* dout;
  long long ld_do;
  int H_total, lse_head0;
  __nv_bfloat16* dqkv;
  long long ld_dqkv;
  int dq_col, dk_col, dv_col;
  float scale, scale_log2;
  int one_issuer;  // fixed-order mode: warp 1 issues both groups' products
  unsigned int* err;
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}


// ===========================================================================
// dK / dV
// ===========================================================================
// A 128 x 128 product with both operands in shared memory takes the whole
// shared-memory bandwidth of the SM, and the compute warps' own shared-memory
// loads then wait behind it.  So P^T is written over S^T and dS^T over dP^T
// in TMEM (bf16 pairs), the A operands of dV = P^T dO and dK = dS^T Q, and
// the compute warps touch no shared memory at all.  For head dims 64 and 80
// K and V are also copied into TMEM once per CTA as the A operands of
// S^T = K Q^T and dP^T = V dO^T, so no product has more than one
// shared-memory operand.  For 96 to 128, dV and dK take 2D TMEM columns and
// the double-buffered S^T and dP^T the other 256, so K and V stay in shared
// memory (loaded once per CTA) and those two products read both operands
// from there.
// The per-query-column terms of the softmax gradient (-LSE and -D) enter
// through the products too: one more contraction step multiplies a 16-column
// chunk appended to K (1, 1, 0, ...) or V (0, 0, 1, 1, 0, ...) with the query
// row (hi(-LSE*sqrt(d)), lo(..), hi(-D), lo(-D), 0, ...), so S^T comes out
// offset by -LSE*sqrt(d) and dP^T by -D: the compute warps read no
// per-column values from shared memory.  The row's 8 nonzero-capable columns
// arrive with the Q/dO stage (16 bytes per query, unswizzled: exactly the
// K-major core-matrix layout); the descriptor points its upper 8 columns at
// one shared 2 KB of zeros.  K's and V's own extra chunks sit in TMEM beside
// them, or (head dims above 80) in shared memory in the same unswizzled
// layout, written by the compute warps.
// TMEM: dV [256, 256+D), dK [256+D, 256+2D), and for head dims 64 and 80
// K' [256+2D, 256+2.5D+8), V' [.., 256+3D+16).  Shared memory: (above 80) K,
// V and their extra chunks, then QS stages of (Q, dO, the 128 query rows'
// 16-byte extra rows), then the zeros.
template <int D>
struct DkdvTmCfg {
  using T = TileGeom<D>;
  // K and V are TMEM operands where their columns fit beside dV and dK (head
  // dims up to 80); above that they stay in shared memory, with their extra
  // chunks
  static constexpr bool KV_TMEM = D <= 80;
  static constexpr int AUX = 128 * 16;                 // 128 rows x 8 bf16
  static constexpr int KV = KV_TMEM ? 0 : 2 * T::TILE + 2 * AUX;  // K, V, K extra, V extra
  static constexpr int STAGE = 2 * T::TILE + AUX;      // Q, dO, extra rows
  static constexpr int ZERO = 2048;                    // the upper 8 columns
  static constexpr int QS_FIT = (232448 - KV - ZERO - 1024 - 256) / STAGE;
  static constexpr int QS = QS_FIT > 4 ? 4 : QS_FIT;
  static constexpr int SMEM = KV + QS * STAGE + ZERO + 1024 + 256;
  static constexpr uint32_t COL_DV = 256, COL_DK = 256 + D, COL_K = 256 + 2 * D, COL_V = 256 + 2 * D + D / 2 + 8;
};

// A step covers 64 queries: sub-tile u is the half u % 2 of
// stage u / 2, and its S^T and dP^T go to buffer b = u % 2 (64 columns each:
// the same 256 columns as one 128-query buffer of each).  Compute warps 2..5
// (group 0) take the even sub-tiles, 6..9 (group 1) the odd ones, each warp
// its lane quarter's 32 key rows by all 64 query columns, so one group's
// exponentials overlap the other group's products instead of alternating
// with them.  Warp 1 issues group 0's products, warp 10 group 1's, in the
// order S(u), dP(u), dV(u) (after P^T(u)), S(u+2), dK(u) (after dS^T(u)),
// dP(u+2): every product that overwrites a buffer comes after its reader
// from the same thread.  Both issuers add into dV and dK, which the compute
// warps zero first; a stage is released once both issuers' products on it
// are done.
// TMEM: S^T [0,64) [64,128), dP^T [128,192) [192,256), then as above.
template <int D>
__global__ void __launch_bounds__(352, 1) attn_dkdv_hs_kernel(const __grid_constant__ AttnBwdParams p) {
  using T = TileGeom<D>;
  using C = DkdvTmCfg<D>;
  constexpr int QS = C::QS;
  constexpr int STAGE = C::STAGE;
  static_assert(C::COL_DK + D <= 512, "TMEM columns");
  static_assert(!C::KV_TMEM || C::COL_V + D / 2 + 8 <= 512, "TMEM columns");
  static_assert(QS >= 2, "Q/dO ring");
  constexpr uint32_t ID_S = idesc_bf16(128, 64, false, false);
  constexpr uint32_t ID_KV = idesc_bf16(128, D, false, true);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKV = smem;                  // K, V, their extra chunks (head dims above 80)
  uint8_t* sStage = smem + C::KV;
  uint8_t* sZero = sStage + QS * STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sZero + C::ZERO);
  uint64_t* kv_ready = bars;            // K', V' in place, dV, dK zeroed (8 compute warps)
  uint64_t* qdo_full = bars + 1;        // [QS]
  uint64_t* qdo_empty = qdo_full + QS;  // [QS], both issuers
  uint64_t* s_full = qdo_empty + QS;    // [2] S^T(u) in buffer u % 2
  uint64_t* dp_full = s_full + 2;       // [2]
  uint64_t* p_full = dp_full + 2;       // [2] P^T(u) written (4 warps of the group)
  uint64_t* ds_full = p_full + 2;       // [2] dS^T(u) written (4 warps)
  uint64_t* all_done = ds_full + 2;     // both issuers' last products done
  uint64_t* drain = all_done + 1;       // [2], one per issuer
  uint64_t* kv_full = drain + 2;        // K, V tiles landed (shared-memory variant)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(kv_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  // head-major, heaviest key tiles (smallest j) of a KV head first, so the
  // CTAs in flight share that head's Q/dO stream in L2
  const int nq_total = (p.s + 127) / 128;
  const int pair = blockIdx.x / nq_total;
  const int j = blockIdx.x % nq_total;
  const int g = pair % p.Hkv;
  const int bi = pair / p.Hkv;
  const int i0 = p.causal ? j : 0;
  const int n_i = nq_total - i0;
  const int T_iter = p.G * n_i;  // stages
  const int U = 2 * T_iter;      // sub-tiles

  if (threadIdx.x == 0) {
    mbar_init(kv_ready, 8);
    for (int i = 0; i < QS; ++i) {
      mbar_init(&qdo_full[i], 1);
      mbar_init(&qdo_empty[i], 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&dp_full[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&ds_full[b], 4);
      mbar_init(&drain[b], 1);
    }
    mbar_init(all_done, 2);
    mbar_init(kv_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&p.map_qkv);
    tma_prefetch(&p.map_do);
    tma_prefetch(&p.map_aux);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  if (threadIdx.x < C::ZERO / 16) {
    reinterpret_cast<uint4*>(sZero)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem;          // + 64 b
  const uint32_t tdP = tmem + 128;   // + 64 b
  const uint32_t tdV = tmem + C::COL_DV;
  const uint32_t tdK = tmem + C::COL_DK;
  const uint32_t tKA = tmem + C::COL_K;
  const uint32_t tVA = tmem + C::COL_V;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      if constexpr (!C::KV_TMEM) {
        mbar_expect_tx(kv_full, 2 * T::TILE);
#pragma unroll
        for (int c = 0; c < T::NCH; ++c) {
          tma_load_3d(sKV + c * T::CHUNK, &p.map_qkv, kv_full, p.k_col + g * D + c * T::CW, j * 128, bi);
          tma_load_3d(sKV + T::TILE + c * T::CHUNK, &p.map_qkv, kv_full, p.v_col + g * D + c * T::CW, j * 128,
                      bi);
        }
      }
      int issued = 0;
      for (int t = 0; t < T_iter; ++t) {
        const int st = t % QS;
        if (t >= QS && !bounded_wait(&qdo_empty[st], ((t / QS) & 1) ^ 1, abort_flag, 631, p.err)) break;
        const int hn = g * p.G + t / n_i;
        const int i = i0 + t % n_i;
        uint8_t* sQ = sStage + st * STAGE;
        uint8_t* sdO = sQ + T::TILE;
        mbar_expect_tx(&qdo_full[st], STAGE);
#pragma unroll
        for (int c = 0; c < T::NCH; ++c) {
          tma_load_3d(sQ + c * T::CHUNK, &p.map_qkv, &qdo_full[st], p.q_col + hn * D + c * T::CW, i * 128, bi);
          tma_load_3d(sdO + c * T::CHUNK, &p.map_do, &qdo_full[st], p.do_col + hn * D + c * T::CW, i * 128, bi);
        }
        const int row = (bi * p.H + hn) * p.s_pad + i * 128;
        tma_load_2d(sQ + 2 * T::TILE, &p.map_aux, &qdo_full[st], 0, row);
        issued = t + 1;
      }
      if (*abort_flag) {
        if constexpr (!C::KV_TMEM) drain_wait(kv_full, 0);
        for (int t = (issued > QS ? issued - QS : 0); t < issued; ++t)
          drain_wait(&qdo_full[t % QS], (t / QS) & 1);
      }
    }
  } else if (warp == 1 || warp == 10) {
    // the whole warp runs the issue loop, one elected lane issues.  One
    // issuer (fixed-order mode): warp 1 issues every sub-tile's products
    // in sub-tile order, so dV and dK take their products in a fixed order
    if (!(p.one_issuer && warp == 10)) {
      // ------------------------------------------------ MMA issuers
      const int b0 = warp == 1 ? 0 : 1;  // this issuer's first sub-tile
      const int ustep = p.one_issuer ? 1 : 2;
      const uint32_t uZero = smem_u32(sZero);
      // the 64 query rows of sub-tile half b start 64 b rows into every
      // chunk of the stage's tiles (whole swizzle atoms), and 64 b rows into
      // its extra rows; sub-tile u uses buffer b = u % 2
      auto stage_u = [&](int u) { return smem_u32(sStage + ((u >> 1) % QS) * STAGE); };
      // K, V and their extra chunks in shared memory (head dims above 80):
      // the extra chunk is 128 rows of 16 bytes, K-major core matrices
      // without swizzle, its upper 8 columns the zeros
      const uint32_t uK = smem_u32(sKV), uV = uK + T::TILE;
      const uint32_t uKx = uK + 2 * T::TILE, uVx = uKx + C::AUX;
      auto issue_s = [&](int u) {
        const int b = u & 1;
        const uint32_t tSb = tS + 64 * b;
        const uint32_t uQ = stage_u(u) + 64 * T::SWB * b;
        const uint32_t uA = stage_u(u) + 2 * T::TILE + 64 * 16 * b;
        if constexpr (C::KV_TMEM) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) umma_bf16_tmem_a_w(tSb, tKA + kk * 8, T::kmajor(uQ, kk), ID_S, kk > 0);
          umma_bf16_tmem_a_w(tSb, tKA + D / 2, sdesc(uA, uZero - uA, 128, 0u), ID_S, 1);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) umma_bf16_w(tSb, T::kmajor(uK, kk), T::kmajor(uQ, kk), ID_S, kk > 0);
          umma_bf16_w(tSb, sdesc(uKx, uZero - uKx, 128, 0u), sdesc(uA, uZero - uA, 128, 0u), ID_S, 1);
        }
        umma_commit_w(&s_full[b]);
      };
      auto issue_dp = [&](int u) {
        const int b = u & 1;
        const uint32_t tdPb = tdP + 64 * b;
        const uint32_t udO = stage_u(u) + T::TILE + 64 * T::SWB * b;
        const uint32_t uA = stage_u(u) + 2 * T::TILE + 64 * 16 * b;
        if constexpr (C::KV_TMEM) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_bf16_tmem_a_w(tdPb, tVA + kk * 8, T::kmajor(udO, kk), ID_S, kk > 0);
          umma_bf16_tmem_a_w(tdPb, tVA + D / 2, sdesc(uA, uZero - uA, 128, 0u), ID_S, 1);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) umma_bf16_w(tdPb, T::kmajor(uV, kk), T::kmajor(udO, kk), ID_S, kk > 0);
          umma_bf16_w(tdPb, sdesc(uVx, uZero - uVx, 128, 0u), sdesc(uA, uZero - uA, 128, 0u), ID_S, 1);
        }
        umma_commit_w(&dp_full[b]);
      };
      auto wait_stage = [&](int u) {
        const int t = u >> 1;
        return bounded_wait_w(&qdo_full[t % QS], (t / QS) & 1, abort_flag, 641, p.err);
      };
      bool ok = bounded_wait_w(kv_ready, 0, abort_flag, 642, p.err) &&
                (C::KV_TMEM || bounded_wait_w(kv_full, 0, abort_flag, 646, p.err)) && wait_stage(b0);
      if (ok) {
        tc_fence_after();
        // sub-tiles 0 and 1 share stage 0 (U is even)
        for (int u = b0; u < 2; u += ustep) {
          issue_s(u);
          issue_dp(u);
        }
      }
      for (int u = b0; ok && u < U; u += ustep) {
        const int b = u & 1;
        const uint32_t tSb = tS + 64 * b, tdPb = tdP + 64 * b;
        const int st = (u >> 1) % QS;
        const uint32_t uQ = stage_u(u);
        const uint32_t udO = uQ + T::TILE;
        const bool more = u + 2 < U;
        // dV += P^T(u) dO(u): the P^T pairs sit over the first 32 columns of
        // buffer b; dO rows 64b.. are K blocks 4b..4b+3 of the stage's tile
        if (!bounded_wait_w(&p_full[b], (u >> 1) & 1, abort_flag, 643, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a_w(tdV, tSb + kk * 8, T::mnmajor(udO, 4 * b + kk), ID_KV, 1);
        if (more) {
          // S(u+2) overwrites P^T(u), after dV(u) in issue order
          if (!wait_stage(u + 2)) { ok = false; break; }
          tc_fence_after();
          issue_s(u + 2);
        }
        // dK += dS^T(u) Q(u)
        if (!bounded_wait_w(&ds_full[b], (u >> 1) & 1, abort_flag, 644, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a_w(tdK, tdPb + kk * 8, T::mnmajor(uQ, 4 * b + kk), ID_KV, 1);
        umma_commit_w(&qdo_empty[st]);
        // dP(u+2) overwrites dS^T(u), after dK(u) in issue order
        if (more) issue_dp(u + 2);
      }
      if (ok) {
        // all_done counts two commits: one per issuer, or both from one
        umma_commit_w(all_done);
        if (p.one_issuer) umma_commit_w(all_done);
      }
      if (!ok) {
        umma_commit_w(&drain[b0]);
        drain_wait(&drain[b0], 0);
      }
    }
  } else {
    // ------------------------------------------------ compute (warps 2..9;
    // warp 10 in the one-issuer mode falls through to the final barrier)
    const int quarter = warp & 3;
    const int b = (warp - 2) >> 2;  // group = buffer = sub-tile parity
    const int r = quarter * 32 + lane;
    const int kvp = j * 128 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    if constexpr (!C::KV_TMEM) {
      // the extra chunk of this thread's K row (group 0: 1, 1 in columns 0,
      // 1) or V row (group 1: in columns 2, 3), which pick the (hi, lo)
      // pairs of the query's extra row; and the group's accumulator (dV,
      // dK) zeroed: both issuers add into it
      reinterpret_cast<uint4*>(sKV + 2 * T::TILE + b * C::AUX)[r] =
          b ? make_uint4(0u, 0x3F803F80u, 0u, 0u) : make_uint4(0x3F803F80u, 0u, 0u, 0u);
      fence_proxy_async_smem();
      uint32_t z[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) z[c] = 0u;
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc) tmem_st16_nw((b ? tdK : tdV) + lane_off + cc * 16, z);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(kv_ready);
    } else {
      // K (group 0) or V (group 1) row of this thread into TMEM as bf16
      // pairs with the extra chunk (rows past the sequence are zero), and
      // the group's accumulator (dV, dK) zeroed: both issuers add into it
      uint32_t w[D / 2 + 8];
      const __nv_bfloat16* src = p.qkv + ((long long)bi * p.s + kvp) * p.ld_qkv + (b ? p.v_col : p.k_col) +
                                 (long long)g * D;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (kvp < p.s) v = *reinterpret_cast<const uint4*>(src + c * 8);
        w[4 * c] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
      }
      // the extra chunk: K picks the (hi, lo) pair of -LSE*sqrt(d) (columns
      // 0, 1 of the query's extra row), V that of -D (columns 2, 3)
      w[D / 2] = b ? 0u : 0x3F803F80u;
      w[D / 2 + 1] = b ? 0x3F803F80u : 0u;
#pragma unroll
      for (int c = 2; c < 8; ++c) w[D / 2 + c] = 0u;
      tmem_store_row<D / 2 + 8>((b ? tVA : tKA) + lane_off, w);
      uint32_t z[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) z[c] = 0u;
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc) tmem_st16_nw((b ? tdK : tdV) + lane_off + cc * 16, z);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(kv_ready);
    }
    const float c = p.scale_log2;
    const uint32_t tSb = tS + 64 * b, tdPb = tdP + 64 * b;
    bool ok = true;
    for (int u = b; u < U; u += 2) {
      const int t = u >> 1;
      const int q0 = (i0 + t % n_i) * 128 + 64 * b;
      ok = bounded_wait(&s_full[b], (u >> 1) & 1, abort_flag, 651, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // ---- phase 1: P^T = exp2(S'^T * scale*log2(e)) (S' offset by
      // -LSE*sqrt(d)); query columns [lo, hi) of the 64 are unmasked
      int lo = 0, hi = min(64, p.s - q0);
      if (p.causal) lo = max(0, kvp - q0);
      if (kvp >= p.s) lo = 64;
      const bool edge = lo > 0 || hi < 64;
      uint32_t sv[64];
      tmem_ld32_nw(tSb + lane_off, sv);
      tmem_ld32_nw(tSb + lane_off + 32, sv + 32);
      tmem_wait_ld(sv);
      // P^T in fp32 (for dS^T) and as bf16 pairs (the dV operand)
      float pe[64];
      if (!edge) {
        const uint64_t c2 = f2(c, c);
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float2 e = f2split(mul2(f2(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), c2));
          pe[k] = ex2(e.x);
          pe[k + 1] = ex2(e.y);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) pe[k] = (k < lo || k >= hi) ? 0.f : ex2(__uint_as_float(sv[k]) * c);
      }
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 64; k += 2) pk[k / 2] = pack_bf16(pe[k], pe[k + 1]);
      tmem_st32(tSb + lane_off, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
      // ---- phase 2: dS^T = P^T dP'^T (dP' offset by -D)
      ok = bounded_wait(&dp_full[b], (u >> 1) & 1, abort_flag, 652, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t dr[64];
      tmem_ld32_nw(tdPb + lane_off, dr);
      tmem_ld32_nw(tdPb + lane_off + 32, dr + 32);
      tmem_wait_ld(dr);
      uint32_t o[32];
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        const float2 v = f2split(mul2(f2(pe[k], pe[k + 1]), f2(__uint_as_float(dr[k]), __uint_as_float(dr[k + 1]))));
        o[k / 2] = pack_bf16(v.x, v.y);
      }
      tmem_st32(tdPb + lane_off, o);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[b]);
    }
    // epilogue: group 0 writes dV, group 1 dK, once both issuers' products
    // are done (TMEM loads by every lane, stores only for rows inside the
    // sequence)
    if (ok) ok = __all_sync(0xffffffffu, bounded_wait(all_done, 0, abort_flag, 653, p.err));
    if (ok) {
      tc_fence_after();
      const bool valid = kvp < p.s;
      const uint32_t tsrc = (b == 0 ? tdV : tdK) + lane_off;
      __nv_bfloat16* row = p.dqkv + ((long long)bi * p.s + kvp) * p.ld_dqkv +
                           (b == 0 ? p.dv_col : p.dk_col) + (long long)g * D;
      const float sc = b == 0 ? 1.f : p.scale;
      if constexpr (D <= 80) {
        uint32_t acc[D];
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) tmem_ld16_nw(tsrc + cc * 16, acc + cc * 16);
        tmem_wait_ld(acc);
        if (valid) {
#pragma unroll
          for (int cc = 0; cc < D / 16; ++cc) store_row16(row + cc * 16, acc + cc * 16, sc);
        }
      } else {
        for (int cc = 0; cc < D / 16; ++cc) {
          uint32_t v[16];
          tmem_ld16_nw(tsrc + cc * 16, v);
          tmem_wait_ld(v);
          if (valid) store_row16(row + cc * 16, v, sc);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// Shared memory of the dQ kernel: the K/V ring.
template <int D>
struct DqCfg {
  using T = TileGeom<D>;
  static constexpr int KVS_FIT = (232448 - 1280) / (2 * T::TILE);
  static constexpr int KVS = KVS_FIT > 5 ? 5 : KVS_FIT;
  static constexpr int SMEM = KVS * 2 * T::TILE + 1024 + 256;
};

// ===========================================================================
// dQ in 64-key sub-tiles with double-buffered S and dP
// ===========================================================================
// One CTA per 128-row query tile of one head, looping over the key/value
// tiles j <= i in 64-key sub-tiles: sub-tile u is the half u % 2 of tile
// u / 2, and its S and dP go to buffer b = u % 2 (64 columns each).  Q and dO
// sit in TMEM as the A operands of S = Q K^T and dP = dO V^T; dS goes over
// the first 32 columns of its dP buffer as the A operand of dQ += dS K.
// Compute warps 2..5 (group 0) take the even sub-tiles and 6..9 (group 1) the
// odd ones, each warp its lane quarter's 32 query rows by the 64 key
// columns; warp 1 issues group 0's products and warp 10 group 1's, in the
// order S(u), dP(u), S(u+2) (once the group has read S(u)), dQ(u) (after
// dS(u)), dP(u+2) (which overwrites dS(u), after dQ(u) from the same
// thread).  Both issuers add into dQ, which group 0 zeroes first; a K/V
// stage is released once both issuers' products on it are done.  The row's
// log-sum-exp and dO.O sum are per-thread scalars.
// TMEM: S [0,64) [64,128), dP [128,192) [192,256), dQ [256, 256+D),
//       Q [256+D, 256+1.5D), dO [256+1.5D, 256+2D).
template <int D>
__global__ void __launch_bounds__(352, 1) attn_dq_hs_kernel(const __grid_constant__ AttnBwdParams p) {
  using T = TileGeom<D>;
  using C = DqCfg<D>;
  constexpr int KVS = C::KVS;
  static_assert(256 + 2 * D <= 512, "TMEM columns");
  constexpr uint32_t ID_S = idesc_bf16(128, 64, false, false);
  constexpr uint32_t ID_DQ = idesc_bf16(128, D, false, true);
  constexpr uint32_t COL_DQ = 256, COL_Q = 256 + D, COL_DO = 256 + D + D / 2;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKV = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + KVS * 2 * T::TILE);
  uint64_t* qo_ready = bars;           // Q, dO in TMEM and dQ zeroed (8 compute warps)
  uint64_t* kv_full = bars + 1;        // [KVS]
  uint64_t* kv_empty = kv_full + KVS;  // [KVS], both issuers
  uint64_t* s_full = kv_empty + KVS;   // [2] S(u) in buffer u % 2
  uint64_t* s_free = s_full + 2;       // [2] S(u) read (4 warps of the group)
  uint64_t* dp_full = s_free + 2;      // [2]
  uint64_t* ds_full = dp_full + 2;     // [2] dS(u) written (4 warps)
  uint64_t* all_done = ds_full + 2;    // both issuers' last products done
  uint64_t* drain = all_done + 1;      // [2], one per issuer
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  // head-major, heaviest query tiles of a head first; the query heads of one
  // KV group are adjacent, so the CTAs in flight share K/V in L2
  const int n_qt = (p.s + 127) / 128;
  const int pair = blockIdx.x / n_qt;
  const int i = n_qt - 1 - (int)(blockIdx.x % n_qt);
  const int n = pair % p.H;
  const int bi = pair / p.H;
  const int g = n / p.G;
  const int q0 = i * 128;
  const int nkv = p.causal ? min(i + 1, n_qt) : n_qt;
  const int U = 2 * nkv;

  if (threadIdx.x == 0) {
    mbar_init(qo_ready, 8);
    for (int k = 0; k < KVS; ++k) {
      mbar_init(&kv_full[k], 1);
      mbar_init(&kv_empty[k], 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 4);
      mbar_init(&dp_full[b], 1);
      mbar_init(&ds_full[b], 4);
      mbar_init(&drain[b], 1);
    }
    mbar_init(all_done, 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch(&p.map_qkv);
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem;         // + 64 b
  const uint32_t tdP = tmem + 128;  // + 64 b
  const uint32_t tdQ = tmem + COL_DQ;
  const uint32_t tQA = tmem + COL_Q;
  const uint32_t tOA = tmem + COL_DO;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int issued = 0;
      for (int jt = 0; jt < nkv; ++jt) {
        const int st = jt % KVS;
        if (jt >= KVS && !bounded_wait(&kv_empty[st], ((jt / KVS) & 1) ^ 1, abort_flag, 661, p.err)) break;
        uint8_t* sK = sKV + st * 2 * T::TILE;
        uint8_t* sV = sK + T::TILE;
        mbar_expect_tx(&kv_full[st], 2 * T::TILE);
#pragma unroll
        for (int c = 0; c < T::NCH; ++c) {
          tma_load_3d(sK + c * T::CHUNK, &p.map_qkv, &kv_full[st], p.k_col + g * D + c * T::CW, jt * 128, bi);
          tma_load_3d(sV + c * T::CHUNK, &p.map_qkv, &kv_full[st], p.v_col + g * D + c * T::CW, jt * 128, bi);
        }
        issued = jt + 1;
      }
      if (*abort_flag) {
        for (int jt = (issued > KVS ? issued - KVS : 0); jt < issued; ++jt)
          drain_wait(&kv_full[jt % KVS], (jt / KVS) & 1);
      }
    }
  } else if (warp == 1 || warp == 10) {
    // the whole warp runs the issue loop, one elected lane issues.  One
    // issuer (fixed-order mode): warp 1 issues every sub-tile's products
    // in sub-tile order, so dQ takes its products in a fixed order
    if (!(p.one_issuer && warp == 10)) {
      // ------------------------------------------------ MMA issuers
      const int b0 = warp == 1 ? 0 : 1;  // this issuer's first sub-tile
      const int ustep = p.one_issuer ? 1 : 2;
      const uint32_t uKV = smem_u32(sKV);
      // the 64 key rows of half b start 64 b rows into every chunk of the
      // stage's K and V tiles (whole swizzle atoms); sub-tile u uses buffer
      // b = u % 2
      auto uK = [&](int u) { return uKV + ((u >> 1) % KVS) * 2 * T::TILE; };
      auto issue_s = [&](int u) {
        const int b = u & 1;
        const uint32_t tSb = tS + 64 * b;
        const uint32_t k = uK(u) + 64 * T::SWB * b;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) umma_bf16_tmem_a_w(tSb, tQA + kk * 8, T::kmajor(k, kk), ID_S, kk > 0);
        umma_commit_w(&s_full[b]);
      };
      auto issue_dp = [&](int u) {
        const int b = u & 1;
        const uint32_t tdPb = tdP + 64 * b;
        const uint32_t v = uK(u) + T::TILE + 64 * T::SWB * b;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) umma_bf16_tmem_a_w(tdPb, tOA + kk * 8, T::kmajor(v, kk), ID_S, kk > 0);
        umma_commit_w(&dp_full[b]);
      };
      auto wait_stage = [&](int u) {
        const int jt = u >> 1;
        return bounded_wait_w(&kv_full[jt % KVS], (jt / KVS) & 1, abort_flag, 671, p.err);
      };
      bool ok = bounded_wait_w(qo_ready, 0, abort_flag, 672, p.err) && wait_stage(b0);
      if (ok) {
        tc_fence_after();
        // sub-tiles 0 and 1 share stage 0 (U is even)
        for (int u = b0; u < 2; u += ustep) {
          issue_s(u);
          issue_dp(u);
        }
      }
      for (int u = b0; ok && u < U; u += ustep) {
        const int b = u & 1;
        const uint32_t tdPb = tdP + 64 * b;
        const int st = (u >> 1) % KVS;
        const bool more = u + 2 < U;
        if (more) {
          // S(u+2) once the group has read S(u)
          if (!bounded_wait_w(&s_free[b], (u >> 1) & 1, abort_flag, 673, p.err) || !wait_stage(u + 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(u + 2);
        }
        // dQ += dS(u) K_u: key rows 64b.. are K blocks 4b..4b+3 of the tile
        if (!bounded_wait_w(&ds_full[b], (u >> 1) & 1, abort_flag, 674, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a_w(tdQ, tdPb + kk * 8, T::mnmajor(uK(u), 4 * b + kk), ID_DQ, 1);
        umma_commit_w(&kv_empty[st]);
        // dP(u+2) overwrites dS(u), after dQ(u) in issue order
        if (more) issue_dp(u + 2);
      }
      if (ok) {
        // all_done counts two commits: one per issuer, or both from one
        umma_commit_w(all_done);
        if (p.one_issuer) umma_commit_w(all_done);
      }
      if (!ok) {
        umma_commit_w(&drain[b0]);
        drain_wait(&drain[b0], 0);
      }
    }
  } else {
    // ------------------------------------------------ compute (warps 2..9;
    // warp 10 in the one-issuer mode falls through to the final barrier)
    const int quarter = warp & 3;
    const int b = (warp - 2) >> 2;  // group = buffer = sub-tile parity
    const int r = quarter * 32 + lane;
    const int qpos = q0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    {
      // Q (group 0) or dO (group 1) row of this thread into TMEM as bf16
      // pairs (rows past the sequence are zero); group 0 also zeroes dQ
      uint32_t w[D / 2];
      const __nv_bfloat16* src = b == 0
          ? p.qkv + ((long long)bi * p.s + qpos) * p.ld_qkv + p.q_col + (long long)n * D
          : p.dout + ((long long)bi * p.s + qpos) * p.ld_do + p.do_col + (long long)n * D;
#pragma unroll
      for (int cc = 0; cc < D / 8; ++cc) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (qpos < p.s) v = *reinterpret_cast<const uint4*>(src + cc * 8);
        w[4 * cc] = v.x;
        w[4 * cc + 1] = v.y;
        w[4 * cc + 2] = v.z;
        w[4 * cc + 3] = v.w;
      }
      tmem_store_row<D / 2>((b == 0 ? tQA : tOA) + lane_off, w);
      if (b == 0) {
        uint32_t z[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) z[k] = 0u;
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) tmem_st16_nw(tdQ + lane_off + cc * 16, z);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(qo_ready);
    }
    const float c = p.scale_log2;
    // this row's -LSE*log2(e) and dO.O sum (finite filler past the sequence)
    const float nl = p.nl2[((long long)bi * p.H + n) * p.s_pad + qpos];
    const float dsum = p.Dsum[((long long)bi * p.H + n) * p.s_pad + qpos];
    const uint32_t tSb = tS + 64 * b, tdPb = tdP + 64 * b;
    bool ok = true;
    for (int u = b; u < U; u += 2) {
      ok = bounded_wait(&s_full[b], (u >> 1) & 1, abort_flag, 681, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // ---- phase 1: P = exp2(S * scale*log2(e) - LSE*log2(e)); key columns
      // [0, hi) of the 64 are unmasked
      const int kv0 = (u >> 1) * 128 + 64 * b;
      int hi = min(64, p.s - kv0);
      if (p.causal) hi = min(hi, qpos - kv0 + 1);
      if (qpos >= p.s) hi = 0;
      uint32_t sv[64];
      tmem_ld32_nw(tSb + lane_off, sv);
      tmem_ld32_nw(tSb + lane_off + 32, sv + 32);
      tmem_wait_ld(sv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[b]);
      // P stays in fp32 registers: no product here reads it, only dS
      float pe[64];
      if (hi >= 64) {
        const uint64_t c2 = f2(c, c), nl2 = f2(nl, nl);
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float2 e = f2split(fma2(f2(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), c2, nl2));
          pe[k] = ex2(e.x);
          pe[k + 1] = ex2(e.y);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) pe[k] = k < hi ? ex2(fmaf(__uint_as_float(sv[k]), c, nl)) : 0.f;
      }
      // ---- phase 2: dS = P (dP - D), over the first 32 columns of buffer b
      ok = bounded_wait(&dp_full[b], (u >> 1) & 1, abort_flag, 682, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t dr[64];
      tmem_ld32_nw(tdPb + lane_off, dr);
      tmem_ld32_nw(tdPb + lane_off + 32, dr + 32);
      tmem_wait_ld(dr);
      uint32_t o[32];
      const uint64_t ds2 = f2(dsum, dsum);
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        const float2 v = f2split(
            mul2(f2(pe[k], pe[k + 1]), sub2(f2(__uint_as_float(dr[k]), __uint_as_float(dr[k + 1])), ds2)));
        o[k / 2] = pack_bf16(v.x, v.y);
      }
      tmem_st32(tdPb + lane_off, o);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[b]);
    }
    // epilogue: the two groups split dQ's 16-column chunks once both
    // issuers' products are done
    if (ok) ok = __all_sync(0xffffffffu, bounded_wait(all_done, 0, abort_flag, 683, p.err));
    if (ok) {
      tc_fence_after();
      constexpr int NC = D / 16;
      constexpr int NC0 = (NC + 1) / 2;
      const int cbeg = b == 0 ? 0 : NC0, cend = b == 0 ? NC0 : NC;
      const bool valid = qpos < p.s;
      __nv_bfloat16* qrow = p.dqkv + ((long long)bi * p.s + qpos) * p.ld_dqkv + p.dq_col + (long long)n * D;
      const uint32_t tq = tdQ + lane_off;
      for (int cc = cbeg; cc < cend; ++cc) {
        uint32_t v[16];
        tmem_ld16_nw(tq + cc * 16, v);
        tmem_wait_ld(v);
        if (valid) store_row16(qrow + cc * 16, v, p.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
int launch_dkdv_hs(AttnBwdParams& prm, int grid, cudaStream_t st) {
  constexpr int SMEM = DkdvTmCfg<D>::SMEM;
  static_assert(SMEM <= 232448, "dK/dV tile set exceeds shared memory");
  static std::atomic<uint64_t> attr{0};  // devices whose limit is set
  if (smem_limit_once(reinterpret_cast<const void*>(attn_dkdv_hs_kernel<D>), SMEM, &attr)) return 3;
  attn_dkdv_hs_kernel<D><<<grid, 352, SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

template <int D>
int launch_dq(AttnBwdParams& prm, int grid, cudaStream_t st) {
  constexpr int SMEM = DqCfg<D>::SMEM;
  static_assert(SMEM <= 232448, "dQ tile set exceeds shared memory");
  static std::atomic<uint64_t> attr{0};  // devices whose limit is set
  if (smem_limit_once(reinterpret_cast<const void*>(attn_dq_hs_kernel<D>), SMEM, &attr)) return 3;
  attn_dq_hs_kernel<D><<<grid, 352, SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

template <int D>
int launch_both(AttnBwdParams& prm, const AttnShape& f, cudaStream_t st) {
  const double pairs = f.causal ? (double)f.s * (f.s + 1) / 2 : (double)f.s * f.s;
  int rc;
  {
    // S, dP, dV, dK over the unmasked pairs
    ProfScope prof(PROF_ATTN_BWD, 8.0 * f.d * pairs * f.H * f.b, 0.0, st);
    const int grid = ((f.s + 127) / 128) * f.Hkv * f.b;
    rc = launch_dkdv_hs<D>(prm, grid, st);
  }
  if (rc) return rc;
  // dQ only: the S and dP this kernel rebuilds for its query-major order are
  // not part of the method's algorithmic work (S, dP, dV, dK, dQ = 2.5x the
  // forward attention), so they are not credited
  ProfScope prof(PROF_ATTN_BWD, 2.0 * f.d * pairs * f.H * f.b, 0.0, st);
  return launch_dq<D>(prm, ((f.s + 127) / 128) * f.H * f.b, st);
}

}  // namespace

int make_attn_map(CUtensorMap* map, const void* qkv, int b, int s, int64_t ld, int d);
int attn_dsum(const AttnBwdShape& sh, const void* o, const void* dout, const float* lse, float* Dsum,
              float* NL2, void* AUX, int s_pad, cudaStream_t st);

// workspace: the per-row dO.O sums D and -LSE*log2(e), both [b, H, s_pad]
// fp32, then the dK/dV kernel's extra query rows [b, H, s_pad, 8] bf16
size_t attention_bwd_ws_bytes(const AttnBwdShape& sh) {
  const int64_t s_pad = ((int64_t)sh.f.s + 127) / 128 * 128;
  return (size_t)sh.f.b * sh.f.H * s_pad * (8 + 16);
}

// lse: [b, H_total, s_pad] fp32 (head offset lse_head0)
int attention_bwd(const AttnBwdShape& sh, const void* qkv, const void* o, const float* lse,
                  const void* dout, void* dqkv, void* ws, cudaStream_t st) {
  const AttnShape& f = sh.f;
  const int s_pad = (f.s + 127) / 128 * 128;
  const size_t nrow = (size_t)f.b * f.H * s_pad;
  float* Dsum = reinterpret_cast<float*>(ws);
  float* NL2 = Dsum + nrow;
  __nv_bfloat16* AUX = reinterpret_cast<__nv_bfloat16*>(NL2 + nrow);
  if (nrow > (size_t)INT32_MAX) return BPT_EUNSUPPORTED;  // the extra rows' TMA row coordinate
  int rc;
  {
    ProfScope prof(PROF_MISC, 0.0, 4.0 * f.b * f.s * f.H * f.d + 28.0 * f.b * f.H * s_pad, st);
    rc = attn_dsum(sh, o, dout, lse, Dsum, NL2, AUX, s_pad, st);
    if (rc) return rc;
  }

  AttnBwdParams prm;
  memset(&prm, 0, sizeof(prm));
  if (make_attn_map(&prm.map_qkv, qkv, f.b, f.s, f.ld_qkv, f.d)) return 1;
  if (make_attn_map(&prm.map_do, dout, f.b, f.s, sh.ld_do, f.d)) return 1;
  if (make_map_2d(&prm.map_aux, AUX, nrow, 8, 8, 8, 128, 0)) return 1;
  prm.s = f.s;
  prm.s_pad = s_pad;
  prm.H = f.H;
  prm.Hkv = f.Hkv;
  prm.G = f.H / f.Hkv;
  prm.causal = f.causal;
  prm.b = f.b;
  prm.q_col = (int)f.q_col;
  prm.k_col = (int)f.k_col;
  prm.v_col = (int)f.v_col;
  prm.do_col = (int)sh.do_col;
  prm.lse = lse;
  prm.Dsum = Dsum;
  prm.nl2 = NL2;
  prm.qkv = reinterpret_cast<const __nv_bfloat16*>(qkv);
  prm.ld_qkv = f.ld_qkv;
  prm.dout = reinterpret_cast<const __nv_bfloat16*>(dout);
  prm.ld_do = sh.ld_do;
  prm.H_total = f.H_total;
  prm.lse_head0 = f.lse_head0;
  prm.dqkv = reinterpret_cast<__nv_bfloat16*>(dqkv);
  prm.ld_dqkv = sh.ld_dqkv;
  prm.dq_col = (int)sh.dq_col;
  prm.dk_col = (int)sh.dk_col;
  prm.dv_col = (int)sh.dv_col;
  prm.scale = 1.f / sqrtf((float)f.d);
  prm.scale_log2 = prm.scale * 1.4426950408889634f;
  prm.one_issuer = sh.deterministic ? 1 : 0;
  prm.err = device_error_word();
  if (!prm.err) return 3;
  switch (f.d) {
    case 64: return launch_both<64>(prm, f, st);
    case 80: return launch_both<80>(prm, f, st);
    case 96: return launch_both<96>(prm, f, st);
    case 112: return launch_both<112>(prm, f, st);
    case 128: return launch_both<128>(prm, f, st);
    default: return 5;
  }
}

}  // namespace bpt
