// attn_fwd.cu -- blockwise causal attention with online softmax on tcgen05.
//
// "Blockwise Parallel Transformer for Long Context Large Models", section 3.4,
// "Blockwise Self-Attention with Online Softmax" and "The Nested-Loop
// Algorithm in Detail (Algorithm 1)": for one query block, loop over the
// key/value blocks; keep a running row max m, denominator l and numerator
// (here O in TMEM); for each block S = Q K_j^T / sqrt(d) with the causal bias,
// m' = max(m, rowmax S), correction exp(m - m'), l = l*corr + rowsum exp(S - m'),
// O = O*corr + exp(S - m') V_j; finally O / l.  The log-sum-exp m + ln l of
// every row is written for the recompute backward.
//
// One CTA = one 128-row query tile of one head (GQA: key/value head n / G);
// warp 0 streams K/V tiles through a ring.  Two kernels:
//  * head dims 64 and 80 (attn_fwd_sk_kernel): the keys of every tile are
//    split in halves, and two groups of four softmax warps (2..5, 6..9),
//    each with its own MMA-issuing warp (1, 10), run independent online
//    softmaxes over their halves -- own running max, own O accumulator --
//    merged once at the end by the log-sum-exp rule;
//  * head dims 96 to 128 (attn_fwd_kernel), whose two O accumulators would
//    not fit in TMEM: warp 1 issues S_{j+1} = Q K_{j+1}^T into one of two
//    TMEM S buffers, then O += P_j V_j, and warps 2..5 do the softmax.
// Softmax, one query row per thread: copy the Q row into TMEM once; per tile
// read the S row, mask, update m, write P (bf16 pairs) over the S buffer,
// rescale the O row in TMEM when the max moved by more than 2^8 (otherwise
// keep the stale max: exact, since O and l are scaled alike); at the end
// normalise and store O.  Up to d = 112 the row sums l come from the tensor
// core (an extra chunk of V), else from fp32 adds.
// The s x s score matrix never leaves TMEM/registers.
#include <math.h>
#include <string.h>

#include <algorithm>

#include "attn_common.cuh"
#include "internal.h"

namespace bpt {

namespace {

struct AttnFwdParams {
  CUtensorMap map_qkv;  // 3-D {ld_qkv, s, b}, box {CW, 128, 1}
  int s, s_pad, H, G, causal;
  int q_col, k_col, v_col;
  __nv_bfloat16* o;
  long long ld_o, o_row0;
  int o_col;
  float* lse;
  int H_total, lse_head0;
  // output head of local head n (O column block and LSE row):
  // (n / o_seg) * o_seg_stride + n % o_seg -- n itself unless the call's
  // heads are spread over the output in segments (interleaved stages)
  int o_seg, o_seg_stride;
  int qt_begin, n_qt, b;
  float scale_log2;  // log2(e) / sqrt(d)
  float scale;       // 1 / sqrt(d)
  const __nv_bfloat16* qkv;  // the packed projection (Q rows copied into TMEM)
  long long ld_qkv;
  unsigned int* err;
};

__device__ __forceinline__ int out_head(const AttnFwdParams& p, int n) {
  return (n / p.o_seg) * p.o_seg_stride + n % p.o_seg;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// TMEM: two 128-column S buffers [0,256), O [256, 256+D+EXT), Q after it
// (D/2 columns).  Q is copied into TMEM once per CTA (the A operand of
// S = Q K_j^T) and each P is written over its own S buffer as bf16 pairs (the
// A operand of O += P V_j), so every product reads only its B operand from
// shared memory, which holds just the K/V ring.
//
// Row sums on the tensor core (EXT = 16): each ring stage carries, right after
// V's column chunks, one more chunk whose every 16-byte unit is (1, 0, ..., 0)
// in bf16, so P V reads N = D + 16 columns and writes the row sum of P (the
// same bf16 P the numerator uses) into O's columns D and D + 8 whatever the
// swizzle permutes.  The sum is rescaled with O, and the softmax does no
// adds.  Not for d = 128, whose 16 KB chunks would cost a ring stage.
template <int D>
struct FwdCfg {
  using T = TileGeom<D>;
  static constexpr int EXT = (T::CW == 16 || D == 64) ? 16 : 0;
  static constexpr int EXT_BYTES = EXT ? T::CHUNK : 0;
  static constexpr int STAGE = 2 * T::TILE + EXT_BYTES;
  static constexpr int KVS_FIT = (232448 - 1280) / STAGE;
  static constexpr int KVS = KVS_FIT > 5 ? 5 : KVS_FIT;
  static constexpr int SMEM = KVS * STAGE + 1024 + 256;
  static constexpr uint32_t COL_O = 256, COL_Q = 256 + D + EXT;
};

template <int D>
__global__ void __launch_bounds__(192, 1) attn_fwd_kernel(const __grid_constant__ AttnFwdParams p) {
  using T = TileGeom<D>;
  using C = FwdCfg<D>;
  constexpr int KVS = C::KVS;
  constexpr int EXT = C::EXT;
  constexpr int STAGE = C::STAGE;
  static_assert(C::COL_Q + D / 2 <= 512, "TMEM columns");
  constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
  constexpr uint32_t IDESC_PV = idesc_bf16(128, D + EXT, false, true);
  constexpr float NEG_INF = -INFINITY;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKV = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + KVS * STAGE);
  uint64_t* q_ready = bars;            // Q copied into TMEM (4 softmax warps)
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + KVS;
  uint64_t* s_full = kv_empty + KVS;   // [2]
  uint64_t* p_full = s_full + 2;       // [2], 4 softmax warps
  uint64_t* pv_done = p_full + 2;
  uint64_t* drain = pv_done + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = warp_id();
  const int lane = lane_id();

  // tile scheduling: head-major, heaviest query tiles of a head first.  The
  // CTAs in flight then share one or two heads' K/V (10 MB per head at
  // s=32K, d=80), which stays in L2; tile-major order spread them over every
  // head and re-read K/V from HBM on each wave.
  const int pair = blockIdx.x / p.n_qt;
  const int qt_rev = blockIdx.x % p.n_qt;
  const int n = pair % p.H;
  const int bi = pair / p.H;
  const int qt = p.qt_begin + p.n_qt - 1 - qt_rev;
  const int q0 = qt * 128;
  const int g = n / p.G;
  const int kv_tiles_total = (p.s + 127) / 128;
  const int nkv = p.causal ? min(qt + 1, kv_tiles_total) : kv_tiles_total;

  if (threadIdx.x == 0) {
    mbar_init(q_ready, 4);
    for (int i = 0; i < KVS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch(&p.map_qkv);
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  if constexpr (EXT > 0) {
    // the row-sum chunk of every stage (never written by TMA)
    constexpr int UNITS = C::EXT_BYTES / 16;
    for (int i = threadIdx.x; i < KVS * UNITS; i += blockDim.x)
      reinterpret_cast<uint4*>(sKV + (i / UNITS) * STAGE + 2 * T::TILE)[i % UNITS] = make_uint4(0x3F80u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem;  // two 128-column S / P buffers
  const uint32_t tO = tmem + C::COL_O;
  const uint32_t tQA = tmem + C::COL_Q;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % KVS;
        if (j >= KVS && !bounded_wait(&kv_empty[st], ((j / KVS) & 1) ^ 1, abort_flag, 201, p.err)) break;
        uint8_t* sK = sKV + st * STAGE;
        uint8_t* sV = sK + T::TILE;
        mbar_expect_tx(&kv_full[st], 2 * T::TILE);
#pragma unroll
        for (int c = 0; c < T::NCH; ++c)
          tma_load_3d(sK + c * T::CHUNK, &p.map_qkv, &kv_full[st], p.k_col + g * D + c * T::CW, j * 128, bi);
#pragma unroll
        for (int c = 0; c < T::NCH; ++c)
          tma_load_3d(sV + c * T::CHUNK, &p.map_qkv, &kv_full[st], p.v_col + g * D + c * T::CW, j * 128, bi);
        issued = j + 1;
      }
      if (*abort_flag) {
        for (int j = (issued > KVS ? issued - KVS : 0); j < issued; ++j)
          drain_wait(&kv_full[j % KVS], (j / KVS) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (the
    // whole warp runs the loop, one elected lane issues)
    // order: S(0); per j: S(j+1), PV(j).  S(j+1) overwrites the buffer of
    // P(j-1) after PV(j-1) in issue order.
    const uint32_t uKV = smem_u32(sKV);
    auto issue_s = [&](int j) -> bool {
      if (!bounded_wait_w(&kv_full[j % KVS], (j / KVS) & 1, abort_flag, 213, p.err)) return false;
      tc_fence_after();
      const uint32_t kt = uKV + (j % KVS) * STAGE;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma_bf16_tmem_a_w(tS + (j & 1) * 128, tQA + kk * 8, T::kmajor(kt, kk), IDESC_S, kk > 0);
      umma_commit_w(&s_full[j & 1]);
      return true;
    };
    bool ok = bounded_wait_w(q_ready, 0, abort_flag, 211, p.err) && issue_s(0);
    for (int j = 0; ok && j < nkv; ++j) {
      if (j + 1 < nkv && !issue_s(j + 1)) { ok = false; break; }
      if (!bounded_wait_w(&p_full[j & 1], (j >> 1) & 1, abort_flag, 212, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t vt = uKV + (j % KVS) * STAGE + T::TILE;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_bf16_tmem_a_w(tO, tS + (j & 1) * 128 + kk * 8, T::mnmajor(vt, kk), IDESC_PV, (j > 0 || kk > 0));
      umma_commit_w(&kv_empty[j % KVS]);
      umma_commit_w(pv_done);
    }
    if (!ok) {
      umma_commit_w(drain);
      drain_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------ softmax (warps 2..5)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qpos = q0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    {
      // this thread's Q row into TMEM as bf16 pairs (zero past the sequence)
      uint32_t w[D / 2];
      const __nv_bfloat16* src =
          p.qkv + ((long long)bi * p.s + qpos) * p.ld_qkv + p.q_col + (long long)n * D;
#pragma unroll
      for (int cc = 0; cc < D / 8; ++cc) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (qpos < p.s) v = *reinterpret_cast<const uint4*>(src + cc * 8);
        w[4 * cc] = v.x;
        w[4 * cc + 1] = v.y;
        w[4 * cc + 2] = v.z;
        w[4 * cc + 3] = v.w;
      }
      tmem_store_row<D / 2>(tQA + lane_off, w);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    const float c = p.scale_log2;
    float m_run = NEG_INF, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      const uint32_t tb = tS + sb * 128 + lane_off;
      ok = bounded_wait(&s_full[sb], (j >> 1) & 1, abort_flag, 221, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[128];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld32_nw(tb + q4 * 32, sv + q4 * 32);
      tmem_wait_ld(sv);
      // key columns [0, hi) are unmasked
      const int kv0 = j * 128;
      int hi = min(128, p.s - kv0);
      if (p.causal) hi = min(hi, qpos - kv0 + 1);
      const bool edge = hi < 128;
      float mx = NEG_INF;
      if (!edge) {
        // four independent chains of three-input maxima
        float m4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
        for (int i = 0; i < 128; i += 2)
          m4[(i >> 1) & 3] = max3f(m4[(i >> 1) & 3], __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
        mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i < hi) mx = fmaxf(mx, __uint_as_float(sv[i]));
      }
      const float m_new = fmaxf(m_run, mx);
      const bool need = (m_new - m_run) * c > 8.f;
      const bool rescale = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (rescale) {
        alpha = (m_run == NEG_INF) ? 0.f : ex2((m_run - m_new) * c);
        m_run = m_new;
      }
      // a row with no unmasked key yet keeps m = -inf; its exponent offset
      // is then 0 and every P entry below is masked to zero
      const float mc = (m_run == NEG_INF) ? 0.f : m_run * c;
      float rs = 0.f;
      uint32_t pk[64];
      if (!edge) {
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
          const float e0 = ex2(fmaf(__uint_as_float(sv[i]), c, -mc));
          const float e1 = ex2(fmaf(__uint_as_float(sv[i + 1]), c, -mc));
          if constexpr (EXT == 0) rs += e0 + e1;
          pk[i / 2] = pack_bf16(e0, e1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
          const float e0 = i < hi ? ex2(fmaf(__uint_as_float(sv[i]), c, -mc)) : 0.f;
          const float e1 = i + 1 < hi ? ex2(fmaf(__uint_as_float(sv[i + 1]), c, -mc)) : 0.f;
          if constexpr (EXT == 0) rs += e0 + e1;
          pk[i / 2] = pack_bf16(e0, e1);
        }
      }
      l_run = l_run * alpha + rs;
      // P over the first 64 columns of its own S buffer (all read above)
      tmem_st32(tb, *reinterpret_cast<const uint32_t(*)[32]>(pk));
      tmem_st32(tb + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
      // PV(j-1) must be done before O is rescaled.  Having seen S(j), which
      // was issued after PV(j-2), these warps know pv_done is in phase j-1
      // or j (PV(j) waits for this step's P), so a wait on the parity of
      // j - 1 is exact however many phases went by unwaited.  The last step
      // always waits, so the wait after the loop is exact too.
      if (j > 0 && (rescale || j == nkv - 1)) {
        ok = bounded_wait(pv_done, (j - 1) & 1, abort_flag, 222, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if (rescale) {
          // the row (and its row-sum columns)
          uint32_t ro[D + EXT];
#pragma unroll
          for (int cc = 0; cc < (D + EXT) / 16; ++cc) tmem_ld16_nw(tO + lane_off + cc * 16, ro + cc * 16);
          tmem_wait_ld(ro);
#pragma unroll
          for (int i = 0; i < D + EXT; ++i) ro[i] = __float_as_uint(__uint_as_float(ro[i]) * alpha);
#pragma unroll
          for (int cc = 0; cc < (D + EXT) / 16; ++cc) tmem_st16_nw(tO + lane_off + cc * 16, ro + cc * 16);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    if (ok) {
      ok = bounded_wait(pv_done, (nkv - 1) & 1, abort_flag, 223, p.err);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const bool valid = qpos < p.s;
      __nv_bfloat16* orow = p.o + ((long long)bi * p.s + qpos - p.o_row0) * p.ld_o + p.o_col + (long long)out_head(p, n) * D;
      uint32_t oall[D + EXT];
#pragma unroll
      for (int cc = 0; cc < (D + EXT) / 16; ++cc) tmem_ld16_nw(tO + lane_off + cc * 16, oall + cc * 16);
      tmem_wait_ld(oall);
      if constexpr (EXT > 0) l_run = __uint_as_float(oall[D]);
      const float inv_l = 1.f / l_run;
      if (valid) {
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) store_row16(orow + cc * 16, oall + cc * 16, inv_l);
      }
      // every row of the padded tile gets a finite value (rows past s see the
      // zero-filled query), so the backward pass never reads garbage
      if (p.lse)
        p.lse[((long long)bi * p.H_total + p.lse_head0 + out_head(p, n)) * p.s_pad + qpos] = m_run * p.scale + logf(l_run);
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

// ---------------------------------------------------------------------------
// Split keys (head dims 64 and 80): two independent online softmaxes per CTA.
// The 128 keys of every K/V tile are split in two halves; softmax group b
// (warps 2..5 for b = 0, 6..9 for b = 1) runs the whole online-softmax loop
// over the keys 64b..64b+63 of every tile, with its own running max, its own
// O accumulator (its row sums in O's extra columns) and its own MMA-issuing
// warp (1 or 10).  The two partial results of a row are merged once, at the
// end, by the log-sum-exp rule: m = max(m0, m1), O = sum_b O_b 2^((m_b - m)c)
// / sum_b l_b 2^((m_b - m)c).  Each SM sub-partition then runs two
// independent softmax warps over 64 columns instead of one over 128, with no
// exchange between them before the merge.
// TMEM: S of group b in [128b, 128b+128) as two 64-column buffers; O_b at
// 256 + b (D + 16); Q at 256 + 2 (D + 16).
template <int D>
struct FwdSkCfg {
  using T = TileGeom<D>;
  static constexpr int EXT = FwdCfg<D>::EXT;
  static constexpr int STAGE = FwdCfg<D>::STAGE;
  static constexpr int RED = 2 * 128 * 4;  // [group][row] running max, for the merge
  static constexpr int KVS_FIT = (232448 - RED - 1280) / STAGE;
  static constexpr int KVS = KVS_FIT > 5 ? 5 : KVS_FIT;
  static constexpr int SMEM = KVS * STAGE + RED + 1024 + 256;
  static constexpr uint32_t COL_O = 256, OW = D + EXT, COL_Q = 256 + 2 * OW;
};

template <int D>
__global__ void __launch_bounds__(352, 1) attn_fwd_sk_kernel(const __grid_constant__ AttnFwdParams p) {
  using T = TileGeom<D>;
  using C = FwdSkCfg<D>;
  constexpr int KVS = C::KVS;
  constexpr int EXT = C::EXT;
  constexpr int STAGE = C::STAGE;
  static_assert(EXT == 16, "the split-key kernel keeps its row sums in O's extra columns");
  static_assert(C::COL_Q + D / 2 <= 512, "TMEM columns");
  constexpr uint32_t IDESC_S = idesc_bf16(128, 64, false, false);
  constexpr uint32_t IDESC_PV = idesc_bf16(128, D + EXT, false, true);
  constexpr float NEG_INF = -INFINITY;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKV = smem;
  float* red = reinterpret_cast<float*>(sKV + KVS * STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + C::RED);
  uint64_t* q_ready = bars;             // Q copied into TMEM (group 0's 4 warps)
  uint64_t* kv_full = bars + 1;         // [KVS]
  uint64_t* kv_empty = kv_full + KVS;   // [KVS], both issuers
  uint64_t* s_full = kv_empty + KVS;    // [group][buffer]
  uint64_t* p_full = s_full + 4;        // [group][buffer], 4 warps
  uint64_t* pv_done = p_full + 4;       // [group]
  uint64_t* drain = pv_done + 2;        // [group]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = warp_id();
  const int lane = lane_id();

  // tile scheduling: head-major, heaviest query tiles of a head first
  const int pair = blockIdx.x / p.n_qt;
  const int qt_rev = blockIdx.x % p.n_qt;
  const int n = pair % p.H;
  const int bi = pair / p.H;
  const int qt = p.qt_begin + p.n_qt - 1 - qt_rev;
  const int q0 = qt * 128;
  const int g = n / p.G;
  const int kv_tiles_total = (p.s + 127) / 128;
  const int nkv = p.causal ? min(qt + 1, kv_tiles_total) : kv_tiles_total;

  if (threadIdx.x == 0) {
    mbar_init(q_ready, 4);
    for (int i = 0; i < KVS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 2);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pv_done[b], 1);
      mbar_init(&drain[b], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch(&p.map_qkv);
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  {
    // the row-sum chunk of every stage (never written by TMA)
    constexpr int UNITS = C::T::CHUNK / 16;
    for (int i = threadIdx.x; i < KVS * UNITS; i += blockDim.x)
      reinterpret_cast<uint4*>(sKV + (i / UNITS) * STAGE + 2 * T::TILE)[i % UNITS] = make_uint4(0x3F80u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tQA = tmem + C::COL_Q;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % KVS;
        if (j >= KVS && !bounded_wait(&kv_empty[st], ((j / KVS) & 1) ^ 1, abort_flag, 231, p.err)) break;
        uint8_t* sK = sKV + st * STAGE;
        uint8_t* sV = sK + T::TILE;
        mbar_expect_tx(&kv_full[st], 2 * T::TILE);
#pragma unroll
        for (int c = 0; c < T::NCH; ++c)
          tma_load_3d(sK + c * T::CHUNK, &p.map_qkv, &kv_full[st], p.k_col + g * D + c * T::CW, j * 128, bi);
#pragma unroll
        for (int c = 0; c < T::NCH; ++c)
          tma_load_3d(sV + c * T::CHUNK, &p.map_qkv, &kv_full[st], p.v_col + g * D + c * T::CW, j * 128, bi);
        issued = j + 1;
      }
      if (*abort_flag) {
        for (int j = (issued > KVS ? issued - KVS : 0); j < issued; ++j)
          drain_wait(&kv_full[j % KVS], (j / KVS) & 1);
      }
    }
  } else if (warp == 1 || warp == 10) {
    // ------------------------------------------------ MMA issuers (the
    // whole warp runs the loop, one elected lane issues)
    // group b's products: S_b(j+1) = Q K_j[64b..]^T into its buffer
    // (j+1) % 2, then O_b += P_b(j) V_j[64b..] (+ the row-sum chunk).
    // S_b(j+1) overwrites P_b(j-1) after PV_b(j-1) from the same thread.
    const int b = warp == 1 ? 0 : 1;
    const uint32_t uKV = smem_u32(sKV);
    const uint32_t tSb = tmem + 128 * b;
    const uint32_t tOb = tmem + C::COL_O + b * C::OW;
    auto issue_s = [&](int j) -> bool {
      if (!bounded_wait_w(&kv_full[j % KVS], (j / KVS) & 1, abort_flag, 233, p.err)) return false;
      tc_fence_after();
      const uint32_t kt = uKV + (j % KVS) * STAGE + 64 * T::SWB * b;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma_bf16_tmem_a_w(tSb + (j & 1) * 64, tQA + kk * 8, T::kmajor(kt, kk), IDESC_S, kk > 0);
      umma_commit_w(&s_full[2 * b + (j & 1)]);
      return true;
    };
    bool ok = bounded_wait_w(q_ready, 0, abort_flag, 234, p.err) && issue_s(0);
    for (int j = 0; ok && j < nkv; ++j) {
      if (j + 1 < nkv && !issue_s(j + 1)) { ok = false; break; }
      if (!bounded_wait_w(&p_full[2 * b + (j & 1)], (j >> 1) & 1, abort_flag, 235, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t vt = uKV + (j % KVS) * STAGE + T::TILE;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16_tmem_a_w(tOb, tSb + (j & 1) * 64 + kk * 8, T::mnmajor(vt, 4 * b + kk), IDESC_PV, (j > 0 || kk > 0));
      umma_commit_w(&kv_empty[j % KVS]);
      umma_commit_w(&pv_done[b]);
    }
    if (!ok) {
      umma_commit_w(&drain[b]);
      drain_wait(&drain[b], 0);
    }
  } else {
    // ------------------------------------------------ softmax (warps 2..9)
    const int quarter = warp & 3;
    const int b = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int qpos = q0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tSb = tmem + 128 * b;
    const uint32_t tOb = tmem + C::COL_O + b * C::OW;
    if (b == 0) {
      // this thread's Q row into TMEM as bf16 pairs (zero past the sequence)
      uint32_t w[D / 2];
      const __nv_bfloat16* src =
          p.qkv + ((long long)bi * p.s + qpos) * p.ld_qkv + p.q_col + (long long)n * D;
#pragma unroll
      for (int cc = 0; cc < D / 8; ++cc) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (qpos < p.s) v = *reinterpret_cast<const uint4*>(src + cc * 8);
        w[4 * cc] = v.x;
        w[4 * cc + 1] = v.y;
        w[4 * cc + 2] = v.z;
        w[4 * cc + 3] = v.w;
      }
      tmem_store_row<D / 2>(tQA + lane_off, w);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    const float c = p.scale_log2;
    float m_run = NEG_INF;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      const uint32_t tb = tSb + sb * 64 + lane_off;
      ok = bounded_wait(&s_full[2 * b + sb], (j >> 1) & 1, abort_flag, 241, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld32_nw(tb, sv);
      tmem_ld32_nw(tb + 32, sv + 32);
      tmem_wait_ld(sv);
      // this group's key columns [0, hi) of the 64 are unmasked
      const int kv0 = j * 128 + 64 * b;
      int hi = min(64, p.s - kv0);
      if (p.causal) hi = min(hi, qpos - kv0 + 1);
      const bool edge = hi < 64;
      float mx = NEG_INF;
      if (!edge) {
        float m4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
        for (int i = 0; i < 64; i += 2)
          m4[(i >> 1) & 3] = max3f(m4[(i >> 1) & 3], __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
        mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i < hi) mx = fmaxf(mx, __uint_as_float(sv[i]));
      }
      const float m_new = fmaxf(m_run, mx);
      const bool need = (m_new - m_run) * c > 8.f;
      const bool rescale = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (rescale) {
        alpha = (m_run == NEG_INF) ? 0.f : ex2((m_run - m_new) * c);
        m_run = m_new;
      }
      // a row with no unmasked key yet keeps m = -inf; its exponent offset
      // is then 0 and every P entry below is masked to zero
      const float mc = (m_run == NEG_INF) ? 0.f : m_run * c;
      uint32_t pk[32];
      if (!edge) {
        const uint64_t c2 = f2(c, c), nmc2 = f2(-mc, -mc);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 e = f2split(fma2(f2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2, nmc2));
          pk[i / 2] = pack_bf16(ex2(e.x), ex2(e.y));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float e0 = i < hi ? ex2(fmaf(__uint_as_float(sv[i]), c, -mc)) : 0.f;
          const float e1 = i + 1 < hi ? ex2(fmaf(__uint_as_float(sv[i + 1]), c, -mc)) : 0.f;
          pk[i / 2] = pack_bf16(e0, e1);
        }
      }
      // P over the first 32 columns of its own S buffer (all read above)
      tmem_st32(tb, pk);
      // PV(j-1) must be done before O is rescaled; the wait is exact
      // without the skipped ones, as in the one-group kernel
      if (j > 0 && (rescale || j == nkv - 1)) {
        ok = bounded_wait(&pv_done[b], (j - 1) & 1, abort_flag, 242, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if (rescale) {
          // the row and its row-sum columns
          uint32_t ro[D + EXT];
#pragma unroll
          for (int cc = 0; cc < (D + EXT) / 16; ++cc) tmem_ld16_nw(tOb + lane_off + cc * 16, ro + cc * 16);
          tmem_wait_ld(ro);
#pragma unroll
          for (int i = 0; i < D + EXT; ++i) ro[i] = __float_as_uint(__uint_as_float(ro[i]) * alpha);
#pragma unroll
          for (int cc = 0; cc < (D + EXT) / 16; ++cc) tmem_st16_nw(tOb + lane_off + cc * 16, ro + cc * 16);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[2 * b + sb]);
    }
    if (ok) ok = __all_sync(0xffffffffu, bounded_wait(&pv_done[b], (nkv - 1) & 1, abort_flag, 243, p.err));
    // merge: both groups always reach this barrier (id 1 + quarter, the two
    // warps of this lane quarter), which also ANDs their status
    red[b * 128 + r] = m_run;
    bool merge = named_bar_and(1 + quarter, 64, ok);
    // the other group's last PV has completed too (it waited for it before
    // the barrier; its barrier has no later phase, so this returns at once)
    if (merge)
      merge = __all_sync(0xffffffffu, bounded_wait(&pv_done[b ^ 1], (nkv - 1) & 1, abort_flag, 244, p.err));
    if (merge) {
      tc_fence_after();
      const float m_o = red[(b ^ 1) * 128 + r];
      const float m_self = m_run;
      const float m = fmaxf(m_self, m_o);
      const float a_self = (m_self == NEG_INF) ? 0.f : ex2((m_self - m) * c);
      const float a_o = (m_o == NEG_INF) ? 0.f : ex2((m_o - m) * c);
      const uint32_t tOo = tmem + C::COL_O + (b ^ 1) * C::OW;
      // row sums from the extra columns of both O's
      uint32_t ls[16], lo[16];
      tmem_ld16_nw(tOb + lane_off + D, ls);
      tmem_ld16_nw(tOo + lane_off + D, lo);
      tmem_wait_ld(ls);
      tmem_wait_ld(lo);
      const float l = __uint_as_float(ls[0]) * a_self + __uint_as_float(lo[0]) * a_o;
      const float inv_l = 1.f / l;
      const float w_self = a_self * inv_l, w_o = a_o * inv_l;
      // each group writes half of the row's 16-column chunks
      constexpr int NC = D / 16;
      constexpr int NC0 = (NC + 1) / 2;
      const int cbeg = b == 0 ? 0 : NC0, cend = b == 0 ? NC0 : NC;
      const bool valid = qpos < p.s;
      __nv_bfloat16* orow = p.o + ((long long)bi * p.s + qpos - p.o_row0) * p.ld_o + p.o_col + (long long)out_head(p, n) * D;
      for (int cc = cbeg; cc < cend; ++cc) {
        uint32_t vs[16], vo[16];
        tmem_ld16_nw(tOb + lane_off + cc * 16, vs);
        tmem_ld16_nw(tOo + lane_off + cc * 16, vo);
        tmem_wait_ld(vs);
        tmem_wait_ld(vo);
        uint32_t vm[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          vm[k] = __float_as_uint(__uint_as_float(vs[k]) * w_self + __uint_as_float(vo[k]) * w_o);
        if (valid) store_row16(orow + cc * 16, vm, 1.f);
      }
      // every row of the padded tile gets a finite value (rows past s see the
      // zero-filled query), so the backward pass never reads garbage
      if (b == 0 && p.lse)
        p.lse[((long long)bi * p.H_total + p.lse_head0 + out_head(p, n)) * p.s_pad + qpos] = m * p.scale + logf(l);
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
int launch_fwd_sk(AttnFwdParams& prm, int grid, cudaStream_t st) {
  constexpr int SMEM = FwdSkCfg<D>::SMEM;
  static_assert(SMEM <= 232448, "attention forward tile set exceeds shared memory");
  static std::atomic<uint64_t> attr{0};  // devices whose limit is set
  if (smem_limit_once(reinterpret_cast<const void*>(attn_fwd_sk_kernel<D>), SMEM, &attr)) return 3;
  attn_fwd_sk_kernel<D><<<grid, 352, SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

template <int D>
int launch_fwd(AttnFwdParams& prm, int grid, cudaStream_t st) {
  constexpr int SMEM = FwdCfg<D>::SMEM;
  static_assert(SMEM <= 232448, "attention forward tile set exceeds shared memory");
  static std::atomic<uint64_t> attr{0};  // devices whose limit is set
  if (smem_limit_once(reinterpret_cast<const void*>(attn_fwd_kernel<D>), SMEM, &attr)) return 3;
  attn_fwd_kernel<D><<<grid, 192, SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

int make_attn_map(CUtensorMap* map, const void* qkv, int b, int s, int64_t ld, int d);

int attention_fwd(const AttnShape& sh, const void* qkv, void* o, float* lse, cudaStream_t st) {
  if (sh.q_end <= sh.q_begin) return 0;
  AttnFwdParams prm;
  memset(&prm, 0, sizeof(prm));
  if (make_attn_map(&prm.map_qkv, qkv, sh.b, sh.s, sh.ld_qkv, sh.d)) return 1;
  prm.s = sh.s;
  prm.s_pad = (sh.s + 127) / 128 * 128;
  prm.H = sh.H;
  prm.G = sh.H / sh.Hkv;
  prm.causal = sh.causal;
  prm.q_col = (int)sh.q_col;
  prm.k_col = (int)sh.k_col;
  prm.v_col = (int)sh.v_col;
  prm.o = reinterpret_cast<__nv_bfloat16*>(o);
  prm.ld_o = sh.ld_o;
  prm.o_row0 = sh.o_row0;
  prm.o_col = (int)sh.o_col;
  prm.lse = lse;
  prm.H_total = sh.H_total;
  prm.lse_head0 = sh.lse_head0;
  prm.o_seg = sh.o_seg > 0 ? sh.o_seg : sh.H;
  prm.o_seg_stride = sh.o_seg > 0 ? sh.o_seg_stride : sh.H;
  prm.qt_begin = sh.q_begin / 128;
  prm.n_qt = (sh.q_end + 127) / 128 - prm.qt_begin;
  prm.b = sh.b;
  prm.scale = 1.f / sqrtf((float)sh.d);
  prm.scale_log2 = prm.scale * 1.4426950408889634f;
  prm.qkv = reinterpret_cast<const __nv_bfloat16*>(qkv);
  prm.ld_qkv = sh.ld_qkv;
  prm.err = device_error_word();
  if (!prm.err) return 3;
  const int grid = prm.n_qt * sh.H * sh.b;
  // algorithmic work: QK^T and PV over the unmasked (query, key) pairs
  const double q0 = sh.q_begin, q1 = std::min(sh.q_end, sh.s);
  const double pairs = sh.causal ? (q1 * (q1 + 1) - q0 * (q0 + 1)) / 2 : (q1 - q0) * sh.s;
  ProfScope prof(PROF_ATTN_FWD, 4.0 * sh.d * pairs * sh.H * sh.b, 0.0, st);
  switch (sh.d) {
    case 64: return launch_fwd_sk<64>(prm, grid, st);
    case 80: return launch_fwd_sk<80>(prm, grid, st);
    case 96: return launch_fwd<96>(prm, grid, st);
    case 112: return launch_fwd<112>(prm, grid, st);
    case 128: return launch_fwd<128>(prm, grid, st);
    default: return 5;
  }
}

}  // namespace bpt
