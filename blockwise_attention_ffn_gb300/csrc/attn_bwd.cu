// attn_bwd.cu -- attention backward with the probabilities rebuilt tile by
// tile from Q, K and the saved log-sum-exp (nothing of size s x s is stored).
//
// Gradient rules ("Training memory: model states, activations and
// checkpointing", section 2, the softmax and product rows): with
// S = Q K^T / sqrt(d), P = softmax(S) = exp(S - LSE), O = P V,
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D) with D = rowsum(dO * O)
//   (= rowsum(P * dP)),  dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d).
// The rebuild is what "Blockwise Parallel Transformer for Long Context Large
// Models", section 3.4, "Implementation Details (Figure 3)" describes as
// remat of each key/value block step in the backward pass.
//
// One CTA = one 128-row key/value tile j of one key/value head g; it loops
// over the G query heads of the group and, for each, over the query tiles
// i >= j (causal) or all i.  dK and dV accumulate in TMEM over the whole
// loop; each dQ_i tile is reduced into an fp32 accumulator in global memory
// with bulk asynchronous reductions.
//   warp 0      TMA: K_j, V_j once; Q_i, dO_i, LSE_i, D_i per step
//   warp 1      MMA issuer: S^T = K Q^T, dP^T = V dO^T, dV += P^T dO,
//               dK += dS^T Q, dQ = dS K
//   warps 2..5  one key/value row per thread: P^T and dS^T (bf16) into
//               shared memory; drain dQ (one query row per thread)
#include <math.h>
#include <string.h>

#include "attn_common.cuh"
#include "internal.h"

namespace bpt {

namespace {

struct AttnBwdParams {
  CUtensorMap map_qkv;  // 3-D {ld_qkv, s, b}, box {CW, 128, 1}
  CUtensorMap map_do;   // 3-D {ld_do, s, b}, box {CW, 128, 1}
  int s, s_pad, H, Hkv, G, causal, b;
  int q_col, k_col, v_col, do_col;
  const float* lse;     // [b, H_total, s_pad] at head offset lse_head0
  const float* Dsum;    // [b, H, s_pad]
  int H_total, lse_head0;
  float* dq_acc;        // [b*s, H*d] fp32
  __nv_bfloat16* dqkv;
  long long ld_dqkv;
  int dk_col, dv_col;
  float scale, scale_log2;
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
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <int D>
struct BwdCfg {
  using T = TileGeom<D>;
  static constexpr int QS = (D >= 112) ? 1 : 2;
  static constexpr bool DQ_SEP = (256 + 3 * D) <= 512;  // dQ has its own TMEM columns
  static constexpr int STAGE = 2 * T::TILE + 2 * 512;  // Q, dO, LSE, D
  static constexpr int SMEM = 2 * T::TILE + QS * STAGE + 2 * SqTile::BYTES + 1024 + 256;
};

template <int D>
__global__ void __launch_bounds__(192, 1) attn_bwd_kernel(const __grid_constant__ AttnBwdParams p) {
  using T = TileGeom<D>;
  constexpr int QS = BwdCfg<D>::QS;
  constexpr bool DQ_SEP = BwdCfg<D>::DQ_SEP;
  constexpr int STAGE = BwdCfg<D>::STAGE;
  constexpr uint32_t ID_SQ = idesc_bf16(128, 128, false, false);  // S^T, dP^T
  constexpr uint32_t ID_KV = idesc_bf16(128, D, false, true);     // dV, dK
  constexpr uint32_t ID_DQ = idesc_bf16(128, D, true, true);      // dQ

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + T::TILE;
  uint8_t* sStage = sV + T::TILE;
  uint8_t* sP = sStage + QS * STAGE;       // P^T tile, then dS^T tile; both reused for dQ staging
  uint8_t* sDS = sP + SqTile::BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sDS + SqTile::BYTES);
  uint64_t* kv_full = bars;
  uint64_t* qdo_full = bars + 1;
  uint64_t* qdo_empty = qdo_full + QS;
  uint64_t* s_full = qdo_empty + QS;
  uint64_t* s_free = s_full + 1;
  uint64_t* dp_full = s_free + 1;
  uint64_t* dp_free = dp_full + 1;
  uint64_t* p_full = dp_free + 1;
  uint64_t* ds_full = p_full + 1;
  uint64_t* dq_full = ds_full + 1;
  uint64_t* dq_free = dq_full + 1;
  uint64_t* grp = dq_free + 1;  // compute-warp group barrier
  uint64_t* drain = grp + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  const int hb = p.Hkv * p.b;
  const int j = blockIdx.x / hb;
  const int g = (blockIdx.x % hb) % p.Hkv;
  const int bi = (blockIdx.x % hb) / p.Hkv;
  const int nq_total = (p.s + 127) / 128;
  const int i0 = p.causal ? j : 0;
  const int n_i = nq_total - i0;
  const int T_iter = p.G * n_i;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < QS; ++i) {
      mbar_init(&qdo_full[i], 1);
      mbar_init(&qdo_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 4);
    mbar_init(p_full, 4);
    mbar_init(ds_full, 4);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);
    mbar_init(grp, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&p.map_qkv);
    tma_prefetch(&p.map_do);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem;               // S^T, 128 columns
  const uint32_t tdP = tmem + 128;        // dP^T, 128 columns
  const uint32_t tdV = tmem + 256;        // D columns
  const uint32_t tdK = tmem + 256 + D;    // D columns
  const uint32_t tdQ = DQ_SEP ? tmem + 256 + 2 * D : tmem;  // D columns

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      mbar_expect_tx(kv_full, 2 * T::TILE);
#pragma unroll
      for (int c = 0; c < T::NCH; ++c) {
        tma_load_3d(sK + c * T::CHUNK, &p.map_qkv, kv_full, p.k_col + g * D + c * T::CW, j * 128, bi);
        tma_load_3d(sV + c * T::CHUNK, &p.map_qkv, kv_full, p.v_col + g * D + c * T::CW, j * 128, bi);
      }
      int issued = 0;
      for (int t = 0; t < T_iter; ++t) {
        const int st = t % QS;
        if (t >= QS && !bounded_wait(&qdo_empty[st], ((t / QS) & 1) ^ 1, abort_flag, 301, p.err)) break;
        const int hn = g * p.G + t / n_i;
        const int i = i0 + t % n_i;
        uint8_t* sQ = sStage + st * STAGE;
        uint8_t* sdO = sQ + T::TILE;
        uint8_t* sL = sdO + T::TILE;
        mbar_expect_tx(&qdo_full[st], STAGE);
#pragma unroll
        for (int c = 0; c < T::NCH; ++c) {
          tma_load_3d(sQ + c * T::CHUNK, &p.map_qkv, &qdo_full[st], p.q_col + hn * D + c * T::CW, i * 128, bi);
          tma_load_3d(sdO + c * T::CHUNK, &p.map_do, &qdo_full[st], p.do_col + hn * D + c * T::CW, i * 128, bi);
        }
        bulk_load(sL, p.lse + ((long long)bi * p.H_total + p.lse_head0 + hn) * p.s_pad + i * 128, 512,
                  &qdo_full[st]);
        bulk_load(sL + 512, p.Dsum + ((long long)bi * p.H + hn) * p.s_pad + i * 128, 512, &qdo_full[st]);
        issued = t + 1;
      }
      if (*abort_flag) {
        bounded_wait(kv_full, 0, abort_flag, 302, p.err);
        for (int t = (issued > QS ? issued - QS : 0); t < issued; ++t)
          mbar_try_wait(&qdo_full[t % QS], (t / QS) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t uK = smem_u32(sK), uV = smem_u32(sV);
      const uint32_t uP = smem_u32(sP), uDS = smem_u32(sDS);
      bool ok = bounded_wait(kv_full, 0, abort_flag, 311, p.err);
      for (int t = 0; ok && t < T_iter; ++t) {
        const int st = t % QS;
        const uint32_t uQ = smem_u32(sStage + st * STAGE);
        const uint32_t udO = uQ + T::TILE;
        if (!bounded_wait(&qdo_full[st], (t / QS) & 1, abort_flag, 312, p.err)) { ok = false; break; }
        if (t >= 1) {
          if (DQ_SEP) {
            if (!bounded_wait(s_free, (t - 1) & 1, abort_flag, 313, p.err)) { ok = false; break; }
          } else {
            if (!bounded_wait(dq_free, (t - 1) & 1, abort_flag, 314, p.err)) { ok = false; break; }
          }
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) umma_bf16(tS, T::kmajor(uK, kk), T::kmajor(uQ, kk), ID_SQ, kk > 0);
        umma_commit(s_full);
        if (t >= 1 && !bounded_wait(dp_free, (t - 1) & 1, abort_flag, 315, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) umma_bf16(tdP, T::kmajor(uV, kk), T::kmajor(udO, kk), ID_SQ, kk > 0);
        umma_commit(dp_full);
        // dV += P^T dO
        if (!bounded_wait(p_full, t & 1, abort_flag, 316, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tdV, SqTile::kmajor(uP, kk), T::mnmajor(udO, kk), ID_KV, (t > 0 || kk > 0));
        // dK += dS^T Q
        if (!bounded_wait(ds_full, t & 1, abort_flag, 317, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tdK, SqTile::kmajor(uDS, kk), T::mnmajor(uQ, kk), ID_KV, (t > 0 || kk > 0));
        umma_commit(&qdo_empty[st]);
        // dQ = dS K  (the S^T columns are free: the compute warps read S^T
        // before they published dS^T)
        if (DQ_SEP && t >= 1 && !bounded_wait(dq_free, (t - 1) & 1, abort_flag, 318, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tdQ, SqTile::mnmajor(uDS, kk), T::mnmajor(uK, kk), ID_DQ, kk > 0);
        umma_commit(dq_full);
      }
      if (!ok) {
        umma_commit(drain);
        bounded_wait(drain, 0, abort_flag, 319, p.err);
      }
    }
  } else {
    // ------------------------------------------------ compute (warps 2..5)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int kvp = j * 128 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float c = p.scale_log2;
    const float LOG2E = 1.4426950408889634f;
    bool ok = true;
    for (int t = 0; t < T_iter; ++t) {
      const int st = t % QS;
      const int hn = g * p.G + t / n_i;
      const int i = i0 + t % n_i;
      const int q0 = i * 128;
      const float* sL = reinterpret_cast<const float*>(sStage + st * STAGE + 2 * T::TILE);
      const float* sDsum = sL + 128;
      ok = bounded_wait(&qdo_full[st], (t / QS) & 1, abort_flag, 321, p.err) &&
           bounded_wait(s_full, t & 1, abort_flag, 322, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float pv[128];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t rr[32];
        tmem_ld32(tS + lane_off + q4 * 32, rr);
#pragma unroll
        for (int k = 0; k < 32; ++k) pv[q4 * 32 + k] = __uint_as_float(rr[k]);
      }
      tc_fence_before();
      __syncwarp();
      if (DQ_SEP && lane == 0) mbar_arrive(s_free);
      const bool edge = (p.causal && kvp > q0) || (q0 + 128 > p.s) || (kvp >= p.s);
#pragma unroll
      for (int k = 0; k < 128; ++k) {
        float e = ex2(fmaf(pv[k], c, -sL[k] * LOG2E));
        if (edge) {
          const int qp = q0 + k;
          if (qp >= p.s || kvp >= p.s || (p.causal && kvp > qp)) e = 0.f;
        }
        pv[k] = e;
      }
      // the previous step's dQ bulk reductions must have finished reading the
      // staging area (it overlaps the P^T / dS^T tiles)
      bulk_wait_read0();
      __syncwarp();
      if (lane == 0) mbar_arrive(grp);
      ok = bounded_wait(grp, t & 1, abort_flag, 325, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        uint4 u;
        u.x = pack_bf16(pv[ch * 8 + 0], pv[ch * 8 + 1]);
        u.y = pack_bf16(pv[ch * 8 + 2], pv[ch * 8 + 3]);
        u.z = pack_bf16(pv[ch * 8 + 4], pv[ch * 8 + 5]);
        u.w = pack_bf16(pv[ch * 8 + 6], pv[ch * 8 + 7]);
        *reinterpret_cast<uint4*>(sP + SqTile::off(r, ch)) = u;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);

      ok = bounded_wait(dp_full, t & 1, abort_flag, 323, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t rr[32];
        tmem_ld32(tdP + lane_off + q4 * 32, rr);
#pragma unroll
        for (int k = 0; k < 32; ++k) pv[q4 * 32 + k] *= (__uint_as_float(rr[k]) - sDsum[q4 * 32 + k]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dp_free);
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        uint4 u;
        u.x = pack_bf16(pv[ch * 8 + 0], pv[ch * 8 + 1]);
        u.y = pack_bf16(pv[ch * 8 + 2], pv[ch * 8 + 3]);
        u.z = pack_bf16(pv[ch * 8 + 4], pv[ch * 8 + 5]);
        u.w = pack_bf16(pv[ch * 8 + 6], pv[ch * 8 + 7]);
        *reinterpret_cast<uint4*>(sDS + SqTile::off(r, ch)) = u;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);

      // drain dQ_i: TMEM lane r is query row q0 + r
      ok = bounded_wait(dq_full, t & 1, abort_flag, 324, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float* stage = reinterpret_cast<float*>(sP) + r * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 16; ++cc) {
        uint32_t rr[16];
        tmem_ld16(tdQ + lane_off + cc * 16, rr);
        float4* dst = reinterpret_cast<float4*>(stage + cc * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_float4(__uint_as_float(rr[4 * k]), __uint_as_float(rr[4 * k + 1]),
                               __uint_as_float(rr[4 * k + 2]), __uint_as_float(rr[4 * k + 3]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      fence_proxy_async_smem();
      if (q0 + r < p.s) {
        float* gdst = p.dq_acc + ((long long)bi * p.s + q0 + r) * ((long long)p.H * D) + (long long)hn * D;
        bulk_reduce_add_f32(gdst, stage, D * 4);
      }
      bulk_commit();
    }
    bulk_wait0();
    if (ok) {
      // dV and dK of this key/value tile: every MMA completed before the last
      // dq_full phase
      tc_fence_after();
      // the TMEM loads are warp-collective: every lane issues them, only the
      // stores depend on the row being inside the sequence
      const bool valid = kvp < p.s;
      __nv_bfloat16* vrow = p.dqkv + ((long long)bi * p.s + kvp) * p.ld_dqkv + p.dv_col + (long long)g * D;
      __nv_bfloat16* krow = p.dqkv + ((long long)bi * p.s + kvp) * p.ld_dqkv + p.dk_col + (long long)g * D;
      const float sc = p.scale;
#pragma unroll 1
      for (int cc = 0; cc < D / 16; ++cc) {
        uint32_t rv[16], rk[16];
        tmem_ld16(tdV + lane_off + cc * 16, rv);
        tmem_ld16(tdK + lane_off + cc * 16, rk);
        if (valid) {
          uint4 v0, v1, k0, k1;
          v0.x = pack_bf16(__uint_as_float(rv[0]), __uint_as_float(rv[1]));
          v0.y = pack_bf16(__uint_as_float(rv[2]), __uint_as_float(rv[3]));
          v0.z = pack_bf16(__uint_as_float(rv[4]), __uint_as_float(rv[5]));
          v0.w = pack_bf16(__uint_as_float(rv[6]), __uint_as_float(rv[7]));
          v1.x = pack_bf16(__uint_as_float(rv[8]), __uint_as_float(rv[9]));
          v1.y = pack_bf16(__uint_as_float(rv[10]), __uint_as_float(rv[11]));
          v1.z = pack_bf16(__uint_as_float(rv[12]), __uint_as_float(rv[13]));
          v1.w = pack_bf16(__uint_as_float(rv[14]), __uint_as_float(rv[15]));
          k0.x = pack_bf16(__uint_as_float(rk[0]) * sc, __uint_as_float(rk[1]) * sc);
          k0.y = pack_bf16(__uint_as_float(rk[2]) * sc, __uint_as_float(rk[3]) * sc);
          k0.z = pack_bf16(__uint_as_float(rk[4]) * sc, __uint_as_float(rk[5]) * sc);
          k0.w = pack_bf16(__uint_as_float(rk[6]) * sc, __uint_as_float(rk[7]) * sc);
          k1.x = pack_bf16(__uint_as_float(rk[8]) * sc, __uint_as_float(rk[9]) * sc);
          k1.y = pack_bf16(__uint_as_float(rk[10]) * sc, __uint_as_float(rk[11]) * sc);
          k1.z = pack_bf16(__uint_as_float(rk[12]) * sc, __uint_as_float(rk[13]) * sc);
          k1.w = pack_bf16(__uint_as_float(rk[14]) * sc, __uint_as_float(rk[15]) * sc);
          reinterpret_cast<uint4*>(vrow + cc * 16)[0] = v0;
          reinterpret_cast<uint4*>(vrow + cc * 16)[1] = v1;
          reinterpret_cast<uint4*>(krow + cc * 16)[0] = k0;
          reinterpret_cast<uint4*>(krow + cc * 16)[1] = k1;
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

template <int D>
int launch_bwd(AttnBwdParams& prm, int grid, cudaStream_t st) {
  constexpr int SMEM = BwdCfg<D>::SMEM;
  static_assert(SMEM <= 232448, "attention backward tile set exceeds shared memory");
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess)
      return 3;
    attr = true;
  }
  attn_bwd_kernel<D><<<grid, 192, SMEM, st>>>(prm);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

int make_attn_map(CUtensorMap* map, const void* qkv, int b, int s, int64_t ld, int d);
int attn_dsum(const AttnBwdShape& sh, const void* o, const void* dout, float* Dsum, int s_pad,
              cudaStream_t st);

size_t attention_bwd_ws_bytes(const AttnBwdShape& sh) {
  const int64_t s_pad = ((int64_t)sh.f.s + 127) / 128 * 128;
  const size_t dq = (size_t)sh.f.b * sh.f.s * sh.f.H * sh.f.d * 4;
  const size_t dsum = (size_t)sh.f.b * sh.f.H * s_pad * 4;
  return ((dq + 255) / 256) * 256 + dsum;
}

// lse: [b, H_total, s_pad] fp32 (head offset lse_head0)
int attention_bwd(const AttnBwdShape& sh, const void* qkv, const void* o, const float* lse,
                  const void* dout, void* dqkv, void* ws, cudaStream_t st) {
  const AttnShape& f = sh.f;
  const int s_pad = (f.s + 127) / 128 * 128;
  const size_t dq_bytes = (size_t)f.b * f.s * f.H * f.d * 4;
  float* dq_acc = reinterpret_cast<float*>(ws);
  float* Dsum = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + ((dq_bytes + 255) / 256) * 256);
  int rc;
  {
    ProfScope prof(PROF_MISC, 0.0, (double)dq_bytes + 4.0 * f.b * f.s * f.H * f.d + 4.0 * f.b * f.H * s_pad, st);
    if (cudaMemsetAsync(dq_acc, 0, dq_bytes, st) != cudaSuccess) return 3;
    rc = attn_dsum(sh, o, dout, Dsum, s_pad, st);
    if (rc) return rc;
  }

  AttnBwdParams prm;
  memset(&prm, 0, sizeof(prm));
  if (make_attn_map(&prm.map_qkv, qkv, f.b, f.s, f.ld_qkv, f.d)) return 1;
  if (make_attn_map(&prm.map_do, dout, f.b, f.s, sh.ld_do, f.d)) return 1;
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
  prm.H_total = f.H_total;
  prm.lse_head0 = f.lse_head0;
  prm.dq_acc = dq_acc;
  prm.dqkv = reinterpret_cast<__nv_bfloat16*>(dqkv);
  prm.ld_dqkv = sh.ld_dqkv;
  prm.dk_col = (int)sh.dk_col;
  prm.dv_col = (int)sh.dv_col;
  prm.scale = 1.f / sqrtf((float)f.d);
  prm.scale_log2 = prm.scale * 1.4426950408889634f;
  prm.err = device_error_word();
  if (!prm.err) return 3;
  const int grid = ((f.s + 127) / 128) * f.Hkv * f.b;
  {
  // algorithmic work: S, dP, dV, dK, dQ over the unmasked (query, key) pairs
  const double pairs = f.causal ? (double)f.s * (f.s + 1) / 2 : (double)f.s * f.s;
  ProfScope prof(PROF_ATTN_BWD, 10.0 * f.d * pairs * f.H * f.b, 0.0, st);
  switch (f.d) {
    case 64: rc = launch_bwd<64>(prm, grid, st); break;
    case 80: rc = launch_bwd<80>(prm, grid, st); break;
    case 96: rc = launch_bwd<96>(prm, grid, st); break;
    case 112: rc = launch_bwd<112>(prm, grid, st); break;
    case 128: rc = launch_bwd<128>(prm, grid, st); break;
    default: return 5;
  }
  }
  if (rc) return rc;
  // dQ = scale * accumulated dS K, into the bf16 gradient buffer
  ProfScope prof(PROF_MISC, 0.0, 6.0 * f.b * f.s * f.H * f.d, st);
  return f32_to_bf16((int64_t)f.b * f.s, (int64_t)f.H * f.d, dq_acc, (int64_t)f.H * f.d,
                     reinterpret_cast<__nv_bfloat16*>(dqkv) + sh.dq_col, sh.ld_dqkv, prm.scale, st);
}

}  // namespace bpt
