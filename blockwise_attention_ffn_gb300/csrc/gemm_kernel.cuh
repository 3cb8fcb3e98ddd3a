// gemm_kernel.cuh -- the tcgen05 GEMM behind gemm() (gemm_tc.cu), with fused
// epilogues for the layer's dense contractions: the Q/K/V and output
// projections, the FFN's fc1 (GeLU or the SwiGLU gate/up pair) and fc2, every
// backward product (activation gradients and fp32 weight gradients) and the
// language-model loss's vocabulary products.
//
// Persistent: each CTA (or pair of CTAs) walks tiles of C.  Warp roles:
//   warp 0      TMA producer: K-tiles of A and B into a smem ring
//   warp 1      TMEM owner and MMA issuer (K = 16 per product): the warp runs
//               the loop, one elected lane issues into one of two
//               256-column accumulators
//   warps 2..9  epilogue: TMEM -> registers (one row per thread, half the
//               columns per warp) -> fused bias / residual / activation ->
//               global, overlapped with the next tile's main loop
// Two forms share this code:
//   one SM (PAIR = false): a 128 x BN tile per CTA, 4 ring stages of 48 KB;
//   a pair of SMs (PAIR = true): a 256 x BN tile per cluster of two CTAs and
//     one product over both (cta_group::2, M = 256).  Each CTA stages its 128
//     rows of A and half of B's BN rows, holds its 128 rows of the
//     accumulator and runs their epilogue; rank 0 waits for both CTAs' loads
//     and issues.  Per 128 x BN x 16 of output an SM's shared memory then
//     feeds 8 KB to the tensor core instead of 12, and a stage is 32 KB, so
//     the ring holds 6.
// Operands are staged with 128-byte swizzle; K-major tiles are [rows x 64]
// boxes, MN-major tiles are [64 K-rows x 64] boxes side by side.
// Work units are tiles, or tiles x K ranges for fp32 weight gradients whose
// whole tiles would leave most of the last wave of SMs idle (each range adds
// its share in L2).  The epilogue moves whole 32-byte sectors per thread
// where every operand allows it.
#pragma once

#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace bpt {
namespace gk {

constexpr int BM = 128;  // rows of A (and of the accumulator) per CTA
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
// ring stages: 48 KB each for one SM (A and 256 rows of B), 32 KB each for
// a pair (A and 128 rows of B per CTA)
template <bool PAIR>
constexpr int stages() {
  return PAIR ? 6 : 4;
}
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;

struct GemmParams {
  CUtensorMap mapA;
  CUtensorMap mapB[3];
  int M, N, K;
  int nkt;          // number of BK tiles of K
  int seg_kt[3];    // first k-tile of segments 1 and 2 (large if absent)
  int epi, act;
  void* out;
  long long ldo;
  void* out2;
  long long ldo2;
  void* out3;
  long long ldo3;
  const __nv_bfloat16* bias;
  const void* res;
  long long ldr;
  int res_f32;
  const __nv_bfloat16* aux;
  long long ldaux;
  const __nv_bfloat16* aux2;
  long long ldaux2;
  float beta;
  int mt, nt, ntiles;  // tile grid; ntiles counts work units (tiles x ksplit)
  int m_fast;          // walk tiles along M first
  int group;           // > 0: bands of `group` tile rows (group_m) or tile
  int group_m;         //      columns, each walked whole before the next
  int ksplit;          // K ranges per tile (> 1: EPI_F32 added atomically)
  int vec32;           // every epilogue operand allows 32-byte accesses
  const float* rowf;   // loss epilogues: per-row log-sum-exp
  const int* rowi;     // loss epilogues: per-row target id
  float scale;
  long long col0;      // vocabulary id of column 0
  unsigned int* err;
};

// Phi(z) = 0.5 (1 + erf(z / sqrt 2)) and e = exp(-z^2 / 2) for the erf GeLU,
// with erf from Abramowitz & Stegun, "Handbook of Mathematical Functions",
// formula 7.1.26: erf(x) = 1 - (a1 t + a2 t^2 + ... + a5 t^5) exp(-x^2),
// t = 1 / (1 + p x), x >= 0, absolute error at most 1.5e-7 (far below the
// bf16 outputs' rounding).  exp(-x^2) at x = z / sqrt 2 is the same e the
// derivative needs, so both come from one exp2 and one reciprocal.
__device__ __forceinline__ void gelu_erf_parts(float z, float& cdf, float& e) {
  const float x = fabsf(z) * 0.70710678118654752f;
  float t;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, x, 1.f)));
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  poly *= t;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-0.72134752044448170f * z * z));  // exp(-z^2/2)
  const float tail = 0.5f * poly * e;  // 0.5 (1 - erf(|x|))
  cdf = z >= 0.f ? 1.f - tail : tail;
}
__device__ __forceinline__ float gelu_f(float z, int act) {
  if (act == 0) {
    float cdf, e;
    gelu_erf_parts(z, cdf, e);
    return z * cdf;
  }
  const float c = 0.7978845608028654f;
  return 0.5f * z * (1.f + tanhf(c * (z + 0.044715f * z * z * z)));
}
// gelu(z) and gelu'(z) sharing the erf (or tanh)
__device__ __forceinline__ void gelu_and_grad_f(float z, int act, float& g, float& d) {
  if (act == 0) {
    float cdf, e;
    gelu_erf_parts(z, cdf, e);
    g = z * cdf;
    d = fmaf(z * e, 0.3989422804014327f, cdf);  // Phi(z) + z phi(z)
  } else {
    const float c = 0.7978845608028654f;
    const float t = tanhf(c * (z + 0.044715f * z * z * z));
    g = 0.5f * z * (1.f + t);
    d = 0.5f * (1.f + t) + 0.5f * z * (1.f - t * t) * c * (1.f + 3.f * 0.044715f * z * z);
  }
}
__device__ __forceinline__ float sigmoid_f(float z) { return 1.f / (1.f + expf(-z)); }

// W consecutive values (W = 8: 16-byte accesses; W = 16 or 32: 32-byte
// accesses, a whole sector per thread, for the epilogue's one-row-per-thread
// pattern)
__device__ __forceinline__ void ld32B(const void* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}
__device__ __forceinline__ void st32B(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
template <int W>
__device__ __forceinline__ void loadw_bf16(const __nv_bfloat16* p, float (&v)[W]) {
  if constexpr (W == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_lo(w[i]);
      v[2 * i + 1] = bf16_hi(w[i]);
    }
  } else {
    // W = 16 or 32: every 32-byte piece loaded before any is used
    uint32_t w[W / 16][8];
#pragma unroll
    for (int h = 0; h < W / 16; ++h) ld32B(p + 16 * h, w[h]);
#pragma unroll
    for (int h = 0; h < W / 16; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[16 * h + 2 * i] = bf16_lo(w[h][i]);
        v[16 * h + 2 * i + 1] = bf16_hi(w[h][i]);
      }
  }
}
template <int W>
__device__ __forceinline__ void storew_bf16(__nv_bfloat16* p, const float (&v)[W]) {
  if constexpr (W == 8) {
    uint4 u;
    u.x = pack_bf16(v[0], v[1]);
    u.y = pack_bf16(v[2], v[3]);
    u.z = pack_bf16(v[4], v[5]);
    u.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
  } else {
#pragma unroll
    for (int h = 0; h < W / 16; ++h) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = pack_bf16(v[16 * h + 2 * i], v[16 * h + 2 * i + 1]);
      st32B(p + 16 * h, w);
    }
  }
}
template <int W>
__device__ __forceinline__ void loadw_f32(const float* p, float (&v)[W]) {
  uint32_t w[W / 8][8];
#pragma unroll
  for (int h = 0; h < W / 8; ++h) {
    if constexpr (W == 8) {
      const float4 a = reinterpret_cast<const float4*>(p)[0];
      const float4 b = reinterpret_cast<const float4*>(p)[1];
      w[h][0] = __float_as_uint(a.x); w[h][1] = __float_as_uint(a.y);
      w[h][2] = __float_as_uint(a.z); w[h][3] = __float_as_uint(a.w);
      w[h][4] = __float_as_uint(b.x); w[h][5] = __float_as_uint(b.y);
      w[h][6] = __float_as_uint(b.z); w[h][7] = __float_as_uint(b.w);
    } else {
      ld32B(p + 8 * h, w[h]);
    }
  }
#pragma unroll
  for (int h = 0; h < W / 8; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * h + i] = __uint_as_float(w[h][i]);
}
template <int W>
__device__ __forceinline__ void storew_f32(float* p, const float (&v)[W]) {
#pragma unroll
  for (int h = 0; h < W / 8; ++h) {
    if constexpr (W == 8) {
      reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(v[8 * h + i]);
      st32B(p + 8 * h, w);
    }
  }
}

template <int W>
__device__ __forceinline__ void loadw_res(const GemmParams& p, int m, int n, float (&v)[W]) {
  if (p.res_f32)
    loadw_f32<W>(reinterpret_cast<const float*>(p.res) + (long long)m * p.ldr + n, v);
  else
    loadw_bf16<W>(reinterpret_cast<const __nv_bfloat16*>(p.res) + (long long)m * p.ldr + n, v);
}
__device__ __forceinline__ float load1_res(const GemmParams& p, int m, int n) {
  const long long i = (long long)m * p.ldr + n;
  return p.res_f32 ? reinterpret_cast<const float*>(p.res)[i]
                   : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.res)[i]);
}

// Applies the epilogue to W consecutive columns n..n+W-1 of row m (all in
// range) given the accumulators a (and a second accumulator b for the dual
// kinds).
template <int W>
__device__ __forceinline__ void epiw(const GemmParams& p, int m, int n, const float (&a)[W],
                                     const float (&b)[W]) {
  float v[W];
  switch (p.epi) {
    case EPI_BF16: {
#pragma unroll
      for (int j = 0; j < W; ++j) v[j] = a[j];
      if (p.bias) {
        float t[W];
        loadw_bf16<W>(p.bias + n, t);
#pragma unroll
        for (int j = 0; j < W; ++j) v[j] += t[j];
      }
      if (p.res) {
        float t[W];
        loadw_res<W>(p, m, n, t);
#pragma unroll
        for (int j = 0; j < W; ++j) v[j] += t[j];
      }
      storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out) + (long long)m * p.ldo + n, v);
      break;
    }
    case EPI_GELU: {
      float z[W];
#pragma unroll
      for (int j = 0; j < W; ++j) z[j] = a[j];
      if (p.bias) {
        float t[W];
        loadw_bf16<W>(p.bias + n, t);
#pragma unroll
        for (int j = 0; j < W; ++j) z[j] += t[j];
      }
      if (p.out2) {
        // out2 = gelu'(z), the factor the backward multiplies dA by
        float d[W];
#pragma unroll
        for (int j = 0; j < W; ++j) gelu_and_grad_f(z[j], p.act, v[j], d[j]);
        storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out) + (long long)m * p.ldo + n, v);
        storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out2) + (long long)m * p.ldo2 + n, d);
      } else {
#pragma unroll
        for (int j = 0; j < W; ++j) v[j] = gelu_f(z[j], p.act);
        storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out) + (long long)m * p.ldo + n, v);
      }
      break;
    }
    case EPI_SWIGLU: {
#pragma unroll
      for (int j = 0; j < W; ++j) v[j] = a[j] * sigmoid_f(a[j]) * b[j];
      storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out) + (long long)m * p.ldo + n, v);
      if (p.out2) storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out2) + (long long)m * p.ldo2 + n, a);
      if (p.out3) storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out3) + (long long)m * p.ldo3 + n, b);
      break;
    }
    case EPI_GELU_BWD: {
      float gd[W];
      loadw_bf16<W>(p.aux + (long long)m * p.ldaux + n, gd);
#pragma unroll
      for (int j = 0; j < W; ++j) v[j] = a[j] * gd[j];
      storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out) + (long long)m * p.ldo + n, v);
      break;
    }
    case EPI_SWIGLU_BWD: {
      float g[W], u[W], w2[W];
      loadw_bf16<W>(p.aux + (long long)m * p.ldaux + n, g);
      loadw_bf16<W>(p.aux2 + (long long)m * p.ldaux2 + n, u);
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const float sg = sigmoid_f(g[j]);
        v[j] = a[j] * u[j] * sg * (1.f + g[j] * (1.f - sg));
        w2[j] = a[j] * g[j] * sg;
      }
      storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out) + (long long)m * p.ldo + n, v);
      storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out2) + (long long)m * p.ldo2 + n, w2);
      break;
    }
    case EPI_CE_GRAD: {
      // (softmax - onehot) * scale from the logit and the row's log-sum-exp
      const float l2 = p.rowf[m] * 1.4426950408889634f;
      const long long t = (long long)p.rowi[m] - p.col0 - n;  // target column within the W
#pragma unroll
      for (int j = 0; j < W; ++j) {
        float e;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fmaf(a[j], 1.4426950408889634f, -l2)));
        v[j] = (e - (t == j ? 1.f : 0.f)) * p.scale;
      }
      storew_bf16<W>(reinterpret_cast<__nv_bfloat16*>(p.out) + (long long)m * p.ldo + n, v);
      break;
    }
    default: {  // EPI_F32
      float* o = reinterpret_cast<float*>(p.out) + (long long)m * p.ldo + n;
      float t[W];
#pragma unroll
      for (int j = 0; j < W; ++j) t[j] = a[j];
      if (p.bias) {
        float bb[W];
        loadw_bf16<W>(p.bias + n, bb);
#pragma unroll
        for (int j = 0; j < W; ++j) t[j] += bb[j];
      }
      if (p.res) {
        float rr[W];
        loadw_res<W>(p, m, n, rr);
#pragma unroll
        for (int j = 0; j < W; ++j) t[j] += rr[j];
      }
      if (p.ksplit > 1) {
        // one K range's share: added in L2 (the host zeroed out when beta = 0)
#pragma unroll
        for (int j = 0; j < W; j += 4) red_add_v4(o + j, t[j], t[j + 1], t[j + 2], t[j + 3]);
        break;
      }
      if (p.beta != 0.f) {
        float ov[W];
        loadw_f32<W>(o, ov);
#pragma unroll
        for (int j = 0; j < W; ++j) t[j] += p.beta * ov[j];
      }
      storew_f32<W>(o, t);
      break;
    }
  }
}

// Scalar version for the ragged N tail.
__device__ __forceinline__ void epi1(const GemmParams& p, int m, int n, float a, float b) {
  switch (p.epi) {
    case EPI_BF16: {
      float v = a;
      if (p.bias) v += __bfloat162float(p.bias[n]);
      if (p.res) v += load1_res(p, m, n);
      reinterpret_cast<__nv_bfloat16*>(p.out)[(long long)m * p.ldo + n] = __float2bfloat16(v);
      break;
    }
    case EPI_GELU: {
      float z = a + (p.bias ? __bfloat162float(p.bias[n]) : 0.f);
      float g, d;
      gelu_and_grad_f(z, p.act, g, d);
      reinterpret_cast<__nv_bfloat16*>(p.out)[(long long)m * p.ldo + n] = __float2bfloat16(g);
      if (p.out2)
        reinterpret_cast<__nv_bfloat16*>(p.out2)[(long long)m * p.ldo2 + n] = __float2bfloat16(d);
      break;
    }
    case EPI_SWIGLU: {
      reinterpret_cast<__nv_bfloat16*>(p.out)[(long long)m * p.ldo + n] =
          __float2bfloat16(a * sigmoid_f(a) * b);
      if (p.out2)
        reinterpret_cast<__nv_bfloat16*>(p.out2)[(long long)m * p.ldo2 + n] = __float2bfloat16(a);
      if (p.out3)
        reinterpret_cast<__nv_bfloat16*>(p.out3)[(long long)m * p.ldo3 + n] = __float2bfloat16(b);
      break;
    }
    case EPI_GELU_BWD: {
      const float gd = __bfloat162float(p.aux[(long long)m * p.ldaux + n]);
      reinterpret_cast<__nv_bfloat16*>(p.out)[(long long)m * p.ldo + n] = __float2bfloat16(a * gd);
      break;
    }
    case EPI_SWIGLU_BWD: {
      const float g = __bfloat162float(p.aux[(long long)m * p.ldaux + n]);
      const float u = __bfloat162float(p.aux2[(long long)m * p.ldaux2 + n]);
      const float sg = sigmoid_f(g);
      reinterpret_cast<__nv_bfloat16*>(p.out)[(long long)m * p.ldo + n] =
          __float2bfloat16(a * u * sg * (1.f + g * (1.f - sg)));
      reinterpret_cast<__nv_bfloat16*>(p.out2)[(long long)m * p.ldo2 + n] =
          __float2bfloat16(a * g * sg);
      break;
    }
    case EPI_CE_GRAD: {
      float e;
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fmaf(a, 1.4426950408889634f, -p.rowf[m] * 1.4426950408889634f)));
      const float v = (e - ((long long)p.rowi[m] == p.col0 + n ? 1.f : 0.f)) * p.scale;
      reinterpret_cast<__nv_bfloat16*>(p.out)[(long long)m * p.ldo + n] = __float2bfloat16(v);
      break;
    }
    default: {
      float* o = reinterpret_cast<float*>(p.out) + (long long)m * p.ldo + n;
      float v = a;
      if (p.bias) v += __bfloat162float(p.bias[n]);
      if (p.res) v += load1_res(p, m, n);
      if (p.ksplit > 1) {
        atomicAdd(o, v);
        break;
      }
      *o = v + (p.beta != 0.f ? p.beta * *o : 0.f);
      break;
    }
  }
}

// Tile origin of persistent work unit `unit` (tile = unit mod the tile count;
// with a split K, the K range is unit / tile count, so the CTAs in flight
// share a K range).  The walk runs fastest along the dimension of the smaller
// operand, so the CTAs in flight share that operand in L2 while the larger
// one streams through once.
__device__ __forceinline__ void k_range(const GemmParams& p, int unit, int& kb, int& ke) {
  const int ks = unit / (p.mt * p.nt);
  kb = (int)((long long)p.nkt * ks / p.ksplit);
  ke = (int)((long long)p.nkt * (ks + 1) / p.ksplit);
}

__device__ __forceinline__ void tile_origin(const GemmParams& p, int unit, int bm, int bn, int& m0, int& n0) {
  const int tile = unit % (p.mt * p.nt);
  int mb, nb;
  if (p.group > 0) {
    // a band of `group` tile rows (or columns) of the operand that would
    // otherwise be re-read stays in L2 while the band is walked across the
    // other dimension, its own dimension fastest; the other operand is read
    // once per band
    const int nmaj = p.group_m ? p.mt : p.nt;
    const int nmin = p.group_m ? p.nt : p.mt;
    const int g = tile / (p.group * nmin);
    const int r = tile - g * (p.group * nmin);
    const int gs = min(p.group, nmaj - g * p.group);
    const int a = g * p.group + r % gs, b = r / gs;
    mb = p.group_m ? a : b;
    nb = p.group_m ? b : a;
  } else if (p.m_fast) {
    mb = tile % p.mt;
    nb = tile / p.mt;
  } else {
    nb = tile % p.nt;
    mb = tile / p.nt;
  }
  m0 = mb * bm;
  n0 = nb * bn;
}

// Pairs of CTAs of `kernel` (one CTA per SM, `smem` bytes of dynamic shared
// memory) that the device holds at once, cached per device in fit[].
inline int pair_slots(const void* kernel, int smem, std::atomic<int>* fit) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int known = fit[dev].load(std::memory_order_acquire);
  if (known > 0) return known;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) return 0;
  fit[dev].store(n, std::memory_order_release);
  return n;
}

// The epilogue of one accumulator for one warp: this thread's row m of the
// tile starting at column n0, the half `half` of its BN columns, read from
// TMEM at tbase (the warp's lane quarter, the accumulator's first column).
template <int BN, bool DUAL>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t tbase, int m, int n0, int half) {
  constexpr int EPI_COLS = BN / 2;  // columns of one accumulator half per epilogue warp
  if (!DUAL && p.epi == EPI_LSE) {
    // this thread's row over its half of the tile: online max and sum of
    // exp over the valid columns, 32 at a time, and the target's logit
    float mx = -INFINITY, sm = 0.f;
    const int t = m < p.M ? p.rowi[m] - (int)p.col0 : -1;
#pragma unroll 1
    for (int c = 0; c < EPI_COLS / 32; ++c) {
      const int col = half * EPI_COLS + c * 32;
      const int nb = n0 + col;
      uint32_t ra[32];
      tmem_ld32(tbase + col, ra);
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (nb + j < p.N) cm = fmaxf(cm, __uint_as_float(ra[j]));
      if (cm > -INFINITY) {
        const float nm = fmaxf(mx, cm);
        const float nl2 = nm * 1.4426950408889634f;
        float e, part = 0.f;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fmaf(mx, 1.4426950408889634f, -nl2)));
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float x;
          asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(x) : "f"(fmaf(__uint_as_float(ra[j]), 1.4426950408889634f, -nl2)));
          part += nb + j < p.N ? x : 0.f;
        }
        sm = fmaf(sm, e, part);
        mx = nm;
      }
      if (m < p.M && t >= nb && t < nb + 32 && t < p.N) {
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (t - nb == j) z = __uint_as_float(ra[j]);
        reinterpret_cast<float*>(p.out2)[m] = z;
      }
    }
    if (m < p.M) {
      const long long part_idx = 2 * (long long)(n0 / BN) + half;
      reinterpret_cast<float2*>(p.out)[part_idx * p.ldo + m] = make_float2(mx, sm);
    }
    return;
  }
#pragma unroll 1
  for (int c = 0; c < EPI_COLS / 32; ++c) {
    const int col = half * EPI_COLS + c * 32;
    uint32_t ra[32], rb[32];
    tmem_ld32(tbase + col, ra);
    if (DUAL) tmem_ld32(tbase + BN + col, rb);
    if (m < p.M) {
      const int nb = n0 + col;
      if (nb + 32 <= p.N) {
        if (p.vec32) {
          // whole 32-byte sectors per access (the warp's 32 rows make 32
          // separate segments either way), and the chunk's inputs all
          // loaded before its first store
          float a32[32], b32[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            a32[j] = __uint_as_float(ra[j]);
            b32[j] = DUAL ? __uint_as_float(rb[j]) : 0.f;
          }
          epiw<32>(p, m, nb, a32, b32);
        } else {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            float a8[8], b8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              a8[j] = __uint_as_float(ra[g * 8 + j]);
              b8[j] = DUAL ? __uint_as_float(rb[g * 8 + j]) : 0.f;
            }
            epiw<8>(p, m, nb + g * 8, a8, b8);
          }
        }
      } else {
        // unrolled so the accumulators stay in registers
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (nb + j < p.N) epi1(p, m, nb + j, __uint_as_float(ra[j]), DUAL ? __uint_as_float(rb[j]) : 0.f);
      }
    }
  }
}

// BN: tile width (columns of C).  DUAL: BN columns of g and BN of u.
// PAIR: a 256-row tile per cluster of two CTAs (see the file comment).
// Persistent: each CTA (or pair) walks work units u0, u0 + units in flight,
// ... with two TMEM accumulators, so the epilogue of one tile overlaps the
// main loop of the next.
template <int BN, bool A_MN, bool B_MN, bool DUAL, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr int STAGES = stages<PAIR>();
  constexpr int BNS = PAIR ? BN / 2 : BN;  // rows of each B this CTA stages
  constexpr int B_BYTES = (DUAL ? 2 : 1) * BNS * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int ACC_COLS = (DUAL ? 2 : 1) * BN;
  static_assert(ACC_COLS == 256, "two accumulators must fill the 512 TMEM columns");
  constexpr uint32_t TMEM_COLS = 512;
  constexpr int TM = PAIR ? 2 * BM : BM;  // rows of C per tile
  constexpr uint32_t IDESC = idesc_bf16(TM, BN, A_MN, B_MN);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  // rank in the pair (0 issues); work units of this CTA (or pair)
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units_in_flight = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      // a pair's accumulator is drained by the epilogue warps of both CTAs
      mbar_init(&acc_empty[a], (PAIR ? 2 : 1) * NUM_EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&p.mapA);
    tma_prefetch(&p.mapB[0]);
    if (DUAL || p.seg_kt[0] < p.nkt) tma_prefetch(&p.mapB[1]);
    if (p.seg_kt[1] < p.nkt) tma_prefetch(&p.mapB[2]);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_holder, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  // a pair: the other CTA's barriers are initialised before anything of this
  // one can arrive on them
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ producer
      // a pair's loads (both CTAs') complete on rank 0's barriers, which
      // expect both CTAs' bytes
      const uint32_t full0 = PAIR ? cluster_addr(smem_u32(full), 0) : smem_u32(full);
      uint32_t it = 0;  // k-tiles issued, across this CTA's tiles
      bool ok = true;
      for (int unit = unit0; ok && unit < p.ntiles; unit += units_in_flight) {
        int m0, n0, kb, ke;
        tile_origin(p, unit, TM, BN, m0, n0);
        k_range(p, unit, kb, ke);
        const int ma = m0 + (int)rank * BM;    // this CTA's rows of A
        const int nbs = n0 + (int)rank * BNS;  // this CTA's rows of each B
        for (int kt = kb; kt < ke; ++kt) {
          const int s = it % STAGES;
          if (it >= STAGES && !bounded_wait(&empty[s], ((it / STAGES) & 1) ^ 1, abort_flag, 101, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          if (rank == 0) mbar_expect_tx(&full[s], (PAIR ? 2 : 1) * STAGE_BYTES);
          const uint32_t fb = full0 + 8u * (uint32_t)s;
          auto load = [&](void* dst, const CUtensorMap* map, int x, int y) {
            if constexpr (PAIR) tma_load_2d_pair(dst, map, fb, x, y);
            else tma_load_2d(dst, map, &full[s], x, y);
          };
          if (!A_MN) {
            load(sa, &p.mapA, kt * BK, ma);
          } else {
            load(sa, &p.mapA, ma, kt * BK);
            load(sa + 8192, &p.mapA, ma + 64, kt * BK);
          }
          if (DUAL) {
            load(sb, &p.mapB[0], kt * BK, nbs);
            load(sb + BNS * BK * 2, &p.mapB[1], kt * BK, nbs);
          } else {
            const int seg = (kt >= p.seg_kt[1]) ? 2 : (kt >= p.seg_kt[0]) ? 1 : 0;
            const int kl = (kt - (seg == 0 ? 0 : p.seg_kt[seg - 1])) * BK;
            if (!B_MN) {
              load(sb, &p.mapB[seg], kl, nbs);
            } else {
#pragma unroll
              for (int c = 0; c < BNS / 64; ++c) load(sb + c * 8192, &p.mapB[seg], nbs + c * 64, kl);
            }
          }
          ++it;
        }
      }
      if (*abort_flag) {
        // let every load issued land before the CTA goes away (a pair's
        // rank 1 waits at the final cluster barrier meanwhile)
        if (rank == 0)
          for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
            drain_wait(&full[j % STAGES], (j / STAGES) & 1);
        // a pair: the loads of rank 1 complete on rank 0's barriers, so
        // neither side can wait for the other's stragglers; both give them
        // a fixed 10^6 cycles (about half a millisecond) before the final
        // cluster barrier
        if (PAIR) {
          const long long t0 = clock64();
          while (clock64() - t0 < 1000000) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (rank == 0) {
      const uint32_t smem_base = smem_u32(smem);
      uint32_t it = 0;
      int tc = 0;  // tiles done by this CTA
      bool ok = true;
      for (int unit = unit0; unit < p.ntiles; unit += units_in_flight, ++tc) {
        const int acc = tc & 1;
        // the epilogue must have drained this accumulator's previous tile
        if (tc >= 2) {
          const uint32_t par = ((tc >> 1) - 1) & 1;
          const bool w = PAIR ? bounded_wait_cluster_w(&acc_empty[acc], par, abort_flag, 106, p.err)
                              : bounded_wait_w(&acc_empty[acc], par, abort_flag, 106, p.err);
          if (!w) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * ACC_COLS);
        int kb, ke;
        k_range(p, unit, kb, ke);
        for (int kt = kb; kt < ke; ++kt) {
          const int s = it % STAGES;
          if (!bounded_wait_w(&full[s], (it / STAGES) & 1, abort_flag, 103, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc(sa + kk * 2048, 8192, 1024, 2) : sdesc(sa + kk * 32, 16, 1024, 2);
            const uint64_t bd = B_MN ? sdesc(sb + kk * 2048, 8192, 1024, 2) : sdesc(sb + kk * 32, 16, 1024, 2);
            const bool accum = kt != kb || kk != 0;
            if constexpr (PAIR) umma_bf16_pair_w(d, ad, bd, IDESC, accum);
            else umma_bf16_w(d, ad, bd, IDESC, accum);
            if (DUAL) {
              const uint64_t bd2 = sdesc(sb + BNS * BK * 2 + kk * 32, 16, 1024, 2);
              if constexpr (PAIR) umma_bf16_pair_w(d + BN, ad, bd2, IDESC, accum);
              else umma_bf16_w(d + BN, ad, bd2, IDESC, accum);
            }
          }
          // the stage is free in both CTAs once these products have read it
          if constexpr (PAIR) umma_commit_pair_w(&empty[s], 3);
          else umma_commit_w(&empty[s]);
          ++it;
        }
        if (!ok) break;
        if constexpr (PAIR) umma_commit_pair_w(&acc_full[acc], 3);
        else umma_commit_w(&acc_full[acc]);
      }
      if (!ok) {
        // wait until nothing issued is still in flight
        if constexpr (PAIR) umma_commit_pair_w(drain, 1);
        else umma_commit_w(drain);
        drain_wait(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..9)
    // warp w reads TMEM lanes 32*(w%4)..+31 (its row quarter) and one half of
    // the accumulator's columns; a pair's rank r holds rows 128 r .. of the tile
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = (int)rank * BM + q * 32 + lane;
    const uint32_t acc_empty0 = PAIR ? cluster_addr(smem_u32(acc_empty), 0) : 0u;
    int tc = 0;
    for (int unit = unit0; unit < p.ntiles; unit += units_in_flight, ++tc) {
      const int acc = tc & 1;
      // the TMEM loads below are warp-collective, so the decision is too
      const bool ok = __all_sync(0xffffffffu, bounded_wait(&acc_full[acc], (tc >> 1) & 1, abort_flag, 105, p.err));
      if (!ok) break;
      tc_fence_after();
      int m0, n0;
      tile_origin(p, unit, TM, BN, m0, n0);
      const uint32_t tbase = tmem + (uint32_t)(acc * ACC_COLS) + ((uint32_t)(q * 32) << 16);
      epilogue_tile<BN, DUAL>(p, tbase, m0 + row, n0, half);
      // this warp's part of the accumulator has been read: hand it back
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR) mbar_arrive_cluster(acc_empty0 + 8u * (uint32_t)acc);
        else mbar_arrive(&acc_empty[acc]);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  // a pair: neither CTA leaves (or frees its TMEM) while the other may still
  // use its barriers, shared memory or tensor memory
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem, TMEM_COLS);
    else tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Units in flight (CTAs, or pairs) and the L2-aware walk, then the launch.
template <int BN, bool A_MN, bool B_MN, bool DUAL, bool PAIR>
int launch(GemmParams& p, cudaStream_t st) {
  constexpr int BNS = PAIR ? BN / 2 : BN;
  constexpr int B_BYTES = (DUAL ? 2 : 1) * BNS * BK * 2;
  constexpr int SMEM = stages<PAIR>() * (A_BYTES + B_BYTES) + 1024 + 256;
  constexpr int TM = PAIR ? 2 * BM : BM;
  auto kern = gemm_kernel<BN, A_MN, B_MN, DUAL, PAIR>;
  static std::atomic<uint64_t> attr{0};  // per instantiation: devices whose limit is set
  if (smem_limit_once(reinterpret_cast<const void*>(kern), SMEM, &attr)) return 3;
  int slots;
  if constexpr (PAIR) {
    static std::atomic<int> fit[64];  // per instantiation and device: pairs resident at once (0: unknown)
    slots = pair_slots(reinterpret_cast<const void*>(kern), SMEM, fit);
  } else {
    slots = sm_count();
  }
  if (slots <= 0) return 3;
  p.mt = (p.M + TM - 1) / TM;
  p.nt = (p.N + BN - 1) / BN;
  p.ntiles = p.mt * p.nt * p.ksplit;
  // the smaller operand's tiles vary fastest (the wave in flight shares the
  // larger operand's tiles)
  p.m_fast = (double)p.M <= (double)p.N * (DUAL ? 2 : 1);
  {
    // Both operands past what L2 keeps while the wave in flight uses them:
    // walk bands of tiles instead.  Band along M (A's rows): A is read once,
    // B once per band; along N the other way round.  The band's slice of its
    // operand is kept to about a quarter of L2, and the side that moves fewer
    // bytes in total is taken.  No bands when the smaller operand is within
    // half of L2: the plain order (its tiles fastest, each tile of the larger
    // one shared by the wave in flight) reads the larger operand once, and
    // the smaller one at most once per wave (measured for the dQKV Wqkv
    // product of the GPT-3B layer: 1.07 GB read against 1.35 GB in bands).
    const double a_bytes = (double)p.M * p.K * 2, b_bytes = (double)p.N * p.K * 2 * (DUAL ? 2 : 1);
    constexpr double L2_KEEP = 32.0 * 1024 * 1024;
    constexpr double L2_RESIDENT = 64.0 * 1024 * 1024;
    p.group = 0;
    if (a_bytes + b_bytes > 3 * L2_KEEP && std::min(a_bytes, b_bytes) > L2_RESIDENT && p.mt > 1 && p.nt > 1) {
      const double row_a = (double)TM * p.K * 2, row_b = (double)BN * p.K * 2 * (DUAL ? 2 : 1);
      const int gm = (int)std::max(1.0, std::min((double)p.mt, L2_KEEP / row_a));
      const int gn = (int)std::max(1.0, std::min((double)p.nt, L2_KEEP / row_b));
      const double tm = a_bytes + b_bytes * ((p.mt + gm - 1) / gm);
      const double tn = b_bytes + a_bytes * ((p.nt + gn - 1) / gn);
      p.group_m = tm <= tn;
      p.group = p.group_m ? gm : gn;
    }
  }
  const int units = p.ntiles < slots ? p.ntiles : slots;
  if constexpr (!PAIR) {
    kern<<<units, NUM_THREADS, SMEM, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * units), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? 0 : 3;
  }
}

// The pair-of-SMs launches (gemm_pair.cu), and the pairs of CTAs the
// device holds at once (every pair instance has the same shared memory and
// threads; 0 when the device cannot hold one, and then gemm() takes the
// one-SM form).
int launch_pair(GemmParams& p, bool a_mn, bool b_mn, bool dual, cudaStream_t st);
int pair_units();

}  // namespace gk
}  // namespace bpt
