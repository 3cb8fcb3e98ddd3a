// norm_misc.cu -- the memory-bound pieces of the layer: LayerNorm / RMSNorm
// forward and backward, column sums (bias gradients), the per-row dO . O sums
// of the attention backward, and an fp32 -> bf16 scaled copy.
//
// Norms follow "Training memory: model states, activations and checkpointing",
// section 3 (pre-LN layer, LayerNorm with scale and shift; Llama-style layer
// with RMSNorm, scale only): y = (x - mean) * rstd * w + b with the biased
// variance, or y = x * rstd * w with rstd = 1/sqrt(mean(x^2) + eps).  One warp
// per row, 16-byte vector accesses; rows are re-read from L1/L2 between passes.
#include <math.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace bpt {

namespace {

__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
  v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
  v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void ld8f(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  u.x = pack_bf16(v[0], v[1]);
  u.y = pack_bf16(v[2], v[3]);
  u.z = pack_bf16(v[4], v[5]);
  u.w = pack_bf16(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 8 consecutive values of a bf16 or fp32 row
__device__ __forceinline__ void ld8x(const void* base, int f32, int64_t idx, float (&v)[8]) {
  if (f32) ld8f(reinterpret_cast<const float*>(base) + idx, v);
  else ld8(reinterpret_cast<const __nv_bfloat16*>(base) + idx, v);
}

// mean (LayerNorm) and rstd of one row, reading it twice
__device__ __forceinline__ void row_stats(const void* x, int x_f32, int64_t row_off, int h, int kind,
                                          float eps, float& mean, float& rstd) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  for (int c = lane * 8; c < h; c += 256) {
    float v[8];
    ld8x(x, x_f32, row_off + c, v);
#pragma unroll
    for (int k = 0; k < 8; ++k) s += (kind == 0) ? v[k] : v[k] * v[k];
  }
  s = warp_sum(s);
  if (kind == 0) {
    mean = s / h;
    float q = 0.f;
    for (int c = lane * 8; c < h; c += 256) {
      float v[8];
      ld8x(x, x_f32, row_off + c, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float t = v[k] - mean;
        q += t * t;
      }
    }
    q = warp_sum(q);
    rstd = rsqrtf(q / h + eps);
  } else {
    mean = 0.f;
    rstd = rsqrtf(s / h + eps);
  }
}

__global__ void norm_fwd_kernel(int64_t rows, int h, int kind, float eps, const void* x, int x_f32,
                                int64_t ldx, const __nv_bfloat16* w, const __nv_bfloat16* b,
                                __nv_bfloat16* y, int64_t ldy) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    float mean, rstd;
    row_stats(x, x_f32, r * ldx, h, kind, eps, mean, rstd);
    for (int c = lane * 8; c < h; c += 256) {
      float v[8], wv[8], bv[8];
      ld8x(x, x_f32, r * ldx + c, v);
      ld8(w + c, wv);
      if (b) ld8(b + c, bv);
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = (v[k] - mean) * rstd * wv[k] + (b ? bv[k] : 0.f);
      st8(y + r * ldy + c, v);
    }
  }
}

// dx = res + rstd * (g - mean(g) - xhat * mean(g * xhat))    (LayerNorm)
//    = res + rstd * (g - xhat * mean(g * xhat))              (RMSNorm)
// with g = dy * w; dw += sum_rows dy * xhat, db += sum_rows dy.
// A block takes a band of rows (one band per resident block: one wave) in
// sub-bands of two rows per warp, each in two phases:
//  1. one warp per row: the row's mean and rstd (as the forward computes
//     them), and the two row sums of the gradient, into shared memory;
//  2. each thread owns 8 columns (the block spans the row up to h = 4096):
//     for every row of the sub-band it forms dx and accumulates dw, db in
//     registers, so the scale/shift gradients take one global atomic per
//     column per block and no shared-memory atomics at all.
// Phase 2 re-reads the rows phase 1 has just read, so they come from L2.
// The loops store through pointers the compiler must assume alias the
// inputs, so they load a group of chunks (phase 1) or two rows (phase 2)
// before any store: one load in flight per thread would leave HBM idle.
// With `part` (the fixed-order mode) each block writes its column sums to
// part[blockIdx.x][0, h) (dw) and [h, 2h) (db) instead of adding them.
__global__ void __launch_bounds__(512) norm_bwd_kernel(int64_t rows, int h, int kind, float eps, NormBwdIO io,
                                                        const __nv_bfloat16* w, float* dw, float* db,
                                                        int64_t band, float* part) {
  extern __shared__ float stat[];  // [sub-band row][4]: mean, rstd, mean(g), mean(g * xhat)
  constexpr int NB1 = 2;           // chunk groups of phase 1 (the accumulators stay live)
  const int lane = threadIdx.x & 31;
  const int nwarp = blockDim.x >> 5;
  const int sub = 2 * nwarp;  // rows per sub-band: two per warp in phase 1
  const int64_t r0 = (int64_t)blockIdx.x * band;
  const int64_t r1 = min(rows, r0 + band);
  // every thread walks the same number of column groups (the barriers below)
  const int ngroups = (h + 8 * (int)blockDim.x - 1) / (8 * (int)blockDim.x);
  for (int gi = 0; gi < ngroups; ++gi) {
    const int c = (gi * (int)blockDim.x + (int)threadIdx.x) * 8;
    const bool active = c < h;
    float adw[8], adb[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) adw[k] = adb[k] = 0.f;
    // sub-bands: phase 2 re-reads the rows phase 1 just read, from L2
    for (int64_t s0 = r0; s0 < r1; s0 += sub) {
      const int64_t s1 = min(r1, s0 + sub);
      for (int64_t r = s0 + (threadIdx.x >> 5); r < s1; r += nwarp) {
        // mean first (LayerNorm), then one pass over x and dy for the
        // variance and the gradient sums: sum g*xhat = rstd * (sum g*x -
        // mean * sum g)
        float mean = 0.f;
        if (kind == 0) {
          float sx = 0.f;
          for (int c0 = lane * 8; c0 < h; c0 += NB1 * 256) {
            float v[NB1][8];
#pragma unroll
            for (int u = 0; u < NB1; ++u)
              if (c0 + u * 256 < h) ld8x(io.x, io.x_f32, r * io.ldx + c0 + u * 256, v[u]);
#pragma unroll
            for (int u = 0; u < NB1; ++u)
              if (c0 + u * 256 < h) {
#pragma unroll
                for (int k = 0; k < 8; ++k) sx += v[u][k];
              }
          }
          mean = warp_sum(sx) / h;
        }
        float q = 0.f, sg = 0.f, sgx = 0.f;
        for (int c0 = lane * 8; c0 < h; c0 += NB1 * 256) {
          float v[NB1][8], gv[NB1][8];
#pragma unroll
          for (int u = 0; u < NB1; ++u)
            if (c0 + u * 256 < h) {
              ld8x(io.x, io.x_f32, r * io.ldx + c0 + u * 256, v[u]);
              ld8x(io.dy, io.dy_f32, r * io.lddy + c0 + u * 256, gv[u]);
            }
#pragma unroll
          for (int u = 0; u < NB1; ++u)
            if (c0 + u * 256 < h) {
              float w8[8];
              ld8(w + c0 + u * 256, w8);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float t = v[u][k] - mean;
                const float g = gv[u][k] * w8[k];
                q += t * t;
                sg += g;
                sgx += g * t;
              }
            }
        }
        q = warp_sum(q);
        const float rstd = rsqrtf(q / h + eps);
        sg = warp_sum(sg) / h;
        sgx = warp_sum(sgx) * rstd / h;
        if (lane == 0) {
          float* o = stat + (r - s0) * 4;
          o[0] = mean;
          o[1] = rstd;
          o[2] = (kind == 0) ? sg : 0.f;
          o[3] = sgx;
        }
      }
      __syncthreads();
      if (active) {
        // two rows per iteration, every load before any store
        for (int64_t r = s0; r < s1; r += 2) {
          const int nr = r + 1 < s1 ? 2 : 1;
          float v[2][8], gv[2][8], rv[2][8], wv[8];
          ld8(w + c, wv);  // from L1: cheaper than holding it live
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (u < nr) {
              ld8x(io.x, io.x_f32, (r + u) * io.ldx + c, v[u]);
              ld8x(io.dy, io.dy_f32, (r + u) * io.lddy + c, gv[u]);
              if (io.res) ld8x(io.res, io.res_f32, (r + u) * io.ldres + c, rv[u]);
            }
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (u < nr) {
              const float4 s4 = *reinterpret_cast<const float4*>(stat + (r + u - s0) * 4);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float xh = (v[u][k] - s4.x) * s4.y;
                adw[k] += gv[u][k] * xh;
                adb[k] += gv[u][k];
                v[u][k] = s4.y * (gv[u][k] * wv[k] - s4.z - xh * s4.w) + (io.res ? rv[u][k] : 0.f);
              }
              st8(reinterpret_cast<__nv_bfloat16*>(io.dx) + (r + u) * io.lddx + c, v[u]);
              if (io.dx_f32) {
                float4* o = reinterpret_cast<float4*>(io.dx_f32 + (r + u) * io.lddx + c);
                o[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
                o[1] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
              }
            }
        }
      }
      __syncthreads();
    }
    if (active) {
      if (part) {
        float* pw = part + (int64_t)blockIdx.x * 2 * h + c;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          pw[k] = adw[k];
          pw[h + k] = adb[k];
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (dw) atomicAdd(&dw[c + k], adw[k]);
          if (db) atomicAdd(&db[c + k], adb[k]);
        }
      }
    }
  }
}

// rows per group of the staged norm backward, at most
constexpr int NB_MAX_R = 8;

// 4 consecutive values of a bf16 or fp32 row (8- or 16-byte accesses)
__device__ __forceinline__ void ld4x(const void* base, int f32, int64_t idx, float (&v)[4]) {
  if (f32) {
    const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + idx);
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
    v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  }
}

// The same backward with its rows staged in shared memory by the copy engine.
// A block takes a contiguous band of rows in groups of R; `ns` ring stages of
// R rows (x, dy and res of each row side by side) are filled by 1-D bulk
// copies issued by thread 0, ns - 1 groups ahead of the group being
// processed, so the loads stay in flight whatever the block does meanwhile.
// Each thread owns 4 consecutive columns (h / 4 threads, up to 1024), so a
// warp's shared-memory accesses are contiguous 8- or 16-byte pieces, free of
// bank conflicts.  Per group:
//  1. the rows' statistics from shared memory, as the forward computes them
//     (mean, then the centred sums), and the two row sums of the gradient,
//     each row split over P = warps / R warps whose partial sums are added
//     in a fixed order (each warp adds its row's partial sums of x itself,
//     one thread per row the rest);
//  2. for every row of the group each thread forms dx for its columns
//     (stored straight to global memory) and accumulates dw, db in
//     registers.
// Every row is read from HBM once.  Rows, the row strides and every pointer
// are 16-byte aligned (the host checks; it takes norm_bwd_kernel otherwise).
__global__ void __launch_bounds__(1024, 1) norm_bwd_staged_kernel(int64_t rows, int h, int kind, float eps,
                                                                  NormBwdIO io, const __nv_bfloat16* w, float* dw,
                                                                  float* db, int64_t band, float* part, int R, int ns,
                                                                  unsigned int* err) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int xe = io.x_f32 ? 4 : 2, de = io.dy_f32 ? 4 : 2, re = io.res ? (io.res_f32 ? 4 : 2) : 0;
  const int xb = h * xe, dyb = h * de, rb = h * re;
  const int row_bytes = xb + dyb + rb;
  const int stage_bytes = R * row_bytes;
  float* stat = reinterpret_cast<float*>(sm + (size_t)ns * stage_bytes);  // [R][4]
  float* red = stat + 4 * NB_MAX_R;                                       // [R][P][3] partial sums
  float* red1 = red + 3 * 32;                                             // [R][P] partial sums of x
  uint64_t* full = reinterpret_cast<uint64_t*>(red1 + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + ns);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarp = blockDim.x >> 5;  // at most 32
  const int P = nwarp / R;             // warps per row for the statistics (R <= warps)
  const int64_t r0 = (int64_t)blockIdx.x * band;
  const int64_t r1 = min(rows, r0 + band);
  const int ngroups = r0 < r1 ? (int)((r1 - r0 + R - 1) / R) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // group g into stage g % ns (thread 0)
  auto issue = [&](int g) {
    const int s = g % ns;
    const int64_t gr = r0 + (int64_t)g * R;
    const int nr = (int)min((int64_t)R, r1 - gr);
    uint8_t* base = sm + (size_t)s * stage_bytes;
    mbar_expect_tx(&full[s], (uint32_t)(nr * row_bytes));
    for (int i = 0; i < nr; ++i) {
      uint8_t* rp = base + (size_t)i * row_bytes;
      const int64_t r = gr + i;
      bulk_load(rp, reinterpret_cast<const uint8_t*>(io.x) + r * io.ldx * xe, (uint32_t)xb, &full[s]);
      bulk_load(rp + xb, reinterpret_cast<const uint8_t*>(io.dy) + r * io.lddy * de, (uint32_t)dyb, &full[s]);
      if (rb) bulk_load(rp + xb + dyb, reinterpret_cast<const uint8_t*>(io.res) + r * io.ldres * re, (uint32_t)rb,
                        &full[s]);
    }
  };
  if (threadIdx.x == 0)
    for (int g = 0; g < min(ns, ngroups); ++g) issue(g);

  const int c = threadIdx.x * 4;
  const bool active = c < h;
  float adw[4], adb[4], wv[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) adw[k] = adb[k] = wv[k] = 0.f;
  if (active) ld4x(w, 0, c, wv);
  int g = 0;
  for (; g < ngroups; ++g) {
    const int s = g % ns;
    const int64_t gr = r0 + (int64_t)g * R;
    const int nr = (int)min((int64_t)R, r1 - gr);
    // one warp polls the stage's barrier, the others wait at the block
    // barrier (and see the copied rows through it)
    const bool ok =
        __syncthreads_and(warp != 0 || bounded_wait(&full[s], (uint32_t)(g / ns) & 1u, abort_flag, 301, err));
    if (!ok) break;
    const uint8_t* base = sm + (size_t)s * stage_bytes;
    // 1. statistics: P warps per row (warp w takes part w % P of row w / P,
    //    every P-th 128-column chunk), partial sums combined in a fixed order
    {
      const int i = warp / P, p = warp % P;
      const bool mine = i < nr;
      const uint8_t* xs = base + (size_t)i * row_bytes;
      const uint8_t* ds = xs + xb;
      if (kind == 0) {
        float sx = 0.f;
        if (mine)
          for (int c0 = (p * 32 + lane) * 4; c0 < h; c0 += P * 128) {
            float v[4];
            ld4x(xs, io.x_f32, c0, v);
            sx += (v[0] + v[1]) + (v[2] + v[3]);
          }
        sx = warp_sum(sx);
        if (mine && lane == 0) red1[i * P + p] = sx;
        __syncthreads();
      }
      // each warp of a row adds the row's partial sums itself (same order);
      // red1 is rewritten only after the barrier that ends the group
      float mean = 0.f;
      if (kind == 0 && mine) {
        for (int u = 0; u < P; ++u) mean += red1[i * P + u];
        mean /= h;
      }
      float q = 0.f, sg = 0.f, sgx = 0.f;
      if (mine)
        for (int c0 = (p * 32 + lane) * 4; c0 < h; c0 += P * 128) {
          float v[4], gv[4], w4[4];
          ld4x(xs, io.x_f32, c0, v);
          ld4x(ds, io.dy_f32, c0, gv);
          ld4x(w, 0, c0, w4);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float t = v[k] - mean;
            const float gg = gv[k] * w4[k];
            q += t * t;
            sg += gg;
            sgx += gg * t;
          }
        }
      q = warp_sum(q);
      sg = warp_sum(sg);
      sgx = warp_sum(sgx);
      if (mine && lane == 0) {
        float* o = red + (i * P + p) * 3;
        o[0] = q;
        o[1] = sg;
        o[2] = sgx;
      }
      __syncthreads();
      if ((int)threadIdx.x < nr) {
        const int r = threadIdx.x;
        float M = 0.f, Q = 0.f, SG = 0.f, SGX = 0.f;
        for (int u = 0; u < P; ++u) {
          const float* o = red + (r * P + u) * 3;
          if (kind == 0) M += red1[r * P + u];
          Q += o[0];
          SG += o[1];
          SGX += o[2];
        }
        const float rstd = rsqrtf(Q / h + eps);
        float* o = stat + r * 4;
        o[0] = (kind == 0) ? M / h : 0.f;
        o[1] = rstd;
        o[2] = (kind == 0) ? SG / h : 0.f;
        o[3] = SGX * rstd / h;
      }
    }
    __syncthreads();
    // 2. dx and the scale/shift gradients, 4 columns per thread
    if (active) {
      for (int i = 0; i < nr; ++i) {
        const uint8_t* xs = base + (size_t)i * row_bytes;
        const float4 s4 = *reinterpret_cast<const float4*>(stat + i * 4);
        float v[4], gv[4], rv[4];
        ld4x(xs, io.x_f32, c, v);
        ld4x(xs + xb, io.dy_f32, c, gv);
        if (rb) ld4x(xs + xb + dyb, io.res_f32, c, rv);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float xh = (v[k] - s4.x) * s4.y;
          adw[k] += gv[k] * xh;
          adb[k] += gv[k];
          v[k] = s4.y * (gv[k] * wv[k] - s4.z - xh * s4.w) + (rb ? rv[k] : 0.f);
        }
        const int64_t r = gr + i;
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(io.dx) + r * io.lddx + c) =
            make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
        if (io.dx_f32) *reinterpret_cast<float4*>(io.dx_f32 + r * io.lddx + c) = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
    // stage s and the statistics are free again
    __syncthreads();
    if (threadIdx.x == 0 && g + ns < ngroups) {
      fence_proxy_async_smem();
      issue(g + ns);
    }
  }
  if (g < ngroups) {
    // gave up waiting: let the copies already issued land before the block
    // (and its shared memory) goes away
    if (threadIdx.x == 0)
      for (int j = g; j < min(ngroups, g + ns); ++j) drain_wait(&full[j % ns], (uint32_t)(j / ns) & 1u);
    return;
  }
  if (active) {
    if (part) {
      float* pw = part + (int64_t)blockIdx.x * 2 * h + c;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pw[k] = adw[k];
        pw[h + k] = adb[k];
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (dw) atomicAdd(&dw[c + k], adw[k]);
        if (db) atomicAdd(&db[c + k], adb[k]);
      }
    }
  }
}

// out[n] += sum_r in[r, n]; 8 columns per thread, rows split over gridDim.y
// Column sums of a bf16 [rows x n] matrix, added atomically into fp32 out.
// A block covers 256 columns (8 per lane of a warp) and a band of rows; its 8
// warps take every 8th row of the band, four rows in flight at a time, and
// combine their partial sums in shared memory so the block issues one atomic
// per column.  n and ld are multiples of 8 (16-byte row segments).  With
// `part` (the fixed-order mode) the block's sums go to part[blockIdx.y][.]
// instead.
constexpr int COLSUM_WARPS = 8;
__global__ void __launch_bounds__(32 * COLSUM_WARPS) colsum_kernel(int64_t rows, int64_t n, const __nv_bfloat16* in,
                                                                   int64_t ld, int64_t band, float* out, float* part) {
  __shared__ float part_s[COLSUM_WARPS][256 + 4];
  float* dst_part = part;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 256 + lane * 8;
  const int64_t r0 = (int64_t)blockIdx.y * band;
  const int64_t r1 = min(rows, r0 + band);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (c < n) {
    int64_t r = r0 + w;
    for (; r + 3 * COLSUM_WARPS < r1; r += 4 * COLSUM_WARPS) {
      float v0[8], v1[8], v2[8], v3[8];
      ld8(in + r * ld + c, v0);
      ld8(in + (r + COLSUM_WARPS) * ld + c, v1);
      ld8(in + (r + 2 * COLSUM_WARPS) * ld + c, v2);
      ld8(in + (r + 3 * COLSUM_WARPS) * ld + c, v3);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += (v0[k] + v1[k]) + (v2[k] + v3[k]);
    }
    for (; r < r1; r += COLSUM_WARPS) {
      float v[8];
      ld8(in + r * ld + c, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += v[k];
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) part_s[w][lane * 8 + k] = acc[k];
  __syncthreads();
  const int col = threadIdx.x;  // 256 threads, one column each
  const int64_t gc = (int64_t)blockIdx.x * 256 + col;
  if (gc < n) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < COLSUM_WARPS; ++i) t += part_s[i][col];
    if (dst_part)
      dst_part[(int64_t)blockIdx.y * n + gc] = t;
    else
      atomicAdd(&out[gc], t);
  }
}

// out[c] += sum over p = 0, 1, ..., nparts - 1 (in that order) of
// part[p * ldp + c]: the second half of the fixed-order column sums.
__global__ void reduce_parts_kernel(int nparts, int64_t n, const float* part, int64_t ldp, float* out) {
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= n) return;
  float t = 0.f;
  for (int p = 0; p < nparts; ++p) t += part[(int64_t)p * ldp + c];
  out[c] += t;
}

__global__ void f32_to_bf16_kernel(int64_t rows, int64_t n, const float* src, int64_t lds,
                                   __nv_bfloat16* dst, int64_t ldd, float scale) {
  const int64_t per_row = n / 8;
  const int64_t total = rows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row;
    const int64_t c = (i % per_row) * 8;
    float v[8];
    ld8f(src + r * lds + c, v);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] *= scale;
    st8(dst + r * ldd + c, v);
  }
}

// Dsum[b, h, q] = sum_k dO[b*s + q, h*d + k] * O[b*s + q, h*d + k]  (0 for q >= s)
// and NL2[b, h, q] = -LSE[b, h, q] * log2(e), the exponent offset of the
// probabilities in base 2 (every padded row too), and one 8-column bf16 row
// per (b, h, q): (hi, lo) of -LSE * sqrt(d), (hi, lo) of -D, four zeros, with
// hi + lo the value to about 2^-16 relative.  Appended to the Q and dO rows
// as one more contraction step against (1, 1, 0, ...) resp. (0, 0, 1, 1, ...),
// it makes the tensor core emit S - LSE/scale and dP - D directly.
// v as the bf16 pair (hi, lo) with hi + lo = v to about 16 significant bits
__device__ __forceinline__ uint32_t hi_lo_pair(float v) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
  return (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(lo) << 16);
}

__global__ void dsum_kernel(int b, int s, int s_pad, int H, int d, const __nv_bfloat16* o,
                            int64_t ld_o, int64_t o_col, const __nv_bfloat16* dout, int64_t ld_do,
                            int64_t do_col, const float* lse, int H_total, int lse_head0, float* Dsum,
                            float* NL2, __nv_bfloat16* AUX) {
  const int64_t total = (int64_t)b * s_pad * H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int hn = (int)(i % H);
    const int64_t t = i / H;
    const int q = (int)(t % s_pad);
    const int bi = (int)(t / s_pad);
    float acc = 0.f;
    if (q < s) {
      const __nv_bfloat16* orow = o + ((int64_t)bi * s + q) * ld_o + o_col + (int64_t)hn * d;
      const __nv_bfloat16* drow = dout + ((int64_t)bi * s + q) * ld_do + do_col + (int64_t)hn * d;
      for (int k = 0; k < d; k += 8) {
        float a[8], c[8];
        ld8(orow + k, a);
        ld8(drow + k, c);
#pragma unroll
        for (int m = 0; m < 8; ++m) acc += a[m] * c[m];
      }
    }
    const int64_t row = ((int64_t)bi * H + hn) * s_pad + q;
    const float l = lse[((int64_t)bi * H_total + lse_head0 + hn) * s_pad + q];
    Dsum[row] = acc;
    NL2[row] = -1.4426950408889634f * l;
    // the row the dK/dV products append to Q and dO: -LSE/scale (scale =
    // 1/sqrt(d)) and -D, each as a (hi, lo) bf16 pair, then four zeros
    reinterpret_cast<uint4*>(AUX)[row] = make_uint4(hi_lo_pair(-l * sqrtf((float)d)), hi_lo_pair(-acc), 0u, 0u);
  }
}


// Rotary position embedding ("Untied Ulysses ...", "Composability with Other
// Memory Optimizations": fused RoPE, rotated in place without an fp32 copy of
// Q and K), in place, on n_heads consecutive heads of d
// columns starting at column col0 of a row-major bf16 buffer [rows, ld]
// (rows = b*s; the position of row r is r % s).  Element i of a head is
// paired with element i + d/2 and the pair turns by the angle p * theta[i],
// theta[i] = base^(-2i/d) (computed on the host in double); inverse turns by
// the negated angle: the transpose of the rotation, hence its gradient.
// The angle is formed and reduced to [-pi, pi] in double -- p * theta reaches
// 1.3e5 rad at s = 128K, where a float product would carry ~4e-3 rad of
// error -- and only its sine and cosine are taken in float.  One thread per
// row and pair of consecutive elements (i, i+1): a bf16x2 load and store per
// half of every head.
struct RopeTheta {
  double t[64];
};

__global__ void rope_kernel(int64_t rows, int s, __nv_bfloat16* buf, int64_t ld, int col0, int n_heads, int d,
                            const __grid_constant__ RopeTheta th, int inverse) {
  const int half = d / 2;
  const int per_row = half / 2;
  const int64_t total = rows * per_row;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / per_row;
    const int i = (int)(idx % per_row) * 2;
    const double p = (double)(r % s);
    float c[2], sn[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const double a = p * th.t[i + u];
      const double k = rint(a * 0.15915494309189535);  // turns: a / (2 pi)
      const float red = (float)fma(-k, 6.283185307179586, a);
      sincosf(red, &sn[u], &c[u]);
      if (inverse) sn[u] = -sn[u];
    }
    __nv_bfloat16* row = buf + r * ld + col0 + i;
    for (int hd = 0; hd < n_heads; ++hd) {
      __nv_bfloat162* pa = reinterpret_cast<__nv_bfloat162*>(row + (int64_t)hd * d);
      __nv_bfloat162* pb = reinterpret_cast<__nv_bfloat162*>(row + (int64_t)hd * d + half);
      const float2 a = __bfloat1622float2(*pa);
      const float2 b = __bfloat1622float2(*pb);
      *pa = __floats2bfloat162_rn(a.x * c[0] - b.x * sn[0], a.y * c[1] - b.y * sn[1]);
      *pb = __floats2bfloat162_rn(a.x * sn[0] + b.x * c[0], a.y * sn[1] + b.y * c[1]);
    }
  }
}

// blocks for a grid-stride loop over `work` items: enough for the work, at
// most 16 per SM of the current device
int grid_for(int64_t work, int per_block) {
  const int nsm = sm_count();
  const int64_t cap = (int64_t)(nsm > 0 ? nsm : 152) * 16;
  int64_t g = (work + per_block - 1) / per_block;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

int norm_fwd(int64_t rows, int h, int kind, float eps, const void* x, int x_f32, int64_t ldx,
             const void* w, const void* b, void* y, int64_t ldy, cudaStream_t st) {
  if (rows <= 0) return 0;
  const int threads = 256;
  ProfScope prof(PROF_NORM, 0.0, (double)rows * h * ((x_f32 ? 4 : 2) + 2), st);
  norm_fwd_kernel<<<grid_for(rows, threads / 32), threads, 0, st>>>(
      rows, h, kind, eps, x, x_f32, ldx, (const __nv_bfloat16*)w, (const __nv_bfloat16*)b,
      (__nv_bfloat16*)y, ldy);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// blocks of the fixed-order norm backward, whose partial sums (dw and db:
// 2h floats per block) the caller's workspace holds
constexpr int64_t NORM_DET_BLOCKS = 256;
// bands (row ranges, one per block row) of the fixed-order column sums
constexpr int64_t COLSUM_DET_BANDS = 64;

int64_t norm_bwd_part_floats(int h) { return NORM_DET_BLOCKS * 2 * (int64_t)h; }
int64_t colsum_part_floats(int64_t n) { return COLSUM_DET_BANDS * n; }

int reduce_parts(int nparts, int64_t n, const float* part, int64_t ldp, float* out, cudaStream_t st) {
  if (nparts <= 0 || n <= 0) return 0;
  reduce_parts_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(nparts, n, part, ldp, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// The staged form when every row starts on a 16-byte boundary and at least
// two ring stages of a row each fit the shared-memory budget; returns -1
// when it does not apply.
static int norm_bwd_staged(int64_t rows, int h, int kind, float eps, const NormBwdIO& io, const void* w,
                           float* dw, float* db, cudaStream_t st, float* part) {
  constexpr int BUDGET = 200 * 1024;  // bytes of ring stages per block (one block per SM)
  auto al = [](const void* p, int64_t ld, int elem) {
    return p == nullptr || ((reinterpret_cast<uintptr_t>(p) & 15) == 0 && ((ld * elem) & 15) == 0);
  };
  const int xe = io.x_f32 ? 4 : 2, de = io.dy_f32 ? 4 : 2, re = io.res ? (io.res_f32 ? 4 : 2) : 0;
  if (h % 8 || h > 4096 || !al(io.x, io.ldx, xe) || !al(io.dy, io.lddy, de) || !al(io.res, io.ldres, re ? re : 2) ||
      !al(io.dx, io.lddx, 2) || !al(io.dx_f32, io.lddx, 4) || (reinterpret_cast<uintptr_t>(w) & 7))
    return -1;
  const int row_bytes = h * (xe + de + re);
  // one thread per 4 columns; two stages of as many rows as fit (never more
  // rows than warps: each row's statistics take at least one).  Larger groups
  // beat deeper rings: a group costs four or five block barriers whatever its size
  // (measured per GPT-3B s=32K step: 1.01 ms of norms with two stages of 5
  // and 4 rows, 1.14 with three of 3 and 2, 1.60 with single rows).
  const int threads = std::max(64, (h / 4 + 31) / 32 * 32);
  const int R = std::min(std::min(NB_MAX_R, threads / 32), BUDGET / (2 * row_bytes));
  const int ns = 2;
  if (R < 1) return -1;
  const int smem = ns * R * row_bytes + 16 * NB_MAX_R + 4 * 4 * 32 + 8 * ns + 16;
  // the limit is raised once per device, to the largest size any call asks for
  static std::atomic<uint64_t> attr{0};
  if (smem_limit_once(reinterpret_cast<const void*>(norm_bwd_staged_kernel), BUDGET + 1024, &attr)) return 3;
  const int64_t nsm = sm_count() > 0 ? sm_count() : 1;
  // one block per SM, contiguous bands of rows; the fixed-order mode keeps
  // the unstaged kernel's bands (at most NORM_DET_BLOCKS partial sums)
  int64_t band;
  if (part) {
    band = std::max<int64_t>(8, (rows + NORM_DET_BLOCKS - 1) / NORM_DET_BLOCKS);
  } else {
    const int64_t g0 = std::min<int64_t>(nsm, (rows + R - 1) / R);
    band = (rows + g0 - 1) / g0;
  }
  const int64_t grid = (rows + band - 1) / band;
  unsigned int* err = device_error_word();
  if (!err) return 3;
  ProfScope prof(PROF_NORM, 0.0,
                 (double)rows * h * ((io.dy_f32 ? 4 : 2) + (io.x_f32 ? 4 : 2) + (io.res ? (io.res_f32 ? 4 : 2) : 0) + 2 +
                                     (io.dx_f32 ? 4 : 0)),
                 st);
  norm_bwd_staged_kernel<<<(unsigned)grid, threads, smem, st>>>(rows, h, kind, eps, io, (const __nv_bfloat16*)w,
                                                                dw, db, band, part, R, ns, err);
  if (cudaGetLastError() != cudaSuccess) return 3;
  if (part) {
    if (dw && reduce_parts((int)grid, h, part, 2 * (int64_t)h, dw, st)) return 3;
    if (db && reduce_parts((int)grid, h, part + h, 2 * (int64_t)h, db, st)) return 3;
  }
  return 0;
}

int norm_bwd(int64_t rows, int h, int kind, float eps, const NormBwdIO& io, const void* w, float* dw,
             float* db, cudaStream_t st, float* part) {
  if (rows <= 0) return 0;
  {
    const int rc = norm_bwd_staged(rows, h, kind, eps, io, w, dw, db, st, part);
    if (rc >= 0) return rc;
  }
  // one thread per 8 columns (a whole row per block up to h = 4096), 64..512
  // threads
  int threads = (h / 8 + 31) / 32 * 32;
  if (threads < 64) threads = 64;
  if (threads > 512) threads = 512;
  // one full wave: as many blocks as the SMs hold at once (registers bound
  // it), bands of at least 8 rows
  const int64_t nsm = sm_count() > 0 ? sm_count() : 1;
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, norm_bwd_kernel, threads, 2 * (threads / 32) * 16) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t band = (rows + nsm * per_sm - 1) / (nsm * per_sm);
  if (band < 8) band = 8;
  if (band > 2048) band = 2048;
  // fixed order: at most NORM_DET_BLOCKS blocks, one partial row each
  if (part) band = std::max<int64_t>(8, (rows + NORM_DET_BLOCKS - 1) / NORM_DET_BLOCKS);
  const int64_t grid = (rows + band - 1) / band;
  const size_t smem = (size_t)2 * (threads / 32) * 4 * sizeof(float);  // one sub-band of statistics
  ProfScope prof(PROF_NORM, 0.0,
                 (double)rows * h * ((io.dy_f32 ? 4 : 2) + (io.x_f32 ? 4 : 2) + (io.res ? (io.res_f32 ? 4 : 2) : 0) + 2 +
                                     (io.dx_f32 ? 4 : 0)),
                 st);
  norm_bwd_kernel<<<(unsigned)grid, threads, smem, st>>>(rows, h, kind, eps, io, (const __nv_bfloat16*)w, dw, db,
                                                         band, part);
  if (cudaGetLastError() != cudaSuccess) return 3;
  if (part) {
    if (dw && reduce_parts((int)grid, h, part, 2 * (int64_t)h, dw, st)) return 3;
    if (db && reduce_parts((int)grid, h, part + h, 2 * (int64_t)h, db, st)) return 3;
  }
  return 0;
}

int colsum(int64_t rows, int64_t n, const void* in, int64_t ld, float* out, int accumulate,
           cudaStream_t st, float* part) {
  if (!accumulate && cudaMemsetAsync(out, 0, n * sizeof(float), st) != cudaSuccess) return 3;
  if (rows <= 0 || n <= 0) return 0;
  ProfScope prof(PROF_MISC, 0.0, (double)rows * n * 2, st);
  // about four blocks per SM in all, each band a multiple of the 8 warps' rows
  const int nsm = sm_count();
  const int64_t gx = (n + 255) / 256;
  int64_t gy = (4 * (nsm > 0 ? nsm : 1) + gx - 1) / gx;
  if (part) gy = std::min(gy, COLSUM_DET_BANDS);
  int64_t band = (rows + gy - 1) / gy;
  band = (band + COLSUM_WARPS - 1) / COLSUM_WARPS * COLSUM_WARPS;
  if (band < 4 * COLSUM_WARPS) band = 4 * COLSUM_WARPS;
  gy = (rows + band - 1) / band;
  dim3 grid((unsigned)gx, (unsigned)gy);
  colsum_kernel<<<grid, 32 * COLSUM_WARPS, 0, st>>>(rows, n, (const __nv_bfloat16*)in, ld, band, out, part);
  if (cudaGetLastError() != cudaSuccess) return 3;
  return part ? reduce_parts((int)gy, n, part, n, out, st) : 0;
}

int f32_to_bf16(int64_t rows, int64_t n, const float* src, int64_t ld_src, void* dst, int64_t ld_dst,
                float scale, cudaStream_t st) {
  if (rows <= 0 || n <= 0) return 0;
  f32_to_bf16_kernel<<<grid_for(rows * (n / 8), 256), 256, 0, st>>>(rows, n, src, ld_src,
                                                                     (__nv_bfloat16*)dst, ld_dst, scale);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

int attn_dsum(const AttnBwdShape& sh, const void* o, const void* dout, const float* lse, float* Dsum,
              float* NL2, void* AUX, int s_pad, cudaStream_t st) {
  const AttnShape& f = sh.f;
  const int64_t total = (int64_t)f.b * s_pad * f.H;
  dsum_kernel<<<grid_for(total, 256), 256, 0, st>>>(f.b, f.s, s_pad, f.H, f.d, (const __nv_bfloat16*)o,
                                                    f.ld_o, f.o_col, (const __nv_bfloat16*)dout, sh.ld_do,
                                                    sh.do_col, lse, f.H_total, f.lse_head0, Dsum, NL2,
                                                    (__nv_bfloat16*)AUX);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

int rope_apply(int64_t rows, int s, void* buf, int64_t ld, int col0, int n_heads, int d, float base, int inverse,
               cudaStream_t st) {
  if (rows <= 0 || n_heads <= 0) return 0;
  if (d % 4 || d > 128 || s <= 0 || !(base > 1.f)) return 1;
  RopeTheta th;
  for (int i = 0; i < 64; ++i) th.t[i] = i < d / 2 ? pow((double)base, -2.0 * i / d) : 0.0;
  ProfScope prof(PROF_MISC, 0.0, (double)rows * n_heads * d * 2 * 2, st);
  rope_kernel<<<grid_for(rows * (d / 4), 256), 256, 0, st>>>(rows, s, (__nv_bfloat16*)buf, ld, col0, n_heads, d, th,
                                                             inverse);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace bpt
