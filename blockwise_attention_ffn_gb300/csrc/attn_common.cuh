// attn_common.cuh -- shared-memory geometry of the attention tiles.
//
// A [128 rows x D] bf16 tile (Q, K, V, dO) is stored as D/CW column chunks of
// [128 rows x CW] each, swizzled the way TMA writes them and tcgen05 reads
// them: CW = 64 (128-byte swizzle) when D is a multiple of 64, else CW = 16
// (32-byte swizzle).  The same chunked tile serves as a K-major operand (the
// head dimension is the contraction: Q K^T, V dO^T) and as an MN-major operand
// (the head dimension is N: P V, P^T dO, dS^T Q, dS K).
#pragma once

#include "ptx.cuh"

namespace bpt {

template <int D>
struct TileGeom {
  static constexpr int CW = (D % 64 == 0) ? 64 : 16;  // chunk width (elements)
  static constexpr int SWB = CW * 2;                   // bytes per chunk row
  static constexpr int NCH = D / CW;                   // chunks per tile
  static constexpr int CHUNK = 128 * SWB;              // bytes per chunk
  static constexpr int TILE = 128 * D * 2;             // bytes per tile
  static constexpr uint32_t LAYOUT = (SWB == 128) ? 2u : 6u;  // descriptor swizzle code
  static constexpr int TMA_SWZ = SWB;                  // swizzle bytes for the map

  // K-major use: 16 columns of the head dimension starting at 16*kk
  static __device__ __forceinline__ uint64_t kmajor(uint32_t tile, int kk) {
    const int c = (kk * 16) / CW;
    const int off = ((kk * 16) % CW) * 2;
    return sdesc(tile + c * CHUNK + off, 16, 8 * SWB, LAYOUT);
  }
  // MN-major use (N = D): 16 rows (the contraction) starting at 16*kk
  static __device__ __forceinline__ uint64_t mnmajor(uint32_t tile, int kk) {
    return sdesc(tile + kk * 16 * SWB, CHUNK, 8 * SWB, LAYOUT);
  }
};

// 16 TMEM fp32 columns of this thread's row -> 16 bf16 values (scaled)
__device__ __forceinline__ void store_row16(__nv_bfloat16* dst, const uint32_t* v, float sc) {
  uint4 a, b;
  a.x = pack_bf16(__uint_as_float(v[0]) * sc, __uint_as_float(v[1]) * sc);
  a.y = pack_bf16(__uint_as_float(v[2]) * sc, __uint_as_float(v[3]) * sc);
  a.z = pack_bf16(__uint_as_float(v[4]) * sc, __uint_as_float(v[5]) * sc);
  a.w = pack_bf16(__uint_as_float(v[6]) * sc, __uint_as_float(v[7]) * sc);
  b.x = pack_bf16(__uint_as_float(v[8]) * sc, __uint_as_float(v[9]) * sc);
  b.y = pack_bf16(__uint_as_float(v[10]) * sc, __uint_as_float(v[11]) * sc);
  b.z = pack_bf16(__uint_as_float(v[12]) * sc, __uint_as_float(v[13]) * sc);
  b.w = pack_bf16(__uint_as_float(v[14]) * sc, __uint_as_float(v[15]) * sc);
  reinterpret_cast<uint4*>(dst)[0] = a;
  reinterpret_cast<uint4*>(dst)[1] = b;
}

// N = D/2 consecutive 32-bit TMEM columns of this thread's lane from w
template <int N>
__device__ __forceinline__ void tmem_store_row(uint32_t taddr, const uint32_t* w) {
  static_assert(N % 8 == 0 && N <= 64, "row width");
  if constexpr (N >= 32) tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(w));
  if constexpr (N == 64) tmem_st32(taddr + 32, *reinterpret_cast<const uint32_t(*)[32]>(w + 32));
  if constexpr (N % 32 >= 16) tmem_st16_nw(taddr + (N / 32) * 32, w + (N / 32) * 32);
  if constexpr (N % 16 == 8) tmem_st8_nw(taddr + (N / 16) * 16, w + (N / 16) * 16);
}

// max of three (sm_100 family: one instruction)
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two fp32 lanes per instruction (the sm_100 family's packed .f32x2 forms):
// the per-element scale, offset and products of the softmax loops, at half
// the instruction count.  Each lane rounds exactly as the scalar form does.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2split(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace bpt
