// gemm_tc.cu -- gemm(): tensor maps, epilogue parameters, the K split and
// the choice between the one-SM and the pair-of-SMs form of the tcgen05 GEMM
// kernel (gemm_kernel.cuh); the one-SM launches.
#include "gemm_kernel.cuh"

namespace bpt {

using namespace gk;

int gemm(int64_t M, int64_t N, int64_t K, const MatView& A, bool a_mn, const MatView* B,
         const int64_t* b_seg_k, int nseg, bool b_mn, const MatView* B2, const Epilogue& e,
         cudaStream_t stream) {
  if (M <= 0 || N <= 0) return 0;
  if (K <= 0 || nseg < 1 || nseg > 3) return 1;
  const bool dual = (B2 != nullptr);
  if (dual && (b_mn || nseg != 1 || a_mn)) return 1;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.nkt = (int)((K + BK - 1) / BK);
  p.seg_kt[0] = p.seg_kt[1] = p.seg_kt[2] = 1 << 30;
  {
    int64_t acc = 0;
    for (int i = 0; i < nseg; ++i) {
      if (i < nseg - 1 && (b_seg_k[i] % BK) != 0) return 1;
      acc += b_seg_k[i];
      if (i < nseg - 1) p.seg_kt[i] = (int)(acc / BK);
    }
    if (acc != K) return 1;
  }
  const int BN = dual ? 128 : 256;
  // a pair of SMs per 256-row tile wherever there are two row tiles (and
  // the device can hold a pair of CTAs)
  const int pairs = M > BM ? pair_units() : 0;
  const bool pair = pairs > 0;
  const int TM = pair ? 2 * BM : BM;
  const int BNS = pair ? BN / 2 : BN;  // rows of each B one CTA stages
  // A
  if (!a_mn) {
    if (make_map_2d(&p.mapA, A.ptr, A.rows, A.cols, A.ld, BK, BM, 128)) return 1;
  } else {
    if (make_map_2d(&p.mapA, A.ptr, A.rows, A.cols, A.ld, 64, BK, 128)) return 1;
  }
  for (int i = 0; i < nseg; ++i) {
    const MatView& b = B[i];
    if (!b_mn) {
      if (make_map_2d(&p.mapB[i], b.ptr, b.rows, b.cols, b.ld, BK, BNS, 128)) return 1;
    } else {
      if (make_map_2d(&p.mapB[i], b.ptr, b.rows, b.cols, b.ld, 64, BK, 128)) return 1;
    }
  }
  if (dual) {
    if (make_map_2d(&p.mapB[1], B2->ptr, B2->rows, B2->cols, B2->ld, BK, BNS, 128)) return 1;
  }
  p.epi = e.kind;
  p.act = e.act;
  p.out = e.out;
  p.ldo = e.ldo;
  p.out2 = e.out2;
  p.ldo2 = e.ldo2;
  p.out3 = e.out3;
  p.ldo3 = e.ldo3;
  p.bias = reinterpret_cast<const __nv_bfloat16*>(e.bias);
  p.res = e.res;
  p.ldr = e.ldr;
  p.res_f32 = e.res_f32;
  p.aux = reinterpret_cast<const __nv_bfloat16*>(e.aux);
  p.ldaux = e.ldaux;
  p.aux2 = reinterpret_cast<const __nv_bfloat16*>(e.aux2);
  p.ldaux2 = e.ldaux2;
  p.beta = e.beta;
  p.rowf = e.rowf;
  p.rowi = e.rowi;
  p.scale = e.scale;
  p.col0 = e.col0;
  p.err = device_error_word();
  if (!p.err) return 3;
  {
    // 32-byte epilogue accesses need 32-byte aligned operands and row strides
    auto ok32 = [](const void* ptr, int64_t ld, int elem) {
      return ptr == nullptr || ((reinterpret_cast<uintptr_t>(ptr) & 31) == 0 && ((ld * elem) & 31) == 0);
    };
    const int out_elem = e.kind == EPI_F32 ? 4 : 2;
    p.vec32 = ok32(e.out, e.ldo, out_elem) && ok32(e.out2, e.ldo2, 2) && ok32(e.out3, e.ldo3, 2) &&
              ok32(e.res, e.ldr, e.res_f32 ? 4 : 2) && ok32(e.aux, e.ldaux, 2) && ok32(e.aux2, e.ldaux2, 2) &&
              ok32(e.bias, 0, 2);
  }
  ProfScope prof(PROF_GEMM, 2.0 * (double)M * (double)N * (double)K * (dual ? 2 : 1), 0.0, stream);
  // Split K for fp32 outputs with nothing but the product (weight gradients)
  // when whole tiles would leave the last wave of SMs mostly idle: K ranges
  // of at least 16 k-tiles each, added atomically into out (zeroed first
  // unless accumulating).
  p.ksplit = 1;
  {
    const int nsm = pair ? pairs : sm_count();  // units in flight
    const int64_t tiles = ((M + TM - 1) / TM) * ((N + BN - 1) / BN);
    auto fill = [&](int64_t units) { return (double)units / (double)(((units + nsm - 1) / nsm) * nsm); };
    const bool aligned = (e.ldo % 4) == 0 && (reinterpret_cast<uintptr_t>(e.out) & 15) == 0;
    if (!dual && e.kind == EPI_F32 && !e.bias && !e.res && (e.beta == 0.f || e.beta == 1.f) && aligned && nsm > 0 &&
        !e.deterministic && fill(tiles) < 0.8) {
      for (int ks = 2; ks <= 8 && p.nkt / ks >= 16; ++ks)
        if (fill(tiles * ks) >= 0.9) {
          p.ksplit = ks;
          break;
        }
    }
    if (p.ksplit > 1 && e.beta == 0.f) {
      if (cudaMemset2DAsync(e.out, (size_t)e.ldo * 4, 0, (size_t)N * 4, (size_t)M, stream) != cudaSuccess) return 3;
    }
  }
  if (pair) return launch_pair(p, a_mn, b_mn, dual, stream);
  if (dual) return launch<128, false, false, true, false>(p, stream);
  if (!a_mn && !b_mn) return launch<256, false, false, false, false>(p, stream);
  if (!a_mn && b_mn) return launch<256, false, true, false, false>(p, stream);
  if (a_mn && b_mn) return launch<256, true, true, false, false>(p, stream);
  return launch<256, true, false, false, false>(p, stream);
}

}  // namespace bpt
