// gemm_pair.cu -- the pair-of-SMs launches of the tcgen05 GEMM kernel
// (gemm_kernel.cuh), in a translation unit of their own so that the two
// forms compile in parallel.
#include "gemm_kernel.cuh"

namespace bpt {
namespace gk {

int pair_units() {
  // the same size as launch<256, ..., true> asks for: 128 rows of B per CTA
  constexpr int SMEM = stages<true>() * (A_BYTES + 128 * BK * 2) + 1024 + 256;
  auto kern = gemm_kernel<256, false, false, false, true>;
  static std::atomic<uint64_t> attr{0};
  if (smem_limit_once(reinterpret_cast<const void*>(kern), SMEM, &attr)) return 0;
  static std::atomic<int> fit[64];
  return pair_slots(reinterpret_cast<const void*>(kern), SMEM, fit);
}

int launch_pair(GemmParams& p, bool a_mn, bool b_mn, bool dual, cudaStream_t st) {
  if (dual) return launch<128, false, false, true, true>(p, st);
  if (!a_mn && !b_mn) return launch<256, false, false, false, true>(p, st);
  if (!a_mn && b_mn) return launch<256, false, true, false, true>(p, st);
  if (a_mn && b_mn) return launch<256, true, true, false, true>(p, st);
  return launch<256, true, false, false, true>(p, st);
}

}  // namespace gk
}  // namespace bpt
