// gemm_pair.cu -- the pair-of-SMs launches of the tcgen05 GEMM kernel
// (gemm_kernel.cuh), in a translation unit of their own so that the two
// forms compile in parallel.
#include "gemm_kernel.cuh"

namespace bpt {
namespace gk {

int launch_pair(GemmParams& p, bool a_mn, bool b_mn, bool dual, cudaStream_t st) {
  if (dual) return launch<128, false, false, true, true>(p, st);
  if (!a_mn && !b_mn) return launch<256, false, false, false, true>(p, st);
  if (!a_mn && b_mn) return launch<256, false, true, false, true>(p, st);
  if (a_mn && b_mn) return launch<256, true, true, false, true>(p, st);
  return launch<256, true, false, false, true>(p, st);
}

}  // namespace gk
}  // namespace bpt
