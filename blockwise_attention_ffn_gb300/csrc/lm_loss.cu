// lm_loss.cu -- the language-model loss after the last layer, blockwise:
// logits z = x W^T through the [V, h] vocabulary projection, the mean token
// cross-entropy over the n positions, and its gradients, without the n x V
// logit matrix ever existing.
//
// "Blockwise Parallel Transformer for Long Context Large Models", section 3
// (the note on the cross-entropy loss before Algorithm 1): the blockwise
// schedule covers the final loss too.  "Untied Ulysses ...", the paragraph on
// Arctic Long Sequence Training and its Table 1: the loss is the largest
// activation term (240 S d_model bytes) and is tiled.
//
//   loss = (1/n) sum_i (lse_i - z_i,t_i),   lse_i = log sum_v exp(z_iv)
//   dz_i = dloss * (softmax(z_i) - onehot(t_i)) / n,  dx = dz W,  dW = dz^T x
//
// Forward: one persistent GEMM over the whole vocabulary whose epilogue
// reduces each row's half-tile of 128 logits to an online (max, sum of
// exponentials) pair and picks the target's logit (EPI_LSE); a second kernel
// combines the pairs of a row (the same carry rule as the attention's online
// softmax) into its log-sum-exp and loss term, and a third sums the terms in
// a fixed order.  No more than one pair per row and half-tile is kept (2 x
// ceil(V/256) x n x 8 bytes), against 2 n V bytes of bf16 logits.
//
// Backward: the vocabulary in blocks of c_v columns.  Per block the logits
// are rebuilt with the gradient as the GEMM epilogue (EPI_CE_GRAD, into one
// n x c_v bf16 buffer reused by every block), then dx += dz_blk W_blk (fp32
// accumulator, the last block's epilogue rounding to bf16) and dW_blk =
// dz_blk^T x.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <algorithm>

#include "../../include/bpt.h"
#include "internal.h"
#include "ptx.cuh"

namespace bpt {

namespace {

constexpr int LM_TILE_N = 256;  // the GEMM's tile width: one (max, sum) pair per row and half
constexpr int LM_BAD_TARGET_SITE = 950;

struct LmDims {
  int64_t n, h, V, cv, nparts, nblk;
  bool det, debug, accum;
};

int lm_validate(const bpt_lm_config* c, LmDims* D) {
  if (!c) return BPT_EINVAL;
  if (c->n < 1 || c->h < 8 || (c->h % 8) || c->vocab < 1) return BPT_EINVAL;
  if (c->vocab_block < 0 || (c->vocab_block % LM_TILE_N)) return BPT_EINVAL;
  if (c->flags & ~(BPT_FLAG_ACCUM_GRADS | BPT_FLAG_DETERMINISTIC | BPT_FLAG_DEBUG_CHECKS)) return BPT_EINVAL;
  D->n = c->n;
  D->h = c->h;
  D->V = c->vocab;
  const int64_t vpad = (D->V + LM_TILE_N - 1) / LM_TILE_N * LM_TILE_N;
  D->cv = c->vocab_block ? std::min<int64_t>(c->vocab_block, vpad) : std::min<int64_t>(8192, vpad);
  D->nparts = 2 * ((D->V + LM_TILE_N - 1) / LM_TILE_N);
  D->nblk = (D->V + D->cv - 1) / D->cv;
  D->det = (c->flags & BPT_FLAG_DETERMINISTIC) != 0;
  D->debug = (c->flags & BPT_FLAG_DEBUG_CHECKS) != 0;
  D->accum = (c->flags & BPT_FLAG_ACCUM_GRADS) != 0;
  return BPT_OK;
}

struct LmFwdWs {
  float2* part;
  float *zt, *row_loss, *lse;
};
struct LmBwdWs {
  void* dz;
  float* dx_acc;
};

size_t take(size_t& off, size_t bytes) {
  const size_t at = off;
  off += (bytes + 255) / 256 * 256;
  return at;
}

size_t plan_lm_fwd(const LmDims& D, void* base, LmFwdWs* w, bool need_lse) {
  uint8_t* b = reinterpret_cast<uint8_t*>(base);
  size_t off = 0;
  const size_t p = take(off, (size_t)D.nparts * D.n * sizeof(float2));
  const size_t z = take(off, (size_t)D.n * 4);
  const size_t r = take(off, (size_t)D.n * 4);
  const size_t l = need_lse ? take(off, (size_t)D.n * 4) : 0;
  if (b) {
    w->part = reinterpret_cast<float2*>(b + p);
    w->zt = reinterpret_cast<float*>(b + z);
    w->row_loss = reinterpret_cast<float*>(b + r);
    w->lse = need_lse ? reinterpret_cast<float*>(b + l) : nullptr;
  }
  return off;
}

size_t plan_lm_bwd(const LmDims& D, void* base, LmBwdWs* w) {
  uint8_t* b = reinterpret_cast<uint8_t*>(base);
  size_t off = 0;
  const size_t z = take(off, (size_t)D.n * D.cv * 2);
  const size_t a = D.nblk > 1 ? take(off, (size_t)D.n * D.h * 4) : 0;
  if (b) {
    w->dz = b + z;
    w->dx_acc = D.nblk > 1 ? reinterpret_cast<float*>(b + a) : nullptr;
  }
  return off;
}

// Row i: lse_i from its pairs (m_p, l_p): m = max m_p, l = sum l_p exp(m_p -
// m) (pairs of an empty half are (-inf, 0) and add nothing), and the loss
// term lse_i - z_i,t.  A target outside [0, V) is recorded in the error word
// (BPT_EINVAL at site 950) and its row's term is lse_i alone.
__global__ void lm_combine_kernel(int64_t n, int nparts, int64_t V, const float2* part, const float* zt,
                                  const int* targets, float* lse, float* row_loss, unsigned int* err) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float m = -INFINITY;
  for (int p = 0; p < nparts; ++p) m = fmaxf(m, part[(int64_t)p * n + i].x);
  float l = 0.f;
  for (int p = 0; p < nparts; ++p) {
    const float2 q = part[(int64_t)p * n + i];
    l += q.y * __expf(q.x - m);
  }
  const float v = m + logf(l);
  lse[i] = v;
  const int t = targets[i];
  const bool ok = t >= 0 && (int64_t)t < V;
  if (!ok) report_bad_data(err, LM_BAD_TARGET_SITE);
  row_loss[i] = v - (ok ? zt[i] : 0.f);
}

// loss = (sum of the row terms) / n, summed in a fixed order: thread k takes
// rows k, k + 1024, ... in turn (fp64), then a fixed tree over the threads.
__global__ void __launch_bounds__(1024) lm_mean_kernel(int64_t n, const float* row_loss, float* loss) {
  __shared__ double acc[1024];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += 1024) s += (double)row_loss[i];
  acc[threadIdx.x] = s;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) acc[threadIdx.x] += acc[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = (float)(acc[0] / (double)n);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct Span {
  const void* p;
  int64_t bytes;
};
int check_spans(const Span* sp, int k) {
  for (int i = 0; i < k; ++i)
    if (sp[i].bytes > 0 && check_device_range(sp[i].p, (size_t)sp[i].bytes)) return BPT_EINVAL;
  return BPT_OK;
}
int debug_finish(cudaStream_t st) {
  unsigned int e[4] = {0, 0, 0, 0};
  if (read_device_error(st, e)) return BPT_ECUDA;
  if (!e[0]) return BPT_OK;
  return e[0] == BPT_EINVAL ? BPT_EINVAL : BPT_ETIMEOUT;
}

}  // namespace
}  // namespace bpt

using namespace bpt;

extern "C" {

size_t bpt_lm_workspace_bytes(const bpt_lm_config* cfg, int pass) {
  LmDims D;
  if (lm_validate(cfg, &D)) return 0;
  if (pass == BPT_PASS_FWD) return plan_lm_fwd(D, nullptr, nullptr, true);
  if (pass == BPT_PASS_BWD) return plan_lm_bwd(D, nullptr, nullptr);
  return 0;
}

int bpt_lm_loss_fwd(const bpt_lm_config* cfg, const void* x, const void* w, const int32_t* targets, float* loss,
                    float* lse, void* ws, size_t ws_bytes, void* stream) {
  LmDims D;
  int rc = lm_validate(cfg, &D);
  if (rc) return rc;
  if (!x || !w || !targets || !loss || !ws) return BPT_EINVAL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(targets) & 3) ||
      (reinterpret_cast<uintptr_t>(loss) & 3) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3)))
    return BPT_EINVAL;
  LmFwdWs W;
  const size_t need = plan_lm_fwd(D, nullptr, nullptr, lse == nullptr);
  if (ws_bytes < need) return BPT_ENOSPC;
  if (D.debug) {
    const Span sp[] = {{x, D.n * D.h * 2}, {w, D.V * D.h * 2}, {targets, D.n * 4}, {loss, 4},
                       {lse, lse ? D.n * 4 : 0}, {ws, (int64_t)need}};
    if (check_spans(sp, 6)) return BPT_EINVAL;
  }
  plan_lm_fwd(D, ws, &W, lse == nullptr);
  float* lse_out = lse ? lse : W.lse;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* err = device_error_word();
  if (!err) return BPT_ECUDA;
  {
    // logits of every row against the whole vocabulary, reduced in the
    // epilogue to one (max, sum exp) pair per row and half-tile
    MatView A{x, D.n, D.h, D.h};
    MatView B{w, D.V, D.h, D.h};
    Epilogue e;
    e.kind = EPI_LSE;
    e.out = W.part;
    e.ldo = D.n;
    e.out2 = W.zt;
    e.rowi = targets;
    e.deterministic = D.det;
    const int64_t K = D.h;
    if ((rc = gemm(D.n, D.V, D.h, A, false, &B, &K, 1, false, nullptr, e, st))) return rc;
  }
  {
    ProfScope prof(PROF_MISC, 0.0, (double)D.n * (D.nparts * 8.0 + 16.0), st);
    lm_combine_kernel<<<(unsigned)((D.n + 255) / 256), 256, 0, st>>>(D.n, (int)D.nparts, D.V, W.part, W.zt, targets,
                                                                      lse_out, W.row_loss, err);
    if (cudaGetLastError() != cudaSuccess) return BPT_ECUDA;
    lm_mean_kernel<<<1, 1024, 0, st>>>(D.n, W.row_loss, loss);
    if (cudaGetLastError() != cudaSuccess) return BPT_ECUDA;
  }
  return D.debug ? debug_finish(st) : BPT_OK;
}

int bpt_lm_loss_bwd(const bpt_lm_config* cfg, const void* x, const void* w, const int32_t* targets,
                    const float* lse, float dloss, void* dx, float* dw, void* ws, size_t ws_bytes, void* stream) {
  LmDims D;
  int rc = lm_validate(cfg, &D);
  if (rc) return rc;
  if (!x || !w || !targets || !lse || !dx || !dw || !ws) return BPT_EINVAL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(dx) || !aligned16(dw) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(targets) & 3) || (reinterpret_cast<uintptr_t>(lse) & 3))
    return BPT_EINVAL;
  if (!(fabsf(dloss) < INFINITY)) return BPT_EINVAL;
  LmBwdWs W;
  const size_t need = plan_lm_bwd(D, nullptr, nullptr);
  if (ws_bytes < need) return BPT_ENOSPC;
  if (D.debug) {
    const Span sp[] = {{x, D.n * D.h * 2},  {w, D.V * D.h * 2}, {targets, D.n * 4}, {lse, D.n * 4},
                       {dx, D.n * D.h * 2}, {dw, D.V * D.h * 4}, {ws, (int64_t)need}};
    if (check_spans(sp, 7)) return BPT_EINVAL;
  }
  plan_lm_bwd(D, ws, &W);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const float scale = dloss / (float)D.n;
  for (int64_t k = 0; k < D.nblk; ++k) {
    const int64_t v0 = k * D.cv;
    const int64_t nv = std::min(D.cv, D.V - v0);
    const void* wb = reinterpret_cast<const uint8_t*>(w) + v0 * D.h * 2;
    // dz = dloss (softmax - onehot) / n over the block's columns
    {
      MatView A{x, D.n, D.h, D.h};
      MatView B{wb, nv, D.h, D.h};
      Epilogue e;
      e.kind = EPI_CE_GRAD;
      e.out = W.dz;
      e.ldo = D.cv;
      e.rowf = lse;
      e.rowi = targets;
      e.scale = scale;
      e.col0 = v0;
      e.deterministic = D.det;
      const int64_t K = D.h;
      if ((rc = gemm(D.n, nv, D.h, A, false, &B, &K, 1, false, nullptr, e, st))) return rc;
    }
    // dW[v0 : v0 + nv] (+)= dz^T x
    {
      MatView A{W.dz, D.n, nv, D.cv};  // MN-major: [K = n rows, M = nv columns]
      MatView B{x, D.n, D.h, D.h};     // MN-major: [K = n rows, N = h columns]
      Epilogue e;
      e.kind = EPI_F32;
      e.out = dw + v0 * D.h;
      e.ldo = D.h;
      e.beta = D.accum ? 1.f : 0.f;
      e.deterministic = D.det;
      const int64_t K = D.n;
      if ((rc = gemm(nv, D.h, D.n, A, true, &B, &K, 1, true, nullptr, e, st))) return rc;
    }
    // dx (+)= dz W_blk: fp32 across blocks, the last block rounds to bf16
    {
      MatView A{W.dz, D.n, nv, D.cv};
      MatView B{wb, nv, D.h, D.h};  // MN-major: [K = nv rows, N = h columns]
      Epilogue e;
      e.deterministic = D.det;
      const bool last = k == D.nblk - 1;
      if (last) {
        e.kind = EPI_BF16;
        e.out = dx;
        e.ldo = D.h;
        if (k > 0) {
          e.res = W.dx_acc;
          e.res_f32 = 1;
          e.ldr = D.h;
        }
      } else {
        e.kind = EPI_F32;
        e.out = W.dx_acc;
        e.ldo = D.h;
        e.beta = k > 0 ? 1.f : 0.f;
      }
      const int64_t K = nv;
      if ((rc = gemm(D.n, D.h, nv, A, false, &B, &K, 1, true, nullptr, e, st))) return rc;
    }
  }
  return D.debug ? debug_finish(st) : BPT_OK;
}

}  // extern "C"
