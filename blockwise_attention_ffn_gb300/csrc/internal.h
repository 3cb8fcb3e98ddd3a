// internal.h -- host-side interfaces between the C ABI (bpt_api.cu) and the
// kernel launchers.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/bpt.h"

namespace bpt {

// ---------------------------------------------------------------- profiling
// When enabled (bpt_profile_enable), every launch is bracketed by CUDA events
// on its stream and tagged with its kind and algorithmic work.
enum ProfKind { PROF_GEMM = 0, PROF_ATTN_FWD = 1, PROF_ATTN_BWD = 2, PROF_NORM = 3, PROF_MISC = 4, PROF_KINDS = 5 };
struct ProfScope {
  ProfScope(int kind, double flops, double bytes, cudaStream_t st);
  ~ProfScope();
  int slot;
  cudaStream_t st;
};

// Device address of this device's error word (4 x u32), or NULL.
unsigned int* device_error_word();
int read_device_error(cudaStream_t st, unsigned int out[4]);
// streaming multiprocessors of the current device (0 on error), cached per device
int sm_count();
// 0 if [p, p + bytes) lies inside one device allocation of the current
// device, else 1 (the debug checks of BPT_FLAG_DEBUG_CHECKS)
int check_device_range(const void* p, size_t bytes);

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (the attribute belongs to the kernel's instance in
// that device's context).  `done` is the caller's per-kernel bit mask of
// devices already set.  Returns 0 on success, 3 (BPT_ECUDA) on failure.
inline int smem_limit_once(const void* kernel, int bytes, std::atomic<uint64_t>* done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 3;
  const uint64_t bit = uint64_t(1) << dev;
  if (done->load(std::memory_order_acquire) & bit) return 0;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return 3;
  done->fetch_or(bit, std::memory_order_release);
  return 0;
}

// ---------------------------------------------------------------- TMA maps
// 2-D bf16 (or fp32) tensor map over a row-major matrix view [rows, cols]
// with a leading dimension of `ld` elements.  box = {box_cols, box_rows};
// swizzle_bytes in {0, 32, 64, 128}.  Returns 0 on success.
int make_map_2d(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                uint32_t box_cols, uint32_t box_rows, int swizzle_bytes, int elem_bytes = 2);

// ---------------------------------------------------------------- GEMM
// C[M, N] = A[M, K] * B[N, K]^T with bf16 operands and fp32 accumulation in
// TMEM, followed by a fused epilogue.
//   A: K-major storage [M rows, K cols] (a_mn = false) or MN-major storage
//      [K rows, M cols] (a_mn = true).
//   B: up to three segments that are concatenated along K (b_seg_k[i] rows of
//      K each), each K-major [N rows, K_i cols] or MN-major [K_i rows, N cols].
//      Every segment but the last must hold a multiple of 64 K.
//   dual: a second B (b2, same major/shape) whose product goes to a second
//      accumulator; used by the SwiGLU gate/up pair.
struct MatView {
  const void* ptr;
  int64_t rows, cols, ld;  // elements
};

enum EpiKind {
  EPI_BF16 = 0,        // out = acc (+ bias[n]) (+ res[m, n])            -> bf16
  EPI_GELU = 1,        // z = acc + bias; out = gelu(z); out2 = gelu'(z) (opt) -> bf16
  EPI_SWIGLU = 2,      // dual: out = silu(g) * u; out2 = g, out3 = u (opt) -> bf16
  EPI_GELU_BWD = 3,    // out = acc * aux[m, n] (aux = gelu'(z))          -> bf16
  EPI_SWIGLU_BWD = 4,  // acc = dA; g = aux, u = aux2: out = dA*u*silu'(g), out2 = dA*silu(g)
  EPI_F32 = 5,         // out = acc (+ bias) (+ res) + beta * out        -> fp32
  // language-model loss, logits z = acc of column n (vocabulary id col0 + n):
  EPI_LSE = 6,         // per row and tile half: (max z, sum exp(z - max)) over
                       // the valid columns -> float2 out[part * ldo + m],
                       // part = 2 * tile column + half (tiles are 256 columns
                       // wide, so part = column / 128); z of the row's target
                       // rowi[m] (if in this tile) -> float out2[m]
  EPI_CE_GRAD = 7,     // out = (exp(z - rowf[m]) - [col0 + n == rowi[m]]) * scale -> bf16
};

struct Epilogue {
  int kind = EPI_BF16;
  int act = 0;  // gelu variant: 0 erf, 1 tanh
  void* out = nullptr;
  int64_t ldo = 0;
  void* out2 = nullptr;
  int64_t ldo2 = 0;
  void* out3 = nullptr;
  int64_t ldo3 = 0;
  const void* bias = nullptr;  // bf16 [N]
  const void* res = nullptr;   // [M, N] with ldr: bf16, or fp32 when res_f32
  int64_t ldr = 0;
  int res_f32 = 0;
  const void* aux = nullptr;
  int64_t ldaux = 0;
  const void* aux2 = nullptr;
  int64_t ldaux2 = 0;
  float beta = 0.f;
  // fixed summation order: no K split (a split adds its K ranges' shares in
  // L2 in whatever order they land)
  int deterministic = 0;
  // per-row inputs of the loss epilogues: rowf fp32 [M] (log-sum-exp),
  // rowi int32 [M] (target ids); scale; col0 = vocabulary id of column 0
  const float* rowf = nullptr;
  const int* rowi = nullptr;
  float scale = 1.f;
  int64_t col0 = 0;
};

// Returns 0 or a BPT_* status.
int gemm(int64_t M, int64_t N, int64_t K, const MatView& A, bool a_mn, const MatView* B,
         const int64_t* b_seg_k, int nseg, bool b_mn, const MatView* B2, const Epilogue& epi,
         cudaStream_t stream);

// ---------------------------------------------------------------- attention
struct AttnShape {
  int b, s, H, Hkv, d;
  int causal;
  // packed projection buffer [b*s, ld_qkv]: Q heads at column q_col + n*d,
  // K heads at k_col + g*d, V heads at v_col + g*d (heads local to the call)
  int64_t ld_qkv, q_col, k_col, v_col;
  // output O [b*s, ld_o], head n at column o_col + n*d; LSE [b, H_total, s]
  // at head offset lse_head0 (nullable)
  int64_t ld_o, o_col;
  int H_total, lse_head0;
  // query rows processed: [q_begin, q_end) of every sequence; O row of query
  // q of sequence bi is bi*s + q - o_row0 (o_row0 lets a caller pass a
  // buffer that holds only the processed block)
  int q_begin, q_end;
  int64_t o_row0;
  // heads spread over the output (interleaved stages): local head n goes to
  // output head (n / o_seg) * o_seg_stride + n % o_seg (O columns and LSE
  // rows, both after o_col / lse_head0); o_seg = 0: output head n
  int o_seg = 0, o_seg_stride = 0;
};
int attention_fwd(const AttnShape& sh, const void* qkv, void* o, float* lse, cudaStream_t st);

struct AttnBwdShape {
  AttnShape f;            // forward geometry (q_begin/q_end ignored: all rows)
  int64_t ld_do, do_col;  // dO [b*s, ld_do], head n at do_col + n*d
  int64_t ld_dqkv, dq_col, dk_col, dv_col;  // outputs, bf16
  // one MMA-issuing thread per CTA, so every accumulator takes its products
  // in a fixed order (the default two issuers add in arrival order)
  int deterministic = 0;
};
// ws: fp32 dQ accumulator [b*s, H*d] followed by D [b, H, s_pad] fp32
// (s_pad = s rounded up to 128); lse is [b, H_total, s_pad].
size_t attention_bwd_ws_bytes(const AttnBwdShape& sh);
int attention_bwd(const AttnBwdShape& sh, const void* qkv, const void* o, const float* lse,
                  const void* dout, void* dqkv, void* ws, cudaStream_t st);

// The checks and launches of bpt_attention_bwd with the workspace given;
// ws_is_library: the workspace is the library's own array (the
// no-allocation entry point), which the debug checks do not inspect.
int attention_bwd_call(const bpt_config* cfg, const void* qkv, const void* o, const void* lse, const void* dout,
                       void* dqkv, void* ws, size_t ws_bytes, void* stream, int ws_is_library);

// ---------------------------------------------------------------- norms & misc
// y = norm(x) * w (+ b), rows of width h; x is bf16 or (x_f32) fp32; y bf16.
int norm_fwd(int64_t rows, int h, int kind, float eps, const void* x, int x_f32, int64_t ldx,
             const void* w, const void* b, void* y, int64_t ldy, cudaStream_t st);
// dx = res + d/dx norm (given dy, x, w); dw/db partial sums accumulated into
// the fp32 vectors (they must be zeroed or hold the running sum): with
// atomics, or, when `part` is given, written per block to part and added in
// block order by a second kernel (a fixed summation order; part holds
// norm_bwd_part_floats(h) floats).
// dy, x and res are each bf16 or fp32 (the *_f32 flags); dx is written as
// bf16 and, when dx_f32 is given, also as fp32 (same leading dimension).
struct NormBwdIO {
  const void* dy; int dy_f32; int64_t lddy;
  const void* x; int x_f32; int64_t ldx;
  const void* res; int res_f32; int64_t ldres;
  void* dx; float* dx_f32; int64_t lddx;
};
int norm_bwd(int64_t rows, int h, int kind, float eps, const NormBwdIO& io, const void* w, float* dw,
             float* db, cudaStream_t st, float* part = nullptr);
int64_t norm_bwd_part_floats(int h);
// out[n] (+)= sum over rows of in[row, n]  (bf16 in, fp32 out); with atomics,
// or, when `part` is given (colsum_part_floats(n) floats), per-band partial
// sums added in band order by a second kernel
int colsum(int64_t rows, int64_t n, const void* in, int64_t ld, float* out, int accumulate,
           cudaStream_t st, float* part = nullptr);
int64_t colsum_part_floats(int64_t n);
// Rotary position embedding in place: n_heads heads of d columns from column
// col0 of bf16 buf [rows, ld], row r at position r % s, pair (i, i + d/2)
// turned by (r % s) * base^(-2i/d) (inverse: by minus that).  d % 4 == 0,
// d <= 128.
int rope_apply(int64_t rows, int s, void* buf, int64_t ld, int col0, int n_heads, int d, float base, int inverse,
               cudaStream_t st);
// dst bf16 [rows, n] (ld_dst) = src fp32 [rows, n] (ld_src) * scale
int f32_to_bf16(int64_t rows, int64_t n, const float* src, int64_t ld_src, void* dst,
                int64_t ld_dst, float scale, cudaStream_t st);

}  // namespace bpt
