// bpt_api.cu -- the C ABI (include/bpt.h): argument validation, workspace
// planning and the launch sequences of the forward pass, the recompute
// backward pass and the head-chunked attention.
//
// Forward schedule ("Blockwise Parallel Transformer for Long Context Large
// Models", section 3.2 and Algorithm 1): N1 and the Q/K/V projection for the
// whole sequence (they are position-wise and not part of the memory
// optimisation); then, for every FFN block of c_f query rows: attention of
// those rows over their key/value blocks, output projection + bias +
// residual, N2, fc1 + activation, fc2 + bias + residual -> y.  Only a
// c_f x f block of the FFN intermediate ever exists.
//
// Head-chunk mode ("Untied Ulysses ...", section 3.4 "The Core Mechanism:
// Headwise Chunking via UPipe", restricted to one GPU): the projection and
// attention run in H/U stages of U query heads and U/G key/value heads; the
// stage buffer is reused and the attention output buffer is filled slice by
// slice; the FFN blocks follow.
//
// Backward ("Training memory ...", section 3, full activation checkpointing:
// rerun the forward, then the backward): N1, Q/K/V and attention are rebuilt
// (the saved log-sum-exp is reused by the attention backward); per FFN block
// x1, N2, fc1 are rebuilt and the FFN / N2 gradients formed; then the output
// projection, attention (per stage) and Q/K/V gradients, and N1.
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>

#include "../../include/bpt.h"
#include "internal.h"

using namespace bpt;

namespace {

struct Dims {
  int64_t b, s, h, H, Hkv, d, f, G, U, cf, s_pad, rows, n_stages;
  bool chunked;
  int64_t Uk;      // key/value heads per stage
  int64_t qkv_w;   // columns of the (stage) projection buffer
  float rope;      // rotary embedding base (0: none)
  bool det;        // BPT_FLAG_DETERMINISTIC
  bool debug;      // BPT_FLAG_DEBUG_CHECKS
  bool interleave; // interleaved stages (chunked, BPT_STAGE_INTERLEAVED)
  int64_t m;       // interleaved: query heads of each group per stage (U / H_kv)
  int64_t iw;      // interleaved: columns of the stage buffer, U d + 2 H_kv d
  int save;        // BPT_SAVE_*
  int64_t full_w;  // columns of Q/K/V of every head, (H + 2 H_kv) d
};

int validate(const bpt_config* c, Dims* D) {
  if (!c) return BPT_EINVAL;
  if (c->b < 1 || c->s < 1 || c->h < 8 || (c->h % 8) || c->n_heads < 1 || c->n_kv_heads < 1 ||
      (c->n_heads % c->n_kv_heads) || c->ffn_dim < 8 || (c->ffn_dim % 8))
    return BPT_EINVAL;
  if (c->norm != BPT_NORM_LAYER && c->norm != BPT_NORM_RMS) return BPT_EINVAL;
  if (c->act < 0 || c->act > 2) return BPT_EINVAL;
  if (c->has_bias != 0 && c->has_bias != 1) return BPT_EINVAL;
  if (c->causal != 0 && c->causal != 1) return BPT_EINVAL;
  if (c->rope_base != 0.f && !(c->rope_base > 1.f && c->rope_base < 3.0e38f)) return BPT_EINVAL;
  if (c->q_block <= 0 || (c->q_block % 128) || c->kv_block <= 0 || (c->kv_block % 128)) return BPT_EINVAL;
  if (c->ffn_block < 0 || (c->ffn_block % c->q_block)) return BPT_EINVAL;
  if (!(c->norm_eps > 0.f)) return BPT_EINVAL;
  if (c->act == BPT_ACT_SWIGLU && (c->ffn_dim % 64)) return BPT_EINVAL;
  if (c->flags & ~(BPT_FLAG_ACCUM_GRADS | BPT_FLAG_ONE_STREAM | BPT_FLAG_DETERMINISTIC | BPT_FLAG_DEBUG_CHECKS))
    return BPT_EINVAL;
  const int d = c->head_dim;
  if (d != 64 && d != 80 && d != 96 && d != 112 && d != 128) return BPT_EUNSUPPORTED;
  const int G = c->n_heads / c->n_kv_heads;
  int U = c->head_chunk;
  if (U == 0) U = c->n_heads;
  if (U < 1 || (c->n_heads % U) || (U % G)) return BPT_EINVAL;
  if (c->stage_order != BPT_STAGE_CONTIGUOUS && c->stage_order != BPT_STAGE_INTERLEAVED) return BPT_EINVAL;
  if (c->stage_order == BPT_STAGE_INTERLEAVED && (U % c->n_kv_heads)) return BPT_EINVAL;
  if (c->save_policy < BPT_SAVE_NOTHING || c->save_policy > BPT_SAVE_ATTN_OUT) return BPT_EINVAL;
  if ((int64_t)c->s * c->b >= (int64_t(1) << 31)) return BPT_EINVAL;
  D->b = c->b;
  D->s = c->s;
  D->h = c->h;
  D->H = c->n_heads;
  D->Hkv = c->n_kv_heads;
  D->d = d;
  D->f = c->ffn_dim;
  D->G = G;
  D->U = U;
  D->Uk = U / G;
  D->chunked = U < c->n_heads;
  D->n_stages = c->n_heads / U;
  D->s_pad = (D->s + 127) / 128 * 128;
  D->cf = c->ffn_block ? c->ffn_block : std::min<int64_t>(2048, D->s_pad);
  D->cf = std::min<int64_t>(D->cf, D->s_pad);
  D->rows = D->b * D->s;
  D->qkv_w = (D->U + 2 * D->Uk) * d;
  D->rope = c->rope_base;
  D->det = (c->flags & BPT_FLAG_DETERMINISTIC) != 0;
  D->debug = (c->flags & BPT_FLAG_DEBUG_CHECKS) != 0;
  D->interleave = D->chunked && c->stage_order == BPT_STAGE_INTERLEAVED;
  D->m = U / c->n_kv_heads;
  D->iw = (U + 2 * (int64_t)c->n_kv_heads) * d;
  D->save = c->save_policy;
  D->full_w = (D->H + 2 * D->Hkv) * d;
  return BPT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_weights(const bpt_config* c, const bpt_weights* w) {
  if (!w) return BPT_EINVAL;
  const void* need[] = {w->ln1_w, w->wq, w->wk, w->wv, w->wo, w->ln2_w, w->w1, w->w2};
  for (const void* p : need)
    if (!p || !aligned16(p)) return BPT_EINVAL;
  if (c->norm == BPT_NORM_LAYER && (!w->ln1_b || !w->ln2_b || !aligned16(w->ln1_b) || !aligned16(w->ln2_b)))
    return BPT_EINVAL;
  if (c->act == BPT_ACT_SWIGLU && (!w->w3 || !aligned16(w->w3))) return BPT_EINVAL;
  if (c->has_bias) {
    const void* bs[] = {w->bq, w->bk, w->bv, w->bo, w->b2};
    for (const void* p : bs)
      if (!p || !aligned16(p)) return BPT_EINVAL;
    if (c->act != BPT_ACT_SWIGLU && (!w->b1 || !aligned16(w->b1))) return BPT_EINVAL;
  }
  return BPT_OK;
}

// ---------------------------------------------------------------- debug checks
// BPT_FLAG_DEBUG_CHECKS: every pointer argument, with the bytes the call
// touches through it, must lie inside one device allocation of the current
// device; after the launches the call synchronises and reports the device
// error word itself.
struct Span {
  const void* p;
  int64_t bytes;
};

int check_spans(const Span* sp, int n) {
  for (int i = 0; i < n; ++i)
    if (sp[i].bytes > 0 && check_device_range(sp[i].p, (size_t)sp[i].bytes)) return BPT_EINVAL;
  return BPT_OK;
}

// The parameters a config uses (bpt_weights / bpt_grads field order), `elem`
// bytes per element; returns the count written to out[17].
int param_spans(const bpt_config* c, const Dims& D, const void* const f[17], int elem, Span* out) {
  const bool ln = c->norm == BPT_NORM_LAYER, hb = c->has_bias != 0, sw = c->act == BPT_ACT_SWIGLU;
  const int64_t h = D.h, q = D.H * D.d, kv = D.Hkv * D.d, ff = D.f;
  const int64_t n[17] = {h,          ln ? h : 0,  q * h,  hb ? q : 0,           kv * h, hb ? kv : 0,
                         kv * h,     hb ? kv : 0, h * q,  hb ? h : 0,           h,      ln ? h : 0,
                         ff * h,     hb && !sw ? ff : 0,  h * ff, hb ? h : 0,   sw ? ff * h : 0};
  for (int i = 0; i < 17; ++i) out[i] = Span{f[i], n[i] * elem};
  return 17;
}

int check_weights_range(const bpt_config* c, const Dims& D, const bpt_weights* w) {
  const void* f[17] = {w->ln1_w, w->ln1_b, w->wq, w->bq, w->wk, w->bk, w->wv, w->bv, w->wo,
                       w->bo,    w->ln2_w, w->ln2_b, w->w1, w->b1, w->w2, w->b2, w->w3};
  Span sp[17];
  return check_spans(sp, param_spans(c, D, f, 2, sp));
}

int check_grads_range(const bpt_config* c, const Dims& D, const bpt_grads* g) {
  const void* f[17] = {g->ln1_w, g->ln1_b, g->wq, g->bq, g->wk, g->bk, g->wv, g->bv, g->wo,
                       g->bo,    g->ln2_w, g->ln2_b, g->w1, g->b1, g->w2, g->b2, g->w3};
  Span sp[17];
  return check_spans(sp, param_spans(c, D, f, 4, sp));
}

// After the launches: wait for them and report the error word (which the
// read clears) or the failure of the synchronisation itself.
int debug_finish(cudaStream_t st) {
  unsigned int e[4] = {0, 0, 0, 0};
  if (read_device_error(st, e)) return BPT_ECUDA;
  if (!e[0]) return BPT_OK;
  return e[0] == BPT_EINVAL ? BPT_EINVAL : BPT_ETIMEOUT;
}

// ---------------------------------------------------------------- workspace
struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(reinterpret_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off += (bytes + 255) / 256 * 256;
    return p;
  }
};

// What the forward keeps for the backward (the caller's `saved` buffer):
// the log-sum-exp [b, H, s_pad] fp32, then with BPT_SAVE_PROJECTIONS Q, K, V
// of every head [rows, (H + 2 H_kv) d] (the unchunked packed layout), then
// with BPT_SAVE_ATTN_OUT the attention output O [rows, H d].
struct Saved {
  float* lse;
  void *qkv, *o;
};
size_t plan_saved(const Dims& D, const void* base, Saved* sv) {
  Carve c(const_cast<void*>(base));
  sv->lse = reinterpret_cast<float*>(c.take(D.b * D.H * D.s_pad * 4));
  sv->qkv = D.save >= BPT_SAVE_PROJECTIONS ? c.take(D.rows * D.full_w * 2) : nullptr;
  sv->o = D.save >= BPT_SAVE_ATTN_OUT ? c.take(D.rows * D.H * D.d * 2) : nullptr;
  return c.off;
}

struct FwdWs {
  void *xn, *qkv, *o, *x1, *x1n, *a;
  float* lse;
  void *wq_perm, *bq_perm;  // interleaved stages: Wq (and bq) rows in stage order
};
// saving: whether the call keeps the backward's activations (a `saved`
// buffer is given); the projections and O then live there, not here
size_t plan_fwd(const Dims& D, void* base, FwdWs* w, bool need_lse, bool saving) {
  Carve c(base);
  const bool keep_qkv = saving && D.save >= BPT_SAVE_PROJECTIONS;
  const bool keep_o = saving && D.save >= BPT_SAVE_ATTN_OUT;
  w->xn = c.take(D.rows * D.h * 2);
  w->qkv = D.interleave ? c.take(D.rows * D.iw * 2) : keep_qkv ? nullptr : c.take(D.rows * D.qkv_w * 2);
  w->o = keep_o ? nullptr : c.take((D.chunked ? D.rows : D.cf) * D.H * D.d * 2);
  w->x1 = c.take(D.cf * D.h * 4);  // fp32 residual stream
  w->x1n = c.take(D.cf * D.h * 2);
  w->a = c.take(D.cf * D.f * 2);
  w->lse = reinterpret_cast<float*>(need_lse ? c.take(D.b * D.H * D.s_pad * 4) : nullptr);
  w->wq_perm = D.interleave ? c.take(D.H * D.d * D.h * 2) : nullptr;
  w->bq_perm = D.interleave ? c.take(D.H * D.d * 2) : nullptr;
  return c.off;
}

struct BwdWs {
  void *xn, *qkv, *o, *x1, *x1n, *gd, *g, *u, *a, *dz, *dx1n, *dx1, *dO, *dqkv, *attn;
  float *dxn, *dx1f;
  // fixed-order mode: per-block partial sums of the norm backward (main
  // stream) and of the bias column sums (second stream); null otherwise
  float *part_main, *part_side;
};
AttnBwdShape stage_bwd_shape(const Dims& D, int64_t k);
size_t plan_bwd(const Dims& D, void* base, BwdWs* w) {
  Carve c(base);
  // the FFN block buffers are sized for the larger (SwiGLU) case; the
  // projections and O come from the saved buffer when the forward kept them
  w->xn = c.take(D.rows * D.h * 2);
  w->qkv = D.save >= BPT_SAVE_PROJECTIONS ? nullptr : c.take(D.rows * D.qkv_w * 2);
  w->o = D.save >= BPT_SAVE_ATTN_OUT ? nullptr : c.take(D.rows * D.H * D.d * 2);
  w->x1 = c.take(D.cf * D.h * 4);  // fp32 residual stream
  w->x1n = c.take(D.cf * D.h * 2);
  w->gd = c.take(D.cf * D.f * 2);  // GeLU: gelu'(z) of the recompute; SwiGLU: gate g
  w->u = c.take(D.cf * D.f * 2);   // SwiGLU: up u
  w->g = w->gd;
  w->a = c.take(D.cf * D.f * 2);
  w->dz = c.take(D.cf * D.f * 2 * 2);  // GeLU: dz [cf, f]; SwiGLU: [dg | du] [cf, 2f]
  w->dx1n = c.take(D.cf * D.h * 2);
  w->dx1 = c.take(D.rows * D.h * 2);
  w->dx1f = reinterpret_cast<float*>(c.take(D.rows * D.h * 4));  // fp32 copy for the final residual sum
  w->dO = c.take(D.rows * D.H * D.d * 2);
  w->dqkv = c.take(D.rows * D.qkv_w * 2);
  w->dxn = reinterpret_cast<float*>(c.take(D.rows * D.h * 4));
  w->attn = c.take(attention_bwd_ws_bytes(stage_bwd_shape(D, 0)));
  w->part_main = w->part_side = nullptr;
  if (D.det) {
    w->part_main = reinterpret_cast<float*>(c.take(norm_bwd_part_floats((int)D.h) * 4));
    const int64_t widest = std::max(std::max(D.h, D.f), D.qkv_w);
    w->part_side = reinterpret_cast<float*>(c.take(colsum_part_floats(widest) * 4));
  }
  return c.off;
}

struct HcWs {
  void *qkv, *wq_perm, *bq_perm;
};
size_t plan_headchunk(const Dims& D, void* base, HcWs* w) {
  Carve c(base);
  w->qkv = c.take(D.rows * (D.interleave ? D.iw : D.qkv_w) * 2);
  w->wq_perm = D.interleave ? c.take(D.H * D.d * D.h * 2) : nullptr;
  w->bq_perm = D.interleave ? c.take(D.H * D.d * 2) : nullptr;
  return c.off;
}

// ---------------------------------------------------------------- pieces
const uint8_t* bf(const void* p, int64_t elems) { return reinterpret_cast<const uint8_t*>(p) + elems * 2; }
uint8_t* bfm(void* p, int64_t elems) { return reinterpret_cast<uint8_t*>(p) + elems * 2; }
float* f32(void* p, int64_t elems) { return reinterpret_cast<float*>(p) + elems; }

// rows of xn projected through n_out rows of a weight matrix (+ bias):
// out[:, 0:n_out] = xn W^T (+ bias), bf16 with row length ldo
int project(const Dims& D, const void* xn, const void* W, const void* bias, int64_t n_out, void* out, int64_t ldo,
            cudaStream_t st) {
  MatView A{xn, D.rows, D.h, D.h};
  MatView B{W, n_out, D.h, D.h};
  Epilogue e;
  e.kind = EPI_BF16;
  e.out = out;
  e.ldo = ldo;
  e.bias = bias;
  int64_t kseg = D.h;
  return gemm(D.rows, n_out, D.h, A, false, &B, &kseg, 1, false, nullptr, e, st);
}

// Where a stage's projections live: a buffer, its row length, and the
// columns of the stage's first query, key and value head.
struct QkvBuf {
  void* p;
  int64_t ld, q_col, k_col, v_col;
};
// the per-stage buffer: Q of the U heads, then K and V of their U/G heads
QkvBuf stage_buf(const Dims& D, void* p) { return QkvBuf{p, D.qkv_w, 0, D.U * D.d, (D.U + D.Uk) * D.d}; }
// stage k's heads inside the buffer of every head's projections that the
// forward keeps for the backward (BPT_SAVE_PROJECTIONS): [Q all | K all | V all]
QkvBuf kept_buf(const Dims& D, void* p, int64_t k) {
  return QkvBuf{p, D.full_w, k * D.U * D.d, D.H * D.d + k * D.Uk * D.d, (D.H + D.Hkv) * D.d + k * D.Uk * D.d};
}

// Q/K/V of stage k (all stages = one stage when not chunked) for all rows:
// Q = xn Wq[kU d : (k+1)U d]^T (+ bq), then K, V of the stage's U/G
// key/value heads, into the columns `b` names.  With rotary embedding, the
// stage's query and key heads are then rotated at their rows' positions.
int stage_qkv(const Dims& D, const bpt_weights* w, bool has_bias, const void* xn, const QkvBuf& b, int64_t k,
              cudaStream_t st) {
  const int64_t d = D.d, h = D.h;
  const int64_t q0 = k * D.U * d, kv0 = k * D.Uk * d;
  struct Piece {
    const void* W;
    const void* bias;
    int64_t row0, n, col;
  } pieces[3] = {{w->wq, w->bq, q0, D.U * d, b.q_col},
                 {w->wk, w->bk, kv0, D.Uk * d, b.k_col},
                 {w->wv, w->bv, kv0, D.Uk * d, b.v_col}};
  for (auto& pc : pieces) {
    int rc = project(D, xn, bf(pc.W, pc.row0 * h), has_bias ? bf(pc.bias, pc.row0) : nullptr, pc.n,
                     bfm(b.p, pc.col), b.ld, st);
    if (rc) return rc;
  }
  if (D.rope == 0.f) return 0;
  if (b.k_col == b.q_col + D.U * d)  // query and key heads adjacent: one pass
    return rope_apply(D.rows, (int)D.s, b.p, b.ld, (int)b.q_col, (int)(D.U + D.Uk), (int)d, D.rope, 0, st);
  int rc = rope_apply(D.rows, (int)D.s, b.p, b.ld, (int)b.q_col, (int)D.U, (int)d, D.rope, 0, st);
  return rc ? rc : rope_apply(D.rows, (int)D.s, b.p, b.ld, (int)b.k_col, (int)D.Uk, (int)d, D.rope, 0, st);
}

AttnShape stage_attn_shape(const Dims& D, int64_t k, int causal, const QkvBuf& b) {
  AttnShape a;
  a.b = (int)D.b;
  a.s = (int)D.s;
  a.H = (int)D.U;
  a.Hkv = (int)D.Uk;
  a.d = (int)D.d;
  a.causal = causal;
  a.ld_qkv = b.ld;
  a.q_col = b.q_col;
  a.k_col = b.k_col;
  a.v_col = b.v_col;
  a.ld_o = D.H * D.d;
  a.o_col = k * D.U * D.d;
  a.H_total = (int)D.H;
  a.lse_head0 = (int)(k * D.U);
  a.q_begin = 0;
  a.q_end = (int)D.s;
  a.o_row0 = 0;
  return a;
}

AttnBwdShape stage_bwd_shape(const Dims& D, int64_t k, const QkvBuf& b) {
  AttnBwdShape s;
  s.f = stage_attn_shape(D, k, 1, b);
  s.ld_do = D.H * D.d;
  s.do_col = k * D.U * D.d;
  s.ld_dqkv = D.qkv_w;
  s.dq_col = 0;
  s.dk_col = D.U * D.d;
  s.dv_col = (D.U + D.Uk) * D.d;
  return s;
}
AttnBwdShape stage_bwd_shape(const Dims& D, int64_t k) { return stage_bwd_shape(D, k, stage_buf(D, nullptr)); }

// Interleaved stages ("Untied Ulysses ...", section 4.1 "The GQA Scheduling
// Algorithm"): stage k takes the m = U / H_kv query heads gG + km .. gG + km
// + m - 1 of every group g.  Every stage needs every key/value head, so
// those are projected once, before the stages, into columns U d .. of the
// stage buffer and stay there; each stage projects only its query heads
// (from a copy of Wq whose rows are in stage order, so one product covers
// the stage) into columns 0 .. U d, and its attention writes O and the
// log-sum-exp at the heads' own places (output head of local head g m + r:
// g G + k m + r).  keep_qkv: every head's Q, K and V are also copied into the
// kept buffer's layout for the backward.
int interleaved_attention(const Dims& D, const bpt_weights* w, bool hb, const void* xn, void* buf, void* wq_perm,
                          void* bq_perm, void* o, float* lse, int causal, void* keep_qkv, cudaStream_t st) {
  const int64_t d = D.d, h = D.h, blk = D.m * d;
  for (int64_t k = 0; k < D.n_stages; ++k)
    for (int64_t g = 0; g < D.Hkv; ++g) {
      const int64_t dst = (k * D.U + g * D.m) * d, src = (g * D.G + k * D.m) * d;  // rows of Wq
      if (cudaMemcpyAsync(bfm(wq_perm, dst * h), bf(w->wq, src * h), (size_t)(blk * h * 2), cudaMemcpyDeviceToDevice,
                          st) != cudaSuccess)
        return BPT_ECUDA;
      if (hb && cudaMemcpyAsync(bfm(bq_perm, dst), bf(w->bq, src), (size_t)(blk * 2), cudaMemcpyDeviceToDevice, st) !=
                    cudaSuccess)
        return BPT_ECUDA;
    }
  const int64_t kc = D.U * d, vc = kc + D.Hkv * d;
  int rc;
  if ((rc = project(D, xn, w->wk, hb ? w->bk : nullptr, D.Hkv * d, bfm(buf, kc), D.iw, st))) return rc;
  if ((rc = project(D, xn, w->wv, hb ? w->bv : nullptr, D.Hkv * d, bfm(buf, vc), D.iw, st))) return rc;
  if (D.rope != 0.f && (rc = rope_apply(D.rows, (int)D.s, buf, D.iw, (int)kc, (int)D.Hkv, (int)d, D.rope, 0, st)))
    return rc;
  if (keep_qkv && cudaMemcpy2DAsync(bfm(keep_qkv, D.H * d), (size_t)(D.full_w * 2), bf(buf, kc), (size_t)(D.iw * 2),
                                    (size_t)(2 * D.Hkv * d * 2), (size_t)D.rows, cudaMemcpyDeviceToDevice,
                                    st) != cudaSuccess)
    return BPT_ECUDA;
  for (int64_t k = 0; k < D.n_stages; ++k) {
    if ((rc = project(D, xn, bf(wq_perm, k * D.U * d * h), hb ? bf(bq_perm, k * D.U * d) : nullptr, D.U * d, buf,
                      D.iw, st)))
      return rc;
    if (D.rope != 0.f && (rc = rope_apply(D.rows, (int)D.s, buf, D.iw, 0, (int)D.U, (int)d, D.rope, 0, st))) return rc;
    if (keep_qkv)
      for (int64_t g = 0; g < D.Hkv; ++g)
        if (cudaMemcpy2DAsync(bfm(keep_qkv, (g * D.G + k * D.m) * d), (size_t)(D.full_w * 2), bf(buf, g * blk),
                              (size_t)(D.iw * 2), (size_t)(blk * 2), (size_t)D.rows, cudaMemcpyDeviceToDevice,
                              st) != cudaSuccess)
          return BPT_ECUDA;
    AttnShape a;
    a.b = (int)D.b;
    a.s = (int)D.s;
    a.H = (int)D.U;
    a.Hkv = (int)D.Hkv;
    a.d = (int)d;
    a.causal = causal;
    a.ld_qkv = D.iw;
    a.q_col = 0;
    a.k_col = kc;
    a.v_col = vc;
    a.ld_o = D.H * d;
    a.o_col = k * blk;
    a.o_seg = (int)D.m;
    a.o_seg_stride = (int)D.G;
    a.H_total = (int)D.H;
    a.lse_head0 = (int)(k * D.m);
    a.q_begin = 0;
    a.q_end = (int)D.s;
    a.o_row0 = 0;
    if ((rc = attention_fwd(a, buf, o, lse, st))) return rc;
  }
  return 0;
}

// out[M, N] (fp32, beta) = sum_i A[:, Kseg_i] B_i  with MN-major B segments;
// one launch when the segment boundaries are multiples of 64, else one per
// segment with accumulation.
// A second stream, per device and host thread, for launches that do not feed
// the next launch of the main chain (weight gradients beside activation
// gradients): they fill the SMs the main chain's kernels leave idle in their
// last, partial wave.  fork: the side stream waits for all work issued on the
// main stream so far; join: the main stream waits for all work issued on the
// side stream so far.  Created on the first backward call of a thread on a
// device.
struct Side {
  cudaStream_t s = nullptr;
  cudaEvent_t ev[8] = {};
  int next = 0;
};

Side* side_stream() {
  static thread_local Side sides[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  Side& sd = sides[dev];
  if (!sd.s) {
    // all or nothing: a half-made Side is destroyed and made again next call
    Side n;
    bool ok = cudaStreamCreateWithFlags(&n.s, cudaStreamNonBlocking) == cudaSuccess;
    for (auto& e : n.ev)
      ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      for (auto e : n.ev)
        if (e) cudaEventDestroy(e);
      if (n.s) cudaStreamDestroy(n.s);
      return nullptr;
    }
    sd = n;
  }
  return &sd;
}

int fork_side(cudaStream_t main, Side* sd) {
  cudaEvent_t e = sd->ev[sd->next++ % 8];
  return (cudaEventRecord(e, main) == cudaSuccess && cudaStreamWaitEvent(sd->s, e, 0) == cudaSuccess) ? 0 : BPT_ECUDA;
}

int join_side(cudaStream_t main, Side* sd) {
  cudaEvent_t e = sd->ev[sd->next++ % 8];
  return (cudaEventRecord(e, sd->s) == cudaSuccess && cudaStreamWaitEvent(main, e, 0) == cudaSuccess) ? 0 : BPT_ECUDA;
}

int gemm_kseg(int64_t M, int64_t N, const MatView& A, const MatView* B, const int64_t* ks, int nseg,
              const Epilogue& e0, cudaStream_t st) {
  bool ok = true;
  int64_t K = 0;
  for (int i = 0; i < nseg; ++i) {
    if (i < nseg - 1 && (ks[i] % 64)) ok = false;
    K += ks[i];
  }
  if (ok) return gemm(M, N, K, A, false, B, ks, nseg, true, nullptr, e0, st);
  int64_t koff = 0;
  for (int i = 0; i < nseg; ++i) {
    MatView Ai{bf(A.ptr, koff), A.rows, ks[i], A.ld};
    Epilogue e = e0;
    if (i > 0) e.beta = 1.f;
    int rc = gemm(M, N, ks[i], Ai, false, &B[i], &ks[i], 1, true, nullptr, e, st);
    if (rc) return rc;
    koff += ks[i];
  }
  return 0;
}

int layer_fwd(const bpt_config* cfg, const Dims& D, const bpt_weights* w, const void* x, void* y, void* saved,
              const FwdWs& W, cudaStream_t st);

}  // namespace

extern "C" {

const char* bpt_status_string(int s) {
  switch (s) {
    case BPT_OK: return "ok";
    case BPT_EINVAL: return "invalid argument (shape, divisibility, pointer or flag)";
    case BPT_ENOSPC: return "workspace too small";
    case BPT_ECUDA: return "CUDA call failed";
    case BPT_ETIMEOUT: return "a bounded device wait ran out";
    case BPT_EUNSUPPORTED: return "unsupported configuration (head_dim must be 64, 80, 96, 112 or 128)";
    default: return "unknown status";
  }
}

int bpt_last_device_error(void* stream, int* detail) {
  unsigned int e[4] = {0, 0, 0, 0};
  int rc = read_device_error(reinterpret_cast<cudaStream_t>(stream), e);
  if (rc) {
    if (detail) *detail = (int)e[1];
    return BPT_ECUDA;
  }
  if (e[0]) {
    if (detail) *detail = (int)e[1];
    return e[0] == BPT_EINVAL ? BPT_EINVAL : BPT_ETIMEOUT;
  }
  if (detail) *detail = 0;
  return BPT_OK;
}

size_t bpt_saved_bytes(const bpt_config* cfg) {
  Dims D;
  if (validate(cfg, &D)) return 0;
  Saved sv;
  return plan_saved(D, nullptr, &sv);
}

size_t bpt_workspace_bytes(const bpt_config* cfg, int pass) {
  Dims D;
  if (validate(cfg, &D)) return 0;
  if (pass == BPT_PASS_FWD) {
    FwdWs w;
    return plan_fwd(D, nullptr, &w, true, false);  // enough with or without `saved`
  }
  if (pass == BPT_PASS_BWD) {
    BwdWs w;
    return plan_bwd(D, nullptr, &w);
  }
  if (pass == BPT_PASS_HEADCHUNK) {
    HcWs w;
    return plan_headchunk(D, nullptr, &w);
  }
  return 0;
}

int bpt_layer_fwd(const bpt_config* cfg, const bpt_weights* w, const void* x, void* y, void* saved,
                  void* ws, size_t ws_bytes, void* stream) {
  Dims D;
  int rc = validate(cfg, &D);
  if (rc) return rc;
  if ((rc = check_weights(cfg, w))) return rc;
  if (!x || !y || !ws || !aligned16(x) || !aligned16(y) || !aligned16(ws) || (saved && !aligned16(saved)))
    return BPT_EINVAL;
  FwdWs W;
  const size_t need = plan_fwd(D, nullptr, &W, saved == nullptr, saved != nullptr);
  if (ws_bytes < need) return BPT_ENOSPC;
  if (D.debug) {
    Saved sv;
    const int64_t act = D.rows * D.h * 2, kept = (int64_t)plan_saved(D, nullptr, &sv);
    const Span sp[] = {{x, act}, {y, act}, {saved, saved ? kept : 0}, {ws, (int64_t)need}};
    if (check_spans(sp, 4) || check_weights_range(cfg, D, w)) return BPT_EINVAL;
  }
  plan_fwd(D, ws, &W, saved == nullptr, saved != nullptr);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = layer_fwd(cfg, D, w, x, y, saved, W, st);
  if (rc) return rc;
  return D.debug ? debug_finish(st) : BPT_OK;
}

}  // extern "C"

namespace {

int layer_fwd(const bpt_config* cfg, const Dims& D, const bpt_weights* w, const void* x, void* y, void* saved,
              const FwdWs& W, cudaStream_t st) {
  int rc;
  Saved sv{nullptr, nullptr, nullptr};
  if (saved) plan_saved(D, saved, &sv);
  float* lse = saved ? sv.lse : W.lse;
  // the projections and O go where the backward will find them when the
  // save policy keeps them
  void* obuf = sv.o ? sv.o : W.o;
  const QkvBuf b0 = sv.qkv ? kept_buf(D, sv.qkv, 0) : stage_buf(D, W.qkv);
  const bool hb = cfg->has_bias != 0;
  const int64_t h = D.h, f = D.f, Hd = D.H * D.d;

  // N1 over the whole sequence
  if ((rc = norm_fwd(D.rows, (int)h, cfg->norm, cfg->norm_eps, x, 0, h, w->ln1_w, w->ln1_b, W.xn, h, st)))
    return rc;
  if (D.interleave) {
    if ((rc = interleaved_attention(D, w, hb, W.xn, W.qkv, W.wq_perm, W.bq_perm, obuf, lse, cfg->causal, sv.qkv,
                                    st)))
      return rc;
  } else if (D.chunked) {
    for (int64_t k = 0; k < D.n_stages; ++k) {
      const QkvBuf b = sv.qkv ? kept_buf(D, sv.qkv, k) : stage_buf(D, W.qkv);
      if ((rc = stage_qkv(D, w, hb, W.xn, b, k, st))) return rc;
      AttnShape a = stage_attn_shape(D, k, cfg->causal, b);
      if ((rc = attention_fwd(a, b.p, obuf, lse, st))) return rc;
    }
  } else {
    if ((rc = stage_qkv(D, w, hb, W.xn, b0, 0, st))) return rc;
  }

  for (int64_t bi = 0; bi < D.b; ++bi) {
    for (int64_t r0 = 0; r0 < D.s; r0 += D.cf) {
      const int64_t nr = std::min(D.cf, D.s - r0);
      const int64_t row = bi * D.s + r0;
      const void* oblk;
      if (D.chunked) {
        oblk = bf(obuf, row * Hd);
      } else {
        // attention of this block's query rows, all heads: into the block
        // buffer, or into the kept O at the rows' own place
        AttnShape a = stage_attn_shape(D, 0, cfg->causal, b0);
        a.b = 1;
        a.q_begin = (int)r0;
        a.q_end = (int)(r0 + nr);
        a.o_row0 = sv.o ? 0 : r0;
        void* odst = sv.o ? bfm(sv.o, bi * D.s * Hd) : W.o;
        if ((rc = attention_fwd(a, bf(b0.p, bi * D.s * b0.ld), odst, lse + bi * D.H * D.s_pad, st))) return rc;
        oblk = sv.o ? bf(sv.o, row * Hd) : W.o;
      }
      // x1 = x + O Wo^T + bo
      {
        MatView A{oblk, nr, Hd, Hd};
        MatView B{w->wo, h, Hd, Hd};
        Epilogue e;
        e.kind = EPI_F32;  // x1 stays fp32: the residual stream is rounded once, at y
        e.out = W.x1;
        e.ldo = h;
        e.bias = hb ? w->bo : nullptr;
        e.res = bf(x, row * h);
        e.ldr = h;
        if ((rc = gemm(nr, h, Hd, A, false, &B, &Hd, 1, false, nullptr, e, st))) return rc;
      }
      if ((rc = norm_fwd(nr, (int)h, cfg->norm, cfg->norm_eps, W.x1, 1, h, w->ln2_w, w->ln2_b, W.x1n, h, st)))
        return rc;
      // a = act(x1n W1^T + b1)  or  silu(x1n W1^T) * (x1n W3^T)
      {
        MatView A{W.x1n, nr, h, h};
        MatView B{w->w1, f, h, h};
        Epilogue e;
        e.out = W.a;
        e.ldo = f;
        if (cfg->act == BPT_ACT_SWIGLU) {
          MatView B2{w->w3, f, h, h};
          e.kind = EPI_SWIGLU;
          if ((rc = gemm(nr, f, h, A, false, &B, &h, 1, false, &B2, e, st))) return rc;
        } else {
          e.kind = EPI_GELU;
          e.act = cfg->act;
          e.bias = hb ? w->b1 : nullptr;
          if ((rc = gemm(nr, f, h, A, false, &B, &h, 1, false, nullptr, e, st))) return rc;
        }
      }
      // y = x1 + a W2^T + b2
      {
        MatView A{W.a, nr, f, f};
        MatView B{w->w2, h, f, f};
        Epilogue e;
        e.out = bfm(y, row * h);
        e.ldo = h;
        e.bias = hb ? w->b2 : nullptr;
        e.res = W.x1;
        e.res_f32 = 1;
        e.ldr = h;
        if ((rc = gemm(nr, h, f, A, false, &B, &f, 1, false, nullptr, e, st))) return rc;
      }
    }
  }
  return BPT_OK;
}

}  // namespace

extern "C" {

int bpt_attn_headchunk(const bpt_config* cfg, const bpt_weights* w, const void* xn, void* o, void* lse,
                       void* ws, size_t ws_bytes, void* stream) {
  Dims D;
  int rc = validate(cfg, &D);
  if (rc) return rc;
  if (!w || !w->wq || !w->wk || !w->wv || !xn || !o || !ws) return BPT_EINVAL;
  if (cfg->has_bias && (!w->bq || !w->bk || !w->bv)) return BPT_EINVAL;
  if (!aligned16(xn) || !aligned16(o) || !aligned16(ws) || (lse && !aligned16(lse))) return BPT_EINVAL;
  HcWs hc;
  const size_t need = plan_headchunk(D, nullptr, &hc);
  if (ws_bytes < need) return BPT_ENOSPC;
  if (D.debug) {
    const int64_t q = D.H * D.d, kv = D.Hkv * D.d, h = D.h;
    const bool hb = cfg->has_bias != 0;
    const Span sp[] = {{xn, D.rows * h * 2},      {o, D.rows * q * 2}, {lse, lse ? D.b * D.H * D.s_pad * 4 : 0},
                       {ws, (int64_t)need},       {w->wq, q * h * 2},  {w->wk, kv * h * 2},
                       {w->wv, kv * h * 2},       {w->bq, hb ? q * 2 : 0}, {w->bk, hb ? kv * 2 : 0},
                       {w->bv, hb ? kv * 2 : 0}};
    if (check_spans(sp, 10)) return BPT_EINVAL;
  }
  plan_headchunk(D, ws, &hc);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool hb = cfg->has_bias != 0;
  if (D.interleave) {
    if ((rc = interleaved_attention(D, w, hb, xn, hc.qkv, hc.wq_perm, hc.bq_perm, o, reinterpret_cast<float*>(lse),
                                    cfg->causal, nullptr, st)))
      return rc;
  } else {
    for (int64_t k = 0; k < D.n_stages; ++k) {
      const QkvBuf b = stage_buf(D, hc.qkv);
      if ((rc = stage_qkv(D, w, hb, xn, b, k, st))) return rc;
      AttnShape a = stage_attn_shape(D, k, cfg->causal, b);
      if ((rc = attention_fwd(a, hc.qkv, o, reinterpret_cast<float*>(lse), st))) return rc;
    }
  }
  return D.debug ? debug_finish(st) : BPT_OK;
}

int bpt_attention_fwd(const bpt_config* cfg, const void* qkv, void* o, void* lse, void* stream) {
  Dims D;
  int rc = validate(cfg, &D);
  if (rc) return rc;
  if (!qkv || !o || !aligned16(qkv) || !aligned16(o) || (lse && !aligned16(lse))) return BPT_EINVAL;
  Dims F = D;
  F.U = D.H;
  F.Uk = D.Hkv;
  F.qkv_w = (D.H + 2 * D.Hkv) * D.d;
  if (D.debug) {
    const Span sp[] = {{qkv, D.rows * F.qkv_w * 2}, {o, D.rows * D.H * D.d * 2},
                       {lse, lse ? D.b * D.H * D.s_pad * 4 : 0}};
    if (check_spans(sp, 3)) return BPT_EINVAL;
  }
  AttnShape a = stage_attn_shape(F, 0, cfg->causal, stage_buf(F, const_cast<void*>(qkv)));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = attention_fwd(a, qkv, o, reinterpret_cast<float*>(lse), st))) return rc;
  return D.debug ? debug_finish(st) : BPT_OK;
}

size_t bpt_attention_bwd_workspace_bytes(const bpt_config* cfg) {
  Dims D;
  if (validate(cfg, &D)) return 0;
  Dims F = D;
  F.U = D.H;
  F.Uk = D.Hkv;
  F.qkv_w = (D.H + 2 * D.Hkv) * D.d;
  AttnBwdShape s = stage_bwd_shape(F, 0);
  s.f.causal = cfg->causal;
  return attention_bwd_ws_bytes(s);
}

int bpt_attention_bwd(const bpt_config* cfg, const void* qkv, const void* o, const void* lse, const void* dout,
                      void* dqkv, void* ws, size_t ws_bytes, void* stream) {
  return bpt::attention_bwd_call(cfg, qkv, o, lse, dout, dqkv, ws, ws_bytes, stream, 0);
}

}  // extern "C"

// The attention backward behind both entry points; ws_is_library: the
// workspace is the library's own array (not checked under the debug flag).
int bpt::attention_bwd_call(const bpt_config* cfg, const void* qkv, const void* o, const void* lse,
                            const void* dout, void* dqkv, void* ws, size_t ws_bytes, void* stream,
                            int ws_is_library) {
  Dims D;
  int rc = validate(cfg, &D);
  if (rc) return rc;
  if (!qkv || !o || !lse || !dout || !dqkv || !ws) return BPT_EINVAL;
  if (!aligned16(qkv) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) || !aligned16(dqkv) ||
      !aligned16(ws))
    return BPT_EINVAL;
  Dims F = D;
  F.U = D.H;
  F.Uk = D.Hkv;
  F.qkv_w = (D.H + 2 * D.Hkv) * D.d;
  AttnBwdShape s = stage_bwd_shape(F, 0);
  s.f.causal = cfg->causal;
  s.deterministic = D.det;
  const size_t need = attention_bwd_ws_bytes(s);
  if (ws_bytes < need) return BPT_ENOSPC;
  if (D.debug) {
    const int64_t packed = D.rows * F.qkv_w * 2, hd = D.rows * D.H * D.d * 2;
    const Span sp[] = {{qkv, packed}, {o, hd}, {lse, D.b * D.H * D.s_pad * 4}, {dout, hd}, {dqkv, packed},
                       {ws, ws_is_library ? 0 : (int64_t)need}};
    if (check_spans(sp, 6)) return BPT_EINVAL;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = attention_bwd(s, qkv, o, reinterpret_cast<const float*>(lse), dout, dqkv, ws, st))) return rc;
  return D.debug ? debug_finish(st) : BPT_OK;
}

extern "C" {

int bpt_layer_bwd(const bpt_config* cfg, const bpt_weights* w, const void* x, const void* saved, const void* dy,
                  void* dx, const bpt_grads* g, void* ws, size_t ws_bytes, void* stream) {
  Dims D;
  int rc = validate(cfg, &D);
  if (rc) return rc;
  if ((rc = check_weights(cfg, w))) return rc;
  if (!x || !saved || !dy || !dx || !g || !ws) return BPT_EINVAL;
  if (!aligned16(x) || !aligned16(saved) || !aligned16(dy) || !aligned16(dx) || !aligned16(ws)) return BPT_EINVAL;
  {
    const void* need[] = {g->ln1_w, g->wq, g->wk, g->wv, g->wo, g->ln2_w, g->w1, g->w2};
    for (const void* p : need)
      if (!p || !aligned16(p)) return BPT_EINVAL;
    if (cfg->norm == BPT_NORM_LAYER && (!g->ln1_b || !g->ln2_b)) return BPT_EINVAL;
    if (cfg->act == BPT_ACT_SWIGLU && !g->w3) return BPT_EINVAL;
    if (cfg->has_bias && (!g->bq || !g->bk || !g->bv || !g->bo || !g->b2 ||
                          (cfg->act != BPT_ACT_SWIGLU && !g->b1)))
      return BPT_EINVAL;
  }
  BwdWs W;
  const size_t need = plan_bwd(D, nullptr, &W);
  if (ws_bytes < need) return BPT_ENOSPC;
  if (D.debug) {
    const int64_t act = D.rows * D.h * 2;
    Saved kv;
    const int64_t kept = (int64_t)plan_saved(D, nullptr, &kv);
    const Span sp[] = {{x, act}, {dy, act}, {dx, act}, {saved, kept}, {ws, (int64_t)need}};
    if (check_spans(sp, 5) || check_weights_range(cfg, D, w) || check_grads_range(cfg, D, g)) return BPT_EINVAL;
  }
  plan_bwd(D, ws, &W);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Side* sd = side_stream();
  if (!sd) return BPT_ECUDA;
  // With BPT_FLAG_ONE_STREAM the weight-gradient products run on the
  // caller's stream in issue order; fork and join become no-ops.
  const bool one = (cfg->flags & BPT_FLAG_ONE_STREAM) != 0;
  cudaStream_t ss = one ? st : sd->s;
  auto fork = [&]() { return one ? 0 : fork_side(st, sd); };
  auto join = [&]() { return one ? 0 : join_side(st, sd); };
  Saved sv;
  plan_saved(D, saved, &sv);
  const float* lse = sv.lse;
  // O and the projections: kept by the forward (save policy) or rebuilt into
  // the workspace
  void* obuf = sv.o ? sv.o : W.o;
  auto qbuf = [&](int64_t k) { return sv.qkv ? kept_buf(D, sv.qkv, k) : stage_buf(D, W.qkv); };
  const bool hb = cfg->has_bias != 0;
  const bool accum = (cfg->flags & BPT_FLAG_ACCUM_GRADS) != 0;
  const bool swiglu = cfg->act == BPT_ACT_SWIGLU;
  const int64_t h = D.h, f = D.f, Hd = D.H * D.d, d = D.d;
  const bool ln = cfg->norm == BPT_NORM_LAYER;

  // The launch sequence; on an early error return the side stream is still
  // joined below, so nothing it was given outlives the call unordered.
  auto run = [&]() -> int {
    if (!accum) {
      if (cudaMemsetAsync(g->ln1_w, 0, h * 4, st) || cudaMemsetAsync(g->ln2_w, 0, h * 4, st)) return BPT_ECUDA;
      if (ln && (cudaMemsetAsync(g->ln1_b, 0, h * 4, st) || cudaMemsetAsync(g->ln2_b, 0, h * 4, st)))
        return BPT_ECUDA;
    }

    // ---- recompute N1, Q/K/V and attention (the saved LSE is not rewritten);
    // what the forward kept is taken from `saved` instead (always contiguous
    // stages here: the result does not depend on the stage order)
    if ((rc = norm_fwd(D.rows, (int)h, cfg->norm, cfg->norm_eps, x, 0, h, w->ln1_w, w->ln1_b, W.xn, h, st)))
      return rc;
    if (!sv.o) {
      for (int64_t k = 0; k < D.n_stages; ++k) {
        const QkvBuf b = qbuf(k);
        if (!sv.qkv && (rc = stage_qkv(D, w, hb, W.xn, b, k, st))) return rc;
        AttnShape a = stage_attn_shape(D, k, cfg->causal, b);
        if ((rc = attention_fwd(a, b.p, obuf, nullptr, st))) return rc;
      }
    }

    // ---- FFN blocks: rebuild x1, N2, fc1 and form the FFN / N2 gradients
    bool first = true;
    for (int64_t bi = 0; bi < D.b; ++bi) {
      for (int64_t r0 = 0; r0 < D.s; r0 += D.cf) {
        const int64_t nr = std::min(D.cf, D.s - r0);
        const int64_t row = bi * D.s + r0;
        const float beta = (accum || !first) ? 1.f : 0.f;
        {
          MatView A{bf(obuf, row * Hd), nr, Hd, Hd};
          MatView B{w->wo, h, Hd, Hd};
          Epilogue e;
          e.deterministic = D.det;
          e.kind = EPI_F32;  // x1 stays fp32: the residual stream is rounded once, at y
          e.out = W.x1;
          e.ldo = h;
          e.bias = hb ? w->bo : nullptr;
          e.res = bf(x, row * h);
          e.ldr = h;
          if ((rc = gemm(nr, h, Hd, A, false, &B, &Hd, 1, false, nullptr, e, st))) return rc;
        }
        // the previous block's weight gradients (side stream) still read x1n,
        // a and dz, which this block now rewrites
        if (!first && (rc = join())) return rc;
        if ((rc = norm_fwd(nr, (int)h, cfg->norm, cfg->norm_eps, W.x1, 1, h, w->ln2_w, w->ln2_b, W.x1n, h, st)))
          return rc;
        {
          MatView A{W.x1n, nr, h, h};
          MatView B{w->w1, f, h, h};
          Epilogue e;
          e.deterministic = D.det;
          e.out = W.a;
          e.ldo = f;
          if (swiglu) {
            MatView B2{w->w3, f, h, h};
            e.kind = EPI_SWIGLU;
            e.out2 = W.g;
            e.ldo2 = f;
            e.out3 = W.u;
            e.ldo3 = f;
            if ((rc = gemm(nr, f, h, A, false, &B, &h, 1, false, &B2, e, st))) return rc;
          } else {
            e.kind = EPI_GELU;
            e.act = cfg->act;
            e.bias = hb ? w->b1 : nullptr;
            e.out2 = W.gd;  // gelu'(z), which the fc2 backward multiplies by
            e.ldo2 = f;
            if ((rc = gemm(nr, f, h, A, false, &B, &h, 1, false, nullptr, e, st))) return rc;
          }
        }
        const void* dyb = bf(dy, row * h);
        // side stream: the fc2 weight gradient needs only dy and a
        if ((rc = fork())) return rc;
        // dW2 (+)= dy^T a ; db2 (+)= colsum(dy)
        {
          MatView A{dyb, nr, h, h};     // MN-major: [K = rows, M = h]
          MatView B{W.a, nr, f, f};     // MN-major: [K = rows, N = f]
          Epilogue e;
          e.deterministic = D.det;
          e.kind = EPI_F32;
          e.out = g->w2;
          e.ldo = f;
          e.beta = beta;
          if ((rc = gemm(h, f, nr, A, true, &B, &nr, 1, true, nullptr, e, ss))) return rc;
          if (hb && (rc = colsum(nr, h, dyb, h, reinterpret_cast<float*>(g->b2), beta != 0.f, ss, W.part_side))) return rc;
        }
        // dA = dy W2, fused with the activation gradient
        {
          MatView A{dyb, nr, h, h};
          MatView B{w->w2, h, f, f};  // [K = h rows, N = f cols]
          Epilogue e;
          e.deterministic = D.det;
          if (swiglu) {
            e.kind = EPI_SWIGLU_BWD;
            e.aux = W.g;
            e.ldaux = f;
            e.aux2 = W.u;
            e.ldaux2 = f;
            e.out = W.dz;
            e.ldo = 2 * f;
            e.out2 = bfm(W.dz, f);
            e.ldo2 = 2 * f;
          } else {
            e.kind = EPI_GELU_BWD;
            e.act = cfg->act;
            e.aux = W.gd;
            e.ldaux = f;
            e.out = W.dz;
            e.ldo = f;
          }
          if ((rc = gemm(nr, f, h, A, false, &B, &h, 1, true, nullptr, e, st))) return rc;
        }
        // side stream: the fc1 weight (and bias) gradients need only dz and x1n
        if ((rc = fork())) return rc;
        // dW1 (+)= dz^T x1n (SwiGLU: dWg from dg, dWu from du) ; db1
        {
          const int64_t ldz = swiglu ? 2 * f : f;
          MatView B{W.x1n, nr, h, h};
          Epilogue e;
          e.deterministic = D.det;
          e.kind = EPI_F32;
          e.ldo = h;
          e.beta = beta;
          MatView A{W.dz, nr, f, ldz};
          e.out = g->w1;
          if ((rc = gemm(f, h, nr, A, true, &B, &nr, 1, true, nullptr, e, ss))) return rc;
          if (swiglu) {
            MatView A2{bf(W.dz, f), nr, f, ldz};
            e.out = g->w3;
            if ((rc = gemm(f, h, nr, A2, true, &B, &nr, 1, true, nullptr, e, ss))) return rc;
          } else if (hb) {
            if ((rc = colsum(nr, f, W.dz, f, reinterpret_cast<float*>(g->b1), beta != 0.f, ss, W.part_side))) return rc;
          }
        }
        // dx1n = dz W1  (SwiGLU: dg Wg + du Wu)
        {
          Epilogue e;
          e.deterministic = D.det;
          e.kind = EPI_BF16;
          e.out = W.dx1n;
          e.ldo = h;
          if (swiglu) {
            MatView A{W.dz, nr, 2 * f, 2 * f};
            MatView Bs[2] = {{w->w1, f, h, h}, {w->w3, f, h, h}};
            int64_t ks[2] = {f, f};
            if (f % 64 == 0) {
              if ((rc = gemm(nr, h, 2 * f, A, false, Bs, ks, 2, true, nullptr, e, st))) return rc;
            } else {
              return BPT_EUNSUPPORTED;
            }
          } else {
            MatView A{W.dz, nr, f, f};
            MatView B{w->w1, f, h, h};
            if ((rc = gemm(nr, h, f, A, false, &B, &f, 1, true, nullptr, e, st))) return rc;
          }
        }
        // dx1 = dy + N2^T(dx1n), as bf16 (operand of the next products) and fp32
        {
          NormBwdIO io{W.dx1n, 0, h, W.x1, 1, h, dyb, 0, h, bfm(W.dx1, row * h), W.dx1f + row * h, h};
          if ((rc = norm_bwd(nr, (int)h, cfg->norm, cfg->norm_eps, io, w->ln2_w, reinterpret_cast<float*>(g->ln2_w),
                             ln ? reinterpret_cast<float*>(g->ln2_b) : nullptr, st, W.part_main)))
            return rc;
        }
        first = false;
      }
    }

    // ---- output projection: dO = dx1 Wo ; dWo (+)= dx1^T O ; dbo
    if ((rc = join())) return rc;
    if ((rc = fork())) return rc;
    {
      // side stream: dWo and dbo need only dx1 and O, and run beside dO and
      // the attention backward
      MatView A2{W.dx1, D.rows, h, h};
      MatView B2{obuf, D.rows, Hd, Hd};
      Epilogue e2;
      e2.deterministic = D.det;
      e2.kind = EPI_F32;
      e2.out = g->wo;
      e2.ldo = Hd;
      e2.beta = accum ? 1.f : 0.f;
      const int64_t K = D.rows;
      if ((rc = gemm(h, Hd, K, A2, true, &B2, &K, 1, true, nullptr, e2, ss))) return rc;
      if (hb && (rc = colsum(D.rows, h, W.dx1, h, reinterpret_cast<float*>(g->bo), accum, ss, W.part_side))) return rc;
      MatView A{W.dx1, D.rows, h, h};
      MatView B{w->wo, h, Hd, Hd};  // [K = h rows, N = Hd cols]
      Epilogue e;
      e.deterministic = D.det;
      e.out = W.dO;
      e.ldo = Hd;
      if ((rc = gemm(D.rows, Hd, h, A, false, &B, &h, 1, true, nullptr, e, st))) return rc;
    }

    // ---- attention and Q/K/V gradients, stage by stage.  Without rotary
    // embedding the key-bias gradient is identically zero: the bias adds
    // Q[q].bk to every logit of query row q alike (masked ones stay -inf),
    // and softmax is invariant to such a shift, so the loss does not depend
    // on bk.  It is then written as exact zeros (left as is when
    // accumulating) instead of summing dK, whose sum of bf16-rounded rows
    // would be rounding noise growing like sqrt(s).  A rotation after the
    // bias makes the added logit depend on the key's position, so with
    // rotary embedding dbk is the column sum of dK like the other biases.
    const bool rope = D.rope != 0.f;
    if (hb && !accum && !rope &&
        cudaMemsetAsync(g->bk, 0, (size_t)(D.Hkv * D.d) * sizeof(float), st) != cudaSuccess)
      return BPT_ECUDA;
    for (int64_t k = 0; k < D.n_stages; ++k) {
      const QkvBuf b = qbuf(k);
      // the projections of stage k: kept by the forward, still in the stage
      // buffer (one stage), or rebuilt (the recompute above made the last
      // stage's, or none of them if O was kept)
      if (!sv.qkv && (D.chunked || sv.o) && (rc = stage_qkv(D, w, hb, W.xn, b, k, st))) return rc;
      // the previous stage's weight gradients (side stream) read dqkv, which
      // this stage's attention backward rewrites
      if (k > 0 && (rc = join())) return rc;
      AttnBwdShape sb = stage_bwd_shape(D, k, b);
      sb.f.causal = cfg->causal;
      sb.deterministic = D.det;
      if ((rc = attention_bwd(sb, b.p, obuf, lse, W.dO, W.dqkv, W.attn, st))) return rc;
      // dQ, dK are gradients of the rotated heads: turn them back
      if (rope && (rc = rope_apply(D.rows, (int)D.s, W.dqkv, D.qkv_w, 0, (int)(D.U + D.Uk), (int)d, D.rope, 1, st)))
        return rc;
      const int64_t q0 = k * D.U * d, kv0 = k * D.Uk * d;
      const int64_t nq = D.U * d, nkv = D.Uk * d;
      // dxn (+)= dQ Wq_s + dK Wk_s + dV Wv_s
      {
        MatView A{W.dqkv, D.rows, D.qkv_w, D.qkv_w};
        MatView Bs[3] = {
            {bf(w->wq, q0 * h), nq, h, h}, {bf(w->wk, kv0 * h), nkv, h, h}, {bf(w->wv, kv0 * h), nkv, h, h}};
        int64_t ks[3] = {nq, nkv, nkv};
        Epilogue e;
        e.deterministic = D.det;
        e.kind = EPI_F32;
        e.out = W.dxn;
        e.ldo = h;
        e.beta = k > 0 ? 1.f : 0.f;
        if ((rc = gemm_kseg(D.rows, h, A, Bs, ks, 3, e, st))) return rc;
      }
      // dWq_s, dWk_s, dWv_s (+)= dQKV_s^T xn ; biases, on the side stream
      // beside dxn
      if ((rc = fork())) return rc;
      {
        struct Piece {
          void* G;
          void* Gb;
          int64_t row0, n, col;
        } pieces[3] = {{g->wq, g->bq, q0, nq, 0}, {g->wk, g->bk, kv0, nkv, nq}, {g->wv, g->bv, kv0, nkv, nq + nkv}};
        MatView B{W.xn, D.rows, h, h};
        const int64_t K = D.rows;
        for (auto& pc : pieces) {
          MatView A{bf(W.dqkv, pc.col), D.rows, pc.n, D.qkv_w};
          Epilogue e;
          e.deterministic = D.det;
          e.kind = EPI_F32;
          e.out = f32(pc.G, pc.row0 * h);
          e.ldo = h;
          e.beta = accum ? 1.f : 0.f;
          if ((rc = gemm(pc.n, h, K, A, true, &B, &K, 1, true, nullptr, e, ss))) return rc;
          if (hb && (pc.Gb != g->bk || rope) &&
              (rc = colsum(D.rows, pc.n, bf(W.dqkv, pc.col), D.qkv_w, f32(pc.Gb, pc.row0), accum, ss, W.part_side)))
            return rc;
        }
      }
    }

    // ---- dx = dx1 + N1^T(dxn)
    {
      NormBwdIO io{W.dxn, 1, h, x, 0, h, W.dx1f, 1, h, dx, nullptr, h};
      if ((rc = norm_bwd(D.rows, (int)h, cfg->norm, cfg->norm_eps, io, w->ln1_w, reinterpret_cast<float*>(g->ln1_w),
                         ln ? reinterpret_cast<float*>(g->ln1_b) : nullptr, st, W.part_main)))
        return rc;
    }
    return BPT_OK;
  };
  rc = run();
  // everything issued on the side stream is ordered before the caller's next
  // work on the main stream
  const int jr = join();
  if (rc) return rc;
  if (jr) return BPT_ECUDA;
  return D.debug ? debug_finish(st) : BPT_OK;
}

}  // extern "C"
