/*
 * bpt.h -- C ABI of libbpt: the fused blockwise attention + FFN layer
 * (Blockwise Parallel Transformer) on one NVIDIA GB300 (sm_103a).
 *
 * What the library computes is the layer these pages define:
 *
 *   x1 = x + Attn(N1(x)) Wo^T + bo
 *   y  = x1 + FFN(N2(x1))
 *   Attn, per query head n with key/value head g = floor(n / G):
 *        softmax(Q_n K_g^T / sqrt(d) + M) V_g,   M_ij = -inf where j > i (causal)
 *   FFN  = GeLU(z W1^T + b1) W2^T + b2           (GPT layer; act 0 erf, 1 tanh)
 *        = (SiLU(z W1^T) * (z W3^T)) W2^T         (Llama layer, act 2; W1 gate, W3 up, W2 down)
 *   N    = LayerNorm(gamma, beta, eps) or RMSNorm(gamma, eps)
 *
 *  - "Blockwise Parallel Transformer for Long Context Large Models", section
 *    3.4: blockwise attention with online softmax ("Blockwise Self-Attention
 *    with Online Softmax", Equation 3), the FFN applied to each finished
 *    query block ("The FFN Memory Bottleneck and Why Fusion Is Possible"),
 *    Algorithm 1 and the Figure 3 implementation notes (remat of each block,
 *    causal bias per block).
 *  - "Training memory: model states, activations and checkpointing", section
 *    3: the pre-LN GPT layer with biases and GeLU, the Llama-style layer,
 *    full activation checkpointing (the backward pass reruns the forward).
 *  - "Untied Ulysses: Memory-Efficient Context Parallelism via Headwise
 *    Chunking", section 3.4 "The Core Mechanism: Headwise Chunking via UPipe"
 *    (U heads per stage, buffers reused, output buffer filled per stage) and
 *    section 4.1 "The GQA Scheduling Algorithm" (query head i uses key/value
 *    head floor(i/G)).  Only the single-GPU part: no all-to-all.
 *
 * Conventions
 *  - Activations and weights are bf16, row-major.  x, y, dy, dx: [b, s, h].
 *    Weights use the nn.Linear layout [out, in]: wq [H*d, h], wk/wv
 *    [H_kv*d, h], wo [h, H*d], w1/w3 [f, h], w2 [h, f]; biases and norm
 *    parameters are vectors.  A pointer a variant does not use is NULL.
 *  - Weight gradients are fp32, same shapes.  They are overwritten unless
 *    BPT_FLAG_ACCUM_GRADS is set, in which case they are accumulated (+=).
 *  - Accumulation is fp32 everywhere; the residual stream inside the layer
 *    (x1 and its gradient) is kept in fp32 so each output is rounded to bf16
 *    once.  The log-sum-exp saved by the forward pass is fp32
 *    [b, H, s_pad] in natural-log units, s_pad = s rounded up to 128 (rows
 *    past s hold finite filler values).
 *  - Every device pointer must be 16-byte aligned and every row length a
 *    multiple of 8 elements.
 *  - Ownership: the caller allocates every buffer (inputs, outputs, the
 *    workspace whose size bpt_workspace_bytes reports).  The library never
 *    allocates device memory.  It keeps one lazily set device error word.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).
 *    Every call is asynchronous on it except bpt_last_device_error.
 *  - Errors: functions return a BPT_* status.  Arguments are validated on
 *    the host before anything is launched; a failed launch returns
 *    BPT_ECUDA.  Device-side waits are bounded: a wait that runs out records
 *    BPT_ETIMEOUT in the device error word, the kernel leaves cleanly, and
 *    bpt_last_device_error reports it.
 */
#ifndef BPT_H_
#define BPT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  BPT_OK = 0,
  BPT_EINVAL = 1,       /* shapes, divisibility, pointers or flags invalid */
  BPT_ENOSPC = 2,       /* workspace smaller than bpt_workspace_bytes() */
  BPT_ECUDA = 3,        /* a CUDA runtime/driver call failed */
  BPT_ETIMEOUT = 4,     /* a bounded device wait ran out (device error word) */
  BPT_EUNSUPPORTED = 5  /* valid but not built: e.g. head_dim not in {64,80,96,112,128} */
};

enum { BPT_NORM_LAYER = 0, BPT_NORM_RMS = 1 };
enum { BPT_ACT_GELU_ERF = 0, BPT_ACT_GELU_TANH = 1, BPT_ACT_SWIGLU = 2 };
/* Flags (bpt_config.flags, OR-ed):
 *  BPT_FLAG_ACCUM_GRADS   weight gradients are added to (+=) instead of
 *                         overwritten.
 *  BPT_FLAG_ONE_STREAM    every launch of bpt_layer_bwd on the caller's
 *                         stream, in issue order (no second stream).
 *  BPT_FLAG_DETERMINISTIC every floating-point sum is taken in an order
 *                         fixed by the shapes and the device's SM count, so
 *                         two calls with the same inputs on the same device
 *                         give bitwise equal results.  Without it, three
 *                         kinds of sums follow the timing of the run: the
 *                         attention backward's two MMA-issuing threads per
 *                         CTA add into one TMEM accumulator in the order
 *                         their products reach the tensor core; weight-
 *                         gradient products split along K add their parts in
 *                         L2; bias and norm-parameter gradients add per-block
 *                         partial sums with atomics.  Each such result is
 *                         then off by at most a rounding step of the
 *                         summation order (one bf16 unit for dQ/dK/dV).  With
 *                         the flag: one issuing warp per CTA, no K split,
 *                         and per-block partial sums written to the workspace
 *                         and added in block order by a second kernel.  The
 *                         attention backward then takes about 1.35-1.5 times
 *                         as long, the layer backward about 1.15-1.25 times
 *                         (measured: 29.1 -> 36.0 ms at the GPT-3B workload,
 *                         166.6 -> 190.8 ms at the Llama-8B one).
 *  BPT_FLAG_DEBUG_CHECKS  before any launch, every device pointer argument
 *                         must lie, with the bytes the call touches through
 *                         it, inside one device allocation of the current
 *                         device (else BPT_EINVAL); after the launches the
 *                         call synchronises `stream` and returns the device
 *                         error word's status (BPT_ETIMEOUT) or a failed
 *                         kernel's (BPT_ECUDA) itself.  The call is then
 *                         synchronous: not for use under stream capture.  */
enum {
  BPT_FLAG_ACCUM_GRADS = 1,
  BPT_FLAG_ONE_STREAM = 2,
  BPT_FLAG_DETERMINISTIC = 4,
  BPT_FLAG_DEBUG_CHECKS = 8
};

enum { BPT_PASS_FWD = 0, BPT_PASS_BWD = 1, BPT_PASS_HEADCHUNK = 2 };
enum { BPT_STAGE_CONTIGUOUS = 0, BPT_STAGE_INTERLEAVED = 1 };
enum { BPT_SAVE_NOTHING = 0, BPT_SAVE_PROJECTIONS = 1, BPT_SAVE_ATTN_OUT = 2 };

/* Shape and schedule of one layer.
 *   b, s, h            batch, sequence length, model width
 *   n_heads, n_kv_heads, head_dim   H, H_kv (H % H_kv == 0, G = H/H_kv), d
 *   ffn_dim            f
 *   q_block, kv_block  attention blocks c_q, c_kv: multiples of 128 (the
 *                      tensor-core tile; a block of 256 is two tiles in turn)
 *   ffn_block          rows per FFN block c_f: a multiple of q_block; 0 means
 *                      min(2048, s rounded up to q_block)
 *   head_chunk         U query heads per stage; U == H (or 0) means no
 *                      chunking; H % U == 0 and U % G == 0
 *   causal             1: key j is masked for query i when j > i; 0: no mask
 *                      (any other value is rejected)
 *   norm, act          BPT_NORM_*, BPT_ACT_*
 *   has_bias           1: every linear has a bias (GPT); 0: none (Llama)
 *                      (any other value is rejected)
 *   norm_eps           epsilon inside the norm's square root
 *   flags              BPT_FLAG_*
 *   rope_base          rotary position embedding ("Untied Ulysses ...",
 *                      "Composability with Other Memory Optimizations": fused
 *                      RoPE, rotated in place with no fp32 copy; the page
 *                      does not state the rotation, this is the standard
 *                      half-split one): 0 = none; else > 1, and Q and K are
 *                      rotated after their projection (and bias): element i
 *                      of a head is paired with i + d/2 and the pair at
 *                      position p (the row's index within its sequence)
 *                      turns by p * rope_base^(-2i/d).  The layer calls and
 *                      bpt_attn_headchunk apply it; the attention-only calls
 *                      take Q/K as given.
 *   stage_order        head-chunk stage order ("Untied Ulysses ...", section
 *                      4.1 "The GQA Scheduling Algorithm"):
 *                      BPT_STAGE_CONTIGUOUS (0): stage k takes query heads
 *                      kU .. kU+U-1 and projects their U/G key/value heads
 *                      itself;
 *                      BPT_STAGE_INTERLEAVED (1): stage k takes the m = U/H_kv
 *                      query heads gG + km .. gG + km + m-1 of every group g,
 *                      and the key/value projections of all H_kv heads are made
 *                      once and stay resident for every stage (U must be a
 *                      multiple of H_kv).  Same result; the forward holds
 *                      U d + 2 H_kv d columns of projections instead of
 *                      (U + 2U/G) d.  The backward always runs the contiguous
 *                      stages.  No effect without chunking.
 *   save_policy        what the forward keeps for the backward, besides the
 *                      log-sum-exp ("Blockwise Parallel Transformer ...",
 *                      Appendix A.2 / Figure 3 notes: the checkpoint policies
 *                      searched for attention; the FFN always recomputes):
 *                      BPT_SAVE_NOTHING (0): nothing else; the backward
 *                      rebuilds N1, Q/K/V and the attention output;
 *                      BPT_SAVE_PROJECTIONS (1): also Q, K, V of every head
 *                      (the contractions without batch dimensions), so the
 *                      backward skips their projection;
 *                      BPT_SAVE_ATTN_OUT (2): also the attention output O
 *                      (the attention's dot products, combined across key
 *                      blocks), so the backward skips the attention forward.
 *                      The per-block score matrices are never kept: together
 *                      they would be the s x s matrix the method avoids.
 *                      bpt_saved_bytes grows accordingly.                    */
typedef struct {
  int32_t b, s, h, n_heads, n_kv_heads, head_dim, ffn_dim;
  int32_t q_block, kv_block, ffn_block, head_chunk;
  int32_t causal;
  int32_t norm;
  int32_t act;
  int32_t has_bias;
  float norm_eps;
  int32_t flags;
  float rope_base;
  int32_t stage_order;
  int32_t save_policy;
} bpt_config;

/* bf16 device pointers, nn.Linear [out, in]; NULL where the variant has none
 * (ln*_b for RMSNorm, every b* when has_bias == 0, w3 unless SwiGLU). */
typedef struct {
  const void *ln1_w, *ln1_b, *wq, *bq, *wk, *bk, *wv, *bv, *wo, *bo;
  const void *ln2_w, *ln2_b, *w1, *b1, *w2, *b2, *w3;
} bpt_weights;

/* fp32 device pointers with the shapes of the matching weights. */
typedef struct {
  void *ln1_w, *ln1_b, *wq, *bq, *wk, *bk, *wv, *bv, *wo, *bo;
  void *ln2_w, *ln2_b, *w1, *b1, *w2, *b2, *w3;
} bpt_grads;

/* Bytes of device workspace a call needs: pass BPT_PASS_FWD for
 * bpt_layer_fwd, BPT_PASS_BWD for bpt_layer_bwd, BPT_PASS_HEADCHUNK for
 * bpt_attn_headchunk.  0 for an invalid config. */
size_t bpt_workspace_bytes(const bpt_config* cfg, int pass);

/* Bytes the forward pass saves for the backward pass: the log-sum-exp of
 * every attention row, fp32 [b, H, s_pad] (with BPT_SAVE_NOTHING the only
 * activation kept besides the layer input x, which the caller keeps); with
 * BPT_SAVE_PROJECTIONS also Q, K, V [b*s, (H + 2 H_kv) d] bf16, with
 * BPT_SAVE_ATTN_OUT also O [b*s, H d] bf16 (each region 256-byte aligned). */
size_t bpt_saved_bytes(const bpt_config* cfg);

/* Forward pass of one layer.
 *   x [b,s,h] bf16 in; y [b,s,h] bf16 out.
 *   saved: bpt_saved_bytes() bytes for the backward pass, or NULL (inference).
 *   ws/ws_bytes: workspace of at least bpt_workspace_bytes(cfg, BPT_PASS_FWD).
 * Schedule: Q/K/V for the whole sequence (per head-chunk stage when
 * head_chunk < H), then for each FFN block of c_f rows: attention of those
 * query rows over their key/value blocks (online softmax, tensor cores), the
 * output projection with bias and residual, N2, fc1 + activation and fc2 with
 * bias and residual into y.  The s x s scores and the s x f FFN intermediate
 * never exist; only one c_f x f block does. */
int bpt_layer_fwd(const bpt_config* cfg, const bpt_weights* w, const void* x, void* y,
                  void* saved, void* ws, size_t ws_bytes, void* stream);

/* Backward pass with recomputation.
 *   x: the forward input; saved: what bpt_layer_fwd wrote; dy [b,s,h] bf16.
 *   dx [b,s,h] bf16 out; grads: fp32 weight gradients (see BPT_FLAG_ACCUM_GRADS).
 *   The key-bias gradient bk is written as exact zeros (left unchanged when
 *   accumulating): the bias shifts every logit of a query row alike, and
 *   softmax is invariant to that, so the gradient is identically zero.
 * The forward pass is rerun blockwise (N1, Q/K/V, attention, output
 * projection, and per FFN block N2 and fc1) and every gradient is formed
 * from the rebuilt blocks: attention probabilities are rebuilt from Q, K and
 * the saved log-sum-exp tile by tile.
 * Weight gradients that the next launch of the chain does not need run on a
 * second stream the library creates (one per device and host thread, on the
 * first call) and joins back into `stream` before returning: all of the
 * call's work is ordered before later work on `stream`.  Make the first call
 * of a thread before capturing `stream` into a graph.  With
 * BPT_FLAG_ONE_STREAM in cfg->flags everything runs on `stream` in issue
 * order instead: same results, no overlap, so that each kernel can be timed
 * on its own. */
int bpt_layer_bwd(const bpt_config* cfg, const bpt_weights* w, const void* x, const void* saved,
                  const void* dy, void* dx, const bpt_grads* grads, void* ws, size_t ws_bytes,
                  void* stream);

/* Headwise-chunked attention on one GPU: for each of H/U stages, project the
 * stage's U query heads and U/G key/value heads from xn (the normalised
 * input, [b,s,h] bf16), run blockwise causal attention for those heads and
 * write their output into o [b,s,H*d] (preallocated, filled slice by slice)
 * and their log-sum-exp into lse [b,H,s_pad] fp32 (nullable).  The per-stage
 * Q/K/V buffer in the workspace is reused by every stage, so peak Q/K/V
 * memory is 2*b*s*(U + 2U/G)*d bytes instead of 2*b*s*(H + 2H_kv)*d. */
int bpt_attn_headchunk(const bpt_config* cfg, const bpt_weights* w, const void* xn, void* o,
                       void* lse, void* ws, size_t ws_bytes, void* stream);

/* Attention alone on a packed projection buffer
 *   qkv [b*s, (H + 2H_kv)*d] bf16: row t holds Q heads 0..H-1, then K heads,
 *   then V heads (the layout the layer's projection writes),
 *   o [b*s, H*d] bf16 out, lse [b,H,s_pad] fp32 out (nullable).
 * Same kernel the layer uses (BPT page section 3.4, Algorithm 1 inner loop). */
int bpt_attention_fwd(const bpt_config* cfg, const void* qkv, void* o, void* lse, void* stream);

/* Attention backward on the same packed layout.
 *   qkv, o, lse as produced by bpt_attention_fwd; dout [b*s, H*d] bf16.
 *   dqkv [b*s, (H + 2H_kv)*d] bf16 out (dQ, then dK, then dV; dK/dV summed
 *   over the G query heads of each group).
 *   ws: at least bpt_attention_bwd_workspace_bytes(cfg) bytes (the fp32
 *   per-row dO.O sums and -LSE*log2(e), and a 16-byte row per query of
 *   both as bf16 (hi, lo) pairs for the dK/dV products: 24*b*H*s_pad bytes).
 *   b*H*s_pad above 2^31 - 1 returns BPT_EUNSUPPORTED.
 * Two kernels: dK/dV with the key/value tile outermost and dQ with the query
 * tile outermost, each accumulating in TMEM (no atomics).  Each CTA has two
 * MMA-issuing threads that add into the same accumulator, so the order of
 * the fp32 sums, and with it the last bit of a bf16 result, follows the
 * timing of the run; BPT_FLAG_DETERMINISTIC in cfg->flags fixes it. */
size_t bpt_attention_bwd_workspace_bytes(const bpt_config* cfg);
int bpt_attention_bwd(const bpt_config* cfg, const void* qkv, const void* o, const void* lse,
                      const void* dout, void* dqkv, void* ws, size_t ws_bytes, void* stream);

/* The attention backward without any device allocation by the caller.
 * This entry point has no counterpart in the paper; it exists for callers
 * that cannot allocate device memory when they call the library: a plugin of
 * an inference or training engine whose enqueue step runs on a memory plan
 * fixed in advance, a hot path that cannot afford cudaMalloc/cudaFree and
 * the device synchronisation they may cause, or a process whose device
 * memory is owned by another allocator.  Same arguments and results as
 * bpt_attention_bwd minus the workspace: the scratch it needs (the per-row
 * dO.O sums and -LSE*log2(e), bpt_attention_bwd_workspace_bytes =
 * 24*b*H*s_pad bytes)
 * lives in a fixed device array of BPT_NOALLOC_SCRATCH_BYTES compiled into
 * the library, which every GPU that loads it keeps until the process exits.
 *  - Returns BPT_ENOSPC, without launching anything, when the problem needs
 *    more scratch than BPT_NOALLOC_SCRATCH_BYTES (192 MiB: b*H*s_pad up to
 *    8M, e.g. 32 heads at s = 256K; 32 heads at s = 512K is too big).
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current) and keeps it for the life of the
 *    process; make that first call before any stream capture.  A device
 *    reset (cudaDeviceReset) after it is not supported: the array would be
 *    reloaded at another address.
 *  - Every call shares the one array.  Nothing in it has to start at zero:
 *    each call writes every byte of the array that it reads before reading
 *    it.  Calls that overlap on the GPU (other streams or host threads on
 *    the same device) race on it: serialise them.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine. */
#define BPT_NOALLOC_SCRATCH_BYTES (192u * 1024u * 1024u)
int bpt_attention_bwd_noalloc(const bpt_config* cfg, const void* qkv, const void* o, const void* lse,
                              const void* dout, void* dqkv, void* stream);

/* ------------------------------------------------------------------------
 * Language-model loss after the last layer, blockwise.
 *
 * "Blockwise Parallel Transformer for Long Context Large Models", section 3
 * (the note on the cross-entropy loss before Algorithm 1): the blockwise
 * schedule covers the final loss as well; "Untied Ulysses ...", the
 * paragraph on Arctic Long Sequence Training and its Table 1: this loss is
 * the largest activation term (240 S d_model bytes) and is computed tiled.
 * The pages do not write the loss out; it is taken as the mean token
 * cross-entropy (natural log) of the logits z = x W^T through a bias-free
 * vocabulary projection:
 *   loss = (1/n) sum_i (logsumexp_v z_iv - z_i,t_i)
 *   dz   = dloss * (softmax(z) - onehot(t)) / n,  dx = dz W,  dW = dz^T x
 * The n x V logits never exist: the forward reduces each 256-column tile of
 * them to per-row partial (max, sum exp) pairs in the GEMM epilogue, the
 * backward rebuilds them one vocabulary block of c_v columns at a time.
 *
 *   n            positions (rows of x; b*s of the layer)
 *   h            model width, a multiple of 8
 *   vocab        V >= 1 (any value; the last tile and block are ragged)
 *   vocab_block  c_v, vocabulary columns per backward block: a multiple of
 *                256; 0 means min(8192, V rounded up to 256).  The
 *                backward's workspace holds one n x c_v bf16 block.
 *   flags        BPT_FLAG_ACCUM_GRADS (dW +=), BPT_FLAG_DETERMINISTIC,
 *                BPT_FLAG_DEBUG_CHECKS (as for the layer); others rejected. */
typedef struct {
  int32_t n, h, vocab, vocab_block, flags;
} bpt_lm_config;

/* Workspace bytes of bpt_lm_loss_fwd (pass BPT_PASS_FWD: 16 n ceil(V/256)
 * bytes of partial pairs plus 12 n; 4 n fewer when lse is given) or
 * bpt_lm_loss_bwd (BPT_PASS_BWD: the n x c_v bf16 block, plus an fp32 n x h
 * accumulator for dx when V spans more than one block).  0 if invalid. */
size_t bpt_lm_workspace_bytes(const bpt_lm_config* cfg, int pass);

/* Forward: x [n, h] bf16, w [V, h] bf16 (nn.Linear layout), targets [n]
 * int32 in [0, V) (device).  Writes loss (one fp32, device) and, if lse is
 * not NULL, the per-row log-sum-exp [n] fp32 that the backward takes.  A
 * target outside [0, V) does not stop the call: the row's term is its
 * log-sum-exp alone, and the device error word records BPT_EINVAL with site
 * BPT_LM_BAD_TARGET_SITE (read with bpt_last_device_error).  The mean is
 * summed in a fixed order (the forward is deterministic in every mode). */
#define BPT_LM_BAD_TARGET_SITE 950
int bpt_lm_loss_fwd(const bpt_lm_config* cfg, const void* x, const void* w, const int32_t* targets,
                    float* loss, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Backward: the gradients of dloss * loss.  lse as the forward wrote it;
 * dx [n, h] bf16 out; dw [V, h] fp32 out (+= with BPT_FLAG_ACCUM_GRADS). */
int bpt_lm_loss_bwd(const bpt_lm_config* cfg, const void* x, const void* w, const int32_t* targets,
                    const float* lse, float dloss, void* dx, float* dw, void* ws, size_t ws_bytes,
                    void* stream);

/* Opt-in launch profiler.  bpt_profile_enable(1) makes every later launch
 * of this process record a pair of CUDA events on its stream, tagged with
 * the launch's kind and its algorithmic work (FLOPs for tensor-core kernels,
 * bytes for memory-bound ones); bpt_profile_enable(0) stops recording.
 * bpt_profile_collect synchronises on the recorded events, writes per kind
 * k < nkinds the summed device time (ms), FLOPs, bytes and launch count, and
 * clears the record.  Kinds: 0 GEMM, 1 attention forward, 2 attention
 * backward, 3 norms, 4 other memory-bound kernels. */
int bpt_profile_enable(int on);
int bpt_profile_collect(int nkinds, double* ms, double* flops, double* bytes, int* launches);
/* The launches recorded since profiling was enabled (or last collected), in
 * launch order: for i < the returned count (at most max), the kind, the
 * algorithmic FLOPs and bytes credited to launch i and its device time in
 * ms.  Synchronises on the recorded events; does not clear the record
 * (bpt_profile_collect does).  Returns the count, or minus a status code.
 * A diagnostic aid: the layer has no such step in the paper. */
int bpt_profile_list(int max, int* kind, double* flops, double* bytes, double* ms);

/* BPT_OK if the bytes [ptr, ptr + bytes) lie inside one device allocation
 * (cudaMalloc, a memory pool's block, managed memory) of the current device,
 * else BPT_EINVAL: host memory, another device's memory, or a range that runs
 * past its allocation's end.  The check BPT_FLAG_DEBUG_CHECKS applies to
 * every pointer argument.  Launches nothing; a diagnostic aid with no
 * counterpart in the paper.  A caching allocator hands out pieces of larger
 * allocations, so a range past the end of its piece but inside the
 * allocation passes. */
int bpt_check_device_range(const void* ptr, size_t bytes);

/* Text of a status code (static storage). */
const char* bpt_status_string(int status);

/* Synchronises `stream`, then reads and clears the device error word.
 * Returns BPT_OK, BPT_ETIMEOUT (a bounded wait ran out; *detail = the wait
 * site id), BPT_EINVAL (a kernel met invalid input data; *detail = its site,
 * e.g. BPT_LM_BAD_TARGET_SITE) or BPT_ECUDA (the synchronisation itself
 * failed; *detail = the cudaError_t).  The first failure of either kind is
 * kept until read.  detail may be NULL. */
int bpt_last_device_error(void* stream, int* detail);

/* Watchdog self-test: exercises the device-side wait limit without faulting
 * anything.  Launches one CTA whose single thread waits, through the same
 * bounded wait every kernel of the library uses, on an mbarrier that nothing
 * arrives at.  After the wait limit (about 4e9 SM cycles, some 2 s) it
 * records BPT_ETIMEOUT with wait site BPT_WATCHDOG_SELFTEST_SITE in the
 * device error word and returns normally; bpt_last_device_error then
 * reports (BPT_ETIMEOUT, BPT_WATCHDOG_SELFTEST_SITE) and clears the word,
 * and later calls run as usual.  Asynchronous on `stream`.  Returns BPT_OK,
 * or BPT_ECUDA if there is no device or the launch fails.  A diagnostic
 * aid: the paper has no such step. */
#define BPT_WATCHDOG_SELFTEST_SITE 900
int bpt_watchdog_selftest(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* BPT_H_ */
