/*
 * moe.h - C ABI of the DeepSeekMoE layer (forward, balancing, training backward)
 * for NVIDIA B300 (sm_103a).
 *
 * One DeepSeekMoE layer: a Sigmoid router with an auxiliary-loss-free
 * balancing bias, hard top-K_r selection, renormalised gates, no-drop dispatch
 * to fine-grained SwiGLU routed experts, always-on shared experts, a
 * gate-weighted combine, and the per-batch load count / sign bias update.
 *
 * Sources ("DeepSeekMoE架构解析", the DeepSeek-V3 walk-through, is "V3";
 * the course chapter "MoE" on blog.zero43.top is "course"):
 *   V3 section 2.1, eqs. (13)-(15)   score, top-K, renormalisation
 *   V3 section 2.2, eq. (16)         bias changes selection only
 *   V3 section 2.2, update rule      b_i -/+ gamma for over/under-loaded experts
 *   V3 section 3.1                   output = u + shared + gate-weighted routed
 *   course section 4                 2024 variant: gates not renormalised
 *   course sections 5, 6             bias applies to the next batch; no drops
 *   V3 section 4.1                   RMSNorm in front of the layer, eps 1e-6
 *   V3 section 4.3                   FP8: 128x128 weight blocks, 1x128 tiles
 *   V3 section 2.2 + chain rule      training backward (moe_backward)
 *
 * Conventions for every entry point
 *   - All tensors are row-major, densely packed, in device memory, unless a
 *     parameter says "host".  The caller allocates and owns every buffer; the
 *     library allocates nothing on any call below.
 *   - Floating tensors use cfg->act_dtype (tokens, activations, outputs) or
 *     cfg->wgt_dtype (centroids, expert weights).  Supported pairs:
 *     (MOE_F32, MOE_F32), (MOE_BF16, MOE_BF16) and (MOE_BF16, MOE_E4M3); the
 *     last is the FP8 layer (block-scaled e4m3 expert weights, bf16 tokens
 *     and centroids) served by the *_fp8 entry points.  Bias, gates and load
 *     statistics are always fp32; indices, counts, offsets are int32.
 *   - For MOE_BF16, d and I must be multiples of 128 and every pointer must be
 *     16-byte aligned.  Limits: 1 <= K <= min(E, 32), E <= 1024, S <= 64,
 *     T*K + S*T < 2^31.  T == 0 is a valid empty batch (nothing is launched).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: argument errors are returned synchronously, launch errors
 *     map to MOE_ERR_CUDA, and faults the kernels detect on the device
 *     (a bounded wait that ran out) are read back with moe_get_status().
 *   - `ws` is caller-owned scratch of at least moe_workspace_size(cfg, which)
 *     bytes, 256-byte aligned; its contents on entry do not matter.
 *   - Calls sharing a workspace must be ordered on one stream.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* bad shape, null or misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2,     /* valid but not built (dtype pair, device) */
  MOE_ERR_WORKSPACE = 3,       /* ws too small */
  MOE_ERR_CUDA = 4,            /* a CUDA runtime/launch error */
  MOE_ERR_DEVICE_TIMEOUT = 5,  /* a device-side bounded wait ran out */
  MOE_ERR_DEVICE_BOUNDS = 6    /* a device-side index check failed */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_E4M3 = 2 } moe_dtype_t;

/* Expert score s_{i,t}.  SIGMOID: V3 eq. (15).  SOFTMAX: the earlier gating
 * that V3 replaced (V3 section 2.1), used by the 2024 16B layer. */
typedef enum { MOE_SCORE_SIGMOID = 0, MOE_SCORE_SOFTMAX = 1 } moe_score_t;

typedef struct {
  int32_t T;            /* tokens in the batch */
  int32_t d;            /* hidden size */
  int32_t E;            /* routed experts */
  int32_t K;            /* routed experts per token, K_r */
  int32_t S;            /* shared experts (always active) */
  int32_t I;            /* intermediate size of every expert (routed and shared) */
  int32_t act_dtype;    /* moe_dtype_t of x, activations, outputs */
  int32_t wgt_dtype;    /* moe_dtype_t of centroids and expert weights */
  int32_t score_func;   /* moe_score_t */
  int32_t normalize;    /* 1: g = g'/sum g' (V3 eq. 13); 0: g = s (course section 4) */
  int32_t add_residual; /* 1: out = u + ... (V3 section 3.1); 0: MoE term only */
  float gamma;          /* bias update speed, 0.001 in V3 section 2.2 */
  int32_t n_groups;     /* node-limited routing (V3 section 2.3): 0 = off, else the
                           experts form n_groups groups of E / n_groups consecutive
                           indices (a multiple of 32, or a power of two below 32;
                           n_groups <= 32) */
  int32_t topk_groups;  /* groups kept per token, ranked by the sum of their
                           experts' scores s (equal sums: lower group); top-K then
                           runs over the kept groups' experts only.  0 when
                           n_groups is 0, else 1..n_groups with K <= topk_groups *
                           E / n_groups */
} moe_cfg_t;

/* Which call a workspace is sized for. */
typedef enum {
  MOE_WS_ROUTE = 0,
  MOE_WS_DISPATCH = 1,
  MOE_WS_EXPERTS = 2,
  MOE_WS_FORWARD = 3,
  MOE_WS_FORWARD_PRENORM = 4,  /* moe_forward_prenorm / moe_forward_fp8_prenorm */
  MOE_WS_FORWARD_W8A16 = 5,    /* moe_forward_w8a16 (FP8 layers) */
  MOE_WS_FORWARD_TRAIN = 6,    /* moe_forward_train */
  MOE_WS_BACKWARD = 7          /* moe_backward */
} moe_ws_kind_t;

/* Bytes of scratch that `which` needs for this cfg (0 on an invalid cfg). */
size_t moe_workspace_size(const moe_cfg_t* cfg, int32_t which);

/* Check cfg alone (shape limits, dtype pair).  No CUDA calls. */
moe_status_t moe_check_cfg(const moe_cfg_t* cfg);

/*
 * moe_route - router of V3 eqs. (15), (16), (14), (13).
 *   x         [T, d]   act_dtype   tokens u_t
 *   centroids [E, d]   wgt_dtype   expert centroids e_i
 *   bias      [E]      fp32        balancing bias b_i (read only)
 *   idx       [T, K]   int32  out  chosen experts, by descending s+b,
 *                                  equal keys to the lower index
 *   gates     [T, K]   fp32   out  g_{i,t}: s_i / sum of chosen s (normalize=1)
 *                                  or s_i (normalize=0); never uses b
 * Scores and keys are fp32; logits are accumulated in fp32.
 */
moe_status_t moe_route(const moe_cfg_t* cfg, const void* x, const void* centroids,
                       const float* bias, int32_t* idx, float* gates,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * moe_dispatch - no-drop dispatch (course section 6): every (t, k) gets a row.
 *   x         [T, d]       act_dtype   tokens
 *   idx       [T, K]       int32       from moe_route
 *   counts    [E]          int32  out  load count c_i = #{(t,k): idx = i}
 *   offsets   [E+1]        int32  out  exclusive prefix sum of counts
 *   xp        [T*K, d]     act_dtype out  rows of expert i at offsets[i] ..,
 *                                  its tokens in ascending token order
 *   perm_tok  [T*K]        int32  out  source token of each xp row
 *   pos       [T, K]       int32  out  xp row of (t, k)
 * Integer results are deterministic.  idx entries must lie in [0, E) and be
 * distinct per token (as moe_route writes them).
 */
moe_status_t moe_dispatch(const moe_cfg_t* cfg, const void* x, const int32_t* idx,
                          int32_t* counts, int32_t* offsets, void* xp,
                          int32_t* perm_tok, int32_t* pos,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * moe_experts - fine-grained SwiGLU experts (V3 section 1 and the section 3.1
 * sketch): y = W2 (SiLU(Wg u) * (Wu u)) for each routed row of xp with its
 * expert's weights, and for every token with each shared expert.
 *   xp       [T*K, d]        act_dtype   dispatched rows (moe_dispatch)
 *   x        [T, d]          act_dtype   tokens (input of the shared experts)
 *   offsets  [E+1]           int32       from moe_dispatch
 *   w13      [E, 2I, d]      wgt_dtype   rows 0..I-1 gate Wg, rows I..2I-1 up Wu
 *   w2       [E, d, I]       wgt_dtype   down projection
 *   ws13     [S, 2I, d], ws2 [S, d, I]   shared experts, same layout (may be
 *                                        NULL when S == 0)
 *   act      [T*K + S*T, I]  act_dtype out  SiLU(gate) * up, rounded to act_dtype
 *   y        [T*K + S*T, d]  act_dtype out  rows 0..T*K-1: routed expert outputs in
 *                                  xp order; row T*K + s*T + t: shared expert s on
 *                                  token t
 * Accumulation is fp32.
 */
moe_status_t moe_experts(const moe_cfg_t* cfg, const void* xp, const void* x,
                         const int32_t* offsets, const void* w13, const void* w2,
                         const void* ws13, const void* ws2, void* act, void* y,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * moe_experts_static - moe_experts without a caller workspace, for callers
 * that cannot allocate device memory: an inference runtime that reserves all
 * of its device memory at start-up and forbids allocation on the request
 * path, or a plugin whose host framework owns the allocator and passes no
 * scratch buffer.  The pages have no counterpart; this is a packaging of the
 * same computation.
 *   Arguments, layouts and results as moe_experts (minus ws, ws_bytes).
 *   Its scratch (the per-expert group table, about 22 KB) is a fixed array
 *   inside the library, sized for E + S <= 1088 groups; larger E + S returns
 *   MOE_ERR_INVALID_ARG.  Every GPU that loads the library holds that array
 *   until the process exits.
 *   The first call on a device looks up the array's device address (no
 *   allocation); make that first call before any stream capture.
 *   Calls share the array: calls that may overlap on the GPU (different
 *   streams without ordering between them) race and give wrong results.
 *   Calls no allocating routine (no cudaMalloc/cudaFree).
 */
moe_status_t moe_experts_static(const moe_cfg_t* cfg, const void* xp, const void* x,
                                const int32_t* offsets, const void* w13, const void* w2,
                                const void* ws13, const void* ws2, void* act, void* y,
                                void* stream);

/*
 * moe_combine - V3 section 3.1: out_t = [u_t] + sum_s y_shared(s,t)
 *               + sum_k g_{t,k} y[pos[t,k]], summed in fp32 in the order
 *               k = 0..K-1, then shared s = 0..S-1, then the residual.
 *   y      [T*K + S*T, d]  act_dtype   from moe_experts
 *   gates  [T, K] fp32, pos [T, K] int32 (moe_route, moe_dispatch)
 *   x      [T, d]          act_dtype   residual u (read only if add_residual)
 *   out    [T, d]          act_dtype out
 */
moe_status_t moe_combine(const moe_cfg_t* cfg, const void* y, const float* gates,
                         const int32_t* pos, const void* x, void* out, void* stream);

/*
 * moe_update_bias - V3 section 2.2 update rule, applied after the batch and
 * used by the next one (course section 5):
 *   counts[i] * E > T*K  ->  bias[i] -= gamma   (overloaded)
 *   counts[i] * E < T*K  ->  bias[i] += gamma   (underloaded)
 *   equal                ->  unchanged
 * Integer comparison, fp32 add (round to nearest even).
 *   counts     [E] int32        load counts of this batch
 *   bias       [E] fp32 in/out  updated in place
 *   load_stats [2] fp32 out     {max c_i / mean, min c_i / mean}, or NULL
 */
moe_status_t moe_update_bias(const moe_cfg_t* cfg, const int32_t* counts, float* bias,
                             float* load_stats, void* stream);

/*
 * moe_forward - the whole layer: moe_route -> moe_dispatch -> moe_experts ->
 * moe_combine on one stream with no host synchronisation.  Dispatched rows,
 * activations and expert outputs live in ws (MOE_WS_FORWARD).  The bias is
 * read, not updated: call moe_update_bias(counts) afterwards to apply the
 * balancing step for the next batch.
 *   x [T,d], centroids [E,d], bias [E], w13, w2, ws13, ws2 as above;
 *   idx [T,K] int32 out, gates [T,K] fp32 out, counts [E] int32 out,
 *   out [T,d] act_dtype out.
 */
moe_status_t moe_forward(const moe_cfg_t* cfg, const void* x, const void* centroids,
                         const float* bias, const void* w13, const void* w2,
                         const void* ws13, const void* ws2, int32_t* idx,
                         float* gates, int32_t* counts, void* out,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * moe_rmsnorm - the RMSNorm in front of the MoE layer (V3 section 4.1: an
 * RMSNorm before and after the MoE layer, eps = 1e-6), per token row:
 *   inv_rms[t] = 1 / sqrt(sum_j x[t,j]^2 / d + eps)
 *   xn[t,j]    = x[t,j] * inv_rms[t] * norm_w[j]
 * in fp32, rounded once (nearest even) to act_dtype.
 *   x [T,d] act_dtype, norm_w [d] fp32 (16-byte aligned), eps > 0;
 *   xn [T,d] act_dtype out (may be x itself), inv_rms [T] fp32 out or NULL.
 */
moe_status_t moe_rmsnorm(const moe_cfg_t* cfg, const void* x, const float* norm_w, float eps,
                         void* xn, float* inv_rms, void* stream);

/*
 * moe_forward_prenorm - the layer behind its RMSNorm, h = x + MoE(RMSNorm(x)):
 * moe_rmsnorm(x) into the workspace, then moe_forward on the normalised
 * tokens (router, dispatch, shared experts), with the residual (add_residual)
 * taken from x itself.  ws: MOE_WS_FORWARD_PRENORM bytes.  Other arguments as
 * moe_forward and moe_rmsnorm.
 */
moe_status_t moe_forward_prenorm(const moe_cfg_t* cfg, const void* x, const float* norm_w,
                                 float eps, const void* centroids, const float* bias,
                                 const void* w13, const void* w2, const void* ws13,
                                 const void* ws2, int32_t* idx, float* gates, int32_t* counts,
                                 void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * FP8 layers (V3 section 4.3): expert weights in e4m3 with one fp32 scale per
 * 128 x 128 block (w = q * scale), activations quantised inside the layer to
 * e4m3 in 1 x 128 tiles along K (scale = max|x| / 448), and tensor-core
 * partial sums promoted to fp32 on the CUDA cores every 128 elements of K.
 * cfg: act_dtype MOE_BF16, wgt_dtype MOE_E4M3; d and I multiples of 128, at most 8192.
 * Centroids are bf16 (the router is not quantised).
 */
typedef struct {
  const void* w13;  const float* w13_scale;   /* [E,2I,d] e4m3; [E, 2I/128, d/128] */
  const void* w2;   const float* w2_scale;    /* [E,d,I]  e4m3; [E, d/128, I/128]  */
  const void* ws13; const float* ws13_scale;  /* [S,2I,d] e4m3; [S, 2I/128, d/128] (NULL if S == 0) */
  const void* ws2;  const float* ws2_scale;   /* [S,d,I]  e4m3; [S, d/128, I/128]  */
} moe_fp8_weights_t;

/*
 * Row layout of the FP8 buffers.  Rows of expert e start at offsets[e], a
 * multiple of 4; the shared experts read their tokens from rows
 * shared_row .. shared_row + T - 1 of xq and write their outputs from row
 * shared_row + s * round_up(T, 4) of act / y.  rows_in: rows of xq (and
 * columns of xq_scale); rows_out: rows of act and y (columns of act_scale).
 */
moe_status_t moe_fp8_rows(const moe_cfg_t* cfg, int64_t* rows_in, int64_t* rows_out,
                          int64_t* shared_row);

/*
 * moe_dispatch_fp8 - moe_dispatch for FP8 layers: the same counts, pos and
 * perm_tok (expert rows in ascending token order), but offsets[e] is the
 * prefix sum of counts rounded up to 4 rows, and the rows are written
 * quantised:
 *   xq       [rows_in, d]         e4m3 out  q = rne_sat(x * 448 / max|tile|)
 *   xq_scale [d/128, rows_in]     fp32 out  max|tile| / 448 (K-block major)
 *   perm_tok [shared_row]         int32 out  source token of each routed row
 * Rows of routed expert e: offsets[e] .. + counts[e]; shared-expert input:
 * rows shared_row .. + T (moe_fp8_rows).  Other rows (and their perm_tok
 * entries) are left unwritten.
 */
moe_status_t moe_dispatch_fp8(const moe_cfg_t* cfg, const void* x, const int32_t* idx,
                              int32_t* counts, int32_t* offsets, void* xq, float* xq_scale,
                              int32_t* perm_tok, int32_t* pos, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * moe_experts_fp8 - moe_experts for FP8 layers on the moe_dispatch_fp8 rows.
 *   act       [rows_out, I]        e4m3 out  SiLU(gate) * up, 1 x 128 tiles
 *   act_scale [I/128, rows_out]    fp32 out
 *   y         [rows_out, d]        bf16 out  expert outputs (routed at
 *                                  offsets[e] + r, shared expert s at
 *                                  shared_row + s * round_up(T, 4) + t)
 * ws: MOE_WS_EXPERTS bytes.  Accumulation is fp32 (promotion every 128 K).
 */
moe_status_t moe_experts_fp8(const moe_cfg_t* cfg, const void* xq, const float* xq_scale,
                             const int32_t* offsets, const int32_t* counts,
                             const moe_fp8_weights_t* w, void* act, float* act_scale, void* y,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward_fp8 - the FP8 layer: moe_route -> moe_dispatch_fp8 ->
 * moe_experts_fp8 -> moe_combine on one stream, no host synchronisation;
 * arguments as moe_forward with the weights in `w`.  moe_combine and
 * moe_update_bias take FP8 cfgs as they are (moe_combine reads the FP8 row
 * layout); moe_dispatch, moe_experts, moe_experts_static and moe_forward
 * return MOE_ERR_UNSUPPORTED for them.
 */
moe_status_t moe_forward_fp8(const moe_cfg_t* cfg, const void* x, const void* centroids,
                             const float* bias, const moe_fp8_weights_t* w, int32_t* idx,
                             float* gates, int32_t* counts, void* out, void* ws,
                             size_t ws_bytes, void* stream);

/*
 * W8A16 form of an FP8 layer: the e4m3 block-scaled expert weights meet bf16
 * tokens and activations.  Each 64-wide slice of a weight tile is brought in
 * as e4m3, dequantised in shared memory to bf16 (q * scale of its 128 x 128
 * block, rounded once) and multiplied on the bf16 tensor cores with fp32
 * accumulation over all of K; nothing else is quantised.  The rows follow the
 * bf16 layer's layout: dispatch and combine are moe_dispatch / moe_combine
 * called with the same cfg but wgt_dtype = MOE_BF16 (they read no weights).
 *   moe_experts_w8a16: xp [T*K, d] bf16 (moe_dispatch), x [T, d] (shared
 *     experts' input), offsets [E+1]; act [T*K+S*T, I] and y [T*K+S*T, d] bf16
 *     out; ws: MOE_WS_EXPERTS bytes.
 *   moe_forward_w8a16: route -> dispatch -> experts -> combine on one stream;
 *     ws: MOE_WS_FORWARD_W8A16 bytes.  Other arguments as moe_forward_fp8.
 */
moe_status_t moe_experts_w8a16(const moe_cfg_t* cfg, const void* xp, const void* x,
                               const int32_t* offsets, const moe_fp8_weights_t* w, void* act,
                               void* y, void* ws, size_t ws_bytes, void* stream);
moe_status_t moe_forward_w8a16(const moe_cfg_t* cfg, const void* x, const void* centroids,
                               const float* bias, const moe_fp8_weights_t* w, int32_t* idx,
                               float* gates, int32_t* counts, void* out, void* ws,
                               size_t ws_bytes, void* stream);

/* moe_forward_fp8 behind the RMSNorm, as moe_forward_prenorm: the router reads
 * the normalised bf16 tokens, the dispatch quantises them to e4m3 1 x 128
 * tiles in its single read, the residual is x.  ws: MOE_WS_FORWARD_PRENORM. */
moe_status_t moe_forward_fp8_prenorm(const moe_cfg_t* cfg, const void* x, const float* norm_w,
                                     float eps, const void* centroids, const float* bias,
                                     const moe_fp8_weights_t* w, int32_t* idx, float* gates,
                                     int32_t* counts, void* out, void* ws, size_t ws_bytes,
                                     void* stream);

/*
 * Training: a forward that keeps what the backward needs, and the backward.
 * bf16 layers only (act_dtype = wgt_dtype = MOE_BF16); other cfgs return
 * MOE_ERR_UNSUPPORTED.  No page writes the backward out: it is the chain rule
 * through the forward of V3 sections 2.1 and 3.1 with the chosen experts held
 * fixed; the balancing bias gets no gradient (V3 section 2.2: it only steers
 * the choice) and is updated by moe_update_bias as in inference.
 *
 * moe_train_state_t - caller-owned device buffers written by moe_forward_train
 * and read by moe_backward (R = T*K + S*T):
 *   idx [T,K] int32, gates [T,K] fp32, scores [T,E] fp32 (s of every expert),
 *   counts [E], offsets [E+1], perm_tok [T*K], pos [T,K] int32 (moe_dispatch),
 *   xp [T*K, d] bf16 (dispatched rows), h [R, 2I] bf16 (gate | up
 *   pre-activations of every row), act [R, I] bf16 (SiLU(gate) * up computed
 *   from the stored h), y [R, d] bf16 (expert outputs).
 */
typedef struct {
  int32_t* idx;
  float* gates;
  float* scores;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm_tok;
  int32_t* pos;
  void* xp;
  void* h;
  void* act;
  void* y;
} moe_train_state_t;

/*
 * moe_grads_t - caller-owned gradient outputs of moe_backward (overwritten):
 *   dx [T,d] bf16, dcentroids [E,d] fp32, dw13 [E,2I,d], dw2 [E,d,I],
 *   dws13 [S,2I,d], dws2 [S,d,I] bf16 (NULL when S == 0).  Experts that no
 *   token chose get zero weight gradients.
 */
typedef struct {
  void* dx;
  float* dcentroids;
  void* dw13;
  void* dw2;
  void* dws13;
  void* dws2;
} moe_grads_t;

/*
 * moe_forward_train - moe_forward that also fills `st`: the router writes
 * every expert's score, the gate/up GEMM writes h instead of act, act =
 * SiLU(gate) * up is formed from the stored bf16 h, then down and combine as
 * in moe_forward.  out [T,d] as moe_forward.  ws: MOE_WS_FORWARD_TRAIN.
 */
moe_status_t moe_forward_train(const moe_cfg_t* cfg, const void* x, const void* centroids,
                               const float* bias, const void* w13, const void* w2,
                               const void* ws13, const void* ws2, const moe_train_state_t* st,
                               void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_backward - gradients of a loss L given dout = dL/d(out) [T,d] bf16, for
 * the batch that moe_forward_train(st) ran on (same x, weights and cfg):
 *   dgates[t,k] = dout_t . y[pos[t,k]];  expert e's output gradient on its
 *   row is gates[t,k] * dout_t (shared experts: dout_t);
 *   experts: da = dy W2, dW2 = dy^T act, [dgate, dup] = [da * up *
 *   SiLU'(gate), da * SiLU(gate)], dW13 = [dgate, dup]^T u, du = [dgate, dup] W13;
 *   router (V3 eqs. 13-15): ds = (dg - sum dg g) / sum s (renormalised gates,
 *   else ds = dg), dlogit = ds s (1 - s) (Sigmoid) or s (ds - sum ds s)
 *   (Softmax), dx += dlogit C, dC = dlogit^T u;  dx += dout (add_residual).
 * Weight gradients are fp32 sums rounded once to bf16; dx sums its terms in
 * fp32; the intermediate gradients (g * dout, da, [dgate, dup], the routed
 * rows' du) are held in bf16.  ws: MOE_WS_BACKWARD.
 */
moe_status_t moe_backward(const moe_cfg_t* cfg, const void* dout, const void* x,
                          const void* centroids, const void* w13, const void* w2,
                          const void* ws13, const void* ws2, const moe_train_state_t* st,
                          const moe_grads_t* grads, void* ws, size_t ws_bytes, void* stream);

/* Waits for `stream`, then returns and clears this device's error word
 * (MOE_OK, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_BOUNDS) or MOE_ERR_CUDA. */
moe_status_t moe_get_status(void* stream);

/*
 * Failure-detection self-test: launches one thread that waits, with the same
 * bounded barrier wait every GEMM role uses, on a barrier nothing arrives on.
 * After limit_ns (1 ns .. 1 s) the wait gives up, the kernel sets the timeout
 * bit of the device error word and returns; the next moe_get_status() on the
 * stream reports MOE_ERR_DEVICE_TIMEOUT (and clears it).  Nothing faults or
 * hangs; the context stays usable.
 */
moe_status_t moe_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Static text for a status code. */
const char* moe_status_string(moe_status_t st);

/*
 * Kernel timing (tracing).  While enabled, every kernel the calls above
 * launch is bracketed by CUDA events on its own stream, and its name, launch
 * count and summed device time are kept per calling thread.  Events come from
 * a pool created on first use; no device memory is allocated.  Calls made
 * while their stream is being captured into a CUDA graph record their events
 * as event-record nodes of the graph: read them after the graph has run.
 */
typedef struct {
  char name[48];
  int32_t launches;
  float total_ms;
} moe_kernel_time_t;

moe_status_t moe_trace_enable(int32_t on);
/* Synchronises the traced events, writes up to `max` entries, sets *n to the
 * number of distinct kernels, and clears the record. */
moe_status_t moe_trace_read(moe_kernel_time_t* out, int32_t max, int32_t* n);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
