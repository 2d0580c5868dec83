// Launchers of the SIMT kernels (router top-K, dispatch, combine, bias update,
// RMSNorm, fp32 expert GEMMs).  Internal.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kDispatchChunk = 256;   // tokens per count/rank CTA (8 warps x 32)

// n_groups > 0: node-limited routing over topk_groups of n_groups groups;
// row_scale [T] (optional) multiplies each token's summed logits
moe_status_t launch_topk(const float* logits, int splits, long long split_stride,
                         const float* bias, int T, int E, int K, int score_func, int normalize,
                         int n_groups, int topk_groups, int32_t* idx, float* gates,
                         cudaStream_t stream, float* scores = nullptr,
                         const float* row_scale = nullptr);
moe_status_t launch_logits_f32(const float* x, const float* c, int T, int d, int E, float* out,
                               cudaStream_t stream);

// hist: [ceil(T/256), E] int32 scratch
moe_status_t launch_dispatch(const void* x, size_t row_bytes, const int32_t* idx, int T, int K,
                             int E, int32_t* counts, int32_t* offsets, void* xp,
                             int32_t* perm_tok, int32_t* pos, int32_t* hist,
                             cudaStream_t stream);

// counts, offsets (padded to `pad` rows per expert), perm_tok, pos only
moe_status_t launch_dispatch_index(const int32_t* idx, int T, int K, int E, int pad,
                                   int32_t* counts, int32_t* offsets, int32_t* perm_tok,
                                   int32_t* pos, int32_t* hist, cudaStream_t stream);

// FP8 rows: xq row pos[t,k] and row shared_row + t (if shared_row >= 0) get
// token t in e4m3, 1 x 128 tiles; scales xs[kb * ld_s + row].
moe_status_t launch_scatter_quant(const void* x, int T, int K, int d, const int32_t* pos,
                                  int shared_row, void* xq, float* xs, long long ld_s,
                                  cudaStream_t stream);

// out_t = sum_k g y[pos[t,k]] + sum_s y[shared0 + s*shared_stride + t] (+ x_t)
moe_status_t launch_combine(int act_dtype, const void* y, const float* gates, const int32_t* pos,
                            const void* x, void* out, int T, int K, int S, int d,
                            long long shared0, long long shared_stride, int add_residual,
                            cudaStream_t stream);

// xn = x * w / sqrt(mean(x^2) + eps) per token row; inv_rms [T] optional
moe_status_t launch_rmsnorm(int act_dtype, const void* x, const float* w, float eps, int T, int d,
                            void* xn, float* inv_rms, cudaStream_t stream);

// ew = w * e per centroid row (weight dtype, rounded once from the exact product)
moe_status_t launch_fold_centroids(int wgt_dtype, const void* e, const float* w, int E, int d,
                                   void* ew, cudaStream_t stream);

// Dispatch of the layer behind its RMSNorm (bf16): token t's row normalised on
// the fly, xn = (x * inv_rms[t]) * w rounded once to bf16, written to its K
// rows of xp (pos) and, when xs is not null, to row t of xs (shared experts).
moe_status_t launch_scatter_norm(const void* x, const float* inv_rms, const float* w, int T,
                                 int K, int d, const int32_t* pos, void* xp, void* xs,
                                 cudaStream_t stream);

// FP8 dispatch behind the RMSNorm: as launch_scatter_quant on the rows
// xn = bf16((x * inv_rms[t]) * w), normalised on the fly.
moe_status_t launch_scatter_quant_norm(const void* x, const float* inv_rms, const float* w, int T,
                                       int K, int d, const int32_t* pos, int shared_row, void* xq,
                                       float* xs, long long ld_s, cudaStream_t stream);

// one bounded wait that runs out after limit_ns: the device error word gets
// the timeout bit (failure-detection self-test)
moe_status_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream);

moe_status_t launch_update_bias(const int32_t* counts, float* bias, float* stats, int E, int T,
                                int K, float gamma, cudaStream_t stream);

// fp32 expert FFNs over the group table (rows of the routed groups in xp,
// shared groups read x).  act [R, I], y [R, d], R = T*K + S*T.
moe_status_t launch_experts_f32(const float* xp, const float* x, const int32_t* offsets,
                                const float* w13, const float* w2, const float* ws13,
                                const float* ws2, float* act, float* y, int T, int K, int E,
                                int S, int d, int I, cudaStream_t stream);

// ---------------------------------------------------------------- training (backward.cu)
// Padded backward rows: expert e from poff[e] (multiple of 16, zero rows up to
// the next one), shared expert s from poff[E] + s * round_up(T, 16).
// rows_max bounds the padded rows (T*K + 15*E + S*round_up(T, 16)).

// act = SiLU(gate) * up from h = [gate | up] (rows x 2I), bf16
moe_status_t launch_swiglu_fwd(const void* h, void* act, long long rows, int I,
                               cudaStream_t stream);
// dy (padded rows) and dgates [T,K] from dout and the forward's y
moe_status_t launch_combine_bwd(const void* dout, const void* y, const float* gates,
                                const int32_t* idx, const int32_t* perm, const int32_t* counts,
                                const int32_t* offsets, const int32_t* poff, int T, int K, int E,
                                int S, int d, long long rows_max, void* dy, float* dgates,
                                cudaStream_t stream);
// dlogits: Sigmoid -> dlk [T,K] and dlrow [T*K] (at pos); Softmax -> dl [T,E]
moe_status_t launch_router_bwd(const float* dgates, const float* gates, const int32_t* idx,
                               const float* scores, const int32_t* pos, int T, int E, int K,
                               int score_func, int normalize, float* dlk, float* dlrow,
                               float* dl, cudaStream_t stream);
// dxr [T,d] fp32 = dl [T,E] C [E,d]
moe_status_t launch_router_dx_dense(const float* dl, const void* cent, int T, int E, int d,
                                    float* dxr, cudaStream_t stream);
// dh (padded rows, 2I) from dact (padded rows, I) and the forward's h
moe_status_t launch_swiglu_bwd(const void* dact, const void* h, const int32_t* counts,
                               const int32_t* offsets, const int32_t* poff, int T, int K, int E,
                               int S, int I, long long rows_max, void* dh, cudaStream_t stream);
// dx [T,d] from dxp (padded rows), the router term (dlk with C, or dxr) and dout
moe_status_t launch_dx(const void* dxp, const int32_t* pos, const int32_t* idx,
                       const int32_t* offsets, const int32_t* poff, const float* dlk,
                       const void* cent, const float* dxr, const void* dout, void* dx, int T,
                       int K, int E, int S, int d, int add_residual, cudaStream_t stream);
// dC [E,d] fp32 = sum over expert e's rows of dlrow * xp (blocks of the
// input-gradient group table: bs, bstart), via part [max_blocks * kDcentSub, d]:
// each token block is summed in kDcentSub row chunks (many small items fill the
// GPU in several waves), and the chunks are added in block and chunk order
constexpr int kDcentSub = 4;
moe_status_t launch_dcent_sparse(const float* dlrow, const void* xp, const int32_t* counts,
                                 const int32_t* offsets, const int32_t* bs,
                                 const int32_t* bstart, int E, int d, int max_blocks,
                                 float* part, float* dc, cudaStream_t stream);
// dC [E,d] fp32 = dl^T x, via part [ceil(T/256), E, d]
moe_status_t launch_dcent_dense(const float* dl, const void* x, int T, int E, int d, float* part,
                                float* dc, cudaStream_t stream);

}  // namespace moe
