// Router epilogue of a DeepSeekMoE layer ("DeepSeekMoE架构解析", section 2.1,
// eqs. (15), (14), (13); section 2.2, eq. (16)):
//   s_i = Sigmoid(u.e_i)   (or Softmax over all experts for the 2024 layer)
//   chosen = top-K_r of s_i + b_i   (bias decides who is chosen, not the weight)
//   g_i = s_i / sum of chosen s     (or g_i = s_i without renormalisation)
// One warp per token sums the K-split partial logits in split order, then
// select_experts (router_select.cuh) picks the experts.  Node-limited routing
// (same page, section 2.3): with n_groups > 0 the experts form n_groups groups
// of consecutive indices; each group's score is the sum of its experts' s
// (summed in a fixed order: within a slot by a butterfly, then over slots);
// the topk_groups best groups (equal sums to the lower group) are kept and
// the K rounds only see their experts.
// Also the fp32 SIMT logits kernel used when tokens are fp32.
#include "common.cuh"
#include "kernels.cuh"
#include "router_select.cuh"

namespace moe {
namespace {

template <int NPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int splits,
                                                   long long split_stride,
                                                   const float* __restrict__ bias, int T, int E,
                                                   int K, int score_func, int normalize,
                                                   int n_groups, int topk_groups,
                                                   int32_t* __restrict__ idx,
                                                   float* __restrict__ gates,
                                                   float* __restrict__ scores,
                                                   const float* __restrict__ row_scale) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  // sum of the K-split partial logits, split by split in a fixed order; the
  // NPL loads of one split are independent, so they are in flight together
  float L[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) L[j] = (j * 32 + lane < E) ? 0.f : -INFINITY;
  const float* row = logits + static_cast<size_t>(t) * E + lane;
  for (int sp = 0; sp < splits; ++sp) {
    float v[NPL];
#pragma unroll
    for (int j = 0; j < NPL; ++j)
      v[j] = (j * 32 + lane < E) ? __ldg(row + sp * split_stride + j * 32) : 0.f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) L[j] += v[j];
  }
  if (row_scale) {   // behind the RMSNorm: logits of x . (w * e_i), times inv_rms
    const float sc = __ldg(row_scale + t);
#pragma unroll
    for (int j = 0; j < NPL; ++j) L[j] *= sc;
  }
  select_experts<NPL>(L, lane, static_cast<size_t>(t), bias, E, K, score_func, normalize,
                      n_groups, topk_groups, idx, gates, scores);
}

// fp32 logits: one warp per (token, expert) dot product, lanes stride over d.
__global__ void logits_f32_kernel(const float* __restrict__ x, const float* __restrict__ c,
                                  int T, int d, int E, float* __restrict__ out) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long long>(T) * E) return;
  const int t = static_cast<int>(w / E), e = static_cast<int>(w % E);
  const float* xr = x + static_cast<size_t>(t) * d;
  const float* cr = c + static_cast<size_t>(e) * d;
  float acc = 0.f;
  for (int j = lane; j < d; j += 32) acc = fmaf(xr[j], cr[j], acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) out[static_cast<size_t>(t) * E + e] = acc;
}

}  // namespace

moe_status_t launch_topk(const float* logits, int splits, long long split_stride,
                         const float* bias, int T, int E, int K, int score_func, int normalize,
                         int n_groups, int topk_groups, int32_t* idx, float* gates,
                         cudaStream_t stream, float* scores, const float* row_scale) {
  if (T <= 0) return MOE_OK;
  TraceScope tr(stream, "router_topk");
  const int grid = ceil_div(T, 8);
#define MOE_TOPK(NPL)                                                                      \
  topk_kernel<NPL><<<grid, 256, 0, stream>>>(logits, splits, split_stride, bias, T, E, K, \
                                             score_func, normalize, n_groups, topk_groups, idx, \
                                             gates, scores, row_scale)
  if (E <= 32) MOE_TOPK(1);
  else if (E <= 64) MOE_TOPK(2);
  else if (E <= 128) MOE_TOPK(4);
  else if (E <= 256) MOE_TOPK(8);
  else if (E <= 512) MOE_TOPK(16);
  else MOE_TOPK(32);
#undef MOE_TOPK
  return launch_status();
}

moe_status_t launch_logits_f32(const float* x, const float* c, int T, int d, int E, float* out,
                               cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  TraceScope tr(stream, "router_logits_f32");
  const long long threads = static_cast<long long>(T) * E * 32;
  const int grid = static_cast<int>((threads + 255) / 256);
  logits_f32_kernel<<<grid, 256, 0, stream>>>(x, c, T, d, E, out);
  return launch_status();
}

}  // namespace moe
