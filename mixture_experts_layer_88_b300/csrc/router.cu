// Router epilogue of a DeepSeekMoE layer ("DeepSeekMoE架构解析", section 2.1,
// eqs. (15), (14), (13); section 2.2, eq. (16)):
//   s_i = Sigmoid(u.e_i)   (or Softmax over all experts for the 2024 layer)
//   chosen = top-K_r of s_i + b_i   (bias decides who is chosen, not the weight)
//   g_i = s_i / sum of chosen s     (or g_i = s_i without renormalisation)
// One warp per token: the logits of its E experts sit in registers, E/32 per
// lane, and K rounds of a 64-bit (key, index) warp argmax pick the experts.
// Node-limited routing (same page, section 2.3): with n_groups > 0 the experts
// form n_groups groups of consecutive indices; each group's score is the sum
// of its experts' s (summed in a fixed order: within a slot by a butterfly,
// then over slots); the topk_groups best groups (equal sums to the lower
// group) are kept and the K rounds only see their experts.
// Also the fp32 SIMT logits kernel used when tokens are fp32.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Bit mask of the kept groups for this warp's token.  Experts per group gs is
// a multiple of 32 or a power of two below 32 (checked by the caller).
template <int NPL>
__device__ __forceinline__ uint32_t kept_groups(const float (&s)[NPL], int E, int n_groups,
                                                int topk_groups, int lane) {
  const int gs = E / n_groups;
  const int seg = gs < 32 ? gs : 32;
  float part[NPL];   // per slot: sum over this lane's segment of seg lanes
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    float v = (j * 32 + lane < E) ? s[j] : 0.f;
    for (int o = 1; o < seg; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    part[j] = v;
  }
  // lane g (< n_groups) gathers group g's score
  float gsum = -INFINITY;
  if (gs >= 32) {
    const int spg = gs >> 5;           // slots per group
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
      if (j / spg == lane) acc += part[j];
    if (lane < n_groups) gsum = acc;
  } else {
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      // group g = j * (32 / gs) + lane / gs lives in slot j, lanes [g*gs % 32, +gs)
      const int g = lane;
      const int src = (g * gs) & 31;
      const float v = __shfl_sync(0xffffffffu, part[j], src);
      if (g < n_groups && (g * gs) >> 5 == j) gsum = v;
    }
  }
  uint32_t mask = 0;
  for (int m = 0; m < topk_groups; ++m) {
    unsigned long long c = 0ull;
    if (lane < n_groups && !((mask >> lane) & 1u))
      c = (static_cast<unsigned long long>(orderable(gsum)) << 32) | (0xFFFFFFFFu - lane);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, c, o);
      c = other > c ? other : c;
    }
    mask |= 1u << (0xFFFFFFFFu - static_cast<uint32_t>(c & 0xFFFFFFFFull));
  }
  return mask;
}

template <int NPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int splits,
                                                   long long split_stride,
                                                   const float* __restrict__ bias, int T, int E,
                                                   int K, int score_func, int normalize,
                                                   int n_groups, int topk_groups,
                                                   int32_t* __restrict__ idx,
                                                   float* __restrict__ gates,
                                                   float* __restrict__ scores) {
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
  float s[NPL];
  if (score_func == MOE_SCORE_SOFTMAX) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NPL; ++j) m = fmaxf(m, L[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      s[j] = (j * 32 + lane < E) ? expf(L[j] - m) : 0.f;
      sum += s[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
    for (int j = 0; j < NPL; ++j) s[j] = s[j] / sum;
  } else {
#pragma unroll
    for (int j = 0; j < NPL; ++j) s[j] = 1.0f / (1.0f + expf(-L[j]));
  }
  if (scores) {   // training forward: every expert's s for the backward
#pragma unroll
    for (int j = 0; j < NPL; ++j)
      if (j * 32 + lane < E) scores[static_cast<size_t>(t) * E + j * 32 + lane] = s[j];
  }
  uint32_t keyo[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = j * 32 + lane;
    keyo[j] = (e < E) ? orderable(s[j] + __ldg(bias + e)) : 0u;
  }
  uint32_t taken = 0;   // per slot: already chosen, or outside the kept groups
  if (n_groups > 0) {
    const uint32_t gm = kept_groups<NPL>(s, E, n_groups, topk_groups, lane);
    const int gs = E / n_groups;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = j * 32 + lane;
      if (e < E && !((gm >> (e / gs)) & 1u)) taken |= 1u << j;
    }
  }
  int my_e = 0;
  float my_s = 0.f, sum_sel = 0.f;
  for (int k = 0; k < K; ++k) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = j * 32 + lane;
      if (e < E && !((taken >> j) & 1u)) {
        const unsigned long long c =
            (static_cast<unsigned long long>(keyo[j]) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
        best = c > best ? c : best;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int e_win = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull));
    const int owner = e_win & 31, jw = e_win >> 5;
    float sv = 0.f;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
      if (j == jw) sv = s[j];
    if (lane == owner) taken |= 1u << jw;
    sv = __shfl_sync(0xffffffffu, sv, owner);
    sum_sel += sv;
    if (lane == k) {
      my_e = e_win;
      my_s = sv;
    }
  }
  if (lane < K) {
    float g = my_s;
    if (normalize) g = sum_sel > 0.f ? my_s / sum_sel : 0.f;
    idx[static_cast<size_t>(t) * K + lane] = my_e;
    gates[static_cast<size_t>(t) * K + lane] = g;
  }
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
                         cudaStream_t stream, float* scores) {
  if (T <= 0) return MOE_OK;
  TraceScope tr(stream, "router_topk");
  const int grid = ceil_div(T, 8);
#define MOE_TOPK(NPL)                                                                      \
  topk_kernel<NPL><<<grid, 256, 0, stream>>>(logits, splits, split_stride, bias, T, E, K, \
                                             score_func, normalize, n_groups, topk_groups, idx, \
                                             gates, scores)
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
