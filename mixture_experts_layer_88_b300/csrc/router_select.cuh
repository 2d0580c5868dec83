// Per-token expert selection of the DeepSeekMoE router ("DeepSeekMoE架构解析",
// section 2.1, eqs. (15), (14), (13); section 2.2, eq. (16); section 2.3 for
// node-limited routing), shared by the top-K kernel and the fused router:
//   s_i = Sigmoid(L_i)   (or Softmax over all experts for the 2024 layer)
//   chosen = top-K_r of s_i + b_i   (bias decides who is chosen, not the weight)
//   g_i = s_i / sum of chosen s     (or g_i = s_i without renormalisation)
// One warp per token: the logits of its E experts sit in registers, E/32 per
// lane (expert j*32 + lane in slot j), and K rounds of a 64-bit (key, index)
// warp argmax pick the experts: equal keys go to the lower index, the chosen
// experts are listed by descending key.  Internal.
#pragma once

#include "common.cuh"

namespace moe {

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

// Selection for token t from its logits L (slot j holds expert j*32 + lane;
// slots of experts >= E are ignored).  Writes idx[t, 0..K), gates[t, 0..K)
// and, when scores is not null, s of every expert to scores[t, 0..E).
template <int NPL>
__device__ __forceinline__ void select_experts(const float (&L)[NPL], int lane, size_t t,
                                               const float* __restrict__ bias, int E, int K,
                                               int score_func, int normalize, int n_groups,
                                               int topk_groups, int32_t* __restrict__ idx,
                                               float* __restrict__ gates,
                                               float* __restrict__ scores) {
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
      if (j * 32 + lane < E) scores[t * E + j * 32 + lane] = s[j];
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
        const unsigned long long c = (static_cast<unsigned long long>(keyo[j]) << 32) |
                                     (0xFFFFFFFFu - static_cast<uint32_t>(e));
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
    idx[t * K + lane] = my_e;
    gates[t * K + lane] = g;
  }
}

}  // namespace moe
