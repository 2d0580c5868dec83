// Gate-weighted combine and the balancing-bias update of a DeepSeekMoE layer.
//
// Combine ("DeepSeekMoE架构解析", section 3.1: output = u + shared + routed):
//   out_t = sum_k g_{t,k} y[pos[t,k]] + sum_s y[shared0 + s*stride + t] (+ u_t)
// (shared rows: shared0 = T*K, stride = T in the bf16/fp32 layout; the FP8
// layout places them after the padded routed rows)
// summed in fp32 in that fixed order.  A (t, k) whose pos is negative (an
// expert id the dispatch rejected and flagged) adds nothing.  One thread owns
// 8 consecutive channels (one 16-byte vector) of one token: the K + S + 1
// source rows are gathered with 16-byte loads, the output written with one
// 16-byte store.
//
// Bias update (same page, section 2.2; applied for the next batch per the
// course chapter "MoE", section 5): b_i -= gamma when c_i * E > T * K,
// b_i += gamma when c_i * E < T * K, decided in integers, added in fp32.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void bf16x8_fma(float (&acc)[8], const uint4& v, float g) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
  }
}
__device__ __forceinline__ void bf16x8_add(float (&acc)[8], const uint4& v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
}

__global__ void __launch_bounds__(128) combine_bf16_kernel(
    const uint4* __restrict__ y, const float* __restrict__ gates, const int32_t* __restrict__ pos,
    const uint4* __restrict__ x, uint4* __restrict__ out, int T, int K, int S, int vpr,
    long long shared0, long long shared_stride, int add_residual) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= vpr) return;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int k = 0; k < K; ++k) {
    const int r = __ldg(pos + static_cast<size_t>(t) * K + k);
    if (r < 0) continue;   // a (t, k) the dispatch rejected (flagged there)
    const float g = __ldg(gates + static_cast<size_t>(t) * K + k);
    bf16x8_fma(acc, __ldg(y + static_cast<size_t>(r) * vpr + v), g);
  }
  for (int s = 0; s < S; ++s)
    bf16x8_add(acc, __ldg(y + static_cast<size_t>(shared0 + s * shared_stride + t) * vpr + v));
  if (add_residual) bf16x8_add(acc, __ldg(x + static_cast<size_t>(t) * vpr + v));
  uint4 o;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  out[static_cast<size_t>(t) * vpr + v] = o;
  }
}

// The same for K <= KMAX: every routed row's index and gate is read first and
// every row load is issued before the first sum, so a thread has up to
// K + S + 1 loads in flight instead of one; the sums run in the same order.
template <int KMAX>
__global__ void __launch_bounds__(128) combine_bf16_unrolled_kernel(
    const uint4* __restrict__ y, const float* __restrict__ gates, const int32_t* __restrict__ pos,
    const uint4* __restrict__ x, uint4* __restrict__ out, int T, int K, int S, int vpr,
    long long shared0, long long shared_stride, int add_residual) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= vpr) return;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    int r[KMAX];
    float g[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      r[k] = k < K ? __ldg(pos + static_cast<size_t>(t) * K + k) : -1;
      g[k] = k < K ? __ldg(gates + static_cast<size_t>(t) * K + k) : 0.f;
    }
    uint4 yv[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (r[k] >= 0) yv[k] = __ldg(y + static_cast<size_t>(r[k]) * vpr + v);   // r < 0: rejected
    uint4 sv = make_uint4(0, 0, 0, 0), xv = make_uint4(0, 0, 0, 0);
    if (S > 0) sv = __ldg(y + static_cast<size_t>(shared0 + t) * vpr + v);
    if (add_residual) xv = __ldg(x + static_cast<size_t>(t) * vpr + v);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (r[k] >= 0) bf16x8_fma(acc, yv[k], g[k]);
    if (S > 0) bf16x8_add(acc, sv);
    for (int s = 1; s < S; ++s)
      bf16x8_add(acc, __ldg(y + static_cast<size_t>(shared0 + s * shared_stride + t) * vpr + v));
    if (add_residual) bf16x8_add(acc, xv);
    uint4 o;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    out[static_cast<size_t>(t) * vpr + v] = o;
  }
}

__global__ void __launch_bounds__(128) combine_f32_kernel(
    const float* __restrict__ y, const float* __restrict__ gates, const int32_t* __restrict__ pos,
    const float* __restrict__ x, float* __restrict__ out, int T, int K, int S, int d,
    long long shared0, long long shared_stride, int add_residual) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
  float acc = 0.f;
  for (int k = 0; k < K; ++k) {
    const int r = __ldg(pos + static_cast<size_t>(t) * K + k);
    if (r < 0) continue;   // a (t, k) the dispatch rejected (flagged there)
    acc = fmaf(__ldg(gates + static_cast<size_t>(t) * K + k), __ldg(y + static_cast<size_t>(r) * d + c), acc);
  }
  for (int s = 0; s < S; ++s)
    acc += __ldg(y + static_cast<size_t>(shared0 + s * shared_stride + t) * d + c);
  if (add_residual) acc += __ldg(x + static_cast<size_t>(t) * d + c);
  out[static_cast<size_t>(t) * d + c] = acc;
  }
}

__global__ void __launch_bounds__(1024) update_bias_kernel(const int32_t* __restrict__ counts,
                                                           float* __restrict__ bias,
                                                           float* __restrict__ stats, int E,
                                                           long long TK, float gamma) {
  __shared__ int smax[32], smin[32];
  const int e = threadIdx.x;
  int cmax = INT_MIN, cmin = INT_MAX;
  if (e < E) {
    const int c = counts[e];
    const long long lhs = static_cast<long long>(c) * E;
    float b = bias[e];
    if (lhs > TK) b = __fsub_rn(b, gamma);        // overloaded
    else if (lhs < TK) b = __fadd_rn(b, gamma);   // underloaded
    bias[e] = b;
    cmax = cmin = c;
  }
  if (stats == nullptr) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    cmin = min(cmin, __shfl_xor_sync(0xffffffffu, cmin, o));
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) {
    smax[w] = cmax;
    smin[w] = cmin;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) {
      cmax = max(cmax, smax[i]);
      cmin = min(cmin, smin[i]);
    }
    const double mean = static_cast<double>(TK) / E;
    stats[0] = static_cast<float>(cmax / mean);
    stats[1] = static_cast<float>(cmin / mean);
  }
}

}  // namespace

moe_status_t launch_combine(int act_dtype, const void* y, const float* gates, const int32_t* pos,
                            const void* x, void* out, int T, int K, int S, int d,
                            long long shared0, long long shared_stride, int add_residual,
                            cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  TraceScope tr(stream, "combine");
  if (act_dtype == MOE_BF16) {
    const int vpr = d / 8;
    dim3 grid(ceil_div(vpr, 128), T < 65535 ? T : 65535);
    if (K <= 8)
      combine_bf16_unrolled_kernel<8><<<grid, 128, 0, stream>>>(
          static_cast<const uint4*>(y), gates, pos, static_cast<const uint4*>(x),
          static_cast<uint4*>(out), T, K, S, vpr, shared0, shared_stride, add_residual);
    else
      combine_bf16_kernel<<<grid, 128, 0, stream>>>(
          static_cast<const uint4*>(y), gates, pos, static_cast<const uint4*>(x),
          static_cast<uint4*>(out), T, K, S, vpr, shared0, shared_stride, add_residual);
  } else {
    dim3 grid(ceil_div(d, 128), T < 65535 ? T : 65535);
    combine_f32_kernel<<<grid, 128, 0, stream>>>(static_cast<const float*>(y), gates, pos,
                                                  static_cast<const float*>(x),
                                                  static_cast<float*>(out), T, K, S, d,
                                                  shared0, shared_stride, add_residual);
  }
  return launch_status();
}

moe_status_t launch_update_bias(const int32_t* counts, float* bias, float* stats, int E, int T,
                                int K, float gamma, cudaStream_t stream) {
  TraceScope tr(stream, "update_bias");
  update_bias_kernel<<<1, 1024, 0, stream>>>(counts, bias, stats, E,
                                             static_cast<long long>(T) * K, gamma);
  return launch_status();
}

}  // namespace moe
