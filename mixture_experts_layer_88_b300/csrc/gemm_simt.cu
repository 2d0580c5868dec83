// fp32 expert FFNs (SwiGLU) for layers whose tokens and weights are fp32.
// One warp per output element, lanes stride over the reduction dimension.
// Row r of the expert-ordered buffers belongs to routed expert e when
// offsets[e] <= r < offsets[e+1] (r < T*K), else to shared expert
// s = (r - T*K) / T on token t = (r - T*K) % T.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

__device__ __forceinline__ int expert_of_row(const int32_t* offsets, int E, int r) {
  int lo = 0, hi = E - 1;  // largest e with offsets[e] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offsets + mid) <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float warp_dot(const float* a, const float* b, int n) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int j = lane; j < n; j += 32) acc = fmaf(a[j], b[j], acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

__global__ void gateup_f32_kernel(const float* __restrict__ xp, const float* __restrict__ x,
                                  const int32_t* __restrict__ offsets,
                                  const float* __restrict__ w13, const float* __restrict__ ws13,
                                  float* __restrict__ act, int T, int K, int E, int S, int d,
                                  int I) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long R = static_cast<long long>(T) * K;           // routed rows
  const long long Rtot = R + static_cast<long long>(S) * T;    // all rows
  if (w >= Rtot * I) return;                                  // whole warp exits together
  const int r = static_cast<int>(w / I), j = static_cast<int>(w % I);
  const float* in;
  const float* W;
  if (r < R) {
    const int e = expert_of_row(offsets, E, r);
    in = xp + static_cast<size_t>(r) * d;
    W = w13 + static_cast<size_t>(e) * 2 * I * d;
  } else {
    const int rr = r - static_cast<int>(R);
    in = x + static_cast<size_t>(rr % T) * d;
    W = ws13 + static_cast<size_t>(rr / T) * 2 * I * d;
  }
  const float g = warp_dot(in, W + static_cast<size_t>(j) * d, d);
  const float u = warp_dot(in, W + static_cast<size_t>(I + j) * d, d);
  if ((threadIdx.x & 31) == 0) act[static_cast<size_t>(r) * I + j] = g / (1.0f + expf(-g)) * u;
}

__global__ void down_f32_kernel(const float* __restrict__ act, const int32_t* __restrict__ offsets,
                                const float* __restrict__ w2, const float* __restrict__ ws2,
                                float* __restrict__ y, int T, int K, int E, int S, int d,
                                int I) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long R = static_cast<long long>(T) * K;
  if (w >= (R + static_cast<long long>(S) * T) * d) return;
  const int r = static_cast<int>(w / d), c = static_cast<int>(w % d);
  const float* W;
  if (r < R) {
    W = w2 + static_cast<size_t>(expert_of_row(offsets, E, r)) * d * I;
  } else {
    W = ws2 + static_cast<size_t>((r - static_cast<int>(R)) / T) * d * I;
  }
  const float v = warp_dot(act + static_cast<size_t>(r) * I, W + static_cast<size_t>(c) * I, I);
  if ((threadIdx.x & 31) == 0) y[static_cast<size_t>(r) * d + c] = v;
}

}  // namespace

moe_status_t launch_experts_f32(const float* xp, const float* x, const int32_t* offsets,
                                const float* w13, const float* w2, const float* ws13,
                                const float* ws2, float* act, float* y, int T, int K, int E,
                                int S, int d, int I, cudaStream_t stream) {
  const long long R = static_cast<long long>(T) * K + static_cast<long long>(S) * T;
  if (R <= 0) return MOE_OK;
  {
    TraceScope tr(stream, "experts_gateup_f32");
    const long long warps = R * I;
    gateup_f32_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, stream>>>(
        xp, x, offsets, w13, ws13, act, T, K, E, S, d, I);
  }
  {
    TraceScope tr(stream, "experts_down_f32");
    const long long warps = R * d;
    down_f32_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, stream>>>(
        act, offsets, w2, ws2, y, T, K, E, S, d, I);
  }
  return launch_status();
}

}  // namespace moe
