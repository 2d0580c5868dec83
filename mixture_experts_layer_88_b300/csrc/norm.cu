// RMSNorm in front of the MoE layer ("DeepSeekMoE架构解析", section 4.1: an
// RMSNorm sits before and after the MoE layer, eps = 1e-6):
//   inv_rms_t = 1 / sqrt(mean_j x_tj^2 + eps),   xn_tj = x_tj * inv_rms_t * w_j
// in fp32, rounded once to the activation type.
//
// Also the weighted centroids w * e_i of the router behind the RMSNorm (its
// logit is (x * inv_rms * w) . e_i = inv_rms * (x . (w * e_i))).
//
// HBM-bound: one 128-thread CTA per token row.  The first pass sums the
// squares (16-byte loads of bf16), the CTA reduces them in a fixed order, and
// the second pass re-reads the same row (from L1/L2, so DRAM sees it once),
// scales it and writes it with 16-byte stores.  xn may alias x: every thread
// reads an element before it writes it, and all reads of the first pass end
// at the CTA barrier of the reduction.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kNormThreads = 128;

// Sum over the CTA; every thread returns the same value (fixed order).
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) s += red[i];
  return s;
}

__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_bf16_kernel(const uint4* x, const float4* __restrict__ w, float eps, int d,
                        uint4* xn, float* __restrict__ inv_rms) {
  __shared__ float red[kNormThreads / 32];
  const int nv = d >> 3;                       // 8 bf16 per 16-byte vector
  const size_t row = blockIdx.x;
  const uint4* xr = x + row * nv;
  float ss = 0.f;
  for (int i = threadIdx.x; i < nv; i += kNormThreads) {
    const uint4 v = xr[i];
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      ss = fmaf(f.x, f.x, ss);
      ss = fmaf(f.y, f.y, ss);
    }
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  if (threadIdx.x == 0 && inv_rms) inv_rms[row] = inv;
  uint4* orow = xn + row * nv;
  for (int i = threadIdx.x; i < nv; i += kNormThreads) {
    const uint4 v = xr[i];
    const float4 w0 = __ldg(w + 2 * i), w1 = __ldg(w + 2 * i + 1);
    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint4 o;
    __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      oh[k] = __floats2bfloat162_rn((f.x * inv) * wv[2 * k], (f.y * inv) * wv[2 * k + 1]);
    }
    orow[i] = o;
  }
}

__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_f32_kernel(const float* x, const float* __restrict__ w, float eps, int d, float* xn,
                       float* __restrict__ inv_rms) {
  __shared__ float red[kNormThreads / 32];
  const size_t row = blockIdx.x;
  const float* xr = x + row * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += kNormThreads) ss = fmaf(xr[i], xr[i], ss);
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  if (threadIdx.x == 0 && inv_rms) inv_rms[row] = inv;
  float* orow = xn + row * d;
  for (int i = threadIdx.x; i < d; i += kNormThreads) orow[i] = (xr[i] * inv) * __ldg(w + i);
}

// Weighted centroids of the router behind the RMSNorm: ew[i, j] = w_j * e_ij,
// from the exact product (a float times a bf16 or float is exact in double)
// rounded once to the weight type.
__global__ void fold_bf16_kernel(const __nv_bfloat16* __restrict__ e, const float* __restrict__ w,
                                 int d, long long n, __nv_bfloat16* __restrict__ ew) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const double v = static_cast<double>(__ldg(w + i % d)) *
                     static_cast<double>(__bfloat162float(e[i]));
    ew[i] = __double2bfloat16(v);
  }
}

// bf16 of the exact product w * e, rounded once, in fp32 arithmetic: p = w * e
// rounded to fp32 and its error err = w * e - p (exact through an FMA, the
// TwoProduct error-free transformation).  Rounding p to bf16 gives the correctly
// rounded product except when p sits exactly halfway between two bf16 values
// and err is not zero; then the exact product lies on err's side of the
// midpoint and is rounded that way.  (Products here are far from fp32's
// subnormal range, where err could itself round.)
__device__ __forceinline__ __nv_bfloat16 product_bf16(float w, float e) {
  const float p = w * e;
  const float err = fmaf(w, e, -p);
  const uint32_t u = __float_as_uint(p);
  if ((u & 0xffffu) == 0x8000u && err != 0.f) {
    const bool away = (err > 0.f) == (p > 0.f);   // the exact magnitude is larger
    const uint32_t r = away ? (u + 0x8000u) >> 16 : u >> 16;
    return __ushort_as_bfloat16(static_cast<unsigned short>(r));
  }
  return __float2bfloat16_rn(p);
}

// The same fold as fold_bf16_kernel, eight elements per thread with 16-byte
// loads and stores (d a multiple of 8), the product rounded by product_bf16.
__global__ void fold_bf16_x8_kernel(const uint4* __restrict__ e, const float4* __restrict__ w,
                                    int vpr, int nvec, uint4* __restrict__ ew) {
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += gridDim.x * blockDim.x) {
    const int c = v % vpr;                       // 8-element column block of the row
    const uint4 q = __ldg(e + v);
    const float4 w0 = __ldg(w + 2 * c), w1 = __ldg(w + 2 * c + 1);
    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&q);
    uint4 o;
    __nv_bfloat16* oh = reinterpret_cast<__nv_bfloat16*>(&o);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      oh[k] = product_bf16(wv[k], __bfloat162float(h[k]));
    ew[v] = o;
  }
}

__global__ void fold_f32_kernel(const float* __restrict__ e, const float* __restrict__ w, int d,
                                long long n, float* __restrict__ ew) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    ew[i] = static_cast<float>(static_cast<double>(__ldg(w + i % d)) * static_cast<double>(e[i]));
}

}  // namespace

moe_status_t launch_fold_centroids(int wgt_dtype, const void* e, const float* w, int E, int d,
                                   void* ew, cudaStream_t stream) {
  if (E <= 0) return MOE_OK;
  TraceScope tr(stream, "fold_centroids");
  const long long n = static_cast<long long>(E) * d;
  const int grid = static_cast<int>(std::min<long long>((n + 255) / 256, 4 * 148));
  const bool aligned = d % 8 == 0 && n / 8 < (1LL << 31) &&
                       reinterpret_cast<uintptr_t>(e) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(w) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(ew) % 16 == 0;
  if (wgt_dtype == MOE_BF16 && aligned) {
    const int nvec = static_cast<int>(n / 8);
    const int g8 = std::min((nvec + 255) / 256, 8 * 148);
    fold_bf16_x8_kernel<<<g8, 256, 0, stream>>>(static_cast<const uint4*>(e),
                                                reinterpret_cast<const float4*>(w), d / 8, nvec,
                                                static_cast<uint4*>(ew));
  } else if (wgt_dtype == MOE_BF16) {
    fold_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(e), w, d, n,
                                               static_cast<__nv_bfloat16*>(ew));
  } else {
    fold_f32_kernel<<<grid, 256, 0, stream>>>(static_cast<const float*>(e), w, d, n,
                                              static_cast<float*>(ew));
  }
  return launch_status();
}

moe_status_t launch_rmsnorm(int act_dtype, const void* x, const float* w, float eps, int T, int d,
                            void* xn, float* inv_rms, cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  TraceScope tr(stream, "rmsnorm");
  if (act_dtype == MOE_BF16) {
    rmsnorm_bf16_kernel<<<T, kNormThreads, 0, stream>>>(
        static_cast<const uint4*>(x), reinterpret_cast<const float4*>(w), eps, d,
        static_cast<uint4*>(xn), inv_rms);
  } else {
    rmsnorm_f32_kernel<<<T, kNormThreads, 0, stream>>>(static_cast<const float*>(x), w, eps, d,
                                                       static_cast<float*>(xn), inv_rms);
  }
  return launch_status();
}

}  // namespace moe
