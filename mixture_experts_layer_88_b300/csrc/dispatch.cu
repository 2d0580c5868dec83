// No-drop dispatch of a DeepSeekMoE layer (course chapter "MoE", section 6:
// every token reaches all K_r chosen experts, nothing is dropped by capacity).
//
// Deterministic, atomic-free on positions:
//   count   one CTA per 256 tokens; warp w of the CTA owns 32 tokens (one per
//           lane) and marks, per expert, which of its lanes chose it in a
//           32-bit shared-memory mask; the CTA's per-expert totals go to hist
//   scan    per expert, an exclusive scan of hist over CTAs (base of each
//           CTA's rows), the load counts c_i and offsets = exclusive scan of c
//   rank    row of (t, k) = offsets[e] + CTA base + earlier warps' lanes +
//           popc(own mask below this lane): tokens of one expert land in
//           ascending token order; writes pos and perm_tok
//   scatter each token row is read once (16-byte vectors) and written to its
//           K destination rows of xp
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int WARPS = kDispatchChunk / 32;

// True when expert id e is invalid for entry k of a token's idx row: outside
// [0, E), or equal to an earlier entry of the same row (a token reaches each
// chosen expert once).  Such entries get no row and raise the bounds bit.
__device__ __forceinline__ bool bad_entry(const int32_t* __restrict__ row, int k, int e, int E) {
  if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) return true;
  for (int j = 0; j < k; ++j)
    if (__ldg(row + j) == e) return true;
  return false;
}

// Expert ids outside [0, E) and repeats within a token are skipped and
// flagged in the device error word.
__device__ __forceinline__ void build_masks(const int32_t* __restrict__ idx, int T, int K, int E,
                                            uint32_t* mask, unsigned* status) {
  for (int i = threadIdx.x; i < WARPS * E; i += blockDim.x) mask[i] = 0u;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kDispatchChunk + warp * 32 + lane;
  if (t < T) {
    const int32_t* row = idx + static_cast<size_t>(t) * K;
    for (int k = 0; k < K; ++k) {
      const int e = __ldg(row + k);
      if (bad_entry(row, k, e, E)) {
        atomicOr(status, ERRBIT_BOUNDS);
        continue;
      }
      atomicOr(mask + warp * E + e, 1u << lane);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDispatchChunk) count_kernel(const int32_t* __restrict__ idx,
                                                               int T, int K, int E,
                                                               int32_t* __restrict__ hist,
                                                               unsigned* status) {
  extern __shared__ uint32_t mask[];
  build_masks(idx, T, K, E, mask, status);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) c += __popc(mask[w * E + e]);
    hist[static_cast<size_t>(blockIdx.x) * E + e] = c;
  }
}

// offsets = exclusive prefix over experts of counts rounded up to `pad` rows
// (pad = 1: dense; pad = 4: every expert's rows start 16-byte aligned for the
// fp32 scale runs of the FP8 path)
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ hist, int nchunks,
                                                    int E, int pad, int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets) {
  __shared__ int warp_sums[32];
  const int e = threadIdx.x;
  int running = 0;
  if (e < E) {
    int c = 0;
    // batches of independent loads, then the dependent prefix
    for (; c + 8 <= nchunks; c += 8) {
      int h[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) h[u] = hist[static_cast<size_t>(c + u) * E + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        hist[static_cast<size_t>(c + u) * E + e] = running;
        running += h[u];
      }
    }
    for (; c < nchunks; ++c) {
      const int h = hist[static_cast<size_t>(c) * E + e];
      hist[static_cast<size_t>(c) * E + e] = running;
      running += h;
    }
  }
  // exclusive scan of the (padded) counts over experts
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int span = (running + pad - 1) / pad * pad;
  int x = span;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int before = (w > 0 ? warp_sums[w - 1] : 0) + x - span;
  if (e < E) {
    counts[e] = running;
    offsets[e] = before;
    if (e == E - 1) offsets[E] = before + span;
  }
}

__global__ void __launch_bounds__(kDispatchChunk) rank_kernel(
    const int32_t* __restrict__ idx, int T, int K, int E, const int32_t* __restrict__ hist_base,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ pos,
    int32_t* __restrict__ perm_tok, unsigned* status) {
  extern __shared__ uint32_t mask[];
  build_masks(idx, T, K, E, mask, status);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kDispatchChunk + warp * 32 + lane;
  if (t >= T) return;
  const uint32_t below = (1u << lane) - 1u;
  const int32_t* row = idx + static_cast<size_t>(t) * K;
  for (int k = 0; k < K; ++k) {
    const int e = __ldg(row + k);
    if (bad_entry(row, k, e, E)) {
      pos[static_cast<size_t>(t) * K + k] = -1;
      continue;
    }
    int r = __ldg(offsets + e) + __ldg(hist_base + static_cast<size_t>(blockIdx.x) * E + e);
    for (int w = 0; w < warp; ++w) r += __popc(mask[w * E + e]);
    r += __popc(mask[warp * E + e] & below);
    pos[static_cast<size_t>(t) * K + k] = r;
    perm_tok[r] = t;
  }
}

template <typename V>
__global__ void __launch_bounds__(256) scatter_kernel(const V* __restrict__ x, int T, int K,
                                                      int vpr, const int32_t* __restrict__ pos,
                                                      V* __restrict__ xp, int tok_per_cta) {
  __shared__ int dst[8][kMaxK];
  const int t0 = blockIdx.x * tok_per_cta;
  for (int i = threadIdx.x; i < tok_per_cta * K; i += blockDim.x) {
    const int tl = i / K, k = i % K;
    if (t0 + tl < T) dst[tl][k] = __ldg(pos + static_cast<size_t>(t0 + tl) * K + k);
  }
  __syncthreads();
  for (int tl = 0; tl < tok_per_cta; ++tl) {
    const int t = t0 + tl;
    if (t >= T) break;
    const V* src = x + static_cast<size_t>(t) * vpr;
    // up to four of the row's vectors in flight per thread before the stores
    constexpr int kIn = 4;
    V val[kIn];
#pragma unroll
    for (int j = 0; j < kIn; ++j) {
      const int v = threadIdx.x + j * blockDim.x;
      if (v < vpr) val[j] = __ldg(src + v);
    }
#pragma unroll
    for (int j = 0; j < kIn; ++j) {
      const int v = threadIdx.x + j * blockDim.x;
      if (v < vpr)
        for (int k = 0; k < K; ++k)
          if (dst[tl][k] >= 0) xp[static_cast<size_t>(dst[tl][k]) * vpr + v] = val[j];
    }
    for (int v = threadIdx.x + kIn * blockDim.x; v < vpr; v += blockDim.x) {
      const V vv = __ldg(src + v);
      for (int k = 0; k < K; ++k)
        if (dst[tl][k] >= 0) xp[static_cast<size_t>(dst[tl][k]) * vpr + v] = vv;
    }
  }
}

// 8 bf16 of x scaled by inv and the per-channel weights w0 (4) and w1 (4), in
// fp32 as (x * inv) * w, rounded once to bf16 (the RMSNorm kernel's rounding).
__device__ __forceinline__ uint4 norm_bf16x8(const uint4& v, float inv, const float4& w0,
                                             const float4& w1) {
  const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint4 o;
  __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    oh[k] = __floats2bfloat162_rn((f.x * inv) * wv[2 * k], (f.y * inv) * wv[2 * k + 1]);
  }
  return o;
}

// Dispatch behind the RMSNorm: each token row is read once, normalised with
// its inv_rms and the norm weights, and written to its K rows of xp and to its
// shared-expert row of xs (when xs is not null).
__global__ void __launch_bounds__(256) scatter_norm_kernel(
    const uint4* __restrict__ x, const float* __restrict__ inv_rms,
    const float4* __restrict__ w, int T, int K, int vpr, const int32_t* __restrict__ pos,
    uint4* __restrict__ xp, uint4* __restrict__ xs, int tok_per_cta) {
  __shared__ int dst[8][kMaxK];
  const int t0 = blockIdx.x * tok_per_cta;
  for (int i = threadIdx.x; i < tok_per_cta * K; i += blockDim.x) {
    const int tl = i / K, k = i % K;
    if (t0 + tl < T) dst[tl][k] = __ldg(pos + static_cast<size_t>(t0 + tl) * K + k);
  }
  __syncthreads();
  for (int tl = 0; tl < tok_per_cta; ++tl) {
    const int t = t0 + tl;
    if (t >= T) break;
    const float inv = __ldg(inv_rms + t);
    const uint4* src = x + static_cast<size_t>(t) * vpr;
    for (int v = threadIdx.x; v < vpr; v += blockDim.x) {
      const uint4 val = norm_bf16x8(__ldg(src + v), inv, __ldg(w + 2 * v), __ldg(w + 2 * v + 1));
      for (int k = 0; k < K; ++k)
        if (dst[tl][k] >= 0) xp[static_cast<size_t>(dst[tl][k]) * vpr + v] = val;
      if (xs) xs[static_cast<size_t>(t) * vpr + v] = val;
    }
  }
}

// FP8 dispatch: each token row is read once (bf16), cut into 1 x 128 tiles
// (V3 walk-through, section 4.3), each tile scaled by 448 / max|x| and
// rounded to e4m3, and written to the token's K expert rows and to its
// shared-expert row.  Scales (max|x| / 448) go K-block-major:
// xs[kb * ld_s + row].  Sixteen threads hold one tile (8 values each).
// NORM: the row is first normalised as in scatter_norm_kernel (bf16 values
// of the normalised row are what gets quantised).
template <bool NORM>
__global__ void __launch_bounds__(256) scatter_quant_kernel(
    const uint4* __restrict__ x, int T, int K, int d, const int32_t* __restrict__ pos,
    int shared_row, uint2* __restrict__ xq, float* __restrict__ xs, long long ld_s,
    const float* __restrict__ inv_rms, const float4* __restrict__ w) {
  const int t = blockIdx.x;
  if (t >= T) return;
  __shared__ int dst[kMaxK + 1];
  for (int k = threadIdx.x; k < K; k += blockDim.x) dst[k] = __ldg(pos + static_cast<size_t>(t) * K + k);
  if (threadIdx.x == 0) dst[K] = shared_row >= 0 ? shared_row + t : -1;
  __syncthreads();
  const int vpr = d / 8;                        // 8-element vectors per row
  for (int base = 0; base < vpr; base += blockDim.x) {
    const int v = base + threadIdx.x;
    const bool in = v < vpr;                    // a 16-lane group is all in or all out
    float f[8];
    if (in) {
      uint4 raw = __ldg(x + static_cast<size_t>(t) * vpr + v);
      if constexpr (NORM)
        raw = norm_bf16x8(raw, __ldg(inv_rms + t), __ldg(w + 2 * v), __ldg(w + 2 * v + 1));
      const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 ff = __bfloat1622float2(hb[i]);
        f[2 * i] = ff.x;
        f[2 * i + 1] = ff.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.f;
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!in) continue;
    const float inv = m > 0.f ? 448.0f / m : 0.f;
    uint2 q;
    uint16_t* qh = reinterpret_cast<uint16_t*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      qh[i] = __nv_cvt_float2_to_fp8x2(make_float2(f[2 * i] * inv, f[2 * i + 1] * inv),
                                       __NV_SATFINITE, __NV_E4M3);
    const int kb = v >> 4;
    for (int k = 0; k <= K; ++k) {
      const int r = dst[k];
      if (r < 0) continue;
      xq[static_cast<size_t>(r) * vpr + v] = q;
      if ((threadIdx.x & 15) == 0) xs[kb * ld_s + r] = m / 448.0f;
    }
  }
}

}  // namespace

moe_status_t launch_scatter_quant(const void* x, int T, int K, int d, const int32_t* pos,
                                  int shared_row, void* xq, float* xs, long long ld_s,
                                  cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  TraceScope tr(stream, "dispatch_scatter_fp8");
  scatter_quant_kernel<false><<<T, 256, 0, stream>>>(static_cast<const uint4*>(x), T, K, d, pos,
                                                     shared_row, static_cast<uint2*>(xq), xs,
                                                     ld_s, nullptr, nullptr);
  return launch_status();
}

moe_status_t launch_scatter_quant_norm(const void* x, const float* inv_rms, const float* w, int T,
                                       int K, int d, const int32_t* pos, int shared_row, void* xq,
                                       float* xs, long long ld_s, cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  TraceScope tr(stream, "dispatch_scatter_fp8_norm");
  scatter_quant_kernel<true><<<T, 256, 0, stream>>>(
      static_cast<const uint4*>(x), T, K, d, pos, shared_row, static_cast<uint2*>(xq), xs, ld_s,
      inv_rms, reinterpret_cast<const float4*>(w));
  return launch_status();
}

moe_status_t launch_scatter_norm(const void* x, const float* inv_rms, const float* w, int T,
                                 int K, int d, const int32_t* pos, void* xp, void* xs,
                                 cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  TraceScope tr(stream, "dispatch_scatter_norm");
  const int tpc = 4;
  scatter_norm_kernel<<<ceil_div(T, tpc), 256, 0, stream>>>(
      static_cast<const uint4*>(x), inv_rms, reinterpret_cast<const float4*>(w), T, K, d / 8,
      pos, static_cast<uint4*>(xp), static_cast<uint4*>(xs), tpc);
  return launch_status();
}

moe_status_t launch_dispatch_index(const int32_t* idx, int T, int K, int E, int pad,
                                   int32_t* counts, int32_t* offsets, int32_t* perm_tok,
                                   int32_t* pos, int32_t* hist, cudaStream_t stream) {
  if (T <= 0) {
    TraceScope tr(stream, "dispatch_empty");
    cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream);
    cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), stream);
    return launch_status();
  }
  const int nchunks = ceil_div(T, kDispatchChunk);
  const size_t mask_bytes = sizeof(uint32_t) * WARPS * E;
  {
    TraceScope tr(stream, "dispatch_count");
    count_kernel<<<nchunks, kDispatchChunk, mask_bytes, stream>>>(idx, T, K, E, hist,
                                                                  device_status_word());
  }
  {
    TraceScope tr(stream, "dispatch_scan");
    scan_kernel<<<1, 1024, 0, stream>>>(hist, nchunks, E, pad, counts, offsets);
  }
  {
    TraceScope tr(stream, "dispatch_rank");
    rank_kernel<<<nchunks, kDispatchChunk, mask_bytes, stream>>>(idx, T, K, E, hist, offsets,
                                                                 pos, perm_tok,
                                                                 device_status_word());
  }
  return launch_status();
}

moe_status_t launch_dispatch(const void* x, size_t row_bytes, const int32_t* idx, int T, int K,
                             int E, int32_t* counts, int32_t* offsets, void* xp,
                             int32_t* perm_tok, int32_t* pos, int32_t* hist,
                             cudaStream_t stream) {
  if (T <= 0) {
    TraceScope tr(stream, "dispatch_empty");
    cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream);
    cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), stream);
    return launch_status();
  }
  const int nchunks = ceil_div(T, kDispatchChunk);
  const size_t mask_bytes = sizeof(uint32_t) * WARPS * E;
  {
    TraceScope tr(stream, "dispatch_count");
    count_kernel<<<nchunks, kDispatchChunk, mask_bytes, stream>>>(idx, T, K, E, hist,
                                                                  device_status_word());
  }
  {
    TraceScope tr(stream, "dispatch_scan");
    scan_kernel<<<1, 1024, 0, stream>>>(hist, nchunks, E, 1, counts, offsets);
  }
  {
    TraceScope tr(stream, "dispatch_rank");
    rank_kernel<<<nchunks, kDispatchChunk, mask_bytes, stream>>>(idx, T, K, E, hist, offsets,
                                                                 pos, perm_tok,
                                                                 device_status_word());
  }
  {
    TraceScope tr(stream, "dispatch_scatter");
    const int tpc = 4;
    const int grid = ceil_div(T, tpc);
    if (row_bytes % 16 == 0) {
      scatter_kernel<uint4><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(x), T, K,
                                                      static_cast<int>(row_bytes / 16), pos,
                                                      static_cast<uint4*>(xp), tpc);
    } else {
      scatter_kernel<uint32_t><<<grid, 256, 0, stream>>>(static_cast<const uint32_t*>(x), T, K,
                                                         static_cast<int>(row_bytes / 4), pos,
                                                         static_cast<uint32_t*>(xp), tpc);
    }
  }
  return launch_status();
}

}  // namespace moe
