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
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int WARPS = kDispatchChunk / 32;

// Expert ids outside [0, E) are skipped and flagged in the device error word.
__device__ __forceinline__ void build_masks(const int32_t* __restrict__ idx, int T, int K, int E,
                                            uint32_t* mask, unsigned* status) {
  for (int i = threadIdx.x; i < WARPS * E; i += blockDim.x) mask[i] = 0u;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kDispatchChunk + warp * 32 + lane;
  if (t < T) {
    for (int k = 0; k < K; ++k) {
      const int e = __ldg(idx + static_cast<size_t>(t) * K + k);
      if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
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

__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ hist, int nchunks,
                                                    int E, int32_t* __restrict__ counts,
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
  // exclusive scan of counts over experts
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = running;
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
  const int before = (w > 0 ? warp_sums[w - 1] : 0) + x - running;
  if (e < E) {
    counts[e] = running;
    offsets[e] = before;
    if (e == E - 1) offsets[E] = before + running;
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
  for (int k = 0; k < K; ++k) {
    const int e = __ldg(idx + static_cast<size_t>(t) * K + k);
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
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
    for (int v = threadIdx.x; v < vpr; v += blockDim.x) {
      const V val = __ldg(src + v);
      for (int k = 0; k < K; ++k)
        if (dst[tl][k] >= 0) xp[static_cast<size_t>(dst[tl][k]) * vpr + v] = val;
    }
  }
}

}  // namespace

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
    scan_kernel<<<1, 1024, 0, stream>>>(hist, nchunks, E, counts, offsets);
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
