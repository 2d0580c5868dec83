// Training pieces of a DeepSeekMoE layer on the CUDA cores: the SwiGLU of the
// training forward, and every backward step that is not a tensor-core GEMM.
//
// The backward is the chain rule through the forward of "DeepSeekMoE架构解析"
// (V3 walk-through): section 3.1 (output = u + shared + sum_k g_k FFN_k(u)),
// eq. (13) (renormalised gates), eq. (15) (Sigmoid affinity; the 2024 layer's
// Softmax, course chapter "MoE", section 4).  The chosen experts are constants
// and the balancing bias gets no gradient (section 2.2: it only steers the
// choice).  With dL/d(out) = dout:
//   dgates[t,k] = dout_t . y_{t,k}              dy_{t,k} = g_{t,k} dout_t
//   shared rows: dy = dout_t                    residual: dx_t += dout_t
//   ds_k = (dg_k - sum_j dg_j g_j) / sum_j s_j  (renormalised; else ds = dg)
//   Sigmoid: dlogit = ds s (1 - s);  Softmax: dlogit_i = s_i (ds_i - sum ds s)
//   dx_t += sum_i dlogit_i e_i,   de_i = sum_t dlogit_{t,i} u_t
//   SwiGLU: dgate = da * up * SiLU'(gate), dup = da * SiLU(gate)
//
// Row layout of the backward ("padded rows"): the output gradients of the
// rows of routed expert e start at poff[e], a multiple of 16, in the forward's
// order (expert rows by ascending token), and the rows up to the next multiple
// of 16 are zero; shared expert s takes rows poff[E] + s * T16 .. (T16 =
// round_up(T, 16)), token order, zero past T.  The weight-gradient GEMMs run
// their K loop over whole 16-token slices of these rows.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

// routed expert of padded row p < poff[E]: the largest e with poff[e] <= p
__device__ __forceinline__ int padded_group(const int32_t* poff, int E, int p) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(poff + mid) <= p) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Source of padded row p: the packed forward row (routed: offsets[e] + j;
// shared: T*K + s*T + j) and the token, or -1 for a zero row.
struct RowSrc {
  int packed, token, e;   // e = -1 for shared rows
};
__device__ __forceinline__ RowSrc padded_row_source(long long p, const int32_t* poff,
                                                    const int32_t* counts,
                                                    const int32_t* offsets,
                                                    const int32_t* perm, int T, int K, int E,
                                                    int T16) {
  RowSrc r{-1, -1, -1};
  const int P = __ldg(poff + E);
  if (p < P) {
    const int e = padded_group(poff, E, static_cast<int>(p));
    const int j = static_cast<int>(p) - __ldg(poff + e);
    if (j < __ldg(counts + e)) {
      r.packed = __ldg(offsets + e) + j;
      r.token = perm ? __ldg(perm + r.packed) : -1;
      r.e = e;
    }
  } else {
    const long long q = p - P;
    const int s = static_cast<int>(q / T16);
    const int j = static_cast<int>(q - static_cast<long long>(s) * T16);
    if (j < T) {
      r.packed = T * K + s * T + j;
      r.token = j;
    }
  }
  return r;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 o;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return o;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float sigmoidf(float z) { return 1.0f / (1.0f + expf(-z)); }

// ---------------------------------------------------------------- training forward

// act = SiLU(gate) * up from the stored pre-activations h = [gate | up].
// Rows are taken block by block (no per-element division); SiLU(g) * u uses
// the fast exponential and division, as the inference epilogue does.
__global__ void __launch_bounds__(256) swiglu_fwd_kernel(const uint4* __restrict__ h,
                                                         uint4* __restrict__ act, long long rows,
                                                         int vI) {
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* hr = h + r * 2 * vI;
    uint4* ar = act + r * vI;
    for (int v = threadIdx.x; v < vI; v += blockDim.x) {
      float g[8], u[8], a[8];
      unpack8(__ldg(hr + v), g);
      unpack8(__ldg(hr + vI + v), u);
#pragma unroll
      for (int j = 0; j < 8; ++j) a[j] = __fdividef(g[j] * u[j], 1.0f + __expf(-g[j]));
      ar[v] = pack8(a);
    }
  }
}

// ---------------------------------------------------------------- combine backward

// One block per padded row: dy = g * dout (routed), dout (shared) or 0 (pad),
// and for routed rows dgates[t,k] = dout_t . y_row (fp32, fixed order).
__global__ void __launch_bounds__(128) combine_bwd_kernel(
    const uint4* __restrict__ dout, const uint4* __restrict__ y, const float* __restrict__ gates,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ perm,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ poff, int T, int K, int E, int S, int T16, int vpr,
    uint4* __restrict__ dy, float* __restrict__ dgates) {
  __shared__ int s_tok, s_row, s_slot;
  __shared__ float s_g;
  __shared__ float s_part[4];
  const long long p = blockIdx.x;
  if (p >= __ldg(poff + E) + static_cast<long long>(S) * T16) return;
  if (threadIdx.x == 0) {
    const RowSrc r = padded_row_source(p, poff, counts, offsets, perm, T, K, E, T16);
    int slot = -1;
    float g = 1.f;
    if (r.e >= 0) {
      for (int k = 0; k < K; ++k)
        if (__ldg(idx + static_cast<size_t>(r.token) * K + k) == r.e) slot = r.token * K + k;
      g = __ldg(gates + slot);
    }
    s_tok = r.token;
    s_row = r.e >= 0 ? r.packed : -1;
    s_slot = slot;
    s_g = g;
  }
  __syncthreads();
  const int tok = s_tok, row = s_row;
  const float g = s_g;
  uint4* dst = dy + p * vpr;
  if (tok < 0) {
    for (int v = threadIdx.x; v < vpr; v += blockDim.x) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* src = dout + static_cast<size_t>(tok) * vpr;
  if (row < 0) {
    for (int v = threadIdx.x; v < vpr; v += blockDim.x) dst[v] = __ldg(src + v);
    return;
  }
  const uint4* yr = y + static_cast<size_t>(row) * vpr;
  float dot = 0.f;
  for (int v = threadIdx.x; v < vpr; v += blockDim.x) {
    float a[8], b[8], o[8];
    unpack8(__ldg(src + v), a);
    unpack8(__ldg(yr + v), b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      dot = fmaf(a[j], b[j], dot);
      o[j] = g * a[j];
    }
    dst[v] = pack8(o);
  }
  dot = warp_sum(dot);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = dot;
  __syncthreads();
  if (threadIdx.x == 0) dgates[s_slot] = (s_part[0] + s_part[1]) + (s_part[2] + s_part[3]);
}

// ---------------------------------------------------------------- router backward

// One warp per token.  Sigmoid: dlogit of the K chosen experts (dlk [T,K]
// and, at the token's dispatched row, dlrow [T*K]).  Softmax: dense dlogit
// [T, E].
__global__ void __launch_bounds__(256) router_bwd_kernel(
    const float* __restrict__ dgates, const float* __restrict__ gates,
    const int32_t* __restrict__ idx, const float* __restrict__ scores,
    const int32_t* __restrict__ pos, int T, int E, int K, int score_func, int normalize,
    float* __restrict__ dlk, float* __restrict__ dlrow, float* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float dg = 0.f, g = 0.f, s = 0.f;
  int e = -1;
  if (lane < K) {
    const size_t i = static_cast<size_t>(t) * K + lane;
    dg = __ldg(dgates + i);
    g = __ldg(gates + i);
    e = __ldg(idx + i);
    s = __ldg(scores + static_cast<size_t>(t) * E + e);
  }
  float ds = dg;
  if (normalize) {
    const float tot = warp_sum(s);
    const float inner = warp_sum(dg * g);
    ds = tot > 0.f ? (dg - inner) / tot : 0.f;
  }
  if (score_func == MOE_SCORE_SIGMOID) {
    if (lane < K) {
      const float v = ds * s * (1.f - s);
      const size_t i = static_cast<size_t>(t) * K + lane;
      dlk[i] = v;
      dlrow[__ldg(pos + i)] = v;
    }
    return;
  }
  const float c = warp_sum(lane < K ? ds * s : 0.f);
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int ee = e0 + lane;
    float dse = 0.f;
    for (int k = 0; k < K; ++k) {
      const int ek = __shfl_sync(0xffffffffu, e, k);
      const float dk = __shfl_sync(0xffffffffu, ds, k);
      if (ek == ee) dse = dk;
    }
    if (ee < E) {
      const size_t i = static_cast<size_t>(t) * E + ee;
      dl[i] = __ldg(scores + i) * (dse - c);
    }
  }
}

// dxr[t, :] = sum_e dl[t, e] C[e, :] (Softmax), 8 tokens x 1024 columns per block.
__global__ void __launch_bounds__(128) router_dx_dense_kernel(const float* __restrict__ dl,
                                                              const uint4* __restrict__ cent,
                                                              int T, int E, int vpr,
                                                              float* __restrict__ dxr) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= vpr) return;
  for (int t0 = blockIdx.y * 8; t0 < T; t0 += gridDim.y * 8) {
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  const int nt = min(8, T - t0);
  for (int e = 0; e < E; ++e) {
    float c[8];
    unpack8(__ldg(cent + static_cast<size_t>(e) * vpr + v), c);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = i < nt ? __ldg(dl + static_cast<size_t>(t0 + i) * E + e) : 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(w, c[j], acc[i][j]);
    }
  }
  for (int i = 0; i < nt; ++i) {
    float4* o = reinterpret_cast<float4*>(dxr + static_cast<size_t>(t0 + i) * vpr * 8) + 2 * v;
    o[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    o[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
  }
}

// ---------------------------------------------------------------- SwiGLU backward

// One block per padded row: dh = [dact * up * SiLU'(gate), dact * SiLU(gate)]
// from the stored pre-activations of the row's packed forward row; zero rows
// stay zero.
__global__ void __launch_bounds__(128) swiglu_bwd_kernel(
    const uint4* __restrict__ dact, const uint4* __restrict__ h,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ poff, int T, int K, int E, int S, int T16, int vI,
    uint4* __restrict__ dh) {
  __shared__ int s_row;
  const long long p = blockIdx.x;
  if (p >= __ldg(poff + E) + static_cast<long long>(S) * T16) return;
  if (threadIdx.x == 0)
    s_row = padded_row_source(p, poff, counts, offsets, nullptr, T, K, E, T16).packed;
  __syncthreads();
  const int r = s_row;
  uint4* dst = dh + p * 2 * vI;
  if (r < 0) {
    for (int v = threadIdx.x; v < 2 * vI; v += blockDim.x) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* hr = h + static_cast<size_t>(r) * 2 * vI;
  for (int v = threadIdx.x; v < vI; v += blockDim.x) {
    float g[8], u[8], da[8], dgt[8], dup[8];
    unpack8(__ldg(hr + v), g);
    unpack8(__ldg(hr + vI + v), u);
    unpack8(__ldg(dact + p * vI + v), da);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float sg = sigmoidf(g[j]);
      dgt[j] = da[j] * u[j] * sg * (1.f + g[j] * (1.f - sg));
      dup[j] = da[j] * g[j] * sg;
    }
    dst[v] = pack8(dgt);
    dst[vI + v] = pack8(dup);
  }
}

// ---------------------------------------------------------------- dx

// dx_t = sum_k dxp[padded row of (t,k)] + sum_s dxp[shared row] + router term
// (+ dout_t), fp32 in that order.  One thread per 8 channels of a token.
__global__ void __launch_bounds__(128) dx_kernel(
    const uint4* __restrict__ dxp, const int32_t* __restrict__ pos,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ poff, const float* __restrict__ dlk,
    const uint4* __restrict__ cent, const float* __restrict__ dxr,
    const uint4* __restrict__ dout, uint4* __restrict__ dx, int T, int K, int E, int S, int T16,
    int vpr, int add_residual) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= vpr) return;
  const long long P = __ldg(poff + E);
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    float acc[8], f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int k = 0; k < K; ++k) {
      const size_t i = static_cast<size_t>(t) * K + k;
      const int e = __ldg(idx + i);
      const long long pp = __ldg(poff + e) + (__ldg(pos + i) - __ldg(offsets + e));
      unpack8(__ldg(dxp + pp * vpr + v), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += f[j];
    }
    for (int s = 0; s < S; ++s) {
      unpack8(__ldg(dxp + (P + static_cast<long long>(s) * T16 + t) * vpr + v), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += f[j];
    }
    if (dlk) {
      for (int k = 0; k < K; ++k) {
        const size_t i = static_cast<size_t>(t) * K + k;
        const float w = __ldg(dlk + i);
        unpack8(__ldg(cent + static_cast<size_t>(__ldg(idx + i)) * vpr + v), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, f[j], acc[j]);
      }
    }
    if (dxr) {
      const float4* r = reinterpret_cast<const float4*>(dxr + static_cast<size_t>(t) * vpr * 8) + 2 * v;
      const float4 a = __ldg(r), b = __ldg(r + 1);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    if (add_residual) {
      unpack8(__ldg(dout + static_cast<size_t>(t) * vpr + v), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += f[j];
    }
    dx[static_cast<size_t>(t) * vpr + v] = pack8(acc);
  }
}

// ---------------------------------------------------------------- centroid gradients

// Sigmoid: partial[q] = sum over the rows r of chunk q of dlrow[r] xp[r], where
// chunk q = b * kDcentSub + s holds rows [64 s, 64 s + 64) of token block b
// (the input-gradient GEMMs' routed blocks, <= 256 rows of one expert; the
// last chunk takes any rows past 64 kDcentSub).  Chunks without rows write
// zeros.
constexpr int kDcentChunkRows = 64;
__global__ void __launch_bounds__(128) dcent_sparse_partial_kernel(
    const float* __restrict__ dlrow, const uint4* __restrict__ xp,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ bs, const int32_t* __restrict__ bstart, int E, int vpr,
    float* __restrict__ part) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= vpr) return;
  const int nq = __ldg(bstart + E) * kDcentSub;
  for (int q = blockIdx.y; q < nq; q += gridDim.y) {
    const int b = q / kDcentSub, s = q - b * kDcentSub;
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(bstart + mid) <= b) lo = mid; else hi = mid - 1;
    }
    const int lb = b - __ldg(bstart + lo);
    const int sz = __ldg(bs + lo);
    const int nrows = min(sz, __ldg(counts + lo) - lb * sz);   // rows of block b
    const int s0 = s * kDcentChunkRows;
    const int n = s == kDcentSub - 1 ? nrows - s0 : min(kDcentChunkRows, nrows - s0);
    const int r0 = __ldg(offsets + lo) + lb * sz + s0;
    float acc[8], f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int i = 0; i < n; ++i) {
      const float w = __ldg(dlrow + r0 + i);
      unpack8(__ldg(xp + static_cast<size_t>(r0 + i) * vpr + v), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, f[j], acc[j]);
    }
    float4* o = reinterpret_cast<float4*>(part + static_cast<size_t>(q) * vpr * 8) + 2 * v;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// dC[e] = sum of the partials of expert e's chunks, in block and chunk order.
__global__ void __launch_bounds__(128) dcent_sparse_reduce_kernel(const float* __restrict__ part,
                                                                  const int32_t* __restrict__ bstart,
                                                                  int d, float* __restrict__ dc) {
  const int e = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  float acc = 0.f;
  for (int q = __ldg(bstart + e) * kDcentSub; q < __ldg(bstart + e + 1) * kDcentSub; ++q)
    acc += __ldg(part + static_cast<size_t>(q) * d + c);
  dc[static_cast<size_t>(e) * d + c] = acc;
}

// Softmax: partial[tc, e] = sum over the 256 tokens of chunk tc of dl[t, e] x_t,
// 8 experts x 8 channels per thread.
__global__ void __launch_bounds__(128) dcent_dense_partial_kernel(const float* __restrict__ dl,
                                                                  const uint4* __restrict__ x,
                                                                  int T, int E, int vpr,
                                                                  float* __restrict__ part) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  const int e0 = blockIdx.y * 8;
  const int tc = blockIdx.z;
  if (v >= vpr) return;
  float acc[8][8], f[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  const int ne = min(8, E - e0);
  const int t1 = min(T, (tc + 1) * 256);
  for (int t = tc * 256; t < t1; ++t) {
    unpack8(__ldg(x + static_cast<size_t>(t) * vpr + v), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = i < ne ? __ldg(dl + static_cast<size_t>(t) * E + e0 + i) : 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(w, f[j], acc[i][j]);
    }
  }
  for (int i = 0; i < ne; ++i) {
    float4* o = reinterpret_cast<float4*>(
                    part + (static_cast<size_t>(tc) * E + e0 + i) * vpr * 8) + 2 * v;
    o[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    o[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
}

__global__ void __launch_bounds__(128) dcent_dense_reduce_kernel(const float* __restrict__ part,
                                                                 int nchunks, int E, int d,
                                                                 float* __restrict__ dc) {
  const int e = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  float acc = 0.f;
  for (int tc = 0; tc < nchunks; ++tc) acc += __ldg(part + (static_cast<size_t>(tc) * E + e) * d + c);
  dc[static_cast<size_t>(e) * d + c] = acc;
}

int grid_y(int n) { return n < 65535 ? n : 65535; }

}  // namespace

moe_status_t launch_swiglu_fwd(const void* h, void* act, long long rows, int I,
                               cudaStream_t stream) {
  if (rows <= 0) return MOE_OK;
  TraceScope tr(stream, "swiglu_fwd");
  const int grid = static_cast<int>(rows < 148LL * 8 ? rows : 148LL * 8);
  swiglu_fwd_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(h),
                                              static_cast<uint4*>(act), rows, I / 8);
  return launch_status();
}

moe_status_t launch_combine_bwd(const void* dout, const void* y, const float* gates,
                                const int32_t* idx, const int32_t* perm, const int32_t* counts,
                                const int32_t* offsets, const int32_t* poff, int T, int K, int E,
                                int S, int d, long long rows_max, void* dy, float* dgates,
                                cudaStream_t stream) {
  TraceScope tr(stream, "combine_bwd");
  combine_bwd_kernel<<<static_cast<unsigned>(rows_max), 128, 0, stream>>>(
      static_cast<const uint4*>(dout), static_cast<const uint4*>(y), gates, idx, perm, counts,
      offsets, poff, T, K, E, S, round_up(T, 16), d / 8, static_cast<uint4*>(dy), dgates);
  return launch_status();
}

moe_status_t launch_router_bwd(const float* dgates, const float* gates, const int32_t* idx,
                               const float* scores, const int32_t* pos, int T, int E, int K,
                               int score_func, int normalize, float* dlk, float* dlrow,
                               float* dl, cudaStream_t stream) {
  TraceScope tr(stream, "router_bwd");
  router_bwd_kernel<<<ceil_div(T, 8), 256, 0, stream>>>(dgates, gates, idx, scores, pos, T, E, K,
                                                        score_func, normalize, dlk, dlrow, dl);
  return launch_status();
}

moe_status_t launch_router_dx_dense(const float* dl, const void* cent, int T, int E, int d,
                                    float* dxr, cudaStream_t stream) {
  TraceScope tr(stream, "router_dx_dense");
  const dim3 grid(ceil_div(d / 8, 128), grid_y(ceil_div(T, 8)));
  router_dx_dense_kernel<<<grid, 128, 0, stream>>>(dl, static_cast<const uint4*>(cent), T, E,
                                                   d / 8, dxr);
  return launch_status();
}

moe_status_t launch_swiglu_bwd(const void* dact, const void* h, const int32_t* counts,
                               const int32_t* offsets, const int32_t* poff, int T, int K, int E,
                               int S, int I, long long rows_max, void* dh, cudaStream_t stream) {
  TraceScope tr(stream, "swiglu_bwd");
  swiglu_bwd_kernel<<<static_cast<unsigned>(rows_max), 128, 0, stream>>>(
      static_cast<const uint4*>(dact), static_cast<const uint4*>(h), counts, offsets, poff, T, K,
      E, S, round_up(T, 16), I / 8, static_cast<uint4*>(dh));
  return launch_status();
}

moe_status_t launch_dx(const void* dxp, const int32_t* pos, const int32_t* idx,
                       const int32_t* offsets, const int32_t* poff, const float* dlk,
                       const void* cent, const float* dxr, const void* dout, void* dx, int T,
                       int K, int E, int S, int d, int add_residual, cudaStream_t stream) {
  TraceScope tr(stream, "dx_gather");
  const dim3 grid(ceil_div(d / 8, 128), grid_y(T));
  dx_kernel<<<grid, 128, 0, stream>>>(static_cast<const uint4*>(dxp), pos, idx, offsets, poff, dlk,
                                      static_cast<const uint4*>(cent), dxr,
                                      static_cast<const uint4*>(dout), static_cast<uint4*>(dx), T,
                                      K, E, S, round_up(T, 16), d / 8, add_residual);
  return launch_status();
}

moe_status_t launch_dcent_sparse(const float* dlrow, const void* xp, const int32_t* counts,
                                 const int32_t* offsets, const int32_t* bs,
                                 const int32_t* bstart, int E, int d, int max_blocks,
                                 float* part, float* dc, cudaStream_t stream) {
  {
    TraceScope tr(stream, "dcent_partial");
    const dim3 grid(ceil_div(d / 8, 128), grid_y(max_blocks * kDcentSub));
    dcent_sparse_partial_kernel<<<grid, 128, 0, stream>>>(dlrow, static_cast<const uint4*>(xp),
                                                          counts, offsets, bs, bstart, E, d / 8,
                                                          part);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  }
  TraceScope tr(stream, "dcent_reduce");
  dcent_sparse_reduce_kernel<<<dim3(ceil_div(d, 128), E), 128, 0, stream>>>(part, bstart, d, dc);
  return launch_status();
}

moe_status_t launch_dcent_dense(const float* dl, const void* x, int T, int E, int d, float* part,
                                float* dc, cudaStream_t stream) {
  const int nchunks = ceil_div(T, 256);
  {
    TraceScope tr(stream, "dcent_partial");
    const dim3 grid(ceil_div(d / 8, 128), ceil_div(E, 8), nchunks);
    dcent_dense_partial_kernel<<<grid, 128, 0, stream>>>(dl, static_cast<const uint4*>(x), T, E,
                                                         d / 8, part);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  }
  TraceScope tr(stream, "dcent_reduce");
  dcent_dense_reduce_kernel<<<dim3(ceil_div(d, 128), E), 128, 0, stream>>>(part, nchunks, E, d,
                                                                           dc);
  return launch_status();
}

}  // namespace moe
