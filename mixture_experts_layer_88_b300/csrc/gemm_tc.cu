// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMA +
// TMEM) for the expert FFNs and the router of a DeepSeekMoE layer.
//
// Weights sit in the MMA's M slot and tokens in its N slot ("swap-AB"):
//   D[w, t] = sum_k A[w, k] * B[t, k],   A = weight rows, B = token rows,
// so a ragged expert group costs at most 15 padded token columns instead of a
// partly empty 128-row tile, and small decode batches still use M = 128.
//
// One tile = one group g, one weight-row block m and one token block (<= 256
// tokens).  Each tile runs two accumulators that share the token operand:
//   GATEUP: acc0 = gate rows [m, m+128) of W13_g, acc1 = the matching up rows
//           (offset I); epilogue writes act = SiLU(acc0) * acc1   (SwiGLU)
//   DOWN:   acc0 / acc1 = rows [m, m+128) / [m+128, m+256) of W2_g; epilogue
//           writes the expert output y (bf16)
//   ROUTER: acc0 / acc1 = centroids [m, m+128) / [m+128, m+256); epilogue
//           writes fp32 partial logits of one K split
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: A0, A1 (128x64 each) and the token rows (at most
//               five boxes of 256/128/64/32/16 rows) of one 64-wide K block per
//               pipeline stage
//   warp 1      TMEM owner and MMA issuer (one thread issues tcgen05.mma
//               M=128, N=tokens, K=16, twice per K step)
//   warps 2..5  epilogue: tcgen05.ld from TMEM (warp w reads lanes 32*(w%4)..)
//
// Every barrier wait is bounded: after `timeout_ns` without progress the CTA
// raises an abort flag, lets the TMA loads it issued land, waits for its own
// MMAs, frees TMEM, sets the device error word and returns.
#include <cudaTypedefs.h>
#include <stdio.h>

#include "common.cuh"
#include "gemm_tc.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int BM = 128;              // weight rows per accumulator (MMA M)
constexpr int BN_MAX = 256;          // tokens per tile (MMA N, <= 256)
constexpr int BK = 64;               // K elements per stage = one 128-byte row
constexpr int STAGES = 3;
constexpr uint32_t A_BOX_BYTES = BM * BK * 2;             // 16 KB
constexpr uint32_t B_ROW_BYTES = BK * 2;                  // 128 B per token row
constexpr uint32_t STAGE_BYTES = 2 * A_BOX_BYTES + BN_MAX * BK * 2;  // 64 KB
constexpr uint32_t TMEM_COLS = 512;  // acc0 at column 0, acc1 at column 256
constexpr int NUM_THREADS = 192;
constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

struct Tile {
  int g, mb, tok0, ntok, nmma, kb0, kb1, split;
};

__device__ __forceinline__ int total_tiles(const GemmArgs& a, int mode) {
  if (mode == GM_ROUTER) return a.router_nb * a.m_blocks * a.k_splits;
  return a.gt.bstart[a.G] * a.m_blocks;
}

__device__ __forceinline__ void decode_tile(const GemmArgs& a, int mode, int tile, Tile& t) {
  if (mode == GM_ROUTER) {
    const int per_split = a.router_nb * a.m_blocks;
    t.split = tile / per_split;
    const int rem = tile - t.split * per_split;
    t.mb = rem / a.router_nb;
    const int nb = rem - t.mb * a.router_nb;
    t.g = 0;
    t.tok0 = nb * a.router_bs;
    t.ntok = min(a.router_bs, a.router_T - t.tok0);
    t.kb0 = t.split * a.k_per_split;
    t.kb1 = min(a.k_blocks, t.kb0 + a.k_per_split);
  } else {
    // largest g with bstart[g] * m_blocks <= tile (groups with no blocks are skipped)
    int lo = 0, hi = a.G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(a.gt.bstart + mid) * a.m_blocks <= tile) lo = mid; else hi = mid - 1;
    }
    t.g = lo;
    const int b0 = __ldg(a.gt.bstart + lo);
    const int nbk = __ldg(a.gt.bstart + lo + 1) - b0;
    const int local = tile - b0 * a.m_blocks;
    t.mb = local / nbk;
    const int nb = local - t.mb * nbk;
    const int bs = __ldg(a.gt.bs + lo);
    t.tok0 = nb * bs;
    t.ntok = min(bs, __ldg(a.gt.rows + lo) - t.tok0);
    t.split = 0;
    t.kb0 = 0;
    t.kb1 = a.k_blocks;
  }
  t.nmma = (t.ntok + 15) & ~15;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) {
    if (!tc::mbar_try_wait(bar, parity)) {
      const uint64_t deadline = tc::globaltimer_ns() + timeout_ns;
      ok = tc::mbar_wait_bounded(bar, parity, abort_flag, deadline) ? 1 : 0;
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    tc::mbar_init(tfull, 1);
    tc::mbar_init(tempty, 128);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane < 2 + 2 * kTokBoxes) {
    const CUtensorMap* m = lane < 2 ? &maps.a[lane] : &maps.b[(lane - 2) / kTokBoxes][(lane - 2) % kTokBoxes];
    tc::tma_prefetch_desc(m);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = total_tiles(args, MODE);
  const unsigned long long tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    int issued_phase[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued_phase[s] = -1;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      Tile t;
      decode_tile(args, MODE, tile, t);
      const bool second = (MODE != GM_ROUTER) && (t.g >= args.E);
      const CUtensorMap* mA = &maps.a[second ? 1 : 0];
      const CUtensorMap* mB = maps.b[second ? 1 : 0];
      const int gl = second ? t.g - args.E : t.g;
      int a_row0, b_row;
      if (MODE == GM_ROUTER) {
        a_row0 = t.mb * 2 * BM;
        b_row = t.tok0;
      } else {
        a_row0 = gl * args.a_rows_per_group + t.mb * (MODE == GM_GATEUP ? BM : 2 * BM);
        b_row = __ldg(args.gt.brow + t.g) + t.tok0;
      }
      const int a_row1 = a_row0 + args.a1_off;
      const uint32_t bytes = 2 * A_BOX_BYTES + t.nmma * B_ROW_BYTES;
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        if (!warp_wait(empty + stage, phase ^ 1u, abort_flag, tmo)) { ok = false; break; }
        if (lane == 0) {
          uint8_t* sa = smem + stage * STAGE_BYTES;
          tc::mbar_arrive_expect_tx(full + stage, bytes);
          tc::tma_load_2d(sa, mA, full + stage, kb * BK, a_row0);
          tc::tma_load_2d(sa + A_BOX_BYTES, mA, full + stage, kb * BK, a_row1);
          // token rows: one box per set bit of nmma / 16, largest first
          int done = 0;
#pragma unroll
          for (int bi = kTokBoxes - 1; bi >= 0; --bi) {
            const int h = 16 << bi;
            if (t.nmma & h) {
              tc::tma_load_2d(sa + 2 * A_BOX_BYTES + done * B_ROW_BYTES, mB + bi, full + stage,
                              kb * BK, b_row + done);
              done += h;
            }
          }
        }
        issued_phase[stage] = static_cast<int>(phase);
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      // abort: let every load this warp issued land before the CTA exits
      for (int s = 0; s < STAGES; ++s)
        if (issued_phase[s] >= 0)
          warp_wait(full + s, static_cast<uint32_t>(issued_phase[s]), abort_flag, tmo);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0, tphase = 0;
    bool ok = true, issued_any = false;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      Tile t;
      decode_tile(args, MODE, tile, t);
      if (!warp_wait(tempty, tphase ^ 1u, abort_flag, tmo)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(BM, t.nmma);
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        if (!warp_wait(full + stage, phase, abort_flag, tmo)) { ok = false; break; }
        tc::tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = tc::smem_u32(smem + stage * STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t da0 = tc::smem_desc_sw128(sa + kk * 32);
            const uint64_t da1 = tc::smem_desc_sw128(sa + A_BOX_BYTES + kk * 32);
            const uint64_t db = tc::smem_desc_sw128(sa + 2 * A_BOX_BYTES + kk * 32);
            const uint32_t acc = (kb > t.kb0 || kk > 0) ? 1u : 0u;
            tc::mma_bf16(tmem_base, da0, db, idesc, acc);
            tc::mma_bf16(tmem_base + 256, da1, db, idesc, acc);
          }
          tc::mma_commit(empty + stage);   // frees the smem stage when these MMAs finish
        }
        issued_any = true;
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) tc::mma_commit(tfull);  // accumulators complete
      __syncwarp();
      tphase ^= 1u;
    }
    if (!ok && issued_any) {
      if (lane == 0) tc::mma_commit(drain);
      __syncwarp();
      warp_wait(drain, 0, abort_flag, tmo);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;       // accumulator row = weight row in the box
    uint32_t tphase = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      Tile t;
      decode_tile(args, MODE, tile, t);
      if (!warp_wait(tfull, tphase, abort_flag, tmo)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      int out_row0, col0;
      if (MODE == GM_ROUTER) {
        out_row0 = t.tok0;
        col0 = t.mb * 2 * BM + row;
      } else {
        out_row0 = __ldg(args.gt.orow + t.g) + t.tok0;
        col0 = t.mb * (MODE == GM_GATEUP ? BM : 2 * BM) + row;
      }
      for (int j0 = 0; j0 < t.nmma; j0 += 16) {
        uint32_t r0[16], r1[16];
        tc::tmem_ld16(taddr + j0, r0);
        tc::tmem_ld16(taddr + 256 + j0, r1);
        tc::tmem_wait_ld(r0, r1);
        const int jn = min(16, t.ntok - j0);
        if (MODE == GM_GATEUP) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
          for (int j = 0; j < jn; ++j) {
            const float v = silu_mul(__uint_as_float(r0[j]), __uint_as_float(r1[j]));
            out[static_cast<size_t>(out_row0 + j0 + j) * args.out_ld + col0] =
                __float2bfloat16_rn(v);
          }
        } else if (MODE == GM_DOWN) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
          const bool c0ok = col0 < args.out_cols, c1ok = col0 + BM < args.out_cols;
          for (int j = 0; j < jn; ++j) {
            __nv_bfloat16* o = out + static_cast<size_t>(out_row0 + j0 + j) * args.out_ld;
            if (c0ok) o[col0] = __float2bfloat16_rn(__uint_as_float(r0[j]));
            if (c1ok) o[col0 + BM] = __float2bfloat16_rn(__uint_as_float(r1[j]));
          }
        } else {
          float* out = static_cast<float*>(args.out) + t.split * args.out_split_stride;
          const bool c0ok = col0 < args.out_cols, c1ok = col0 + BM < args.out_cols;
          for (int j = 0; j < jn; ++j) {
            float* o = out + static_cast<size_t>(out_row0 + j0 + j) * args.out_ld;
            if (c0ok) o[col0] = __uint_as_float(r0[j]);
            if (c1ok) o[col0 + BM] = __uint_as_float(r1[j]);
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(tempty);
      tphase ^= 1u;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) atomicOr(args.status, ERRBIT_TIMEOUT);
}

// ---------------------------------------------------------------- group table

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  // 1024-thread block scan; returns the exclusive prefix of v
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
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
    warp_sums[lane] = s;  // inclusive prefix of warp sums
  }
  __syncthreads();
  const int before = (w > 0 ? warp_sums[w - 1] : 0) + x - v;
  if (total) *total = warp_sums[(blockDim.x >> 5) - 1];
  return before;
}

__global__ void __launch_bounds__(1024) build_groups_kernel(const int* offsets, int T, int K,
                                                            int E, int S, int* rows,
                                                            int* brow_gu, int* orow, int* bs,
                                                            int* bstart) {
  __shared__ int warp_sums[32];
  const int G = E + S;
  // each thread owns two consecutive groups (G <= kMaxE + kMaxS <= 2048)
  int nb_pair[2];
  int local = 0;
  for (int u = 0; u < 2; ++u) {
    const int g = threadIdx.x * 2 + u;
    int nb = 0;
    if (g < G) {
      int r, br, orw;
      if (g < E) {
        br = offsets[g];
        r = offsets[g + 1] - br;
        orw = br;
      } else {
        r = T;
        br = 0;
        orw = T * K + (g - E) * T;
      }
      int b;
      token_blocks(r, &b, &nb);
      rows[g] = r;
      brow_gu[g] = br;
      orow[g] = orw;
      bs[g] = b;
    }
    nb_pair[u] = nb;
    local += nb;
  }
  int total = 0;
  const int before = block_exclusive_scan(local, warp_sums, &total);
  const int g0 = threadIdx.x * 2;
  if (g0 < G) bstart[g0] = before;
  if (g0 + 1 < G) bstart[g0 + 1] = before + nb_pair[0];
  if (threadIdx.x == 0) bstart[G] = total;
}

template <int MODE>
moe_status_t launch_mode(const GemmMaps& maps, const GemmArgs& args, int grid,
                         cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set[dev] = true;
  }
  static const char* names[3] = {"gemm_gateup_swiglu", "gemm_down", "gemm_router"};
  TraceScope tr(stream, names[MODE]);
  gemm_tc_kernel<MODE><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps, args);
  return launch_status();
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc || !base || rows == 0 || cols == 0) return false;
  const cuuint64_t gdim[2] = {cols, rows};
  const cuuint64_t gstride[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim,
                   gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_gemm_maps(GemmMaps* m, const void* a0, uint64_t a0_rows, const void* a1,
                    uint64_t a1_rows, const void* b0, uint64_t b0_rows, const void* b1,
                    uint64_t b1_rows, uint64_t k) {
  if (!make_tmap_bf16(&m->a[0], a0, a0_rows, k, BM)) return false;
  if (a1) {
    if (!make_tmap_bf16(&m->a[1], a1, a1_rows, k, BM)) return false;
  } else {
    m->a[1] = m->a[0];
  }
  for (int i = 0; i < kTokBoxes; ++i) {
    if (!make_tmap_bf16(&m->b[0][i], b0, b0_rows, k, 16u << i)) return false;
    if (b1) {
      if (!make_tmap_bf16(&m->b[1][i], b1, b1_rows, k, 16u << i)) return false;
    } else {
      m->b[1][i] = m->b[0][i];
    }
  }
  return true;
}

moe_status_t launch_gemm_tc(int mode, const GemmMaps& maps, const GemmArgs& args, int grid,
                            cudaStream_t stream) {
  if (grid <= 0) return MOE_OK;
  switch (mode) {
    case GM_GATEUP: return launch_mode<GM_GATEUP>(maps, args, grid, stream);
    case GM_DOWN: return launch_mode<GM_DOWN>(maps, args, grid, stream);
    case GM_ROUTER: return launch_mode<GM_ROUTER>(maps, args, grid, stream);
    default: return MOE_ERR_INVALID_ARG;
  }
}

moe_status_t launch_build_groups(const int* offsets, int T, int K, int E, int S, int* rows,
                                 int* brow_gu, int* orow, int* bs, int* bstart,
                                 cudaStream_t stream) {
  TraceScope tr(stream, "build_groups");
  build_groups_kernel<<<1, 1024, 0, stream>>>(offsets, T, K, E, S, rows, brow_gu, orow, bs,
                                              bstart);
  return launch_status();
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

}  // namespace moe
