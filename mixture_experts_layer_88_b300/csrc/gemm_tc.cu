// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMA +
// TMEM) for the expert FFNs and the router of a DeepSeekMoE layer.
//
// Weights sit in the MMA's M slot and tokens in its N slot ("swap-AB"):
//   D[w, t] = sum_k A[w, k] * B[t, k],   A = weight rows, B = token rows,
// so a ragged expert group costs at most 15 padded token columns instead of a
// partly empty 128-row tile, and small decode batches still use M = 128.
//
// The expert GEMMs run on CTA pairs (clusters of two, tcgen05 cta_group::2):
// one MMA of M = 256 weight rows spans both CTAs, each CTA holding 128 rows of
// A and of the accumulator and half of the token rows of B.  Per CTA that is
// 48 KB of operands per 64-wide K step instead of 64 KB for the same FLOPs,
// which is what bounds this GEMM: the bytes each SM takes in per FLOP.
// The router runs the single-CTA form (CG = 1) of the same kernel.
//
// One tile = one group g, one weight-row block and one token block (<= 256
// tokens).  Each tile runs two accumulators that share the token operand:
//   GATEUP: acc0 = gate rows of W13_g, acc1 = the matching up rows (offset I);
//           epilogue writes act = SiLU(acc0) * acc1   (SwiGLU)
//   DOWN:   acc0 / acc1 = two row blocks of W2_g; epilogue writes y (bf16)
//   ROUTER: acc0 / acc1 = centroids [m, m+128) / [m+128, m+256); epilogue
//           writes fp32 partial logits of one K split
// CTA r of a pair owns accumulator rows [r*128, r*128+128) of each M = 256
// block, so each CTA's epilogue is independent.
//
// Warp roles (192 threads per CTA):
//   warp 0      TMA producer: its CTA's two 128x64 weight boxes and its half
//               of the token rows (at most five boxes) per pipeline stage; both
//               CTAs' bytes are counted on the even CTA's "full" barrier
//   warp 1      TMEM owner; in the even CTA also the MMA issuer (one thread
//               issues tcgen05.mma K=16, twice per K step, and commits to
//               both CTAs' barriers)
//   warps 2..5  epilogue: tcgen05.ld from this CTA's TMEM (warp w reads lanes
//               32*(w%4)..), then one arrival per warp on the even CTA's
//               "tmem empty" barrier
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

constexpr int BM = 128;              // weight rows per accumulator per CTA (MMA M / CG)
constexpr int BN_MAX = 256;          // tokens per tile (MMA N, <= 256)
constexpr int BK = 64;               // K elements per stage = one 128-byte row
constexpr uint32_t A_BOX_BYTES = BM * BK * 2;             // 16 KB
constexpr uint32_t B_ROW_BYTES = BK * 2;                  // 128 B per token row
constexpr uint32_t TMEM_COLS = 512;  // acc0 at column 0, acc1 at column 256
constexpr int NUM_THREADS = 192;

template <int CG> struct Cfg {
  static constexpr int STAGES = CG == 1 ? 3 : 4;
  // two weight boxes + this CTA's share of the token rows
  static constexpr uint32_t STAGE_BYTES = 2 * A_BOX_BYTES + (BN_MAX / CG) * BK * 2;
  static constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int TOK_BOX0 = 16 / CG;   // smallest token box height
};

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

// First weight row of the tile's M block (both CTAs of a pair; CTA r then
// adds r * 128).  GATEUP blocks are CG*128 gate rows; DOWN and ROUTER blocks
// are 2*CG*128 rows (acc1 = the second half).
template <int CG>
__device__ __forceinline__ int m_block_rows(int mode) {
  return mode == GM_GATEUP ? CG * BM : 2 * CG * BM;
}

// Bounded wait by lane 0, result broadcast to the warp.  CLUSTER: the
// barrier's arrivals come from threads of the peer CTA (acquire at cluster scope).
template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) {
    if (!(CLUSTER ? tc::mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity))) {
      const uint64_t deadline = tc::globaltimer_ns() + timeout_ns;
      ok = tc::mbar_wait_bounded<CLUSTER>(bar, parity, abort_flag, deadline) ? 1 : 0;
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

template <int MODE, int CG>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  constexpr int STAGES = Cfg<CG>::STAGES;
  constexpr uint32_t STAGE_BYTES = Cfg<CG>::STAGE_BYTES;
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
  const uint32_t rank = CG == 2 ? tc::cluster_ctarank() : 0u;
  const int cluster = blockIdx.x / CG, nclusters = gridDim.x / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full + s, 1);     // the even CTA expects both CTAs' bytes
      tc::mbar_init(empty + s, 1);
    }
    tc::mbar_init(tfull, 1);
    tc::mbar_init(tempty, CG * 4);    // every epilogue warp of the pair
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane < 2 + 2 * kTokBoxes) {
    const CUtensorMap* m = lane < 2 ? &maps.a[lane] : &maps.b[(lane - 2) / kTokBoxes][(lane - 2) % kTokBoxes];
    tc::tma_prefetch_desc(m);
  }
  if (warp == 1) {
    tc::tmem_alloc<CG>(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish<CG>();
  }
  tc::tc_fence_before();
  if constexpr (CG == 2) tc::cluster_sync_all(); else __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = total_tiles(args, MODE);
  const unsigned long long tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_par = 0;   // per stage: a load is in flight / its parity
    bool ok = true;
    for (int tile = cluster; tile < ntiles && ok; tile += nclusters) {
      Tile t;
      decode_tile(args, MODE, tile, t);
      const bool second = (MODE != GM_ROUTER) && (t.g >= args.E);
      const CUtensorMap* mA = &maps.a[second ? 1 : 0];
      const CUtensorMap* mB = maps.b[second ? 1 : 0];
      const int gl = second ? t.g - args.E : t.g;
      const int half = t.nmma / CG;                // token rows this CTA loads
      int a_row0, b_row;
      if (MODE == GM_ROUTER) {
        a_row0 = t.mb * 2 * BM;
        b_row = t.tok0;
      } else {
        a_row0 = gl * args.a_rows_per_group + t.mb * m_block_rows<CG>(MODE) + rank * BM;
        b_row = __ldg(args.gt.brow + t.g) + t.tok0 + rank * half;
      }
      const int a_row1 = a_row0 + args.a1_off;
      const uint32_t bytes = 2 * A_BOX_BYTES + half * B_ROW_BYTES;
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        if (!warp_wait(empty + stage, phase ^ 1u, abort_flag, tmo)) { ok = false; break; }
        if (lane == 0) {
          uint8_t* sa = smem + stage * STAGE_BYTES;
          if constexpr (CG == 1) {
            tc::mbar_arrive_expect_tx(full + stage, bytes);
            tc::tma_load_2d(sa, mA, full + stage, kb * BK, a_row0);
            tc::tma_load_2d(sa + A_BOX_BYTES, mA, full + stage, kb * BK, a_row1);
          } else {
            // Only the even CTA arrives, expecting the bytes of both CTAs; the
            // odd CTA's loads just count their bytes on the even CTA's barrier.
            // (The odd CTA reuses stage s only after the MMAs that consumed it
            // completed, so its bytes always land in the phase they belong to.)
            const uint32_t fb = tc::mapa_shared(tc::smem_u32(full + stage), 0);
            if (rank == 0) tc::mbar_arrive_expect_tx(full + stage, CG * bytes);
            tc::tma_load_2d_pair(sa, mA, fb, kb * BK, a_row0);
            tc::tma_load_2d_pair(sa + A_BOX_BYTES, mA, fb, kb * BK, a_row1);
          }
          // token rows: one box per set bit of half / TOK_BOX0, largest first
          int done = 0;
#pragma unroll
          for (int bi = kTokBoxes - 1; bi >= 0; --bi) {
            const int h = Cfg<CG>::TOK_BOX0 << bi;
            if (half & h) {
              uint8_t* dst = sa + 2 * A_BOX_BYTES + done * B_ROW_BYTES;
              if constexpr (CG == 1)
                tc::tma_load_2d(dst, mB + bi, full + stage, kb * BK, b_row + done);
              else
                tc::tma_load_2d_pair(dst, mB + bi, tc::mapa_shared(tc::smem_u32(full + stage), 0),
                                     kb * BK, b_row + done);
              done += h;
            }
          }
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && (CG == 1 || rank == 0)) {
      // abort: let every load counted on this CTA's barriers land before exit
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s))
          warp_wait(full + s, (issued_par >> s) & 1u, abort_flag, tmo);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (CG == 1 || rank == 0) {
      int stage = 0;
      uint32_t phase = 0, tphase = 0;
      bool ok = true, issued_any = false;
      for (int tile = cluster; tile < ntiles && ok; tile += nclusters) {
        Tile t;
        decode_tile(args, MODE, tile, t);
        if (!warp_wait<CG == 2>(tempty, tphase ^ 1u, abort_flag, tmo)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t idesc = tc::idesc_bf16_f32(BM * CG, t.nmma);
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
              tc::mma_bf16<CG>(tmem_base, da0, db, idesc, acc);
              tc::mma_bf16<CG>(tmem_base + 256, da1, db, idesc, acc);
            }
            tc::mma_commit<CG>(empty + stage);   // frees the stage in both CTAs
          }
          issued_any = true;
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) tc::mma_commit<CG>(tfull);  // accumulators complete, both CTAs
        __syncwarp();
        tphase ^= 1u;
      }
      if (!ok && issued_any) {
        if (lane == 0) tc::mma_commit<CG>(drain, 0x1);
        __syncwarp();
        warp_wait(drain, 0, abort_flag, tmo);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;       // accumulator row = weight row in the box
    const uint32_t tempty_addr =
        CG == 2 ? tc::mapa_shared(tc::smem_u32(tempty), 0) : tc::smem_u32(tempty);
    uint32_t tphase = 0;
    for (int tile = cluster; tile < ntiles; tile += nclusters) {
      Tile t;
      decode_tile(args, MODE, tile, t);
      if (!warp_wait(tfull, tphase, abort_flag, tmo)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      int out_row0, col0, col1;
      if (MODE == GM_ROUTER) {
        out_row0 = t.tok0;
        col0 = t.mb * 2 * BM + row;
        col1 = col0 + BM;
      } else {
        out_row0 = __ldg(args.gt.orow + t.g) + t.tok0;
        col0 = t.mb * m_block_rows<CG>(MODE) + static_cast<int>(rank) * BM + row;
        col1 = col0 + CG * BM;   // DOWN: acc1 rows
      }
      const bool c0ok = col0 < args.out_cols, c1ok = col1 < args.out_cols;
      for (int j0 = 0; j0 < t.nmma; j0 += 16) {
        uint32_t r0[16], r1[16];
        tc::tmem_ld16(taddr + j0, r0);
        tc::tmem_ld16(taddr + 256 + j0, r1);
        tc::tmem_wait_ld(r0, r1);
        const int jn = min(16, t.ntok - j0);
        // fully unrolled with a predicate, so r0/r1 stay in registers
        if (MODE == GM_GATEUP) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out) +
                               static_cast<size_t>(out_row0 + j0) * args.out_ld + col0;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0ok && j < jn)
              out[static_cast<size_t>(j) * args.out_ld] = __float2bfloat16_rn(
                  silu_mul(__uint_as_float(r0[j]), __uint_as_float(r1[j])));
        } else if (MODE == GM_DOWN) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out) +
                               static_cast<size_t>(out_row0 + j0) * args.out_ld;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j < jn) {
              __nv_bfloat16* o = out + static_cast<size_t>(j) * args.out_ld;
              if (c0ok) o[col0] = __float2bfloat16_rn(__uint_as_float(r0[j]));
              if (c1ok) o[col1] = __float2bfloat16_rn(__uint_as_float(r1[j]));
            }
          }
        } else {
          float* out = static_cast<float*>(args.out) + t.split * args.out_split_stride +
                       static_cast<size_t>(out_row0 + j0) * args.out_ld;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j < jn) {
              float* o = out + static_cast<size_t>(j) * args.out_ld;
              if (c0ok) o[col0] = __uint_as_float(r0[j]);
              if (c1ok) o[col1] = __uint_as_float(r1[j]);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) tc::mbar_arrive_cluster(tempty_addr); else tc::mbar_arrive(tempty);
      }
      tphase ^= 1u;
    }
  }

  tc::tc_fence_before();
  if constexpr (CG == 2) tc::cluster_sync_all(); else __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<CG>(tmem_base, TMEM_COLS);
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

template <int MODE, int CG>
moe_status_t launch_mode(const GemmMaps& maps, const GemmArgs& args, int grid,
                         cudaStream_t stream) {
  constexpr size_t smem = Cfg<CG>::SMEM_BYTES;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<MODE, CG>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set[dev] = true;
  }
  static const char* names[3] = {"gemm_gateup_swiglu", "gemm_down", "gemm_router"};
  TraceScope tr(stream, names[MODE]);
  cudaLaunchConfig_t lc = {};
  lc.blockDim = dim3(NUM_THREADS, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  // persistent: no more clusters than can be resident at once
  static int max_clusters[64] = {0};
  if (dev < 64 && max_clusters[dev] == 0) {
    lc.gridDim = dim3(static_cast<unsigned>(num_sms() / CG * CG), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<MODE, CG>, &lc) != cudaSuccess ||
        n <= 0)
      return MOE_ERR_CUDA;
    max_clusters[dev] = n;
  }
  int clusters = grid / CG;
  if (dev < 64 && clusters > max_clusters[dev]) clusters = max_clusters[dev];
  if (clusters < 1) clusters = 1;
  lc.gridDim = dim3(static_cast<unsigned>(clusters * CG), 1, 1);
  if (cudaLaunchKernelEx(&lc, gemm_tc_kernel<MODE, CG>, maps, args) != cudaSuccess)
    return MOE_ERR_CUDA;
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
                    uint64_t b1_rows, uint64_t k, uint32_t tok_box0) {
  if (!make_tmap_bf16(&m->a[0], a0, a0_rows, k, BM)) return false;
  if (a1) {
    if (!make_tmap_bf16(&m->a[1], a1, a1_rows, k, BM)) return false;
  } else {
    m->a[1] = m->a[0];
  }
  for (int i = 0; i < kTokBoxes; ++i) {
    if (!make_tmap_bf16(&m->b[0][i], b0, b0_rows, k, tok_box0 << i)) return false;
    if (b1) {
      if (!make_tmap_bf16(&m->b[1][i], b1, b1_rows, k, tok_box0 << i)) return false;
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
    case GM_GATEUP: return launch_mode<GM_GATEUP, 2>(maps, args, grid, stream);
    case GM_DOWN: return launch_mode<GM_DOWN, 2>(maps, args, grid, stream);
    case GM_ROUTER: return launch_mode<GM_ROUTER, 1>(maps, args, grid, stream);
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
