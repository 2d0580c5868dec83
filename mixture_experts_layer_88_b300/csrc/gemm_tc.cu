// Persistent grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMA +
// TMEM) for the expert FFNs and the router of a DeepSeekMoE layer.
//
// Weights sit in the MMA's M slot and tokens in its N slot ("swap-AB"):
//   D[w, t] = sum_k A[w, k] * B[t, k],   A = weight rows, B = token rows,
// so a ragged expert group costs at most 15 padded token columns instead of a
// partly empty 128-row tile, and small decode batches still use M = 128.
//
// Expert GEMMs (expert_gemm_kernel) run on CTA pairs: clusters of two CTAs and
// tcgen05 cta_group::2, so one MMA of M = 256 weight rows spans both CTAs;
// each CTA holds 128 rows of A and of the accumulator and half of the tile's
// token rows of B.  One tile = one group g, one weight-row block and one
// token block of N <= 256 tokens; each CTA runs two accumulators of 128 lanes
// x N fp32 columns (all 512 TMEM columns) that share the token operand:
//   GATEUP: a pair covers 256 intermediate columns c0..c0+255.  CTA r: acc0 =
//           gate rows c0+128r .. +127, acc1 = the matching up rows (offset I);
//           the epilogue writes act = SiLU(acc0) * acc1   (SwiGLU)
//   DOWN:   a pair covers 512 rows m..m+511 of W2.  CTA r: acc0 = rows
//           m+128r .., acc1 = rows m+256+128r ..; the epilogue writes y (bf16)
// Per CTA that is 48 KB of operands per 64-wide K step for 8.4 MFLOP.  The
// two accumulators fill TMEM, so a tile's MMAs wait for the previous tile's
// epilogue; eight epilogue warps keep that drain short.
//
// Training adds two modes of the same kernel: GATEUP_H writes the gate/up
// pre-activations h = [gate | up] (bf16) instead of act, and DGRAD computes
// input gradients (da = dy W2, du = dh W13) with the DOWN tiling and the
// weight operand read MN-major (the weight matrix of a group is [K, M] in
// memory: TMA boxes of 64 K-rows x 64 M-columns, the transpose bit of the
// instruction descriptor).  The weight gradients (dW = A^T B over a group's
// tokens) run in wgrad_gemm_kernel, described at its definition.
//
// The router GEMM (router_gemm_kernel) runs one CTA per tile: two 128-row
// centroid boxes, one token block, one K split; fp32 partial logits out.
//
// Warp roles of the expert kernel (320 threads per CTA):
//   warp 0      TMA producer: per 64-wide K step, this CTA's two 128-row weight
//               boxes and its half of the token rows (at most five boxes); both
//               CTAs' bytes are counted on the even CTA's "full" barrier
//   warp 1      TMEM owner; in the even CTA also the MMA issuer (one thread
//               issues tcgen05.mma M=256 N=tokens K=16 twice per K step and
//               commits to both CTAs)
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4).. of its CTA, the
//               two warps of a lane quadrant take alternate 16-token chunks;
//               each chunk is rounded to bf16, written token-major into a
//               shared-memory box (stmatrix.trans) and copied out with
//               16-byte stores; then one arrival per warp on the even CTA's
//               "tmem empty" barrier
//
// The W8 variant (FP8 layers' e4m3 weights, bf16 tokens) adds eight
// dequantisation warps (warps 10..17): they turn each K step of raw e4m3
// weight boxes into bf16 in TMEM, and the MMAs read A from there (see the
// W8_* constants below).
//
// Every barrier wait is bounded: after `timeout_ns` without progress the CTA
// raises an abort flag, lets the TMA loads it issued land, waits for its own
// MMAs, frees TMEM, sets the device error word and returns.
#include <cudaTypedefs.h>
#include <cuda_fp8.h>
#include <stdio.h>

#include "common.cuh"
#include "gemm_tc.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int BK = 64;                        // K elements per stage = one 128-byte row
constexpr uint32_t ROW_BYTES = BK * 2;        // 128 B per operand row per stage
constexpr uint32_t TMEM_COLS = 512;

struct Tile {
  int g, mb, tok0, ntok, nmma, kb0, kb1, split;
};

__device__ __forceinline__ void decode_group_tile(const GemmArgs& a, int tile, Tile& t) {
  // largest g with bstart[g] * m_blocks <= tile (groups with no blocks are skipped)
  int lo = 0, hi = a.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.gt.bstart + mid) * a.m_blocks <= tile) lo = mid; else hi = mid - 1;
  }
  t.g = lo;
  const int b0 = __ldg(a.gt.bstart + lo);
  // Order inside a group.  Routed experts: weight-block-major, so the tiles
  // that share a weight block (its token blocks) are neighbours and stream it
  // from DRAM once, in step.  Shared experts (T tokens, up to 117 MB of token
  // operand): token-block-major, so a token block stays in L2 while all its
  // weight blocks pass over it instead of streaming the whole batch again for
  // every weight block.
  const int local = tile - b0 * a.m_blocks;
  int nb;
  if (lo < a.E) {
    const int nbk = __ldg(a.gt.bstart + lo + 1) - b0;
    t.mb = local / nbk;
    nb = local - t.mb * nbk;
  } else {
    nb = local / a.m_blocks;
    t.mb = local - nb * a.m_blocks;
  }
  const int bs = __ldg(a.gt.bs + lo);
  t.tok0 = nb * bs;
  t.ntok = min(bs, __ldg(a.gt.rows + lo) - t.tok0);
  t.split = 0;
  t.kb0 = 0;
  t.kb1 = a.k_blocks;
  t.nmma = (t.ntok + 15) & ~15;
}

__device__ __forceinline__ void decode_router_tile(const GemmArgs& a, int tile, Tile& t) {
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
  t.nmma = (t.ntok + 15) & ~15;
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

// Bounded wait of a single thread (roles whose loop runs on one thread).
template <bool CLUSTER = false>
__device__ __forceinline__ bool thread_wait(uint64_t* bar, uint32_t parity,
                                            volatile int* abort_flag,
                                            unsigned long long timeout_ns) {
  if (CLUSTER ? tc::mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity))
    return true;
  return tc::mbar_wait_bounded<CLUSTER>(bar, parity, abort_flag,
                                        tc::globaltimer_ns() + timeout_ns);
}

// Drain wait after an abort: lane 0 waits up to timeout_ns whatever the abort
// flag says, so the loads and MMAs this CTA issued complete before TMEM is
// freed and the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity,
                                           unsigned long long timeout_ns) {
  if ((threadIdx.x & 31) == 0)
    tc::mbar_wait_deadline(bar, parity, tc::globaltimer_ns() + timeout_ns);
  __syncwarp();
}

// SiLU(g) * u with the fast reciprocal: g * u / (1 + e^-g).
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g * u, 1.0f + __expf(-g));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Rounds a 16-lane x 16-column TMEM fragment (tcgen05.ld 16x256b.x2 layout)
// to bf16 and stores it token-major at this lane's stmatrix row address.
__device__ __forceinline__ void stage_bf16(uint32_t saddr, const uint32_t (&r)[8]) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
  tc::stmatrix_x4_trans(saddr, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                        pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

// Same for SiLU(gate) * up of two fragments at the same TMEM positions.
__device__ __forceinline__ void stage_swiglu(uint32_t saddr, const uint32_t (&g)[8],
                                             const uint32_t (&u)[8]) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = silu_mul(__uint_as_float(g[i]), __uint_as_float(u[i]));
  tc::stmatrix_x4_trans(saddr, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                        pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

// Token rows of one stage: one TMA box per set bit of rows / box0, largest first.
template <bool PAIR>
__device__ __forceinline__ void load_token_rows(uint8_t* dst, const CUtensorMap* maps,
                                                uint32_t box0, int rows, uint64_t* bar,
                                                uint32_t bar_caddr, int k0, int row0) {
  int done = 0;
#pragma unroll
  for (int bi = kTokBoxes - 1; bi >= 0; --bi) {
    const int h = static_cast<int>(box0) << bi;
    if (rows & h) {
      if constexpr (PAIR)
        tc::tma_load_2d_pair(dst + done * ROW_BYTES, maps + bi, bar_caddr, k0, row0 + done);
      else
        tc::tma_load_2d(dst + done * ROW_BYTES, maps + bi, bar, k0, row0 + done);
      done += h;
    }
  }
}

// ============================================================================
// Expert GEMMs on CTA pairs
// ============================================================================

constexpr int EX_STAGES = 4;
constexpr uint32_t EX_A_BOX_BYTES = 128 * ROW_BYTES;      // 16 KB: one 128-row weight box
constexpr uint32_t EX_B_BYTES = 128 * ROW_BYTES;          // 16 KB: up to 128 token rows
constexpr uint32_t EX_STAGE_BYTES = 2 * EX_A_BOX_BYTES + EX_B_BYTES;
constexpr uint32_t kMnBoxBytes = 64 * ROW_BYTES;           // 8 KB: 64 K rows x 64 columns
constexpr int EX_EPI_WARPS = 8;
constexpr int EX_QUEUE = 4;                               // tile indices in flight

// W8 variant (e4m3 weights with 128x128 fp32 block scales, bf16 tokens): a
// stage holds this CTA's two raw e4m3 weight boxes (64-byte swizzle) and its
// token rows.  Dequantisation warps (one thread per weight row) turn a K
// step of raw weights into bf16 (q * scale, rounded once) and write it to an
// A slot in tensor memory with tcgen05.st; the MMAs read A from TMEM (the
// "TS" form).  Writing A to shared memory instead needs a proxy fence per K
// step, which cost more than the MMAs.  TMEM: acc0 at column 0, acc1 at 192
// (token blocks of at most 192), two A slots of 2 x 32 columns at 384.  Two
// groups of four warps take alternate K steps (slot = step % 2).
constexpr uint32_t W8_RAW_BOX_BYTES = 128 * BK;                          // 8 KB
constexpr uint32_t W8_STAGE_BYTES = 2 * W8_RAW_BOX_BYTES + EX_B_BYTES;   // 32 KB
constexpr int W8_STAGES = 6;
constexpr int W8_A_SLOTS = 2;
constexpr int W8_DQ_GROUP = 4;                             // warps per dequantisation group
constexpr int W8_DQ_WARPS = W8_A_SLOTS * W8_DQ_GROUP;      // one group per A slot
constexpr uint32_t W8_ACC1_COL = 192;
constexpr uint32_t W8_A_COL = 384;                         // slot j: columns 384 + 64 j
constexpr int W8_MAX_BS = 192;
static_assert(W8_STAGES * W8_STAGE_BYTES == EX_STAGES * EX_STAGE_BYTES,
              "the W8 ring fills the bf16 ring's space");
static_assert(W8_A_COL + W8_A_SLOTS * 64 <= TMEM_COLS && 2 * W8_MAX_BS <= W8_A_COL, "TMEM");
// Small batches (decode): token blocks of at most 64 tokens, so a CTA's token
// rows take 4 KB; stages of 36 KB make a five-stage ring, with four stages of
// weights in flight instead of three (the GEMMs only stream weights there).
constexpr uint32_t SB_STAGE_BYTES = 2 * EX_A_BOX_BYTES + 32 * ROW_BYTES;   // 36 KB
constexpr int SB_STAGES = 5;
constexpr int SB_MAX_BS = 64;
static_assert(SB_STAGE_BYTES == 2 * EX_A_BOX_BYTES + (SB_MAX_BS / 2) * ROW_BYTES,
              "a small stage holds half of a token block per CTA");
static_assert(SB_STAGES * SB_STAGE_BYTES <= EX_STAGES * EX_STAGE_BYTES, "ring space");
constexpr int EX_MAX_STAGES = W8_STAGES;

constexpr int ex_threads(bool w8) { return 64 + 32 * (EX_EPI_WARPS + (w8 ? W8_DQ_WARPS : 0)); }
// readers of each published tile index: the MMA warp and the epilogue warps of
// the even CTA, the producer and the epilogue warps of the odd CTA, and (W8)
// the dequantisation warps of both
constexpr int queue_consumers(bool w8) {
  return 2 + 2 * EX_EPI_WARPS + (w8 ? 2 * W8_DQ_WARPS : 0);
}
// Epilogue staging: per warp, two buffers of NOUT output boxes (16 tokens x 32
// columns of bf16: 64-byte rows whose 16-byte pieces are permuted by row pair,
// so that both the stmatrix writes and the row reads are free of bank
// conflicts), 1024-byte aligned, after the operand ring and 1 KB of barriers.
constexpr uint32_t EX_STG_OFF = EX_STAGES * EX_STAGE_BYTES + 1024;
constexpr uint32_t EX_STG_BOX = 16 * 64;
constexpr int ex_nout(int mode) { return mode == GM_GATEUP ? 1 : 2; }
constexpr size_t ex_smem_bytes(int mode) {
  return EX_STG_OFF + EX_EPI_WARPS * 2 * ex_nout(mode) * EX_STG_BOX + 1024;
}
static_assert(ex_smem_bytes(GM_DOWN) <= 227 * 1024, "expert GEMM shared memory");

// Dynamic tile scheduling for a CTA pair.  The even CTA's producer takes the
// next tile from a global counter (atomicAdd) and publishes it in slot
// i % EX_QUEUE of a small queue held in both CTAs' shared memory; every other
// role reads the same sequence from its own CTA's copy.  An index >= ntiles
// ends the sequence.  Waits are bounded like all others.
struct TileQueue {
  uint64_t* qfull;
  uint64_t* qempty;
  volatile int* tq;
  uint32_t rank;
  volatile int* abort_flag;
  unsigned long long tmo;
  int* counter;
  int i = 0;

  // even CTA, producer warp, lane 0: claim a tile (the value is needed only
  // by the publish that follows, so the atomic's latency overlaps the loads
  // issued in between)
  __device__ __forceinline__ int take() const {
    return (threadIdx.x & 31) == 0 ? atomicAdd(counter, 1) : 0;
  }
  // even CTA, producer thread: publish a claimed tile to both CTAs.  Other
  // single-thread roles: read the next published tile and release the slot.
  __device__ __forceinline__ bool publish1(int t, int& tile) {
    const int s = i % EX_QUEUE;
    const uint32_t ph = static_cast<uint32_t>(i / EX_QUEUE) & 1u;
    if (!thread_wait<true>(qempty + s, ph ^ 1u, abort_flag, tmo)) return false;
    tq[s] = t;
    tc::st_shared_cluster_u32(tc::mapa_shared(tc::smem_u32(const_cast<int*>(tq) + s), 1),
                              static_cast<uint32_t>(t));
    tc::mbar_arrive(qfull + s);
    tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(qfull + s), 1));
    tile = t;
    ++i;
    return true;
  }
  __device__ __forceinline__ bool next1(int& tile) {
    const int s = i % EX_QUEUE;
    const uint32_t ph = static_cast<uint32_t>(i / EX_QUEUE) & 1u;
    if (!thread_wait<true>(qfull + s, ph, abort_flag, tmo)) return false;
    tile = tq[s];
    tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(qempty + s), 0));
    ++i;
    return true;
  }
  // any other role: read the next published tile and release the slot
  __device__ __forceinline__ bool next(int& tile) {
    const int s = i % EX_QUEUE;
    const uint32_t ph = static_cast<uint32_t>(i / EX_QUEUE) & 1u;
    if (!warp_wait<true>(qfull + s, ph, abort_flag, tmo)) return false;
    tile = tq[s];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(qempty + s), 0));
    ++i;
    return true;
  }
};

// e4m3 pair -> bf16 pair of q * scale (one rounding)
__device__ __forceinline__ uint32_t dequant2(uint16_t q2, float sc) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(q2, __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  return pack_bf16x2(f.x * sc, f.y * sc);
}

template <int MODE, bool W8, bool SMALL>
__global__ void __launch_bounds__(ex_threads(W8), 1)
    expert_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  static_assert(!(W8 && SMALL), "one ring variant at a time");
  constexpr int NST = W8 ? W8_STAGES : SMALL ? SB_STAGES : EX_STAGES;   // operand ring stages
  constexpr uint32_t STB = W8 ? W8_STAGE_BYTES : SMALL ? SB_STAGE_BYTES : EX_STAGE_BYTES;
  constexpr uint32_t ACC1 = W8 ? W8_ACC1_COL : 256;           // TMEM column of acc1
  // weight rows (or DGRAD: columns) of a tile: 256 gate rows with their up
  // rows (GATEUP, GATEUP_H), or 512 (DOWN, DGRAD)
  constexpr int kBlockW = (MODE == GM_GATEUP || MODE == GM_GATEUP_H) ? 256 : 512;
  static_assert(MODE != GM_ROUTER && (!W8 || MODE == GM_GATEUP || MODE == GM_DOWN), "variant");
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + EX_STAGES * EX_STAGE_BYTES);
  uint64_t* empty = full + EX_MAX_STAGES;
  uint64_t* tfull = empty + EX_MAX_STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* qfull = drain + 1;           // [EX_QUEUE]: tile index published
  uint64_t* qempty = qfull + EX_QUEUE;   // [EX_QUEUE]: read by every consumer
  uint64_t* raw_full = qempty + EX_QUEUE;      // W8 [NST]: this CTA's raw boxes landed
  uint64_t* a_full = raw_full + EX_MAX_STAGES; // W8 [A slots]: dequantised, both CTAs (even)
  uint64_t* a_empty = a_full + W8_A_SLOTS;     // W8 [A slots]: MMAs done with the slot
  volatile int* tq = reinterpret_cast<volatile int*>(a_empty + W8_A_SLOTS);   // [EX_QUEUE]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tq) + EX_QUEUE);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      tc::mbar_init(full + s, 1);     // the even CTA expects both CTAs' bytes
      tc::mbar_init(empty + s, 1);
    }
    tc::mbar_init(tfull, 1);
    tc::mbar_init(tempty, 2 * EX_EPI_WARPS);  // every epilogue warp of the pair
    tc::mbar_init(drain, 1);
    for (int s = 0; s < EX_QUEUE; ++s) {
      tc::mbar_init(qfull + s, 1);
      tc::mbar_init(qempty + s, queue_consumers(W8));
    }
    if (W8) {
      for (int s = 0; s < NST; ++s) tc::mbar_init(raw_full + s, 1);
      for (int j = 0; j < W8_A_SLOTS; ++j) {
        tc::mbar_init(a_full + j, 2 * W8_DQ_GROUP);   // the slot's group, both CTAs
        tc::mbar_init(a_empty + j, 1);
      }
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane < 2 + 2 * kTokBoxes) {
    const CUtensorMap* m =
        lane < 2 ? &maps.a[lane] : &maps.b[(lane - 2) / kTokBoxes][(lane - 2) % kTokBoxes];
    tc::tma_prefetch_desc(m);
  }
  if (warp == 1) {
    tc::tmem_alloc<2>(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish<2>();
  }
  tc::tc_fence_before();
  tc::cluster_sync_all();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = args.gt.bstart[args.G] * args.m_blocks;
  const unsigned long long tmo = args.timeout_ns;

  TileQueue queue{qfull, qempty, tq, rank, abort_flag, tmo, args.tile_counter};
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // One thread runs the loop: no warp-collective step sits between its
    // barrier tests and its TMA instructions.
    if (lane == 0) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_par = 0;   // per stage: a load is in flight / its parity
    bool ok = true;
    int tile = 0;
    ok = rank == 0 ? queue.publish1(queue.take(), tile) : queue.next1(tile);
    while (ok && tile < ntiles) {
      const int claimed = rank == 0 ? queue.take() : 0;   // the tile after this one
      Tile t;
      decode_group_tile(args, tile, t);
      const bool second = t.g >= args.E;
      const CUtensorMap* mA = &maps.a[second ? 1 : 0];
      const CUtensorMap* mB = maps.b[second ? 1 : 0];
      const int gl = second ? t.g - args.E : t.g;
      const int half = t.nmma >> 1;                // token rows this CTA loads
      // GATEUP: gate rows of this CTA and the matching up rows (+I);
      // DOWN: W2 rows of this CTA in the two 256-row halves of the block
      const int a_row0 = gl * args.a_rows_per_group + t.mb * kBlockW + static_cast<int>(rank) * 128;
      const int a_row1 = a_row0 + args.a1_off;
      const int b_row = __ldg(args.gt.brow + t.g) + t.tok0 + static_cast<int>(rank) * half;
      // bytes of this CTA on the even CTA's "full" barrier (W8: token rows only;
      // the raw weight boxes count on this CTA's own raw_full barrier)
      const uint32_t bytes = (W8 ? 0u : 2 * EX_A_BOX_BYTES) + half * ROW_BYTES;
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        if (!thread_wait(empty + stage, phase ^ 1u, abort_flag, tmo)) { ok = false; break; }
        {
          // Only the even CTA arrives, expecting the bytes of both CTAs; the
          // odd CTA's loads just count their bytes on the even CTA's barrier.
          // (The odd CTA reuses stage s only after the MMAs that consumed it
          // completed, so its bytes always land in the phase they belong to.)
          const uint32_t fb = tc::mapa_shared(tc::smem_u32(full + stage), 0);
          if (rank == 0) tc::mbar_arrive_expect_tx(full + stage, 2 * bytes);
          if (W8) {
            uint8_t* sa = smem + stage * STB;
            tc::mbar_arrive_expect_tx(raw_full + stage, 2 * W8_RAW_BOX_BYTES);
            tc::tma_load_2d(sa, mA, raw_full + stage, kb * BK, a_row0);
            tc::tma_load_2d(sa + W8_RAW_BOX_BYTES, mA, raw_full + stage, kb * BK, a_row1);
            load_token_rows<true>(sa + 2 * W8_RAW_BOX_BYTES, mB, kTokBox0Pair, half, nullptr,
                                  fb, kb * BK, b_row);
          } else if (MODE == GM_DGRAD) {
            // MN-major weights: rows kb*64.. of the group's [K, M] matrix,
            // columns of acc0 (this CTA's 128) and of acc1 (256 further), in
            // boxes of 64 columns
            uint8_t* sa = smem + stage * STB;
            const int krow = gl * args.a_rows_per_group + kb * BK;
            const int c0 = t.mb * 512 + static_cast<int>(rank) * 128;
#pragma unroll
            for (int bx = 0; bx < 4; ++bx)
              tc::tma_load_2d_pair(sa + bx * kMnBoxBytes, mA, fb, c0 + (bx >> 1) * 256 + (bx & 1) * 64,
                                   krow);
            load_token_rows<true>(sa + 2 * EX_A_BOX_BYTES, mB, kTokBox0Pair, half, nullptr, fb,
                                  kb * BK, b_row);
          } else {
            uint8_t* sa = smem + stage * STB;
            tc::tma_load_2d_pair(sa, mA, fb, kb * BK, a_row0);
            tc::tma_load_2d_pair(sa + EX_A_BOX_BYTES, mA, fb, kb * BK, a_row1);
            load_token_rows<true>(sa + 2 * EX_A_BOX_BYTES, mB, kTokBox0Pair, half, nullptr, fb,
                                  kb * BK, b_row);
          }
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == NST) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      ok = rank == 0 ? queue.publish1(claimed, tile) : queue.next1(tile);
    }
    if (!ok) {
      // abort: let every load counted on this CTA's barriers land before exit
      const unsigned long long dl = tc::globaltimer_ns() + tmo;
      for (int s = 0; s < NST; ++s) {
        if (!(issued & (1u << s))) continue;
        if (rank == 0) tc::mbar_wait_deadline(full + s, (issued_par >> s) & 1u, dl);
        if (W8) tc::mbar_wait_deadline(raw_full + s, (issued_par >> s) & 1u, dl);
      }
    }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (rank == 0 && lane == 0) {   // one thread runs the loop
      int stage = 0, aslot = 0;
      uint32_t phase = 0, tphase = 0, aphase = 0;
      bool ok = true, issued_any = false;
      for (;;) {
        int tile;
        if (!queue.next1(tile)) { ok = false; break; }
        if (tile >= ntiles) break;
        Tile t;
        decode_group_tile(args, tile, t);
        if (!thread_wait<true>(tempty, tphase ^ 1u, abort_flag, tmo)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t idesc = tc::idesc_bf16_f32_mn(256, t.nmma, MODE == GM_DGRAD, false);
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!thread_wait(full + stage, phase, abort_flag, tmo)) { ok = false; break; }
          // W8: the dequantised weights of both CTAs (written by threads,
          // published with release at cluster scope)
          if (W8 && !thread_wait<true>(a_full + aslot, aphase, abort_flag, tmo)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          {
            const uint32_t sa = tc::smem_u32(smem + stage * STB);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint32_t acc = (kb > t.kb0 || kk > 0) ? 1u : 0u;
              if constexpr (W8) {
                // A from the TMEM slot: box b at +32 b, K = 16 per MMA = 8 columns
                const uint32_t ta = tmem_base + W8_A_COL + aslot * 64 + kk * 8;
                const uint64_t db = tc::smem_desc_sw128(sa + 2 * W8_RAW_BOX_BYTES + kk * 32);
                tc::mma_bf16_ts<2>(tmem_base, ta, db, idesc, acc);
                tc::mma_bf16_ts<2>(tmem_base + ACC1, ta + 32, db, idesc, acc);
              } else {
                // K-major A: K = 16 is 32 bytes along the row; MN-major A: 16
                // rows of 128 bytes, the second 64 columns one box further
                const uint64_t da0 =
                    MODE == GM_DGRAD
                        ? tc::smem_desc_sw128_mn(sa + kk * 16 * ROW_BYTES, kMnBoxBytes)
                        : tc::smem_desc_sw128(sa + kk * 32);
                const uint64_t da1 =
                    MODE == GM_DGRAD
                        ? tc::smem_desc_sw128_mn(sa + 2 * kMnBoxBytes + kk * 16 * ROW_BYTES,
                                                 kMnBoxBytes)
                        : tc::smem_desc_sw128(sa + EX_A_BOX_BYTES + kk * 32);
                const uint64_t db = tc::smem_desc_sw128(sa + 2 * EX_A_BOX_BYTES + kk * 32);
                tc::mma_bf16<2>(tmem_base, da0, db, idesc, acc);
                tc::mma_bf16<2>(tmem_base + ACC1, da1, db, idesc, acc);
              }
            }
            tc::mma_commit<2>(empty + stage);   // frees the stage in both CTAs
            if (W8) tc::mma_commit<2>(a_empty + aslot);
          }
          issued_any = true;
          if (++stage == NST) { stage = 0; phase ^= 1u; }
          if (W8 && ++aslot == W8_A_SLOTS) { aslot = 0; aphase ^= 1u; }
        }
        if (!ok) break;
        tc::mma_commit<2>(tfull);  // accumulators complete, both CTAs
        tphase ^= 1u;
      }
      if (!ok && issued_any) {
        tc::mma_commit<2>(drain, 0x1);
        tc::mbar_wait_deadline(drain, 0, tc::globaltimer_ns() + tmo);
      }
    }
    __syncwarp();
  } else if (W8 && warp >= 2 + EX_EPI_WARPS) {
    // ------------------------------------------------------------ dequantisation (W8)
    // Group grp takes the K steps ks with ks % 2 == grp (A slot grp).  Thread
    // = weight row r of the CTA's 128 (TMEM lane r; warp w reaches lanes
    // 32 (w % 4)..): per box it reads the row's 64 raw bytes (four 16-byte
    // pieces, 64-byte swizzle: conflict-free), converts them to 32 bf16 pairs
    // and stores them to its TMEM lane in one tcgen05.st.
    const int grp = (warp - 2 - EX_EPI_WARPS) / W8_DQ_GROUP;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t ta_lane = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                             W8_A_COL + grp * 64;
    const uint32_t afull_c = tc::mapa_shared(tc::smem_u32(a_full + grp), 0);
    uint32_t ks = 0;                               // K steps of the sequence so far
    bool ok = true;
    for (;;) {
      int tile;
      if (!queue.next(tile) || tile >= ntiles) break;
      Tile t;
      decode_group_tile(args, tile, t);
      const bool second = t.g >= args.E;
      const int gl = second ? t.g - args.E : t.g;
      const int a_row0 = gl * args.a_rows_per_group + t.mb * kBlockW + static_cast<int>(rank) * 128;
      const int a_row1 = a_row0 + args.a1_off;
      // 128 x 128 block scales of the two boxes' rows, one per 128-wide K block
      const float* scb = second ? args.w_scale[1] : args.w_scale[0];
      const float* sc0 = scb + static_cast<size_t>(a_row0 >> 7) * args.scale_kb;
      const float* sc1 = scb + static_cast<size_t>(a_row1 >> 7) * args.scale_kb;
      for (int kb = t.kb0; kb < t.kb1; ++kb, ++ks) {
        if ((ks & 1u) != static_cast<uint32_t>(grp)) continue;
        const int stage = static_cast<int>(ks % NST);
        const uint32_t phase = (ks / NST) & 1u;
        const uint32_t aphase = (ks / W8_A_SLOTS) & 1u;
        if (!warp_wait(raw_full + stage, phase, abort_flag, tmo)) { ok = false; break; }
        if (!warp_wait(a_empty + grp, aphase ^ 1u, abort_flag, tmo)) { ok = false; break; }
        tc::tc_fence_after();
        const uint8_t* raw = smem + stage * STB + r * 64;
#pragma unroll
        for (int box = 0; box < 2; ++box) {
          const float sc = __ldg((box ? sc1 : sc0) + (kb >> 1));
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(
                raw + box * W8_RAW_BOX_BYTES + ((c ^ ((r >> 1) & 3)) << 4));
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[8 * c + 2 * i] = dequant2(static_cast<uint16_t>(wv[i] & 0xffffu), sc);
              o[8 * c + 2 * i + 1] = dequant2(static_cast<uint16_t>(wv[i] >> 16), sc);
            }
          }
          tc::tmem_st32(ta_lane + box * 32, o);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(afull_c);
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w drains TMEM lanes 32*(w%4).. (its quadrant: 32 output columns of
    // this CTA) in 16-token chunks, alternate chunks per warp of a quadrant.
    // tcgen05.ld 16x256b yields the 8x8 fragment layout that stmatrix.trans
    // writes token-major into a staging box (16 tokens x 64 bytes); the warp
    // then copies the box out with 16-byte loads and stores.  (A TMA store of
    // the box needs a proxy fence first, which cost more than the copy.)
    constexpr int NOUT = ex_nout(MODE);
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t tempty_addr = tc::mapa_shared(tc::smem_u32(tempty), 0);
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    constexpr uint32_t kLanes16 = 16u << 16;     // TMEM lane offset of the upper 16 lanes
    uint8_t* stg_p = smem + EX_STG_OFF + (warp - 2) * (2 * NOUT * EX_STG_BOX);
    const uint32_t stg = tc::smem_u32(stg_p);
    // stmatrix: lane 8i+j addresses row j of matrix i; matrices 0/1 hold
    // tokens 0..7 and 2/3 tokens 8..15, odd ones the upper 8 columns of a
    // 16-lane half; the box row r keeps 16-byte chunk c at c ^ ((r >> 1) & 3)
    const int srow = (lane & 7) + 8 * (lane >> 4);
    uint32_t soff[2];
#pragma unroll
    for (int lh = 0; lh < 2; ++lh) {
      const int chunk = 2 * lh + ((lane >> 3) & 1);
      soff[lh] = static_cast<uint32_t>(srow * 64 + ((chunk ^ ((srow >> 1) & 3)) << 4));
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
    int sbuf = 0;
    uint32_t tphase = 0;
    for (;;) {
      int tile;
      if (!queue.next(tile) || tile >= ntiles) break;
      Tile t;
      decode_group_tile(args, tile, t);
      const int out_row0 = __ldg(args.gt.orow + t.g) + t.tok0;
      // GATEUP: act columns (SiLU(acc0) * acc1); DOWN: y columns of acc0 and,
      // 256 further, of acc1
      const int colbase = t.mb * kBlockW + static_cast<int>(rank) * 128 + q * 32;
      if (!warp_wait(tfull, tphase, abort_flag, tmo)) break;
      tc::tc_fence_after();
      for (int j0 = h * 16; j0 < t.nmma; j0 += 32) {
        uint32_t g0[8], g1[8], u0[8], u1[8];      // acc0 / acc1, lanes 0..15 / 16..31
        tc::tmem_ld16x256_x2(taddr + j0, g0);
        tc::tmem_ld16x256_x2(taddr + kLanes16 + j0, g1);
        tc::tmem_ld16x256_x2(taddr + ACC1 + j0, u0);
        tc::tmem_ld16x256_x2(taddr + kLanes16 + ACC1 + j0, u1);
        tc::tmem_wait_ld4(g0, g1, u0, u1);
        // buffer sbuf was last read two chunks ago, before the previous
        // chunk's __syncwarp
        const uint32_t buf = stg + sbuf * (NOUT * EX_STG_BOX);
        if (MODE == GM_GATEUP) {
          stage_swiglu(buf + soff[0], g0, u0);
          stage_swiglu(buf + soff[1], g1, u1);
        } else {
          stage_bf16(buf + soff[0], g0);
          stage_bf16(buf + soff[1], g1);
          stage_bf16(buf + EX_STG_BOX + soff[0], u0);
          stage_bf16(buf + EX_STG_BOX + soff[1], u1);
        }
        __syncwarp();
        // each box: 16 token rows of 64 bytes, one 16-byte piece per lane
        // and step (a quarter row), rows of tokens past the group skipped
        const int nv = min(16, t.ntok - j0);
        const uint8_t* bp = stg_p + sbuf * (NOUT * EX_STG_BOX);
#pragma unroll
        for (int o = 0; o < NOUT; ++o) {
          // GATEUP_H: gate column colbase.. and its up column a1_off further,
          // both valid while colbase < I (= out_cols)
          const int col = colbase + o * (MODE == GM_GATEUP_H ? args.a1_off : 256);
          const int ccheck = MODE == GM_GATEUP_H ? colbase : col;
#pragma unroll
          for (int u = lane; u < 64; u += 32) {
            const int r = u >> 2, c = u & 3;
            if (r < nv && ccheck < args.out_cols) {
              const uint4 v = *reinterpret_cast<const uint4*>(
                  bp + o * EX_STG_BOX + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
              *reinterpret_cast<uint4*>(
                  out + static_cast<size_t>(out_row0 + j0 + r) * args.out_ld + col + 8 * c) = v;
            }
          }
        }
        sbuf ^= 1;
      }
      // the accumulators are free once this warp's tcgen05.ld completed (waited
      // above); a relaxed arrival does not wait for the output stores to drain
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster_relaxed(tempty_addr);
      tphase ^= 1u;
    }
  }

  tc::tc_fence_before();
  tc::cluster_sync_all();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<2>(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) atomicOr(args.status, ERRBIT_TIMEOUT);
}

// ============================================================================
// Weight gradients on CTA pairs: dW[g] = sum over the group's tokens j of
// A[j, :]^T B[j, :]  (dW2 = dy^T act, dW13 = dh^T u)
// ============================================================================
//
// Both operands are token rows, so both are MN-major for the MMA (K = the
// group's tokens): A rows come from the padded row layout of the output
// gradients (rows of group g start at a 16-row boundary and the rows up to
// the next boundary are zero), B rows from the packed forward rows.  An
// accumulator tile is 256 rows of dW (128 per CTA) x 256 columns, a K step
// 64 tokens.  The last step issues only the MMAs of the 16-token slices that
// hold tokens of the group; their rows past the group's end are zero in A,
// which zeroes the product whatever B holds there.  A group without tokens
// writes zeros without touching the tensor cores.
//
// With about 256 tokens per routed expert a tile has little MMA work for the
// operand bytes it needs, so the kernel keeps A in shared memory: a work unit
// of a routed expert is one 256-row block of dW and ALL its column blocks;
// A (this CTA's 128 rows x the expert's tokens, up to WG_A_SLOTS K steps) is
// loaded once and only B streams, which halves the operand bytes per MMA.
// Experts with more tokens and the shared experts (the whole batch) stream A
// with B through the same slots, one column block per work unit.  The two
// 256-column accumulators in TMEM alternate between consecutive tiles (the
// MMAs of one run while the epilogue drains the other), and the epilogue
// writes whole 128-byte lines: each warp rounds 32 rows x 64 columns to bf16
// into a swizzled shared-memory box, then stores it four rows per instruction.
//
// Warp roles as in the expert kernel (producer, MMA issuer in the even CTA,
// eight epilogue warps: lane quadrant w % 4, column half (w - 2) / 4).

struct WTile {
  int g, mb, nb0, nb1, arow, brow, kn;
};

constexpr int WG_A_SLOTS = 6;                          // K steps of A held at once (384 tokens)
constexpr int WG_B_STAGES = 6;

// Work units: shared experts first (their K is the whole batch), one per
// (expert, row block, column block); then routed experts, one per (expert,
// row block) covering every column block.
__device__ __forceinline__ void decode_wgrad_tile(const WgradArgs& a, int tile, WTile& t) {
  const int nsh = a.S * a.m_blocks * a.n_blocks;
  if (tile < nsh) {
    const int per = a.m_blocks * a.n_blocks;
    const int s = tile / per;
    const int local = tile - s * per;
    t.mb = local / a.n_blocks;
    t.nb0 = t.nb1 = local - t.mb * a.n_blocks;
    t.g = a.E + s;
    t.kn = a.T;
    t.arow = __ldg(a.poff + a.E) + s * a.T16;
    t.brow = a.b_sh0 + s * a.b_shs;
  } else {
    const int r = tile - nsh;
    const int e = r / a.m_blocks;
    t.mb = r - e * a.m_blocks;
    t.nb0 = 0;
    t.nb1 = a.n_blocks - 1;
    t.g = e;
    t.kn = __ldg(a.counts + e);
    t.arow = __ldg(a.poff + e);
    t.brow = __ldg(a.offsets + e);
  }
}

__device__ __forceinline__ bool wgrad_resident(const WTile& t, int E) {
  return t.g < E && (t.kn + BK - 1) / BK <= WG_A_SLOTS;
}

constexpr uint32_t WG_SLOT_BYTES = 2 * kMnBoxBytes;     // 16 KB: 64 tokens x 128 columns
constexpr uint32_t WG_B_OFF = WG_A_SLOTS * WG_SLOT_BYTES;
constexpr uint32_t WG_STG_BYTES = 32 * 128;            // per warp: 32 rows x 64 bf16
constexpr uint32_t WG_BAR_OFF = WG_B_OFF + WG_B_STAGES * WG_SLOT_BYTES;
constexpr uint32_t WG_STG_OFF = WG_BAR_OFF + 1024;
constexpr size_t WG_SMEM_BYTES = WG_STG_OFF + EX_EPI_WARPS * WG_STG_BYTES + 1024;
constexpr int WG_THREADS = 64 + 32 * EX_EPI_WARPS;
static_assert(WG_SMEM_BYTES <= 227 * 1024, "wgrad shared memory");

__global__ void __launch_bounds__(WG_THREADS, 1)
    wgrad_gemm_kernel(const __grid_constant__ WgradMaps maps, const WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + WG_BAR_OFF);
  uint64_t* a_empty = a_full + WG_A_SLOTS;
  uint64_t* b_full = a_empty + WG_A_SLOTS;
  uint64_t* b_empty = b_full + WG_B_STAGES;
  uint64_t* tfull = b_empty + WG_B_STAGES;   // [2] accumulator slot complete
  uint64_t* tempty = tfull + 2;              // [2] accumulator slot drained (even CTA)
  uint64_t* drain = tempty + 2;
  uint64_t* qfull = drain + 1;
  uint64_t* qempty = qfull + EX_QUEUE;
  volatile int* tq = reinterpret_cast<volatile int*>(qempty + EX_QUEUE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tq) + EX_QUEUE);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < WG_A_SLOTS; ++s) {
      tc::mbar_init(a_full + s, 1);
      tc::mbar_init(a_empty + s, 1);
    }
    for (int s = 0; s < WG_B_STAGES; ++s) {
      tc::mbar_init(b_full + s, 1);
      tc::mbar_init(b_empty + s, 1);
    }
    for (int j = 0; j < 2; ++j) {
      tc::mbar_init(tfull + j, 1);
      tc::mbar_init(tempty + j, 2 * EX_EPI_WARPS);
    }
    tc::mbar_init(drain, 1);
    for (int s = 0; s < EX_QUEUE; ++s) {
      tc::mbar_init(qfull + s, 1);
      tc::mbar_init(qempty + s, queue_consumers(false));
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane < 3) tc::tma_prefetch_desc(lane == 0 ? &maps.a : &maps.b[lane - 1]);
  if (warp == 1) {
    tc::tmem_alloc<2>(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish<2>();
  }
  tc::tc_fence_before();
  tc::cluster_sync_all();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = args.S * args.m_blocks * args.n_blocks + args.E * args.m_blocks;
  const unsigned long long tmo = args.timeout_ns;

  TileQueue queue{qfull, qempty, tq, rank, abort_flag, tmo, args.tile_counter};
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // A loads (ai) and B loads (bi) each run through their ring of slots; a
    // slot is refilled after the MMAs committed its "empty" barrier.  One
    // thread runs the loop.
    if (lane == 0) {
    uint32_t ai = 0, bi = 0;
    uint32_t a_iss = 0, a_par = 0, b_iss = 0, b_par = 0;   // per slot: load in flight, parity
    bool ok = true;
    int tile = 0;
    ok = rank == 0 ? queue.publish1(queue.take(), tile) : queue.next1(tile);
    auto load_a = [&](const WTile& t, int kb) -> bool {
      const uint32_t s = ai % WG_A_SLOTS, ph = (ai / WG_A_SLOTS) & 1u;
      if (!thread_wait(a_empty + s, ph ^ 1u, abort_flag, tmo)) return false;
      {
        const uint32_t fb = tc::mapa_shared(tc::smem_u32(a_full + s), 0);
        if (rank == 0) tc::mbar_arrive_expect_tx(a_full + s, 2 * WG_SLOT_BYTES);
        uint8_t* sa = smem + s * WG_SLOT_BYTES;
        const int mcol = t.mb * 256 + static_cast<int>(rank) * 128;
        const int ar = t.arow + kb * BK;
        tc::tma_load_2d_pair(sa, &maps.a, fb, mcol, ar);
        tc::tma_load_2d_pair(sa + kMnBoxBytes, &maps.a, fb, mcol + 64, ar);
      }
      a_iss |= 1u << s;
      a_par = (a_par & ~(1u << s)) | (ph << s);
      ++ai;
      return true;
    };
    auto load_b = [&](const WTile& t, int nb, int kb) -> bool {
      const uint32_t s = bi % WG_B_STAGES, ph = (bi / WG_B_STAGES) & 1u;
      if (!thread_wait(b_empty + s, ph ^ 1u, abort_flag, tmo)) return false;
      {
        const uint32_t fb = tc::mapa_shared(tc::smem_u32(b_full + s), 0);
        if (rank == 0) tc::mbar_arrive_expect_tx(b_full + s, 2 * WG_SLOT_BYTES);
        uint8_t* sb = smem + WG_B_OFF + s * WG_SLOT_BYTES;
        const CUtensorMap* mB = &maps.b[t.g >= args.E ? 1 : 0];
        const int ncol = nb * 256 + static_cast<int>(rank) * 128;
        const int br = t.brow + kb * BK;
        tc::tma_load_2d_pair(sb, mB, fb, ncol, br);
        tc::tma_load_2d_pair(sb + kMnBoxBytes, mB, fb, ncol + 64, br);
      }
      b_iss |= 1u << s;
      b_par = (b_par & ~(1u << s)) | (ph << s);
      ++bi;
      return true;
    };
    while (ok && tile < ntiles) {
      const int claimed = rank == 0 ? queue.take() : 0;
      WTile t;
      decode_wgrad_tile(args, tile, t);
      const int nk = (t.kn + BK - 1) / BK;
      const bool res = wgrad_resident(t, args.E);
      for (int kb = 0; ok && res && kb < nk; ++kb) ok = load_a(t, kb);
      for (int nb = t.nb0; ok && nb <= t.nb1 && nk > 0; ++nb)
        for (int kb = 0; ok && kb < nk; ++kb) {
          if (!res) ok = load_a(t, kb);
          if (ok) ok = load_b(t, nb, kb);
        }
      if (!ok) break;
      ok = rank == 0 ? queue.publish1(claimed, tile) : queue.next1(tile);
    }
    if (!ok && rank == 0) {
      // abort: let every load counted on this CTA's barriers land before exit
      const unsigned long long dl = tc::globaltimer_ns() + tmo;
      for (int s = 0; s < WG_A_SLOTS; ++s)
        if (a_iss & (1u << s)) tc::mbar_wait_deadline(a_full + s, (a_par >> s) & 1u, dl);
      for (int s = 0; s < WG_B_STAGES; ++s)
        if (b_iss & (1u << s)) tc::mbar_wait_deadline(b_full + s, (b_par >> s) & 1u, dl);
    }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (rank == 0 && lane == 0) {   // one thread runs the loop
      uint32_t ai = 0, bi = 0, acc_n = 0;
      bool ok = true, issued_any = false;
      const uint32_t idesc = tc::idesc_bf16_f32_mn(256, 256, true, true);
      for (;;) {
        int tile;
        if (!queue.next1(tile)) { ok = false; break; }
        if (tile >= ntiles) break;
        WTile t;
        decode_wgrad_tile(args, tile, t);
        const int nk = (t.kn + BK - 1) / BK;
        if (nk == 0) continue;                 // no tokens: the epilogue writes zeros
        const bool res = wgrad_resident(t, args.E);
        const uint32_t a0 = ai;                // resident: this unit's A loads a0 .. a0+nk-1
        if (res) ai += nk;
        for (int nb = t.nb0; ok && nb <= t.nb1; ++nb) {
          const uint32_t slot = acc_n & 1u, use = acc_n >> 1;
          if (!thread_wait<true>(tempty + slot, (use & 1u) ^ 1u, abort_flag, tmo)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t dcol = tmem_base + slot * 256;
          for (int kb = 0; kb < nk; ++kb) {
            const uint32_t aj = res ? a0 + kb : ai++;
            const uint32_t as = aj % WG_A_SLOTS, bs = bi % WG_B_STAGES;
            if (!thread_wait(a_full + as, (aj / WG_A_SLOTS) & 1u, abort_flag, tmo) ||
                !thread_wait(b_full + bs, (bi / WG_B_STAGES) & 1u, abort_flag, tmo)) {
              ok = false;
              break;
            }
            ++bi;
            tc::tc_fence_after();
            {
              const uint32_t sa = tc::smem_u32(smem + as * WG_SLOT_BYTES);
              const uint32_t sb = tc::smem_u32(smem + WG_B_OFF + bs * WG_SLOT_BYTES);
              const int left = t.kn - kb * BK;
              const int nmma = left >= BK ? BK / 16 : (left + 15) / 16;
              for (int kk = 0; kk < nmma; ++kk) {
                const uint32_t ko = kk * 16 * ROW_BYTES;
                tc::mma_bf16<2>(dcol, tc::smem_desc_sw128_mn(sa + ko, kMnBoxBytes),
                                tc::smem_desc_sw128_mn(sb + ko, kMnBoxBytes), idesc,
                                (kb > 0 || kk > 0) ? 1u : 0u);
              }
              tc::mma_commit<2>(b_empty + bs);
              if (!res) tc::mma_commit<2>(a_empty + as);
            }
            issued_any = true;
          }
          if (!ok) break;
          tc::mma_commit<2>(tfull + slot);
          ++acc_n;
        }
        if (!ok) break;
        if (res) {
          // the unit's MMAs are issued: its A slots free once they complete
          for (int kb = 0; kb < nk; ++kb) tc::mma_commit<2>(a_empty + (a0 + kb) % WG_A_SLOTS);
        }
      }
      if (!ok && issued_any) {
        tc::mma_commit<2>(drain, 0x1);
        tc::mbar_wait_deadline(drain, 0, tc::globaltimer_ns() + tmo);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // warp w: TMEM lanes 32 (w % 4).. (dW rows), columns 128 h .. of each
    // column block.  The next unit's index is read before the stores of this
    // unit's last tile: releasing the queue slot then has few stores to wait for.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint8_t* stg = smem + WG_STG_OFF + (warp - 2) * WG_STG_BYTES;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    uint32_t acc_n = 0;
    int tile;
    bool ok = queue.next(tile);
    while (ok && tile < ntiles) {
      WTile t;
      decode_wgrad_tile(args, tile, t);
      const int row0 = t.mb * 256 + static_cast<int>(rank) * 128 + q * 32;
      const bool second = t.g >= args.E;
      __nv_bfloat16* out =
          static_cast<__nv_bfloat16*>(second ? args.out_shared : args.out_routed) +
          static_cast<size_t>(second ? t.g - args.E : t.g) * args.out_gstride;
      const bool zero = t.kn <= 0;
      int next_tile = ntiles;
      bool fetched = false;
      for (int nb = t.nb0; nb <= t.nb1; ++nb) {
        const int col0 = nb * 256 + h * 128;
        const uint32_t slot = acc_n & 1u, use = acc_n >> 1;
        if (!zero) {
          if (!warp_wait(tfull + slot, use & 1u, abort_flag, tmo)) { ok = false; break; }
          tc::tc_fence_after();
        }
        // the next unit's index is published once the producer issued every
        // load of this unit, which needs the MMAs (and this epilogue) to be
        // at this unit's last tile: read it there, not earlier
        if (nb == t.nb1) {
          ok = queue.next(next_tile);
          fetched = true;
        }
        const uint32_t taddr = tmem_base + lane_addr + slot * 256 + h * 128;
        for (int c0 = 0; c0 < 128; c0 += 64) {
          // this lane's row: 64 columns -> 32 bf16 pairs -> 8 swizzled 16-byte chunks
          uint32_t p[32];
          if (!zero) {
            uint32_t r0[16], r1[16], r2[16], r3[16];
            tc::tmem_ld16(taddr + c0, r0);
            tc::tmem_ld16(taddr + c0 + 16, r1);
            tc::tmem_wait_ld(r0, r1);
            tc::tmem_ld16(taddr + c0 + 32, r2);
            tc::tmem_ld16(taddr + c0 + 48, r3);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              p[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
              p[8 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
            }
            tc::tmem_wait_ld(r2, r3);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              p[16 + i] = pack_bf16x2(__uint_as_float(r2[2 * i]), __uint_as_float(r2[2 * i + 1]));
              p[24 + i] = pack_bf16x2(__uint_as_float(r3[2 * i]), __uint_as_float(r3[2 * i + 1]));
            }
            if (c0 == 64) {
              // every TMEM read of the slot is complete: hand it back to the MMAs
              tc::tc_fence_before();
              __syncwarp();
              if (lane == 0)
                tc::mbar_arrive_cluster_relaxed(tc::mapa_shared(tc::smem_u32(tempty + slot), 0));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) p[i] = 0u;
          }
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
          __syncwarp();
          // lane: chunk lane % 8 of rows 4 i + lane / 8 -> four whole rows per store
          const int col = col0 + c0 + (lane & 7) * 8;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            const uint4 v =
                *reinterpret_cast<const uint4*>(stg + r * 128 + (((lane & 7) ^ (r & 7)) << 4));
            if (row0 + r < args.M && col < args.N)
              *reinterpret_cast<uint4*>(out + static_cast<size_t>(row0 + r) * args.N + col) = v;
          }
          __syncwarp();
        }
        if (!zero) ++acc_n;
      }
      if (!fetched) ok = false;
      tile = next_tile;
    }
  }

  tc::tc_fence_before();
  tc::cluster_sync_all();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<2>(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) atomicOr(args.status, ERRBIT_TIMEOUT);
}

// ============================================================================
// Router GEMM: one CTA per tile
// ============================================================================

constexpr int RT_STAGES = 3;
constexpr uint32_t RT_A_BOX_BYTES = 128 * ROW_BYTES;                     // 16 KB
constexpr uint32_t RT_STAGE_BYTES = 2 * RT_A_BOX_BYTES + 256 * ROW_BYTES;  // 64 KB
constexpr int RT_THREADS = 192;
constexpr size_t RT_SMEM_BYTES = RT_STAGES * RT_STAGE_BYTES + 1024 + 256;

__global__ void __launch_bounds__(RT_THREADS, 1)
    router_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RT_STAGES * RT_STAGE_BYTES);
  uint64_t* empty = full + RT_STAGES;
  uint64_t* tfull = empty + RT_STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RT_STAGES; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    tc::mbar_init(tfull, 1);
    tc::mbar_init(tempty, 4);    // one arrival per epilogue warp
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane < 1 + kTokBoxes) {
    tc::tma_prefetch_desc(lane == 0 ? &maps.a[0] : &maps.b[0][lane - 1]);
  }
  if (warp == 1) {
    tc::tmem_alloc<1>(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish<1>();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = args.router_nb * args.m_blocks * args.k_splits;
  const unsigned long long tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_par = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      Tile t;
      decode_router_tile(args, tile, t);
      const int a_row0 = t.mb * 256;
      const uint32_t bytes = 2 * RT_A_BOX_BYTES + t.nmma * ROW_BYTES;
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        if (!warp_wait(empty + stage, phase ^ 1u, abort_flag, tmo)) { ok = false; break; }
        if (lane == 0) {
          uint8_t* sa = smem + stage * RT_STAGE_BYTES;
          tc::mbar_arrive_expect_tx(full + stage, bytes);
          tc::tma_load_2d(sa, &maps.a[0], full + stage, kb * BK, a_row0);
          tc::tma_load_2d(sa + RT_A_BOX_BYTES, &maps.a[0], full + stage, kb * BK, a_row0 + 128);
          load_token_rows<false>(sa + 2 * RT_A_BOX_BYTES, maps.b[0], kTokBox0Single, t.nmma,
                                 full + stage, 0, kb * BK, t.tok0);
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        __syncwarp();
        if (++stage == RT_STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      for (int s = 0; s < RT_STAGES; ++s)
        if (issued & (1u << s)) drain_wait(full + s, (issued_par >> s) & 1u, tmo);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0, tphase = 0;
    bool ok = true, issued_any = false;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      Tile t;
      decode_router_tile(args, tile, t);
      if (!warp_wait(tempty, tphase ^ 1u, abort_flag, tmo)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, t.nmma);
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        if (!warp_wait(full + stage, phase, abort_flag, tmo)) { ok = false; break; }
        tc::tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = tc::smem_u32(smem + stage * RT_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t da0 = tc::smem_desc_sw128(sa + kk * 32);
            const uint64_t da1 = tc::smem_desc_sw128(sa + RT_A_BOX_BYTES + kk * 32);
            const uint64_t db = tc::smem_desc_sw128(sa + 2 * RT_A_BOX_BYTES + kk * 32);
            const uint32_t acc = (kb > t.kb0 || kk > 0) ? 1u : 0u;
            tc::mma_bf16<1>(tmem_base, da0, db, idesc, acc);
            tc::mma_bf16<1>(tmem_base + 256, da1, db, idesc, acc);
          }
          tc::mma_commit<1>(empty + stage);
        }
        issued_any = true;
        __syncwarp();
        if (++stage == RT_STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) tc::mma_commit<1>(tfull);
      __syncwarp();
      tphase ^= 1u;
    }
    if (!ok && issued_any) {
      if (lane == 0) tc::mma_commit<1>(drain);
      __syncwarp();
      drain_wait(drain, 0, tmo);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    uint32_t tphase = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      Tile t;
      decode_router_tile(args, tile, t);
      if (!warp_wait(tfull, tphase, abort_flag, tmo)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int col0 = t.mb * 256 + row, col1 = col0 + 128;
      const bool c0ok = col0 < args.out_cols, c1ok = col1 < args.out_cols;
      for (int j0 = 0; j0 < t.nmma; j0 += 16) {
        uint32_t r0[16], r1[16];
        tc::tmem_ld16(taddr + j0, r0);
        tc::tmem_ld16(taddr + 256 + j0, r1);
        tc::tmem_wait_ld(r0, r1);
        float* o = static_cast<float*>(args.out) + t.split * args.out_split_stride +
                   static_cast<size_t>(t.tok0 + j0) * args.out_ld;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j0 + j < t.ntok) {
            if (c0ok) o[static_cast<size_t>(j) * args.out_ld + col0] = __uint_as_float(r0[j]);
            if (c1ok) o[static_cast<size_t>(j) * args.out_ld + col1] = __uint_as_float(r1[j]);
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tempty);
      tphase ^= 1u;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<1>(tmem_base, TMEM_COLS);
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

__global__ void __launch_bounds__(1024) build_groups_kernel(const int* offsets, const int* counts,
                                                            int T, int E, int S, GroupLayout lay,
                                                            int* rows, int* brow, int* orow,
                                                            int* bs, int* bstart) {
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
        r = counts ? counts[g] : offsets[g + 1] - br;
        orw = br;
      } else {
        r = T;
        br = lay.shared_src;
        orw = lay.shared_out0 + (g - E) * lay.shared_stride;
      }
      int b;
      token_blocks(r, &b, &nb, lay.max_bs);
      rows[g] = r;
      brow[g] = br;
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
  if (threadIdx.x == 0) {
    bstart[G] = total;
    bstart[G + 1] = 0;   // tile counter of the gate/up GEMM
    bstart[G + 2] = 0;   // tile counter of the down GEMM
  }
}

__global__ void __launch_bounds__(1024) build_bwd_groups_kernel(const int* counts, int T, int E,
                                                                int S, int* poff, int* rows,
                                                                int* brow, int* orow, int* bs,
                                                                int* bstart, int* counters) {
  __shared__ int warp_sums[32];
  __shared__ int spoff[kMaxE + 1];
  // padded offsets of the routed groups (E <= 1024: one group per thread)
  const int e = threadIdx.x;
  int total = 0;
  const int before =
      block_exclusive_scan(e < E ? (counts[e] + 15) & ~15 : 0, warp_sums, &total);
  if (e < E) {
    poff[e] = before;
    spoff[e] = before;
  }
  if (threadIdx.x == 0) {
    poff[E] = total;
    spoff[E] = total;
    for (int i = 0; i < 4; ++i) counters[i] = 0;
  }
  __syncthreads();
  const int T16 = (T + 15) & ~15;
  const int G = E + S;
  // each thread owns two consecutive groups (G <= kMaxE + kMaxS <= 2048)
  int nb_pair[2];
  int local = 0;
  for (int u = 0; u < 2; ++u) {
    const int g = threadIdx.x * 2 + u;
    int nb = 0;
    if (g < G) {
      const int r = g < E ? counts[g] : T;
      const int br = g < E ? spoff[g] : spoff[E] + (g - E) * T16;
      int b;
      token_blocks(r, &b, &nb, 256);
      rows[g] = r;
      brow[g] = br;
      orow[g] = br;
      bs[g] = b;
    }
    nb_pair[u] = nb;
    local += nb;
  }
  int tot_blocks = 0;
  const int b0 = block_exclusive_scan(local, warp_sums, &tot_blocks);
  const int g0 = threadIdx.x * 2;
  if (g0 < G) bstart[g0] = b0;
  if (g0 + 1 < G) bstart[g0 + 1] = b0 + nb_pair[0];
  if (threadIdx.x == 0) bstart[G] = tot_blocks;
}

// Grid of a persistent kernel: at most one CTA (or pair) per SM, and no more
// clusters than can be resident at once.
// The occupancy query runs on a kernel's first launch on a device only, so
// later launches (and CUDA graph captures after a first eager call) make no
// host query.
template <typename Kern>
int persistent_ctas(Kern kern, int cluster, size_t smem, int threads, int want) {
  struct Entry {
    const void* fn;
    int dev, ctas;
  };
  static Entry cache[32] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const void* fn = reinterpret_cast<const void*>(kern);
  int slot = -1;
  for (int i = 0; i < 32; ++i) {
    if (cache[i].fn == fn && cache[i].dev == dev) { slot = i; break; }
    if (!cache[i].fn) { slot = i; break; }
  }
  if (slot < 0) slot = 31;                        // more kernels x devices than slots: re-query
  int& c = cache[slot].ctas;
  if (cache[slot].fn != fn || cache[slot].dev != dev) {
    cache[slot].fn = fn;
    cache[slot].dev = dev;
    c = 0;
  }
  if (c == 0) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(num_sms() / cluster * cluster), 1, 1);
    lc.blockDim = dim3(threads, 1, 1);
    lc.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &lc) != cudaSuccess || n <= 0) return 0;
    c = n * cluster;
  }
  const int g = want < c ? want : c;
  return g / cluster * cluster;
}

template <typename Kern>
moe_status_t launch_persistent(Kern kern, const char* name, int cluster, size_t smem,
                               int threads, int want, const GemmMaps& maps, const GemmArgs& args,
                               cudaStream_t stream, bool* attr_done) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_done[dev] = true;
  }
  const int grid = persistent_ctas(kern, cluster, smem, threads, want);
  if (grid <= 0) return MOE_ERR_CUDA;
  TraceScope tr(stream, name);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  lc.blockDim = dim3(threads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, kern, maps, args) != cudaSuccess) return MOE_ERR_CUDA;
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

bool make_tmap_e4m3(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc || !base || rows == 0 || cols == 0) return false;
  const cuuint64_t gdim[2] = {cols, rows};
  const cuuint64_t gstride[1] = {cols};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), 128};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_gemm_maps(GemmMaps* m, const void* a0, uint64_t a0_rows, const void* a1,
                    uint64_t a1_rows, uint32_t a_box_rows, const void* b0, uint64_t b0_rows,
                    const void* b1, uint64_t b1_rows, uint64_t k, uint32_t tok_box0) {
  if (!make_tmap_bf16(&m->a[0], a0, a0_rows, k, a_box_rows)) return false;
  if (a1) {
    if (!make_tmap_bf16(&m->a[1], a1, a1_rows, k, a_box_rows)) return false;
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
                            cudaStream_t stream, bool w8, bool small, const char* trace_name) {
  if (grid <= 0) return MOE_OK;
  static bool attr_gu[64], attr_dn[64], attr_rt[64], attr_gu8[64], attr_dn8[64], attr_gus[64],
      attr_dns[64], attr_guh[64], attr_guhs[64], attr_dg[64];
  switch (mode) {
    case GM_GATEUP:
      if (w8)
        return launch_persistent(expert_gemm_kernel<GM_GATEUP, true, false>,
                                 "gemm_w8_gateup_swiglu", 2, ex_smem_bytes(GM_GATEUP),
                                 ex_threads(true), grid, maps, args, stream, attr_gu8);
      if (small)
        return launch_persistent(expert_gemm_kernel<GM_GATEUP, false, true>,
                                 "gemm_gateup_swiglu", 2, ex_smem_bytes(GM_GATEUP),
                                 ex_threads(false), grid, maps, args, stream, attr_gus);
      return launch_persistent(expert_gemm_kernel<GM_GATEUP, false, false>, "gemm_gateup_swiglu",
                               2, ex_smem_bytes(GM_GATEUP), ex_threads(false), grid, maps, args,
                               stream, attr_gu);
    case GM_DOWN:
      if (w8)
        return launch_persistent(expert_gemm_kernel<GM_DOWN, true, false>, "gemm_w8_down", 2,
                                 ex_smem_bytes(GM_DOWN), ex_threads(true), grid, maps, args,
                                 stream, attr_dn8);
      if (small)
        return launch_persistent(expert_gemm_kernel<GM_DOWN, false, true>, "gemm_down", 2,
                                 ex_smem_bytes(GM_DOWN), ex_threads(false), grid, maps, args,
                                 stream, attr_dns);
      return launch_persistent(expert_gemm_kernel<GM_DOWN, false, false>, "gemm_down", 2,
                               ex_smem_bytes(GM_DOWN), ex_threads(false), grid, maps, args,
                               stream, attr_dn);
    case GM_ROUTER:
      return launch_persistent(router_gemm_kernel, "gemm_router", 1, RT_SMEM_BYTES, RT_THREADS,
                               grid, maps, args, stream, attr_rt);
    case GM_GATEUP_H:
      if (w8) return MOE_ERR_UNSUPPORTED;
      if (small)
        return launch_persistent(expert_gemm_kernel<GM_GATEUP_H, false, true>, "gemm_gateup_h",
                                 2, ex_smem_bytes(GM_GATEUP_H), ex_threads(false), grid, maps,
                                 args, stream, attr_guhs);
      return launch_persistent(expert_gemm_kernel<GM_GATEUP_H, false, false>, "gemm_gateup_h", 2,
                               ex_smem_bytes(GM_GATEUP_H), ex_threads(false), grid, maps, args,
                               stream, attr_guh);
    case GM_DGRAD:
      if (w8 || small) return MOE_ERR_UNSUPPORTED;
      return launch_persistent(expert_gemm_kernel<GM_DGRAD, false, false>,
                               trace_name ? trace_name : "gemm_dgrad", 2,
                               ex_smem_bytes(GM_DGRAD), ex_threads(false), grid, maps, args,
                               stream, attr_dg);
    default: return MOE_ERR_INVALID_ARG;
  }
}

moe_status_t launch_build_groups(const int* offsets, const int* counts, int T, int E, int S,
                                 GroupLayout lay, int* rows, int* brow, int* orow, int* bs,
                                 int* bstart, cudaStream_t stream) {
  TraceScope tr(stream, "build_groups");
  build_groups_kernel<<<1, 1024, 0, stream>>>(offsets, counts, T, E, S, lay, rows, brow, orow,
                                              bs, bstart);
  return launch_status();
}

moe_status_t launch_build_bwd_groups(const int* counts, int T, int E, int S, int* poff, int* rows,
                                     int* brow, int* orow, int* bs, int* bstart, int* counters,
                                     cudaStream_t stream) {
  TraceScope tr(stream, "build_bwd_groups");
  build_bwd_groups_kernel<<<1, 1024, 0, stream>>>(counts, T, E, S, poff, rows, brow, orow, bs,
                                                  bstart, counters);
  return launch_status();
}

moe_status_t launch_wgrad(const WgradMaps& maps, const WgradArgs& args, cudaStream_t stream,
                          const char* trace_name) {
  static bool attr[64];
  const int want = num_sms();
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr[dev]) {
    if (cudaFuncSetAttribute(wgrad_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(WG_SMEM_BYTES)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr[dev] = true;
  }
  const int grid = persistent_ctas(wgrad_gemm_kernel, 2, WG_SMEM_BYTES, WG_THREADS, want);
  if (grid <= 0) return MOE_ERR_CUDA;
  TraceScope tr(stream, trace_name);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  lc.blockDim = dim3(WG_THREADS, 1, 1);
  lc.dynamicSmemBytes = WG_SMEM_BYTES;
  lc.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, wgrad_gemm_kernel, maps, args) != cudaSuccess) return MOE_ERR_CUDA;
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
