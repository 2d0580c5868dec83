// FP8 expert GEMMs with block scaling and CUDA-core promotion, on CTA pairs of
// the 5th-generation tensor cores (tcgen05 kind::f8f6f4 cta_group::2 + TMA +
// TMEM).
//
// Quantisation follows the V3 walk-through, section 4.3: expert weights in
// 128 x 128 blocks and activations in 1 x 128 tiles along K, each block with
// its own fp32 scale, and the partial sums promoted to fp32 on the CUDA cores
// every N_C = 128 elements of K.  So for one tile
//   D[w, t] = sum_kb  sw[w / 128, kb] * sx[t, kb] * P_kb[w, t],
//   P_kb[w, t] = sum_{k in block kb} qA[w, k] * qB[t, k]     (e4m3 x e4m3, fp32)
// P_kb comes from the tensor cores into a fresh TMEM buffer; the promotion
// warps read it, scale it and add it into fp32 running sums held in
// registers.  Three TMEM buffers rotate, so the MMAs of blocks kb + 1 and
// kb + 2 run while block kb is promoted.
//
// Layout is swap-AB as in the bf16 kernel (weights in the MMA's M slot, tokens
// in N), and a tile runs on a CTA pair (a cluster of two CTAs): one MMA of
// M = 256 weight rows spans both CTAs, each CTA holding 128 rows of A and of
// the partial sums and half of the tile's token rows.  One tile = group g,
// weight-row block mb, one token block of N <= 160 tokens:
//   GATEUP: the pair covers intermediate columns c = 128 mb .. c + 127; CTA r
//           holds gate rows c + 64 r .. +63 of W13_g in TMEM lanes 0..63 and
//           the matching up rows (+I) in lanes 64..127, so SwiGLU pairs lane l
//           with lane l + 64 through shared memory; the per-token max of act
//           over the pair's 128 columns (one 1 x 128 tile of the down GEMM's
//           K) is exchanged between the two CTAs through distributed shared
//           memory, and act leaves in e4m3 with its scale
//   DOWN:   the pair covers rows m = 256 mb .. of W2_g; CTA r holds rows
//           m + 128 r .. +127; the tile ends with y in bf16
// Per 128-wide K block the even CTA issues four MMAs (K = 32 each, M = 256,
// N = tokens) into partial buffer b = block % 3 (TMEM columns 160 b ..).  Per
// CTA that is 26 KB of operands for 5.2 MFLOP at N = 160, and 128 x 160 fp32
// running sums: up to 64 per thread of the twelve promotion warps (a CTA of
// 14 warps lets a thread hold 128 registers).
//
// Activation scales sit K-block-major ([K/128][rows], fp32), so the scales of
// a tile's tokens for block kb are one contiguous run that TMA brings in.
// Group rows start on multiples of 4 (16 bytes of scales).
//
// Warp roles (448 threads per CTA, one CTA per SM):
//   warp 0       TMA producer (one thread): per K block this CTA's 128 weight
//                rows (GATEUP: two 64-row boxes) and its half of the token
//                rows (bytes counted on the even CTA's "full" barrier), and
//                the scales of all the tile's tokens into an 8-slot ring of
//                this CTA
//   warp 1       TMEM owner; in the even CTA also the MMA issuer (one thread)
//   warps 2..13  promotion + epilogue: warp w reads TMEM lanes 32 (w % 4)..
//                and token columns [64 h, min(64 h + 64, 160)), h = (w - 2) / 4
// Every barrier wait is bounded (abort flag, device error word), as in the
// bf16 kernel.
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_fp8.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int KB = 128;                       // K elements (= bytes) per stage
constexpr uint32_t ROW = 128;                 // bytes per operand row per stage
constexpr int STAGES = 6;
constexpr int MAX_N = kFp8TileTokens;         // tokens per tile
constexpr uint32_t A_BYTES = 128 * ROW;       // 16 KB: this CTA's weight rows
constexpr uint32_t STAGE_BYTES = A_BYTES + (MAX_N / 2) * ROW;   // 26 KB
constexpr int EPI_WARPS = 12;
constexpr int CW = 64;                        // token columns per promotion warp
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr int PBUFS = 3;                      // partial buffers of MAX_N columns
constexpr int SC_SLOTS = 8;
// shared memory after the stages: the gate/up exchange, the token-scale ring,
// per-warp premultiplied scales, the act amax exchange, barriers
constexpr uint32_t XCH_OFF = STAGES * STAGE_BYTES;                 // [MAX_N][64] fp32 up sums
constexpr uint32_t SC_OFF = XCH_OFF + MAX_N * 64 * 4;
constexpr uint32_t PS_OFF = SC_OFF + SC_SLOTS * MAX_N * 4;
constexpr uint32_t AM_OFF = PS_OFF + EPI_WARPS * CW * 4;
constexpr uint32_t BAR_OFF = AM_OFF + 2 * 2 * 2 * MAX_N * 4;       // [2 par][2 rank][2 q][MAX_N]
constexpr size_t SMEM_BYTES = BAR_OFF + 512 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "fp8 GEMM shared memory");
// the last column group of warps is narrow (32 columns) when MAX_N is not a
// multiple of CW
static_assert((EPI_WARPS / 4) * CW >= MAX_N && (EPI_WARPS / 4 - 1) * CW + 32 <= MAX_N &&
                  MAX_N % 32 == 0 && PBUFS * MAX_N <= TMEM_COLS, "TMEM partial buffers");
static_assert(STAGE_BYTES % 1024 == 0, "128B-swizzled stages start on 1 KB");
constexpr int HALF_WARPS = EPI_WARPS / 2;    // GATEUP: up (or gate) warps

__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (0u << 7) | (0u << 10)                    // A, B format: e4m3
         | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T over the pair: M = 256 rows split across
// the two CTAs, N token rows split likewise; issued by one thread of the even CTA.
__device__ __forceinline__ void mma_e4m3_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Tile {
  int g, mb, tok0, ntok, nmma;
};

// Tile order inside a group: routed experts weight-block-major (the token
// blocks that share a weight block run side by side and stream it from DRAM
// once), the shared experts token-block-major (a token block stays in L2
// while the weight blocks pass over it).
__device__ __forceinline__ void decode(const Fp8GemmArgs& a, int tile, Tile& t) {
  int lo = 0, hi = a.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.gt.bstart + mid) * a.m_blocks <= tile) lo = mid; else hi = mid - 1;
  }
  t.g = lo;
  const int b0 = __ldg(a.gt.bstart + lo);
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
  t.nmma = (t.ntok + 15) & ~15;
}

// Non-blocking phase test (mbarrier.test_wait): unlike try_wait it never
// suspends the thread inside the shared-memory pipe.
template <bool CLUSTER>
__device__ __forceinline__ bool test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (CLUSTER)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(tc::smem_u32(bar)), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(tc::smem_u32(bar)), "r"(parity)
        : "memory");
  return ok != 0;
}

// Bounded wait of one thread (the TMA producer or the MMA issuer): try_wait,
// which may suspend the thread until the phase completes; the abort flag and
// the wall clock are checked every 16 polls.
template <bool CLUSTER = false>
__device__ __forceinline__ bool role_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns) {
  if (test_wait<CLUSTER>(bar, parity)) return true;
  const unsigned long long deadline = tc::globaltimer_ns() + timeout_ns;
  uint32_t polls = 0;
  while (!(CLUSTER ? tc::mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity))) {
    if ((++polls & 15u) == 0) {
      if (*abort_flag) return false;
      if (tc::globaltimer_ns() > deadline) {
        *abort_flag = 1;
        return false;
      }
    }
  }
  return true;
}

// Bounded wait of one lane of a promotion warp: polls with test_wait and
// checks the abort flag and the wall clock every 64 polls.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag,
                                             unsigned long long timeout_ns) {
  if (test_wait<CLUSTER>(bar, parity)) return true;
  const unsigned long long deadline = tc::globaltimer_ns() + timeout_ns;
  uint32_t polls = 0;
  while (!test_wait<CLUSTER>(bar, parity)) {
    if ((++polls & 63u) == 0) {
      if (*abort_flag) return false;
      if (tc::globaltimer_ns() > deadline) {
        *abort_flag = 1;
        return false;
      }
    }
  }
  return true;
}

// Bounded wait by lane 0, result broadcast to the warp.  CLUSTER: arrivals
// come from the peer CTA (acquire at cluster scope).
template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) ok = wait_bounded<CLUSTER>(bar, parity, abort_flag, timeout_ns) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Every lane waits (bounded); true when the whole warp saw the phase.
template <bool CLUSTER = false>
__device__ __forceinline__ bool all_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long timeout_ns) {
  return __all_sync(0xffffffffu, wait_bounded<CLUSTER>(bar, parity, abort_flag, timeout_ns));
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g * u, 1.0f + __expf(-g));
}

// Max over the 32 lanes of each of 32 columns (v[c] per lane) by recursive
// halving: after the five exchange steps lane l holds the warp maximum of
// column l in v[0].
__device__ __forceinline__ void warp_colmax32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 16 >> step;            // values kept after this step
    const bool upper = (lane & half) != 0;  // keeps the upper half of the columns
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, half);
      v[i] = fmaxf(keep, got);
    }
  }
}

// acc{0,1} += p{0,1} * s{0,1} as one packed two-lane fp32 FMA (f32x2).
__device__ __forceinline__ void ffma2(float& a0, float& a1, float p0, float p1, float s0,
                                      float s1) {
  uint64_t acc, p, s;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(p0), "f"(p1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(s) : "f"(s0), "f"(s1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(p), "l"(s));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}

// acc[0..32) += p[i] * s[i], the scales read as float4 broadcasts from
// shared memory
__device__ __forceinline__ void promote32(float* acc, const uint32_t (&p)[32], const float* s) {
  const float4* sv = reinterpret_cast<const float4*>(s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 x = sv[i];
    ffma2(acc[4 * i], acc[4 * i + 1], __uint_as_float(p[4 * i]), __uint_as_float(p[4 * i + 1]),
          x.x, x.y);
    ffma2(acc[4 * i + 2], acc[4 * i + 3], __uint_as_float(p[4 * i + 2]),
          __uint_as_float(p[4 * i + 3]), x.z, x.w);
  }
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ Fp8GemmMaps maps, const Fp8GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* xch = reinterpret_cast<float*>(smem + XCH_OFF);        // [MAX_N][64]
  float* sc_ring = reinterpret_cast<float*>(smem + SC_OFF);     // [SC_SLOTS][MAX_N]
  float* psc = reinterpret_cast<float*>(smem + PS_OFF);         // [EPI_WARPS][CW]
  float* amx = reinterpret_cast<float*>(smem + AM_OFF);         // [2 par][2 rank][2 q][MAX_N]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* pfull = empty + STAGES;     // [PBUFS] partial buffer written (MMA commit, both CTAs)
  uint64_t* pempty = pfull + PBUFS;     // [PBUFS] promoted by every warp of the pair (even CTA)
  uint64_t* sfull = pempty + PBUFS;     // [SC_SLOTS] token scales landed
  uint64_t* sempty = sfull + SC_SLOTS;  // [SC_SLOTS] token scales read by every warp
  uint64_t* xup = sempty + SC_SLOTS;    // up sums in the exchange (GATEUP)
  uint64_t* xfree = xup + 1;            // exchange read by the gate warps (GATEUP)
  uint64_t* xam = xfree + 1;            // [2 par] act amax of both CTAs (GATEUP)
  uint64_t* drain = xam + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr bool kGU = MODE == GM_GATEUP;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full + s, 1);                // the even CTA expects both CTAs' bytes
      tc::mbar_init(empty + s, 1);               // MMAs done
    }
    for (int b = 0; b < PBUFS; ++b) {
      tc::mbar_init(pfull + b, 1);
      tc::mbar_init(pempty + b, 2 * EPI_WARPS);
    }
    for (int i = 0; i < SC_SLOTS; ++i) {
      tc::mbar_init(sfull + i, 1);
      tc::mbar_init(sempty + i, EPI_WARPS);
    }
    tc::mbar_init(xup, HALF_WARPS * 32);         // every thread of the up warps
    tc::mbar_init(xfree, HALF_WARPS * 32);       // every thread of the gate warps
    for (int i = 0; i < 2; ++i) tc::mbar_init(xam + i, 2 * HALF_WARPS * 32);   // gate warps of the pair
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane < 3 + 2 * kTokBoxes) {
    const CUtensorMap* m = lane < 2 ? &maps.a[lane]
                           : lane == 2 ? &maps.sx
                                       : &maps.b[(lane - 3) / kTokBoxes][(lane - 3) % kTokBoxes];
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
  const int nkb = args.k_blocks;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const unsigned long long tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // One thread runs the whole loop: no warp-collective step sits between
    // its barrier tests and its TMA instructions.
    if (lane == 0) {
      uint32_t kc = 0;
      uint32_t issued = 0, issued_par = 0, s_issued = 0, s_par = 0;
      bool ok = true;
      const uint32_t full_c = tc::mapa_shared(tc::smem_u32(full), 0);
      for (int tile = pair; tile < ntiles && ok; tile += npairs) {
        Tile t;
        decode(args, tile, t);
        const bool second = t.g >= args.E;
        const CUtensorMap* mA = &maps.a[second ? 1 : 0];
        const CUtensorMap* mB = maps.b[second ? 1 : 0];
        const int gl = second ? t.g - args.E : t.g;
        const int half = t.nmma >> 1;                  // token rows this CTA loads
        // GATEUP: gate rows c + 64 r and the up rows I further (two 64-row
        // boxes); DOWN: rows m + 128 r (one 128-row box)
        const int a_row0 = gl * args.a_rows_per_group + t.mb * (kGU ? 128 : 256) +
                           static_cast<int>(rank) * (kGU ? 64 : 128);
        const int b_tile = __ldg(args.gt.brow + t.g) + t.tok0;
        const int b_row = b_tile + static_cast<int>(rank) * half;
        const uint32_t bytes = A_BYTES + half * ROW;   // this CTA's bytes on the even CTA
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const int stage = kc % STAGES;
          const uint32_t phase = (kc / STAGES) & 1u;
          const int slot = kc % SC_SLOTS;
          const uint32_t sph = (kc / SC_SLOTS) & 1u;
          if (!role_wait(empty + stage, phase ^ 1u, abort_flag, tmo)) { ok = false; break; }
          if (!role_wait(sempty + slot, sph ^ 1u, abort_flag, tmo)) { ok = false; break; }
          // Only the even CTA arrives, expecting both CTAs' bytes; the odd
          // CTA's loads count on it (a stage is reused only after the MMAs
          // that read it completed, so the bytes land in their own phase).
          const uint32_t fb = full_c + stage * 8;
          if (rank == 0) tc::mbar_arrive_expect_tx(full + stage, 2 * bytes);
          uint8_t* sa = smem + stage * STAGE_BYTES;
          tc::tma_load_2d_pair(sa, mA, fb, kb * KB, a_row0);
          if (kGU) tc::tma_load_2d_pair(sa + A_BYTES / 2, mA, fb, kb * KB, a_row0 + args.a1_off);
          int done = 0;
#pragma unroll
          for (int bi = kTokBoxes - 1; bi >= 0; --bi) {
            const int hgt = 8 << bi;
            if (half & hgt) {
              tc::tma_load_2d_pair(sa + A_BYTES + done * ROW, mB + bi, fb, kb * KB,
                                   b_row + done);
              done += hgt;
            }
          }
          // scales of all the tile's tokens for block kb, into this CTA
          tc::mbar_arrive_expect_tx(sfull + slot, MAX_N * 4);
          tc::tma_load_2d(sc_ring + slot * MAX_N, &maps.sx, sfull + slot, b_tile, kb);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          s_issued |= 1u << slot;
          s_par = (s_par & ~(1u << slot)) | (sph << slot);
        }
      }
      if (!ok) {
        // abort: let every load counted on this CTA's barriers land before exit
        const unsigned long long dl = tc::globaltimer_ns() + tmo;
        for (int s = 0; s < STAGES; ++s)
          if (rank == 0 && (issued & (1u << s)))
            tc::mbar_wait_deadline(full + s, (issued_par >> s) & 1u, dl);
        for (int s = 0; s < SC_SLOTS; ++s)
          if (s_issued & (1u << s)) tc::mbar_wait_deadline(sfull + s, (s_par >> s) & 1u, dl);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (rank == 0 && lane == 0) {
      uint32_t kc = 0;
      bool ok = true, issued_any = false;
      for (int tile = pair; tile < ntiles && ok; tile += npairs) {
        Tile t;
        decode(args, tile, t);
        const uint32_t idesc = idesc_e4m3_f32(256, t.nmma);
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const int stage = kc % STAGES;
          const uint32_t phase = (kc / STAGES) & 1u;
          const int pb = kc % PBUFS;
          const uint32_t puse = (kc / PBUFS) & 1u;
          if (!role_wait<true>(pempty + pb, puse ^ 1u, abort_flag, tmo)) { ok = false; break; }
          if (!role_wait(full + stage, phase, abort_flag, tmo)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t d = tmem_base + pb * MAX_N;
#pragma unroll
          for (int kk = 0; kk < KB / 32; ++kk) {
            const uint64_t da = tc::smem_desc_sw128(sa + kk * 32);
            const uint64_t db = tc::smem_desc_sw128(sa + A_BYTES + kk * 32);
            mma_e4m3_pair(d, da, db, idesc, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit<2>(empty + stage);   // operands consumed, both CTAs
          tc::mma_commit<2>(pfull + pb);      // partial sums of block kb ready, both CTAs
          issued_any = true;
        }
      }
      if (!ok && issued_any) {
        tc::mma_commit<2>(drain, 0x1);
        tc::mbar_wait_deadline(drain, 0, tc::globaltimer_ns() + tmo);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ promotion + epilogue
    const int ew = warp - 2;
    const int q = warp & 3;                        // TMEM lane quarter of this warp
    const int h = ew >> 2;                         // token columns [CW h, CW h + CW)
    const int c0 = h * CW;
    const bool wide = c0 + CW <= MAX_N;            // else columns c0 .. c0 + 31 only
    const bool up = kGU && q >= 2;                 // GATEUP: lanes 64..127 hold up rows
    float* my_ps = psc + ew * CW;
    const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t pempty_c = tc::mapa_shared(tc::smem_u32(pempty), 0);
    uint32_t kc = 0;
    int tcount = 0;
    bool ok = true;
    for (int tile = pair; tile < ntiles && ok; tile += npairs, ++tcount) {
      Tile t;
      decode(args, tile, t);
      const bool second = t.g >= args.E;
      const int gl = second ? t.g - args.E : t.g;
      const bool active = c0 < t.nmma;
      // this warp's weight rows: GATEUP gate (or up) rows of intermediate
      // columns col0 .. col0 + 31; DOWN rows col0 .. col0 + 31 of W2 (= y columns)
      const int col0 = kGU ? t.mb * 128 + static_cast<int>(rank) * 64 + (q & 1) * 32
                           : t.mb * 256 + static_cast<int>(rank) * 128 + q * 32;
      const int wrow = (up ? args.a1_off : 0) + col0;          // row within the group
      const bool valid = col0 < args.out_cols;
      const float* wsc = second ? args.w_scale[1] : args.w_scale[0];
      const float* ws = wsc + static_cast<size_t>(gl * (args.a_rows_per_group / 128) +
                                                  (wrow >> 7)) * nkb;
      float acc[CW];
#pragma unroll
      for (int i = 0; i < CW; ++i) acc[i] = 0.f;
      float nsw = valid ? __ldg(ws) : 0.f;
      for (int kb = 0; kb < nkb; ++kb, ++kc) {
        const float sw = nsw;
        if (kb + 1 < nkb) nsw = valid ? __ldg(ws + kb + 1) : 0.f;   // ahead of use
        const int pb = kc % PBUFS;
        const uint32_t puse = (kc / PBUFS) & 1u;
        const int slot = kc % SC_SLOTS;
        const uint32_t sph = (kc / SC_SLOTS) & 1u;
        if (!warp_wait(pfull + pb, puse, abort_flag, tmo)) { ok = false; break; }
        tc::tc_fence_after();
        if (!warp_wait(sfull + slot, sph, abort_flag, tmo)) { ok = false; break; }
        if (active) {
          const float* sx = sc_ring + slot * MAX_N + c0;
#pragma unroll
          for (int j = 0; j < CW / 32; ++j)
            if (j == 0 || wide) my_ps[32 * j + lane] = sw * sx[32 * j + lane];
          __syncwarp();
          // two TMEM round trips of 32 columns (the running sums take 64
          // registers, the loaded partials 32)
          const uint32_t tb = tl + pb * MAX_N + c0;
#pragma unroll
          for (int j = 0; j < CW / 32; ++j) {
            if (j > 0 && !wide) break;
            uint32_t p[32];
            tc::tmem_ld32(tb + 32 * j, p);
            tc::tmem_wait_ld32(p);
            promote32(acc + 32 * j, p, my_ps + 32 * j);
          }
          __syncwarp();
        }
        // the partial buffer is free once this warp's loads completed (waited
        // above): a relaxed arrival; the scale slot after this warp's reads
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive_cluster_relaxed(pempty_c + pb * 8);
          tc::mbar_arrive(sempty + slot);
        }
      }
      if (!ok) break;
      // ---------------------------------------------------------- tile end
      const size_t orow0 = static_cast<size_t>(__ldg(args.gt.orow + t.g) + t.tok0) + c0;
      const int nval = t.ntok - c0;                // valid token columns of this warp
      if (kGU) {
        // Up warps hand their sums to the gate warps of the same lanes - 64
        // through xch ([token][64 rows]); every warp of both kinds takes part
        // in the exchanges on every tile (inactive ones with nothing to
        // move), so barrier phases stay in step.
        const int xr = (q & 1) * 32 + lane;        // row of the exchange
        const uint32_t tpar = static_cast<uint32_t>(tcount) & 1u;
        if (up) {
          if (tcount > 0 && !all_wait(xfree, tpar ^ 1u, abort_flag, tmo)) { ok = false; break; }
          if (active) {
#pragma unroll
            for (int i = 0; i < CW; ++i)
              if (i < 32 || wide) xch[(c0 + i) * 64 + xr] = acc[i];
          }
          tc::mbar_arrive(xup);
          continue;
        }
        if (!all_wait(xup, tpar, abort_flag, tmo)) { ok = false; break; }
        if (active) {
#pragma unroll
          for (int i = 0; i < CW; ++i)
            if (i < 32 || wide) acc[i] = silu_mul(acc[i], xch[(c0 + i) * 64 + xr]);
        }
        tc::mbar_arrive(xfree);
        // per-token max of |act| over this warp's 32 columns, to both CTAs
        const int par = tcount & 1;
        if (active) {
          float* am = amx + ((par * 2 + static_cast<int>(rank)) * 2 + (q & 1)) * MAX_N + c0;
#pragma unroll
          for (int hh = 0; hh < CW / 32; ++hh) {   // tokens c0 + 32 hh + lane
            if (hh > 0 && !wide) break;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = fabsf(acc[32 * hh + i]);
            warp_colmax32(v, lane);
            am[32 * hh + lane] = v[0];
            tc::st_shared_cluster_u32(tc::mapa_shared(tc::smem_u32(am + 32 * hh + lane), rank ^ 1u),
                                      __float_as_uint(v[0]));
          }
        }
        tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(xam + par), rank));
        tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(xam + par), rank ^ 1u));
        if (!all_wait<true>(xam + par, static_cast<uint32_t>(tcount >> 1) & 1u, abort_flag, tmo)) {
          ok = false;
          break;
        }
        if (active && valid) {
          // 1 / scale of tokens c0 + lane, c0 + 32 + lane (max over both CTAs' 64 columns)
          const float* am0 = amx + par * 4 * MAX_N + c0;
          float m[CW / 32];
#pragma unroll
          for (int u = 0; u < CW / 32; ++u) {
            const int i = 32 * u + lane;
            if (u > 0 && !wide) { m[u] = 0.f; my_ps[i] = 0.f; break; }
            m[u] = fmaxf(fmaxf(am0[i], am0[MAX_N + i]), fmaxf(am0[2 * MAX_N + i], am0[3 * MAX_N + i]));
            my_ps[i] = m[u] > 0.f ? 448.0f / m[u] : 0.f;
          }
          __syncwarp();
          uint8_t* oq = static_cast<uint8_t*>(args.out) + orow0 * args.out_ld + col0 + lane;
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            if (i < nval) {
              const __nv_fp8_storage_t b =
                  __nv_cvt_float_to_fp8(acc[i] * my_ps[i], __NV_SATFINITE, __NV_E4M3);
              oq[static_cast<size_t>(i) * args.out_ld] = b;
            }
          }
          // scale of each token for K block mb of the down GEMM: even CTA, q = 0
          if (rank == 0 && q == 0) {
#pragma unroll
            for (int u = 0; u < CW / 32; ++u)
              if (32 * u + lane < nval)
                args.out_scale[static_cast<size_t>(t.mb) * args.out_scale_ld + orow0 + 32 * u + lane] =
                    m[u] / 448.0f;
          }
          __syncwarp();
        }
      } else {
        if (active && valid) {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(args.out) + orow0 * args.out_ld + col0 + lane;
#pragma unroll
          for (int i = 0; i < CW; ++i)
            if (i < nval) o[static_cast<size_t>(i) * args.out_ld] = __float2bfloat16_rn(acc[i]);
        }
      }
    }
  }

  tc::tc_fence_before();
  tc::cluster_sync_all();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<2>(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) atomicOr(args.status, ERRBIT_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// e4m3 matrix [rows, cols] read in boxes of {128 bytes, box_rows} with 128-byte swizzle
bool tmap_e4m3(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
               uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || !base || rows == 0 || cols == 0) return false;
  const cuuint64_t gdim[2] = {cols, rows};
  const cuuint64_t gstride[1] = {cols};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// fp32 scales [k_blocks, rows] read as runs of 128 rows of one K block
bool tmap_scales(CUtensorMap* map, const float* base, uint64_t rows, uint64_t k_blocks) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || !base || rows == 0 || k_blocks == 0) return false;
  const cuuint64_t gdim[2] = {rows, k_blocks};
  const cuuint64_t gstride[1] = {rows * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(MAX_N), 1};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), gdim, gstride,
             box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs of one launch: every pair that fits at once (one CTA per SM)
template <int MODE>
int resident_ctas() {
  static int ctas[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && ctas[dev] > 0) return ctas[dev];
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(num_sms() / 2 * 2), 1, 1);
  lc.blockDim = dim3(THREADS, 1, 1);
  lc.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, fp8_gemm_kernel<MODE>, &lc) != cudaSuccess ||
      clusters <= 0)
    return 0;
  const int n = std::min(clusters * 2, num_sms() / 2 * 2);
  if (dev < 64) ctas[dev] = n;
  return n;
}

template <int MODE>
moe_status_t launch(const Fp8GemmMaps& maps, const Fp8GemmArgs& args, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(fp8_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int grid = resident_ctas<MODE>();
  if (grid <= 0) return MOE_ERR_CUDA;
  TraceScope tr(stream, MODE == GM_GATEUP ? "gemm_fp8_gateup_swiglu" : "gemm_fp8_down");
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  lc.blockDim = dim3(THREADS, 1, 1);
  lc.dynamicSmemBytes = SMEM_BYTES;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, fp8_gemm_kernel<MODE>, maps, args) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_status();
}

}  // namespace

bool make_fp8_maps(Fp8GemmMaps* m, const void* a0, uint64_t a0_rows, const void* a1,
                   uint64_t a1_rows, uint32_t a_box_rows, const void* b, uint64_t b_rows,
                   const float* sx, uint64_t k) {
  if (!tmap_e4m3(&m->a[0], a0, a0_rows, k, a_box_rows)) return false;
  if (a1) {
    if (!tmap_e4m3(&m->a[1], a1, a1_rows, k, a_box_rows)) return false;
  } else {
    m->a[1] = m->a[0];
  }
  for (int i = 0; i < kTokBoxes; ++i) {
    if (!tmap_e4m3(&m->b[0][i], b, b_rows, k, 8u << i)) return false;
    m->b[1][i] = m->b[0][i];
  }
  return tmap_scales(&m->sx, sx, b_rows, k / 128);
}

moe_status_t launch_fp8_gemm(int mode, const Fp8GemmMaps& maps, const Fp8GemmArgs& args,
                             cudaStream_t stream) {
  switch (mode) {
    case GM_GATEUP: return launch<GM_GATEUP>(maps, args, stream);
    case GM_DOWN: return launch<GM_DOWN>(maps, args, stream);
    default: return MOE_ERR_INVALID_ARG;
  }
}

}  // namespace moe
