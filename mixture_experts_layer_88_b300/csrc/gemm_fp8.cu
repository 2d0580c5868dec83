// FP8 expert GEMMs with block scaling and CUDA-core promotion, on the
// 5th-generation tensor cores (tcgen05 kind::f8f6f4 + TMA + TMEM).
//
// Quantisation follows the V3 walk-through, section 4.3: expert weights in
// 128 x 128 blocks and activations in 1 x 128 tiles along K, each block with
// its own fp32 scale, and the partial sums promoted to fp32 on the CUDA cores
// every N_C = 128 elements of K.  So for one tile
//   D[w, t] = sum_kb  sw[w / 128, kb] * sx[t, kb] * P_kb[w, t],
//   P_kb[w, t] = sum_{k in block kb} qA[w, k] * qB[t, k]     (e4m3 x e4m3, fp32)
// P_kb comes from the tensor cores (one K = 128 block = 4 MMAs of K = 32 into
// a fresh TMEM buffer); the epilogue warps read it, scale it and add it into
// fp32 accumulators held in registers.  Two TMEM buffers alternate, so the
// MMAs of block kb+1 run while block kb is promoted.
//
// Layout is swap-AB as in the bf16 kernel: weights in the MMA's M slot,
// tokens in N.  One tile = group g, two 128-row weight boxes, one token block
// of N <= 96 tokens (each epilogue thread keeps 2 x 48 fp32 accumulators in
// registers; with ten warps a thread can hold at most 168 registers):
//   GATEUP: acc0 = gate rows [128 mb, +128) of W13_g, acc1 = the up rows (+I);
//           the tile ends with act = SiLU(acc0) * acc1 quantised to e4m3 per
//           token over its 128 columns (one 1 x 128 tile of the down GEMM's K)
//   DOWN:   acc0 / acc1 = rows [256 mb, +128) / [256 mb + 128, +128) of W2_g;
//           the tile ends with y in bf16
//
// Activation scales sit K-block-major ([K/128][rows], fp32), so the scales of
// a tile's tokens for block kb are one contiguous run that TMA brings in with
// the operands.  Group rows start on multiples of 4 (16 bytes of scales).
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0      TMA producer: weight boxes and token rows per stage, the token
//               scales of the same K block into an 8-slot ring (freed by the
//               promotion, while the stage is freed by the MMAs)
//   warp 1      TMEM owner and MMA issuer
//   warps 2..9  promotion + epilogue: warp w reads TMEM lanes 32*(w%4).. and
//               columns [48 h, 48 h + 48), h = (w - 2) / 4
// Every barrier wait is bounded (abort flag, device error word), as in the
// bf16 kernel.
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "gemm_fp8.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int KB = 128;                       // K elements (= bytes) per stage
constexpr uint32_t ROW = 128;                 // bytes per operand row per stage
constexpr int STAGES = 4;
constexpr uint32_t A_BOX = 128 * ROW;         // 16 KB
constexpr uint32_t STAGE_BYTES = 2 * A_BOX + 128 * ROW;   // 48 KB
constexpr int EPI_WARPS = 8;
constexpr int CW = 48;                        // token columns per epilogue warp (N <= 2 CW)
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
// shared memory after the stages: token-scale ring, per-warp premultiplied
// scales, amax exchange, per-warp weight scales, barriers
// token scales ride in their own, deeper ring: an operand stage is freed as soon
// as its MMAs finish, while the scales of that K block stay until promoted
constexpr int SC_SLOTS = 8;
constexpr uint32_t SC_OFF = STAGES * STAGE_BYTES;
constexpr uint32_t PS_OFF = SC_OFF + SC_SLOTS * 128 * 4;
constexpr uint32_t AM_OFF = PS_OFF + EPI_WARPS * 2 * 64 * 4;
constexpr uint32_t WS_OFF = AM_OFF + 2 * 2 * 4 * 64 * 4;   // per warp: the tile's weight scales
constexpr int MAX_KB = 64;                                  // K blocks per tile (K <= 8192)
constexpr uint32_t BAR_OFF = WS_OFF + EPI_WARPS * 2 * MAX_KB * 4;
constexpr size_t SMEM_BYTES = BAR_OFF + 256 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "fp8 GEMM shared memory");

__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (0u << 7) | (0u << 10)                    // A, B format: e4m3
         | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Tile {
  int g, mb, tok0, ntok, nmma;
};

__device__ __forceinline__ void decode(const Fp8GemmArgs& a, int tile, Tile& t) {
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
  t.nmma = (t.ntok + 15) & ~15;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0 && !tc::mbar_try_wait(bar, parity))
    ok = tc::mbar_wait_bounded(bar, parity, abort_flag, tc::globaltimer_ns() + timeout_ns) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Drain wait after an abort: waits up to timeout_ns whatever the abort flag
// says, so this CTA's own loads and MMAs complete before TMEM is freed.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity,
                                           unsigned long long timeout_ns) {
  if ((threadIdx.x & 31) == 0)
    tc::mbar_wait_deadline(bar, parity, tc::globaltimer_ns() + timeout_ns);
  __syncwarp();
}

__device__ __forceinline__ bool lane_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  return tc::mbar_wait_bounded(bar, parity, abort_flag, tc::globaltimer_ns() + timeout_ns);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g * u, 1.0f + __expf(-g));
}

// Max over the 32 lanes of each of 64 columns (v[c] per lane) by recursive
// halving: after the five exchange steps lane l holds the warp maxima of
// columns 2l and 2l + 1 in v[0], v[1].
__device__ __forceinline__ void warp_colmax64(float (&v)[64], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 32 >> step;            // values kept after this step
    const int bit = 16 >> step;             // partner lane distance
    const bool upper = (lane & bit) != 0;   // keeps the upper half of the columns
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, bit);
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

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ Fp8GemmMaps maps, const Fp8GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* sc_ring = reinterpret_cast<float*>(smem + SC_OFF);     // [SC_SLOTS][128]
  float* psc = reinterpret_cast<float*>(smem + PS_OFF);         // [EPI_WARPS][2][64]
  float* amx = reinterpret_cast<float*>(smem + AM_OFF);         // [2 par][2 h][4 q][64]
  float* wsm = reinterpret_cast<float*>(smem + WS_OFF);         // [EPI_WARPS][2][MAX_KB]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* pfull = empty + STAGES;     // [2]
  uint64_t* pempty = pfull + 2;         // [2]
  uint64_t* xam = pempty + 2;           // [2 par][2 h]
  uint64_t* sempty = xam + 4;           // [SC_SLOTS]: scales promoted by every epilogue warp
  uint64_t* drain = sempty + SC_SLOTS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);               // MMAs done
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(pfull + b, 1);
      tc::mbar_init(pempty + b, EPI_WARPS);
    }
    for (int i = 0; i < 4; ++i) tc::mbar_init(xam + i, 128);
    for (int i = 0; i < SC_SLOTS; ++i) tc::mbar_init(sempty + i, EPI_WARPS);
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
    tc::tmem_alloc<1>(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish<1>();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = args.gt.bstart[args.G] * args.m_blocks;
  const int nkb = args.k_blocks;
  const unsigned long long tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    uint32_t kc = 0;
    uint32_t issued = 0, issued_par = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      Tile t;
      decode(args, tile, t);
      const bool second = t.g >= args.E;
      const CUtensorMap* mA = &maps.a[second ? 1 : 0];
      const CUtensorMap* mB = maps.b[second ? 1 : 0];
      const int gl = second ? t.g - args.E : t.g;
      const int a_row0 = gl * args.a_rows_per_group + t.mb * (MODE == GM_GATEUP ? 128 : 256);
      const int a_row1 = a_row0 + args.a1_off;
      const int b_row = __ldg(args.gt.brow + t.g) + t.tok0;
      const uint32_t bytes = 2 * A_BOX + t.nmma * ROW + 128 * 4;
      for (int kb = 0; kb < nkb; ++kb, ++kc) {
        const int stage = kc % STAGES;
        const uint32_t phase = (kc / STAGES) & 1u;
        const int slot = kc % SC_SLOTS;
        if (!warp_wait(empty + stage, phase ^ 1u, abort_flag, tmo)) { ok = false; break; }
        if (!warp_wait(sempty + slot, ((kc / SC_SLOTS) & 1u) ^ 1u, abort_flag, tmo)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* sa = smem + stage * STAGE_BYTES;
          tc::mbar_arrive_expect_tx(full + stage, bytes);
          tc::tma_load_2d(sa, mA, full + stage, kb * KB, a_row0);
          tc::tma_load_2d(sa + A_BOX, mA, full + stage, kb * KB, a_row1);
          int done = 0;
#pragma unroll
          for (int bi = kTokBoxes - 1; bi >= 0; --bi) {
            const int hgt = 16 << bi;
            if (t.nmma & hgt) {
              tc::tma_load_2d(sa + 2 * A_BOX + done * ROW, mB + bi, full + stage, kb * KB,
                              b_row + done);
              done += hgt;
            }
          }
          // 128 token scales of block kb starting at the tile's first row
          tc::tma_load_2d(sc_ring + slot * 128, &maps.sx, full + stage, b_row, kb);
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        __syncwarp();
      }
    }
    if (!ok) {
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) drain_wait(full + s, (issued_par >> s) & 1u, tmo);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t kc = 0;
    bool ok = true, issued_any = false;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      Tile t;
      decode(args, tile, t);
      const uint32_t idesc = idesc_e4m3_f32(128, t.nmma);
      for (int kb = 0; kb < nkb; ++kb, ++kc) {
        const int stage = kc % STAGES;
        const uint32_t phase = (kc / STAGES) & 1u;
        const int pb = kc & 1;
        const uint32_t puse = (kc >> 1) & 1u;
        if (!warp_wait(pempty + pb, puse ^ 1u, abort_flag, tmo)) { ok = false; break; }
        if (!warp_wait(full + stage, phase, abort_flag, tmo)) { ok = false; break; }
        tc::tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = tc::smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t d0 = tmem_base + pb * 256;
#pragma unroll
          for (int kk = 0; kk < KB / 32; ++kk) {
            const uint64_t da0 = tc::smem_desc_sw128(sa + kk * 32);
            const uint64_t da1 = tc::smem_desc_sw128(sa + A_BOX + kk * 32);
            const uint64_t db = tc::smem_desc_sw128(sa + 2 * A_BOX + kk * 32);
            mma_e4m3(d0, da0, db, idesc, kk > 0 ? 1u : 0u);
            mma_e4m3(d0 + 128, da1, db, idesc, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit<1>(empty + stage);   // operands consumed
          tc::mma_commit<1>(pfull + pb);      // partial sums of block kb ready
        }
        issued_any = true;
        __syncwarp();
      }
    }
    if (!ok && issued_any) {
      if (lane == 0) tc::mma_commit<1>(drain);
      __syncwarp();
      drain_wait(drain, 0, tmo);
    }
  } else {
    // ------------------------------------------------------------ promotion + epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int ew = warp - 2;
    float* my_ps = psc + ew * 128;                 // [2][64]: acc0 and acc1 scales
    const uint32_t tl = static_cast<uint32_t>(q * 32) << 16;
    uint32_t kc = 0;
    int tcount = 0;
    bool ok = true;
    const float* wsc = args.w_scale[0];
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++tcount) {
      Tile t;
      decode(args, tile, t);
      const bool second = t.g >= args.E;
      const int gl = second ? t.g - args.E : t.g;
      wsc = second ? args.w_scale[1] : args.w_scale[0];
      // weight-scale rows of acc0 / acc1 in [groups][row blocks][k blocks]
      const int rb = args.a_rows_per_group / 128;
      const int rb0 = gl * rb + t.mb * (MODE == GM_GATEUP ? 1 : 2);
      const int rb1 = rb0 + (MODE == GM_GATEUP ? args.a1_off / 128 : 1);
      const bool rb1ok = MODE == GM_GATEUP || t.mb * 2 + 1 < rb;
      const int c0 = h * CW;
      const bool active = c0 < t.nmma;
      // the tile's weight scales, one read per tile instead of one per K block
      float* my_ws = wsm + ew * 2 * MAX_KB;
      for (int k = lane; k < nkb; k += 32) {
        my_ws[k] = __ldg(wsc + static_cast<size_t>(rb0) * nkb + k);
        my_ws[MAX_KB + k] = rb1ok ? __ldg(wsc + static_cast<size_t>(rb1) * nkb + k) : 0.f;
      }
      __syncwarp();
      float a0[CW], a1[CW];
#pragma unroll
      for (int i = 0; i < CW; ++i) { a0[i] = 0.f; a1[i] = 0.f; }
      for (int kb = 0; kb < nkb; ++kb, ++kc) {
        const int pb = kc & 1;
        const uint32_t puse = (kc >> 1) & 1u;
        if (!warp_wait(pfull + pb, puse, abort_flag, tmo)) { ok = false; break; }
        tc::tc_fence_after();
        if (active) {
          const float sw0 = my_ws[kb];
          const float sw1 = my_ws[MAX_KB + kb];
          const float* sx = sc_ring + (kc % SC_SLOTS) * 128 + c0;
          my_ps[lane] = sw0 * sx[lane];
          my_ps[64 + lane] = sw1 * sx[lane];
          if (lane + 32 < CW) {
            my_ps[lane + 32] = sw0 * sx[lane + 32];
            my_ps[64 + lane + 32] = sw1 * sx[lane + 32];
          }
          __syncwarp();
          const uint32_t tb = tmem_base + pb * 256 + tl + c0;
#pragma unroll
          for (int j = 0; j < CW / 16; ++j) {
            if (c0 + 16 * j < t.nmma) {
              uint32_t p0[16], p1[16];
              tc::tmem_ld16(tb + 16 * j, p0);
              tc::tmem_ld16(tb + 128 + 16 * j, p1);
              tc::tmem_wait_ld(p0, p1);
              const float4* s0v = reinterpret_cast<const float4*>(my_ps + 16 * j);
              const float4* s1v = reinterpret_cast<const float4*>(my_ps + 64 + 16 * j);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 s0 = s0v[i], s1 = s1v[i];
                float* x0 = a0 + 16 * j + 4 * i;
                float* x1 = a1 + 16 * j + 4 * i;
                ffma2(x0[0], x0[1], __uint_as_float(p0[4 * i]), __uint_as_float(p0[4 * i + 1]),
                      s0.x, s0.y);
                ffma2(x0[2], x0[3], __uint_as_float(p0[4 * i + 2]),
                      __uint_as_float(p0[4 * i + 3]), s0.z, s0.w);
                ffma2(x1[0], x1[1], __uint_as_float(p1[4 * i]), __uint_as_float(p1[4 * i + 1]),
                      s1.x, s1.y);
                ffma2(x1[2], x1[3], __uint_as_float(p1[4 * i + 2]),
                      __uint_as_float(p1[4 * i + 3]), s1.z, s1.w);
              }
            }
          }
          __syncwarp();
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(pempty + pb);
          tc::mbar_arrive(sempty + kc % SC_SLOTS);
        }
      }
      if (!ok) break;
      // ---------------------------------------------------------- tile end
      const size_t orow0 = static_cast<size_t>(__ldg(args.gt.orow + t.g) + t.tok0) + c0;
      if (MODE == GM_GATEUP) {
        // act = SiLU(gate) * up, then e4m3 per token over the CTA's 128
        // columns.  All four warps of a half take part in the amax exchange
        // on every tile (inactive ones with nothing to store), so its
        // barrier phases and buffer parity stay in step.
        float v[64];
        if (active) {
#pragma unroll
          for (int i = 0; i < CW; ++i) a0[i] = silu_mul(a0[i], a1[i]);
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = i < CW ? fabsf(a0[i]) : 0.f;
          warp_colmax64(v, lane);                  // v[0..1]: warp max of cols 2l, 2l+1
        }
        const int par = tcount & 1;
        float* am = amx + (par * 2 + h) * 4 * 64;
        if (active) {
          am[q * 64 + 2 * lane] = v[0];
          am[q * 64 + 2 * lane + 1] = v[1];
        }
        uint64_t* xb = xam + par * 2 + h;
        tc::mbar_arrive(xb);
        if (!lane_wait(xb, (tcount >> 1) & 1u, abort_flag, tmo)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (active) {
          const int col = t.mb * 128 + q * 32 + lane;
          uint8_t* oq = static_cast<uint8_t*>(args.out) + orow0 * args.out_ld + col;
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            const float m = fmaxf(fmaxf(am[i], am[64 + i]), fmaxf(am[128 + i], am[192 + i]));
            const float inv = m > 0.f ? 448.0f / m : 0.f;
            if (c0 + i < t.ntok) {
              const __nv_fp8_storage_t b =
                  __nv_cvt_float_to_fp8(a0[i] * inv, __NV_SATFINITE, __NV_E4M3);
              oq[static_cast<size_t>(i) * args.out_ld] = b;
            }
          }
          // scales of this tile's tokens for K block mb of the down GEMM
          if (q == 0) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int i = 2 * lane + u;
              const float m = fmaxf(fmaxf(am[i], am[64 + i]), fmaxf(am[128 + i], am[192 + i]));
              if (i < CW && c0 + i < t.ntok)
                args.out_scale[static_cast<size_t>(t.mb) * args.out_scale_ld + orow0 + i] =
                    m / 448.0f;
            }
          }
        }
      } else {
        if (active) {
          const int col0 = t.mb * 256 + q * 32 + lane, col1 = col0 + 128;
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(args.out) + orow0 * args.out_ld;
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            if (c0 + i < t.ntok) {
              if (col0 < args.out_cols)
                o[static_cast<size_t>(i) * args.out_ld + col0] = __float2bfloat16_rn(a0[i]);
              if (col1 < args.out_cols)
                o[static_cast<size_t>(i) * args.out_ld + col1] = __float2bfloat16_rn(a1[i]);
            }
          }
        }
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<1>(tmem_base, TMEM_COLS);
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
  const cuuint32_t box[2] = {128, 1};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), gdim, gstride,
             box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  TraceScope tr(stream, MODE == GM_GATEUP ? "gemm_fp8_gateup_swiglu" : "gemm_fp8_down");
  fp8_gemm_kernel<MODE><<<num_sms(), THREADS, SMEM_BYTES, stream>>>(maps, args);
  return launch_status();
}

}  // namespace

bool make_fp8_maps(Fp8GemmMaps* m, const void* a0, uint64_t a0_rows, const void* a1,
                   uint64_t a1_rows, const void* b, uint64_t b_rows, const float* sx,
                   uint64_t k) {
  if (!tmap_e4m3(&m->a[0], a0, a0_rows, k, 128)) return false;
  if (a1) {
    if (!tmap_e4m3(&m->a[1], a1, a1_rows, k, 128)) return false;
  } else {
    m->a[1] = m->a[0];
  }
  for (int i = 0; i < kTokBoxes; ++i) {
    if (!tmap_e4m3(&m->b[0][i], b, b_rows, k, 16u << i)) return false;
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
