// Fused router of a DeepSeekMoE layer on the 5th-generation tensor cores.  One
// kernel computes the affinity logits u_t . e_i ("DeepSeekMoE架构解析", section
// 2.1, eq. (15)) and, per token, the score, the biased top-K and the gates
// (eqs. (13)-(16); node-limited groups of section 2.3), and writes only idx
// and gates (and, for the training forward, every expert's score).  The logits
// never leave the chip.
//
// Behind the layer's RMSNorm (section 4.1) the same kernel reads the raw
// tokens x: its centroids are the weighted centroids w * e_i (made by
// launch_fold_centroids), the idle mover warps sum x^2 of every token from the
// operand tiles while the MMAs run, and the logits are scaled by
// inv_rms = 1 / sqrt(mean(x^2) + eps), since (x * inv_rms * w) . e_i =
// inv_rms * (x . (w * e_i)).  inv_rms is written out for the dispatch.
//
// Tiling: the experts sit in the MMA's M slot (one accumulator of 128 experts,
// two for E <= 256), a block of nb <= 256 tokens in its N slot.  The ck CTAs
// of a thread-block cluster split the hidden dimension of one token block:
// CTA r accumulates, in TMEM, the partial logits over K steps
// [r kps, (r+1) kps).  The partials are reduced through distributed shared
// memory: CTA r owns tokens [r nown, (r+1) nown) of the block (nown = nb / ck,
// a multiple of 8); every CTA stores its partial of each other CTA's tokens
// into that CTA's shared memory (16-byte st.shared::cluster, expert-major
// rows), one cluster barrier later the owner adds the ck partials in rank
// order (partial 0 + partial 1 + ...), in place, and four lanes per token
// select the experts from shared memory.
//
// Warp roles (320 threads): warp 0 TMA producer (per 64-wide K step the
// centroid boxes and the block's token rows), warp 1 TMEM owner and MMA
// issuer, warps 2..9 the movers (two per TMEM lane quadrant: TMEM reads,
// partial exchange, sums; behind the RMSNorm also the sums of squares); all
// ten warps select.  The reduction buffers reuse the operand ring, idle by
// then.  Every mbarrier wait is bounded; a CTA that times out skips its
// remaining work but still passes every cluster barrier, so its cluster never
// waits on it, and it lets its own loads land and its MMAs finish before it
// frees TMEM.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_tc.cuh"
#include "router_select.cuh"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int FR_BK = 64;                                  // K elements per stage
constexpr uint32_t FR_ROW = 128;                           // bytes per operand row per stage
constexpr int FR_MAX_STAGES = 6;                           // operand ring: 3..6 stages
constexpr uint32_t FR_A_BOX = 128 * FR_ROW;                // 16 KB: 128 centroid rows
constexpr uint32_t FR_RING = 220 * 1024;                   // operand ring (stages of A boxes + B rows)
constexpr uint32_t FR_EPI_MAX = 220 * 1024;              // reduction buffers (alias the ring)
constexpr int FR_WARPS = 10;
constexpr int FR_MOVERS = 8;                               // warps 2..9
constexpr int FR_TB = 6;                                   // tokens a warp selects at once
constexpr int FR_THREADS = FR_WARPS * 32;
constexpr uint32_t FR_AREA = FR_EPI_MAX > FR_RING ? FR_EPI_MAX : FR_RING;
constexpr size_t FR_SMEM = 1024 + FR_AREA + 128 + 256 * 4;   // + barriers + bias
constexpr uint32_t FR_TMEM_COLS = 512;
constexpr int FR_TOKBOXES = 5;                             // token boxes of 16 << i rows

struct FusedMaps {
  CUtensorMap a;                  // centroids [E, d], boxes of 64 columns x 128 rows
  CUtensorMap b[FR_TOKBOXES];     // tokens [T, d], boxes of 64 columns x (16 << i) rows
};

struct FusedArgs {
  int T, E, K, nacc, epad, d;
  int k_blocks, kps, ck, nb, nown, nblocks, nclusters;
  int nstages;                    // operand ring depth
  uint32_t stage_bytes, b_off;    // bytes per stage; offset of the token rows in a stage
  int stride;                     // row stride (floats) of the logits buffer
  uint32_t ss_off;                // byte offset of the sum-of-squares slots [ck][nown]
  uint32_t inv_off;               // byte offset of the owned tokens' inv_rms [nown]
  const float* bias;
  int score_func, normalize, n_groups, topk_groups;
  int32_t* idx;
  float* gates;
  float* scores;
  float eps;
  float* inv_rms;                 // not null: behind the RMSNorm (see header)
  unsigned* status;
  unsigned long long timeout_ns;
};

// Bounded wait by lane 0, result broadcast to the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0 && !tc::mbar_try_wait(bar, parity))
    ok = tc::mbar_wait_bounded(bar, parity, abort_flag, tc::globaltimer_ns() + timeout_ns) ? 1
                                                                                            : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded wait of a single thread (the producer and MMA loops run on one thread).
__device__ __forceinline__ bool thread_wait(uint64_t* bar, uint32_t parity,
                                            volatile int* abort_flag,
                                            unsigned long long timeout_ns) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  return tc::mbar_wait_bounded(bar, parity, abort_flag, tc::globaltimer_ns() + timeout_ns);
}

// Drain wait after an abort: bounded by the deadline alone.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity,
                                           unsigned long long timeout_ns) {
  if ((threadIdx.x & 31) == 0)
    tc::mbar_wait_deadline(bar, parity, tc::globaltimer_ns() + timeout_ns);
  __syncwarp();
}

// ---------------------------------------------------------------- selection
// Approximate exponential and reciprocal (the hardware instructions, about
// 2 ulp): the scores they give differ from the correctly rounded ones by a few
// fp32 ulps, far below the 1e-5 margin of the key comparisons and of the gates.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Selection of TB tokens by one warp, interleaved so that the tokens' warp
// reductions overlap.  col[b]: token b's logits in shared memory, expert e at
// col[b][e * stride]; ok[b]: the token exists; t[b]: its index.  No
// node-limited groups, any K <= 32; the rules of select_experts: scores by
// eq. (15) or Softmax over all E, keys s + b, K rounds taking the largest key,
// equal keys to the lower index, g = s / sum of the chosen s or s.  Each round
// takes two single-instruction warp reductions: the maximum of the lanes'
// best 32-bit orderable keys, then the minimum expert index among the lanes
// holding that key; only the winning lane rescans its slots (taken slots in a
// bit mask), and the chosen expert's score is recomputed from its logit with
// the same arithmetic.  bias_s: the bias in shared memory.
template <int NPL, int TB>
__device__ __forceinline__ void select_warp(const float* const (&col)[TB], int stride,
                                            const bool (&ok)[TB], const size_t (&t)[TB],
                                            int lane, const float* __restrict__ bias_s, int E,
                                            int K, int score_func, int normalize,
                                            int32_t* __restrict__ idx, float* __restrict__ gates,
                                            float* __restrict__ scores) {
  constexpr float kLog2e = 1.4426950408889634f;
  const bool softmax = score_func == MOE_SCORE_SOFTMAX;
  float m[TB], r[TB];                 // Softmax: maximum logit and 1 / sum
  uint32_t key[TB][NPL];
  uint32_t best[TB], taken[TB];
  int bj[TB];
#pragma unroll
  for (int b = 0; b < TB; ++b) {
    float L[NPL];
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = j * 32 + lane;
      L[j] = e < E ? col[b][e * stride] : -INFINITY;
    }
    m[b] = 0.f;
    r[b] = 1.f;
    if (softmax) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < NPL; ++j) mx = fmaxf(mx, L[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < NPL; ++j) sum += j * 32 + lane < E ? fast_exp2((L[j] - mx) * kLog2e) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      m[b] = mx;
      r[b] = 1.0f / sum;
    }
    best[b] = 0u;
    bj[b] = 0;
    taken[b] = 0u;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = j * 32 + lane;
      const float sc = softmax ? fast_exp2((L[j] - m[b]) * kLog2e) * r[b]
                               : fast_rcp(1.0f + fast_exp2(-L[j] * kLog2e));
      key[b][j] = e < E ? orderable(sc + bias_s[e]) : 0u;
      if (scores && ok[b] && e < E) scores[t[b] * E + e] = sc;
      // this lane's best key and its slot (lower slot = lower expert on equal keys)
      if (key[b][j] > best[b]) { best[b] = key[b][j]; bj[b] = j; }
    }
  }
  int my_e[TB];
  float my_s[TB], sum_sel[TB];
#pragma unroll
  for (int b = 0; b < TB; ++b) { my_e[b] = 0; my_s[b] = 0.f; sum_sel[b] = 0.f; }
  for (int k = 0; k < K; ++k) {
    uint32_t ew[TB];
#pragma unroll
    for (int b = 0; b < TB; ++b) {
      const uint32_t mx = __reduce_max_sync(0xffffffffu, best[b]);
      ew[b] = best[b] == mx ? static_cast<uint32_t>(bj[b] * 32 + lane) : 0xFFFFFFFFu;
    }
#pragma unroll
    for (int b = 0; b < TB; ++b) ew[b] = __reduce_min_sync(0xffffffffu, ew[b]);
#pragma unroll
    for (int b = 0; b < TB; ++b) {
      if (lane == static_cast<int>(ew[b] & 31u)) {
        taken[b] |= 1u << bj[b];
        best[b] = 0u;
        bj[b] = 0;
#pragma unroll
        for (int j = 0; j < NPL; ++j)
          if (!((taken[b] >> j) & 1u) && key[b][j] > best[b]) { best[b] = key[b][j]; bj[b] = j; }
      }
      const float Lw = col[b][static_cast<int>(ew[b]) * stride];
      const float sv = softmax ? fast_exp2((Lw - m[b]) * kLog2e) * r[b]
                               : fast_rcp(1.0f + fast_exp2(-Lw * kLog2e));
      sum_sel[b] += sv;
      if (lane == k) {
        my_e[b] = static_cast<int>(ew[b]);
        my_s[b] = sv;
      }
    }
  }
#pragma unroll
  for (int b = 0; b < TB; ++b) {
    if (ok[b] && lane < K) {
      float g = my_s[b];
      if (normalize) g = sum_sel[b] > 0.f ? my_s[b] / sum_sel[b] : 0.f;
      idx[t[b] * K + lane] = my_e[b];
      gates[t[b] * K + lane] = g;
    }
  }
}

template <int NPL>
__global__ void __launch_bounds__(FR_THREADS, 1)
    router_fused_kernel(const __grid_constant__ FusedMaps maps, const FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + FR_AREA);
  uint64_t* empty = full + FR_MAX_STAGES;
  uint64_t* tfull = empty + FR_MAX_STAGES;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* bias_s = reinterpret_cast<float*>(smem + FR_AREA + 128);   // [E <= 256]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(tc::cluster_ctarank());
  const int cid = blockIdx.x / a.ck;
  const bool prenorm = a.inv_rms != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.nstages; ++s) {
      tc::mbar_init(full + s, 1);
      // released by the MMA commit, and behind the RMSNorm also by one arrival
      // of each mover warp once it has read the stage's token rows
      tc::mbar_init(empty + s, prenorm ? 1 + FR_MOVERS : 1);
    }
    tc::mbar_init(tfull, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane <= FR_TOKBOXES)
    tc::tma_prefetch_desc(lane == 0 ? &maps.a : &maps.b[lane - 1]);
  if (warp == 1) {
    tc::tmem_alloc<1>(tmem_slot, FR_TMEM_COLS);
    tc::tmem_relinquish<1>();
  }
  for (int e = threadIdx.x; e < a.E; e += FR_THREADS) bias_s[e] = __ldg(a.bias + e);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long tmo = a.timeout_ns;
  const int kb0 = rank * a.kps;
  const int kb1 = min(a.k_blocks, kb0 + a.kps);

  // ring position: producer, MMA issuer and movers walk the same stage sequence
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, issued_par = 0;   // producer: stages that received loads, and their parity
  bool mma_issued = false;
  uint32_t tphase = 0;
  // reduction buffers (alias the operand ring): receive slots [ck - 1][epad]
  // rows (the first doubles as the logits buffer: the owner sums in place),
  // or with ck = 1 the logits buffer [epad] rows; then the sum-of-squares
  // slots [ck][nown] and the owned tokens' inv_rms [nown]
  float* lg = reinterpret_cast<float*>(smem);
  float* ssq = reinterpret_cast<float*>(smem + a.ss_off);
  float* invs = reinterpret_cast<float*>(smem + a.inv_off);
  const int quad = warp & 3;                 // TMEM lane quadrant of a mover warp
  const int half = (warp - 2) >> 2;          // which alternate 8-column chunks it takes
  const int mv = threadIdx.x - 64;           // mover thread index 0..255: token column
  const int nch = a.nown >> 3;               // 8-column chunks per owner
  const size_t slot_floats = static_cast<size_t>(a.epad) * a.stride;

  for (int blk = cid; blk < a.nblocks; blk += a.nclusters) {
    const int tok0 = blk * a.nb;
    const int ntok = min(a.nb, a.T - tok0);
    const int nmma = (ntok + 15) & ~15;
    float ss = 0.f;                          // movers: sum of x^2 of token column mv
    if (warp == 0) {
      // ---------------------------------------------------------------- TMA producer
      // (one thread: no warp-collective step between its waits and its loads)
      if (lane == 0 && !*abort_flag) {
        const uint32_t bytes = a.nacc * FR_A_BOX + nmma * FR_ROW;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!thread_wait(empty + stage, phase ^ 1u, abort_flag, tmo)) break;
          {
            uint8_t* sa = smem + stage * a.stage_bytes;
            tc::mbar_arrive_expect_tx(full + stage, bytes);
            tc::tma_load_2d(sa, &maps.a, full + stage, kb * FR_BK, 0);
            if (a.nacc == 2)
              tc::tma_load_2d(sa + FR_A_BOX, &maps.a, full + stage, kb * FR_BK, 128);
            int done = 0;
#pragma unroll
            for (int bi = FR_TOKBOXES - 1; bi >= 0; --bi) {
              const int h = 16 << bi;
              if (nmma & h) {
                tc::tma_load_2d(sa + a.b_off + done * FR_ROW, &maps.b[bi], full + stage,
                                kb * FR_BK, tok0 + done);
                done += h;
              }
            }
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == a.nstages) { stage = 0; phase ^= 1u; }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      if (lane == 0 && !*abort_flag) {   // one thread
        const uint32_t idesc = tc::idesc_bf16_f32(128, nmma);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!thread_wait(full + stage, phase, abort_flag, tmo)) { ok = false; break; }
          tc::tc_fence_after();
          {
            const uint32_t sa = tc::smem_u32(smem + stage * a.stage_bytes);
#pragma unroll
            for (int kk = 0; kk < FR_BK / 16; ++kk) {
              const uint64_t db = tc::smem_desc_sw128(sa + a.b_off + kk * 32);
              const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
              tc::mma_bf16<1>(tmem, tc::smem_desc_sw128(sa + kk * 32), db, idesc, acc);
              if (a.nacc == 2)
                tc::mma_bf16<1>(tmem + 256, tc::smem_desc_sw128(sa + FR_A_BOX + kk * 32), db,
                                idesc, acc);
            }
            tc::mma_commit<1>(empty + stage);
          }
          mma_issued = true;
          if (++stage == a.nstages) { stage = 0; phase ^= 1u; }
        }
        if (ok) tc::mma_commit<1>(tfull);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------------- movers
      if (prenorm && !*abort_flag) {
        // sum of squares of token row mv over this CTA's K slice, from the
        // landed operand tiles (128-byte rows, 16-byte pieces swizzled by
        // row % 8), summed in the row's element order
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!warp_wait(full + stage, phase, abort_flag, tmo)) break;
          if (mv < nmma) {
            const uint8_t* rowp = smem + stage * a.stage_bytes + a.b_off + mv * FR_ROW;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 q = *reinterpret_cast<const uint4*>(rowp + ((c ^ (mv & 7)) << 4));
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(h2[k]);
                ss = fmaf(f.x, f.x, ss);
                ss = fmaf(f.y, f.y, ss);
              }
            }
          }
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(empty + stage);
          if (++stage == a.nstages) { stage = 0; phase ^= 1u; }
        }
      }
      // this CTA's accumulators
      warp_wait(tfull, tphase, abort_flag, tmo);
      tc::tc_fence_after();
    }
    tphase ^= 1u;

    // B0: this block's MMAs are complete in every CTA of the cluster, so every
    // operand ring is free for the reduction buffers
    tc::tc_fence_before();
    tc::cluster_sync_all();
    tc::tc_fence_after();
    const bool live = !*abort_flag;
    if (warp >= 2 && live) {
      const int row = quad * 32 + lane;      // expert row of this lane within a half
      if (a.ck > 1) {
        // this CTA's partials of every other CTA's tokens, both halves, 8
        // tokens per pair of 16-byte stores, into that CTA's receive slot
        for (int i = half; i < (a.ck - 1) * nch; i += 2) {
          const int oc = i / nch;
          const int c = oc < rank ? oc : oc + 1;
          const int jl = (i - oc * nch) * 8;
          const int slot = rank < c ? rank : rank - 1;
          const uint32_t tq = tmem + (static_cast<uint32_t>(quad * 32) << 16) + c * a.nown + jl;
          uint32_t v0[8], v1[8];
          tc::tmem_ld8(tq, v0);
          if (a.nacc == 2) tc::tmem_ld8(tq + 256, v1);
          tc::tmem_wait_ld8(v0);
          if (a.nacc == 2) tc::tmem_wait_ld8(v1);
          const uint32_t dst = tc::mapa_shared(
              tc::smem_u32(lg) +
                  static_cast<uint32_t>((slot * slot_floats + static_cast<size_t>(row) * a.stride +
                                         jl) * 4),
              static_cast<uint32_t>(c));
          tc::st_shared_cluster_v4(dst, v0[0], v0[1], v0[2], v0[3]);
          tc::st_shared_cluster_v4(dst + 16, v0[4], v0[5], v0[6], v0[7]);
          if (a.nacc == 2) {
            const uint32_t d1 = dst + 128u * static_cast<uint32_t>(a.stride) * 4u;
            tc::st_shared_cluster_v4(d1, v1[0], v1[1], v1[2], v1[3]);
            tc::st_shared_cluster_v4(d1 + 16, v1[4], v1[5], v1[6], v1[7]);
          }
        }
      }
      if (prenorm && mv < a.nb) {
        // this CTA's sum of squares of token column mv, to the column's owner
        const int c = mv / a.nown;
        tc::st_shared_cluster_u32(
            tc::mapa_shared(tc::smem_u32(ssq) +
                                static_cast<uint32_t>((rank * a.nown + mv - c * a.nown) * 4),
                            static_cast<uint32_t>(c)),
            __float_as_uint(ss));
      }
    }
    // B1: every partial of this CTA's tokens has arrived (release / acquire)
    tc::cluster_sync_all();
    if (warp >= 2 && live) {
      const int row = quad * 32 + lane;
      if (prenorm) {
        if (mv < a.nown) {
          float q = 0.f;
          for (int src = 0; src < a.ck; ++src) {
            const float x = ssq[src * a.nown + mv];
            q = src == 0 ? x : q + x;
          }
          const float inv = 1.0f / sqrtf(q / static_cast<float>(a.d) + a.eps);
          invs[mv] = inv;
          const int t = tok0 + rank * a.nown + mv;
          if (t < a.T) a.inv_rms[t] = inv;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(FR_MOVERS * 32) : "memory");
      }
      // owner: the ck partials of each owned token added in rank order (in
      // place over the first receive slot), times inv_rms behind the RMSNorm
      for (int i = half; i < nch; i += 2) {
        const int jl = i * 8;
        const uint32_t tq =
            tmem + (static_cast<uint32_t>(quad * 32) << 16) + rank * a.nown + jl;
        uint32_t v0[8], v1[8];
        tc::tmem_ld8(tq, v0);
        if (a.nacc == 2) tc::tmem_ld8(tq + 256, v1);
        tc::tmem_wait_ld8(v0);
        if (a.nacc == 2) tc::tmem_wait_ld8(v1);
        float sc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sc[k] = prenorm ? invs[jl + k] : 1.f;
        for (int h = 0; h < a.nacc; ++h) {
          const uint32_t* own = h == 0 ? v0 : v1;
          const size_t r_off = static_cast<size_t>(h * 128 + row) * a.stride + jl;
          float acc[8];
          for (int src = 0; src < a.ck; ++src) {
            float x[8];
            if (src == rank) {
#pragma unroll
              for (int k = 0; k < 8; ++k) x[k] = __uint_as_float(own[k]);
            } else {
              const float4* p =
                  reinterpret_cast<const float4*>(lg + (src < rank ? src : src - 1) * slot_floats +
                                                  r_off);
              const float4 x0 = p[0], x1 = p[1];
              x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
              x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = src == 0 ? x[k] : acc[k] + x[k];
          }
          if (prenorm) {
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] *= sc[k];
          }
          float4* o = reinterpret_cast<float4*>(lg + r_off);
          o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
          o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (live) {
      const int own0 = tok0 + rank * a.nown;
      if (a.n_groups == 0) {
        // FR_TB owned tokens per warp at a time
        for (int jb = warp * FR_TB; jb < a.nown; jb += FR_WARPS * FR_TB) {
          const float* colp[FR_TB];
          bool ok[FR_TB];
          size_t t[FR_TB];
#pragma unroll
          for (int b = 0; b < FR_TB; ++b) {
            const int jl = jb + b < a.nown ? jb + b : a.nown - 1;
            ok[b] = jb + b < a.nown && own0 + jb + b < a.T;
            t[b] = static_cast<size_t>(own0 + jl);
            colp[b] = lg + jl;
          }
          select_warp<NPL, FR_TB>(colp, a.stride, ok, t, lane, bias_s, a.E, a.K, a.score_func,
                                  a.normalize, a.idx, a.gates, a.scores);
        }
      } else {
        // node-limited groups: one warp per token (select_experts)
        for (int jl = warp; jl < a.nown; jl += FR_WARPS) {
          const int t = own0 + jl;
          if (t >= a.T) break;
          float L[NPL];
#pragma unroll
          for (int j = 0; j < NPL; ++j) {
            const int e = j * 32 + lane;
            L[j] = e < a.E ? lg[e * a.stride + jl] : -INFINITY;
          }
          select_experts<NPL>(L, lane, static_cast<size_t>(t), a.bias, a.E, a.K, a.score_func,
                              a.normalize, a.n_groups, a.topk_groups, a.idx, a.gates, a.scores);
        }
      }
    }
    // the ring's generic accesses are complete before the next block's TMA
    // writes; the next block's B0 orders them against other CTAs' stores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    tc::tc_fence_after();
  }

  // the producer's and MMA issuer's loop state lives in lane 0: share it
  // with the warp, and take one view of the abort flag per warp
  issued = __shfl_sync(0xffffffffu, issued, 0);
  issued_par = __shfl_sync(0xffffffffu, issued_par, 0);
  mma_issued = __shfl_sync(0xffffffffu, mma_issued ? 1 : 0, 0) != 0;
  if (__shfl_sync(0xffffffffu, *abort_flag, 0)) {
    if (warp == 0) {
      for (int s = 0; s < a.nstages; ++s)
        if (issued & (1u << s)) drain_wait(full + s, (issued_par >> s) & 1u, tmo);
    } else if (warp == 1 && mma_issued) {
      if (lane == 0) tc::mma_commit<1>(drain);
      __syncwarp();
      drain_wait(drain, 0, tmo);
    }
  }
  // the last remote stores were ordered by the last block's B1: no CTA
  // accesses another's shared memory after it, so each CTA leaves on its own
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<1>(tmem, FR_TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) atomicOr(a.status, ERRBIT_TIMEOUT);
}

// Layout of the reduction buffers (bytes from the start of shared memory).
// With ck > 1: ck - 1 receive slots of epad expert rows, row stride = 4
// (mod 32) words, so 16-byte row pieces written and read by one lane per
// expert meet no bank conflict (the first slot becomes the logits buffer);
// with ck = 1 only the logits buffer, row stride = 8 (mod 32) words, so the
// four lanes of a token reading experts 4i + q meet no bank conflict.  Then
// the sum-of-squares slots [ck][nown] and inv_rms [nown].
struct FrLayout {
  int stride;
  uint32_t ss_off, inv_off, bytes;
};
FrLayout fr_layout(int nown, int ck, int epad) {
  FrLayout L{};
  const int m = ck > 1 ? 4 : 8;
  L.stride = nown + (((m - nown % 32) % 32) + 32) % 32;
  const size_t rows = static_cast<size_t>(ck > 1 ? ck - 1 : 1) * epad;
  L.ss_off = static_cast<uint32_t>(align_up(rows * L.stride * 4, 16));
  L.inv_off = static_cast<uint32_t>(align_up(L.ss_off + static_cast<size_t>(ck) * nown * 4, 16));
  L.bytes = static_cast<uint32_t>(align_up(L.inv_off + static_cast<size_t>(nown) * 4, 16));
  return L;
}

template <int NPL>
cudaLaunchConfig_t fused_config(int ck, int grid, cudaStream_t stream, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  lc.blockDim = dim3(FR_THREADS, 1, 1);
  lc.dynamicSmemBytes = FR_SMEM;
  lc.stream = stream;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(ck);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return lc;
}

template <int NPL>
bool set_smem_attr() {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && done[dev]) return true;
  if (cudaFuncSetAttribute(router_fused_kernel<NPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(FR_SMEM)) != cudaSuccess)
    return false;
  if (dev < 64) done[dev] = true;
  return true;
}

// Clusters of ck CTAs that fit on the device at once (0: none).
int max_active_clusters(int ck) {
  static int cache[64][4] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int slot = ck == 1 ? 0 : ck == 2 ? 1 : ck == 4 ? 2 : 3;
  if (dev < 64 && cache[dev][slot]) return cache[dev][slot];
  if (!set_smem_attr<8>()) return 0;
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t lc = fused_config<8>(ck, ck, nullptr, at);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, router_fused_kernel<8>, &lc) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (dev < 64 && n > 0) cache[dev][slot] = n;
  return n;
}

template <int NPL>
moe_status_t launch_fused(const FusedMaps& maps, const FusedArgs& a, cudaStream_t stream) {
  if (!set_smem_attr<NPL>()) return MOE_ERR_CUDA;
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t lc = fused_config<NPL>(a.ck, a.nclusters * a.ck, stream, at);
  if (cudaLaunchKernelEx(&lc, router_fused_kernel<NPL>, maps, a) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_status();
}

}  // namespace

bool fused_router_applies(int act_dtype, int d, int E) {
  return act_dtype == MOE_BF16 && E >= 1 && E <= 256 && d % 64 == 0 && d > 0;
}

// Shape of the launch, by a cost model in SM cycles with rates measured on
// B300: each CTA's operands (centroid rows and token rows of its K slice)
// cross from L2 at about 68 B/cycle, the batch's tokens are read from HBM at
// about 3250 B/cycle for the whole GPU (6.5 TB/s at 2 GHz), the partials move
// between the CTAs of a cluster at about 9 B/cycle per SM, and a warp selects
// FR_TB tokens in about 5000 cycles.  Wider token blocks cut the centroid
// traffic, more K splits cut it further but add exchange: for the V3 prefill
// layer (T = 8192) this picks clusters of two CTAs and blocks of 112 tokens.
bool fused_router_plan(int T, int d, int E, FusedRouterPlan* p) {
  if (T <= 0 || !fused_router_applies(MOE_BF16, d, E)) return false;
  constexpr double kL2BytesPerCycle = 68.0, kHbmBytesPerCycle = 3250.0;
  constexpr double kDsmemBytesPerCycle = 9.0, kSelectCycles = 5000.0;
  const int nacc = E > 128 ? 2 : 1;
  const int epad = 128 * nacc;
  const int kb = d / 64;
  const double hbm = static_cast<double>(T) * d * 2 / kHbmBytesPerCycle;
  bool found = false;
  FusedRouterPlan best{};
  double best_cost = 0.0;
  for (int ck = 1; ck <= 8; ck *= 2) {
    const int kps = ceil_div(kb, ck);
    if ((ck - 1) * kps >= kb) continue;                   // a split would be empty
    const int maxc = max_active_clusters(ck);
    if (maxc <= 0) continue;
    // token blocks: multiples of 16 (MMA N) whose share per CTA is whole
    // 8-column chunks, at most 256, and whose reduction buffers fit
    const int step = std::max(16, 8 * ck);
    int nb = std::min(round_up(ceil_div(T, maxc), step), 256 / step * step);
    while (nb >= step && fr_layout(nb / ck, ck, epad).bytes > FR_EPI_MAX) nb -= step;
    if (nb < step) continue;
    const int nblocks = ceil_div(T, nb);
    const int nclusters = std::min(maxc, nblocks);
    const int waves = ceil_div(nblocks, nclusters);
    const int nown = nb / ck;
    const double kloop = waves * static_cast<double>(kps) * (128.0 * nacc + nb) * 128.0 /
                         kL2BytesPerCycle;
    const double exch =
        waves * static_cast<double>(ck - 1) * nown * epad * 4.0 / kDsmemBytesPerCycle;
    const double sel = waves * static_cast<double>(ceil_div(nown, FR_WARPS * FR_TB)) *
                       kSelectCycles;
    const double cost = std::max(kloop, hbm) + exch + sel;
    if (!found || cost < best_cost) {
      found = true;
      best_cost = cost;
      best.ck = ck;
      best.nb = nb;
      best.kps = kps;
      best.nblocks = nblocks;
      best.nclusters = nclusters;
    }
  }
  if (found) *p = best;
  return found;
}

moe_status_t launch_router_fused(const FusedRouterPlan& p, const void* x, const void* centroids,
                                 const float* bias, int T, int d, int E, int K, int score_func,
                                 int normalize, int n_groups, int topk_groups, int32_t* idx,
                                 float* gates, float* scores, float norm_eps, float* inv_rms,
                                 unsigned* status, unsigned long long timeout_ns,
                                 cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  FusedMaps maps{};
  if (!make_tmap_bf16(&maps.a, centroids, E, d, 128)) return MOE_ERR_CUDA;
  for (int i = 0; i < FR_TOKBOXES; ++i)
    if (!make_tmap_bf16(&maps.b[i], x, T, d, 16u << i)) return MOE_ERR_CUDA;
  FusedArgs a{};
  a.T = T;
  a.E = E;
  a.K = K;
  a.nacc = E > 128 ? 2 : 1;
  a.epad = 128 * a.nacc;
  a.k_blocks = d / 64;
  a.kps = p.kps;
  a.ck = p.ck;
  a.nb = p.nb;
  a.nown = p.nb / p.ck;
  a.nblocks = p.nblocks;
  a.nclusters = p.nclusters;
  // operand ring: A boxes (one per 128 experts) then the block's token rows,
  // 1024-byte aligned for the 128-byte swizzle; as many stages as fit
  a.b_off = static_cast<uint32_t>(a.nacc) * FR_A_BOX;
  a.stage_bytes = static_cast<uint32_t>(align_up(a.b_off + static_cast<size_t>(round_up(a.nb, 16)) *
                                                     FR_ROW, 1024));
  a.nstages = std::min<int>(FR_MAX_STAGES, static_cast<int>(FR_RING / a.stage_bytes));
  const FrLayout L = fr_layout(a.nown, p.ck, a.epad);
  a.stride = L.stride;
  a.ss_off = L.ss_off;
  a.inv_off = L.inv_off;
  a.d = d;
  a.eps = norm_eps;
  a.inv_rms = inv_rms;
  a.bias = bias;
  a.score_func = score_func;
  a.normalize = normalize;
  a.n_groups = n_groups;
  a.topk_groups = topk_groups;
  a.idx = idx;
  a.gates = gates;
  a.scores = scores;
  a.status = status;
  a.timeout_ns = timeout_ns;
  TraceScope tr(stream, "router_fused");
  if (E <= 32) return launch_fused<1>(maps, a, stream);
  if (E <= 64) return launch_fused<2>(maps, a, stream);
  if (E <= 128) return launch_fused<4>(maps, a, stream);
  return launch_fused<8>(maps, a, stream);
}

}  // namespace moe
