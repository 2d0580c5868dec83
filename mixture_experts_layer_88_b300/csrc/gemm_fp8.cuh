// Host-side interface of the FP8 block-scaled expert GEMMs (internal).
#pragma once

#include <cuda.h>
#include "common.cuh"
#include "gemm_tc.cuh"

namespace moe {

// Largest token block of one FP8 tile: the group table is built with blocks of
// at most this many tokens.
constexpr int kFp8TileTokens = 160;

struct Fp8GemmMaps {
  CUtensorMap a[2];               // e4m3 weights: routed (0) / shared (1), boxes of 64 (GATEUP) or 128 rows
  CUtensorMap b[2][kTokBoxes];    // e4m3 token rows, boxes of 8 << i rows (both entries alike)
  CUtensorMap sx;                 // fp32 token scales [K/128, rows], runs of 128 rows
};

struct Fp8GemmArgs {
  GroupTable gt;
  int G, E;
  int m_blocks;                 // pair tiles per group: GATEUP I / 128; DOWN ceil(d / 256)
  int a_rows_per_group;         // 2I (GATEUP) or d (DOWN)
  int a1_off;                   // GATEUP: row offset of the up rows (I); DOWN: unused
  int k_blocks;                 // K / 128
  const float* w_scale[2];      // weight block scales, routed / shared: [groups][rows/128][K/128]
  int out_ld;                   // GATEUP: I (e4m3 act); DOWN: d (bf16 y)
  int out_cols;
  void* out;
  float* out_scale;             // GATEUP: act scales [I/128][out_scale_ld]
  long long out_scale_ld;
  unsigned* status;
  unsigned long long timeout_ns;
};

// a0/a1: routed / shared e4m3 weights [rows, k]; b: e4m3 token rows [b_rows, k]
// with scales sx [k/128, b_rows] (b_rows a multiple of 4).
bool make_fp8_maps(Fp8GemmMaps* m, const void* a0, uint64_t a0_rows, const void* a1,
                   uint64_t a1_rows, uint32_t a_box_rows, const void* b, uint64_t b_rows,
                   const float* sx, uint64_t k);

moe_status_t launch_fp8_gemm(int mode, const Fp8GemmMaps& maps, const Fp8GemmArgs& args,
                             cudaStream_t stream);

}  // namespace moe
