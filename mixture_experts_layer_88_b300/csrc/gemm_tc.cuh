// Host-side interface of the tcgen05 grouped GEMM (internal).
#pragma once

#include <cuda.h>
#include "common.cuh"

namespace moe {

// GATEUP: gate/up GEMM with the SwiGLU epilogue (act out).  DOWN: down GEMM
// (y out).  ROUTER: router logits.  GATEUP_H: the gate/up GEMM writing the
// pre-activations h = [gate | up] instead of act (training forward).  DGRAD:
// the DOWN tiling with the weight operand read MN-major, for input gradients
// (dact = dy W2 and dxp = dh W13): A is the weight matrix of a group viewed as
// [K rows, M columns].
enum GemmMode : int { GM_GATEUP = 0, GM_DOWN = 1, GM_ROUTER = 2, GM_GATEUP_H = 3, GM_DGRAD = 4 };

// Per-group table on the device (G groups; bstart has G+1 entries).
struct GroupTable {
  const int* rows;    // tokens of the group
  const int* brow;    // first row of the group in the B (token) source
  const int* orow;    // first output row of the group
  const int* bs;      // token-block size of the group (multiple of 16, <= 256)
  const int* bstart;  // exclusive prefix of token blocks per group
};

struct GemmArgs {
  GroupTable gt;
  int G;                     // groups (grouped modes)
  int E;                     // groups g < E read A/B map 0, others map 1
  int m_blocks;              // weight-row blocks per group (a block spans the CTA pair)
  int a_rows_per_group;      // rows of A per group (2I or d; 0 in router mode)
  int a1_off;                // GATEUP: row offset of the up rows (I)
  int k_blocks;              // K / 64
  int k_splits;              // router mode: K splits (1 otherwise)
  int k_per_split;           // k-blocks per split
  int router_T;              // router mode: tokens
  int router_bs;             // router mode: token-block size
  int router_nb;             // router mode: token blocks
  int out_ld;                // output leading dimension (elements)
  int out_cols;              // valid output columns
  long long out_split_stride;  // router mode: elements between split partials
  void* out;
  int* tile_counter;         // expert GEMMs: next tile to hand out, 0 at launch
  const float* w_scale[2];   // W8: routed / shared 128x128 block scales [groups, rows/128, K/128]
  int scale_kb;              // W8: K / 128
  unsigned* status;
  unsigned long long timeout_ns;  // bound of every barrier wait
};

// Tensor map of a row-major bf16 matrix [rows, cols] read in boxes of
// {64 columns, box_rows rows} with 128-byte swizzle.  False on failure.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);

// Token-operand boxes come in five heights h0 << i, so a CTA's share of a
// token block is fetched with at most five TMA loads: h0 = 16 (16..256 rows)
// when one CTA loads the whole block (router), h0 = 8 (8..128 rows) when
// each CTA of a pair loads half of a block (expert GEMMs).
constexpr int kTokBoxes = 5;
constexpr uint32_t kTokBox0Single = 16;
constexpr uint32_t kTokBox0Pair = 8;

struct GemmMaps {
  CUtensorMap a[2];               // weight operand: routed (0) / shared (1), 128-row boxes
  CUtensorMap b[2][kTokBoxes];    // token operand: routed (0) / shared (1), box 16 << i rows
};

// Fills `m`: a[i] over the [a_rows[i], k] weight matrices in boxes of
// a_box_rows rows, b[i][*] over the [b_rows[i], k] token matrices in boxes of
// tok_box0 << j rows (a null pointer reuses entry 0).
bool make_gemm_maps(GemmMaps* m, const void* a0, uint64_t a0_rows, const void* a1,
                    uint64_t a1_rows, uint32_t a_box_rows, const void* b0, uint64_t b0_rows,
                    const void* b1, uint64_t b1_rows, uint64_t k, uint32_t tok_box0);

// Launches a persistent grouped GEMM on at most `grid` CTAs: GATEUP and DOWN
// on CTA pairs (clusters of two), ROUTER on single CTAs.  w8: the expert
// weights are e4m3 (maps.a from make_tmap_e4m3) with args.w_scale block
// scales, dequantised to bf16 on the way to the tensor cores.  small: token
// blocks of at most 64 tokens (decode batches), a deeper ring of smaller stages.
moe_status_t launch_gemm_tc(int mode, const GemmMaps& maps, const GemmArgs& args, int grid,
                            cudaStream_t stream, bool w8 = false, bool small = false,
                            const char* trace_name = nullptr);

// Tensor map of a row-major e4m3 matrix [rows, cols] read in boxes of {64
// columns, 128 rows} with 64-byte swizzle (the dequantisation warps read it,
// one 64-byte row per thread).
bool make_tmap_e4m3(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);

// Where the rows of each group live.  Routed group g < E: counts[g] rows
// starting at offsets[g] in both the token source and the outputs.  Shared
// expert s: T rows read from source row shared_src and written from output
// row shared_out0 + s * shared_stride.  Token blocks hold at most max_bs rows.
struct GroupLayout {
  int shared_src, shared_out0, shared_stride, max_bs;
};

// Builds the group table of the expert GEMMs from the dispatch offsets (E+1
// entries; group g has counts[g] rows, or offsets[g+1] - offsets[g] when
// counts is NULL), and zeroes the two tile counters (gate/up, down) that
// follow bstart (bstart[G + 1], bstart[G + 2]):
// groups 0..E-1 are routed experts, E..E+S-1 the shared experts.  Writes
// rows, brow (token source row), orow (output row), bs, bstart.
moe_status_t launch_build_groups(const int* offsets, const int* counts, int T, int E, int S,
                                 GroupLayout lay, int* rows, int* brow, int* orow, int* bs,
                                 int* bstart, cudaStream_t stream);

// Weight-gradient GEMM (wgrad_gemm_kernel): dW[g] [M, N] = sum over the
// group's tokens j of A[arow_g + j, 0..M)^T B[brow_g + j, 0..N), bf16 out.
// Routed group e: counts[e] tokens, A rows from poff[e] (padded layout: zero
// rows up to the next multiple of 16), B rows from offsets[e].  Shared expert
// s: T tokens, A rows from poff[E] + s * T16, B rows from b_sh0 + s * b_shs.
struct WgradArgs {
  const int* counts;
  const int* offsets;
  const int* poff;
  int E, S, T, T16;
  int b_sh0, b_shs;
  int m_blocks, n_blocks;     // ceil(M / 256), ceil(N / 256)
  int M, N;
  long long out_gstride;      // elements between groups' dW (M * N)
  void* out_routed;           // [E, M, N]
  void* out_shared;           // [S, M, N]
  int* tile_counter;          // 0 at launch
  unsigned* status;
  unsigned long long timeout_ns;
};
struct WgradMaps {
  CUtensorMap a;       // padded output-gradient rows [rows, M], boxes {64, 64}
  CUtensorMap b[2];    // routed / shared forward rows [rows, N], boxes {64, 64}
};
moe_status_t launch_wgrad(const WgradMaps& maps, const WgradArgs& args, cudaStream_t stream,
                          const char* trace_name = "gemm_wgrad");

// Backward row layout and the input-gradient GEMMs' group table: poff[e] =
// sum of round_up(counts[j], 16) over j < e (E+1 entries, poff[E] = start of
// the shared segments, T16 = round_up(T, 16) rows each); group g < E has
// counts[g] rows at brow = orow = poff[g], shared expert s has T rows at
// poff[E] + s * T16; token blocks of at most 256.  Zeroes `counters` (4 ints).
moe_status_t launch_build_bwd_groups(const int* counts, int T, int E, int S, int* poff, int* rows,
                                     int* brow, int* orow, int* bs, int* bstart, int* counters,
                                     cudaStream_t stream);

int num_sms();

// Fused router (router_fused.cu): logits, score, biased top-K and gates in one
// kernel; the K splits of a token block form a thread-block cluster of ck
// CTAs and reduce through distributed shared memory.  Applies to bf16 tokens
// with E <= 256 experts (d a multiple of 64).
struct FusedRouterPlan {
  int ck;          // CTAs per cluster = K splits
  int nb;          // tokens per block (multiple of 16, <= 256)
  int kps;         // K steps (64 wide) per split
  int nblocks;     // token blocks
  int nclusters;   // clusters launched (each walks blocks cid, cid + nclusters, ...)
};
bool fused_router_applies(int act_dtype, int d, int E);
// False when the fused router does not apply or no cluster shape fits.
bool fused_router_plan(int T, int d, int E, FusedRouterPlan* p);
// inv_rms not null: the layer behind its RMSNorm.  centroids must then be the
// weighted centroids w * e_i (launch_fold_centroids); the logits are scaled by
// 1 / sqrt(mean(x^2) + norm_eps) of each raw token row x, written to inv_rms [T].
moe_status_t launch_router_fused(const FusedRouterPlan& p, const void* x, const void* centroids,
                                 const float* bias, int T, int d, int E, int K, int score_func,
                                 int normalize, int n_groups, int topk_groups, int32_t* idx,
                                 float* gates, float* scores, float norm_eps, float* inv_rms,
                                 unsigned* status, unsigned long long timeout_ns,
                                 cudaStream_t stream);

// Token-block size and count for `rows` tokens: blocks of at most max_bs
// (256 or 128) tokens, balanced, each a multiple of 16.
__host__ __device__ inline void token_blocks(int rows, int* bs, int* nb, int max_bs = 256) {
  if (rows <= 0) { *bs = 16; *nb = 0; return; }
  int n0 = (rows + max_bs - 1) / max_bs;
  int b = ((rows + n0 - 1) / n0 + 15) / 16 * 16;
  *bs = b;
  *nb = (rows + b - 1) / b;
}

}  // namespace moe
