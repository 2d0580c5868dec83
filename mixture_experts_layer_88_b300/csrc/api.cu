// C ABI of the DeepSeekMoE layer library: argument checks, workspace layout,
// tensor maps, launch sequencing, device error word and kernel tracing.
#include <cuda.h>
#include <string.h>

#include <string>
#include <vector>

#include "common.cuh"
#include "gemm_fp8.cuh"
#include "gemm_tc.cuh"
#include "kernels.cuh"

// Device error word, one per device (module-scope variable).
__device__ unsigned g_moe_status_word;

namespace moe {

unsigned* device_status_word() {
  static unsigned* cached[64] = {nullptr};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cached[dev]) return cached[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_moe_status_word) != cudaSuccess) return nullptr;
  if (dev < 64) cached[dev] = static_cast<unsigned*>(p);
  return static_cast<unsigned*>(p);
}

// ---------------------------------------------------------------- tracing
namespace {
struct TraceRec {
  const char* name;
  cudaEvent_t ev0, ev1;
};
struct TraceState {
  bool on = false;
  std::vector<TraceRec> recs;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
thread_local TraceState g_trace;
}  // namespace

// While the stream is being captured into a CUDA graph the events become
// event-record nodes of the graph, recorded each time the graph runs.
void trace_record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}
void trace_begin(cudaStream_t s, const char* name) {
  if (!g_trace.on) return;
  TraceRec r{name, g_trace.get(), g_trace.get()};
  trace_record(r.ev0, s);
  g_trace.recs.push_back(r);
}
void trace_end(cudaStream_t s) {
  if (!g_trace.on || g_trace.recs.empty()) return;
  trace_record(g_trace.recs.back().ev1, s);
}

// ---------------------------------------------------------------- plans
namespace {

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s per barrier wait
constexpr int kRouterTargetCtas = 148;

size_t esize(int dt) { return dt == MOE_BF16 ? 2 : 4; }

struct RouterPlan {
  int bs, nb, eb, k_blocks, splits, kps;
};

// Router tiles: token blocks x expert blocks x K splits, chosen to fill the
// SMs in one wave: the most tiles that fit, then the largest token blocks
// (fewer re-reads of the centroids), then the fewest splits (fewer partials).
RouterPlan router_plan(const moe_cfg_t& c) {
  RouterPlan p{};
  p.eb = ceil_div(c.E, 256);
  p.k_blocks = c.d / 64;
  const int sms = kRouterTargetCtas;
  int best_tiles = -1;
  for (int s = 1; s <= 16 && s <= p.k_blocks; ++s) {
    const int nb_max = sms / (p.eb * s);
    if (nb_max < 1) break;
    int bs = round_up(ceil_div(c.T > 0 ? c.T : 1, nb_max), 16);
    if (bs > 256) continue;                 // too few blocks for T with s splits
    const int nb = ceil_div(c.T > 0 ? c.T : 1, bs);
    const int kps = ceil_div(p.k_blocks, s);
    const int splits = ceil_div(p.k_blocks, kps);
    const int tiles = nb * p.eb * splits;
    if (tiles > best_tiles || (tiles == best_tiles && bs > p.bs)) {
      best_tiles = tiles;
      p.bs = bs;
      p.nb = nb;
      p.kps = kps;
      p.splits = splits;
    }
  }
  if (best_tiles < 0) {                     // more tokens than one wave holds
    token_blocks(c.T, &p.bs, &p.nb);
    p.kps = p.k_blocks;
    p.splits = 1;
  }
  return p;
}

size_t route_ws(const moe_cfg_t& c) {
  if (c.act_dtype == MOE_BF16) {
    const RouterPlan p = router_plan(c);
    return align_up(static_cast<size_t>(p.splits) * c.T * c.E * sizeof(float), 256);
  }
  return align_up(static_cast<size_t>(c.T) * c.E * sizeof(float), 256);
}
size_t dispatch_ws(const moe_cfg_t& c) {
  return align_up(static_cast<size_t>(ceil_div(c.T, kDispatchChunk)) * c.E * sizeof(int32_t) + 4,
                  256);
}
size_t experts_ws(const moe_cfg_t& c) {
  const size_t G = static_cast<size_t>(c.E) + c.S;
  // group table (5 x (G+1) int32) + two tile counters after bstart
  return align_up((5 * (G + 1) + 2) * sizeof(int32_t), 256);
}

// FP8 layers: rows of expert e start at offsets[e], a multiple of 4 (the
// scales of a token block are a 16-byte aligned fp32 run); the shared
// experts' input rows sit at a fixed row P after every routed row, and their
// outputs at P + s * Tp.
struct Fp8Rows {
  long long P, Tp, rows_in, rows_out;
};

bool is_fp8(const moe_cfg_t& c) { return c.wgt_dtype == MOE_E4M3; }

// The W8A16 path of an FP8 layer keeps every activation in bf16 and uses the
// bf16 layer's row layout: the same cfg with bf16 weights describes it.
moe_cfg_t bf16_layout(const moe_cfg_t& c) {
  moe_cfg_t v = c;
  v.wgt_dtype = MOE_BF16;
  return v;
}

Fp8Rows fp8_rows(const moe_cfg_t& c) {
  Fp8Rows r;
  const long long TK = static_cast<long long>(c.T) * c.K;
  r.P = (TK + 3LL * c.E + 3) / 4 * 4;
  r.Tp = (c.T + 3LL) / 4 * 4;
  r.rows_in = r.P + r.Tp;
  r.rows_out = r.P + c.S * r.Tp;
  return r;
}

struct ForwardLayout {
  size_t route, dispatch, experts, offsets, perm, pos, xp, act, y, total;
  size_t xs, act_s;   // FP8 layers: activation scales
};

ForwardLayout forward_layout(const moe_cfg_t& c) {
  ForwardLayout L{};
  const size_t es = esize(c.act_dtype);
  const size_t TK = static_cast<size_t>(c.T) * c.K;
  const size_t R = TK + static_cast<size_t>(c.S) * c.T;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes, 256);
    return o;
  };
  L.route = take(route_ws(c));
  L.dispatch = take(dispatch_ws(c));
  L.experts = take(experts_ws(c));
  L.offsets = take((c.E + 1) * sizeof(int32_t));
  // perm_tok spans the row space of the routed rows (padded in FP8 layers)
  L.perm = take((is_fp8(c) ? static_cast<size_t>(fp8_rows(c).P) : TK) * sizeof(int32_t));
  L.pos = take(TK * sizeof(int32_t));
  if (is_fp8(c)) {
    const Fp8Rows fr = fp8_rows(c);
    L.xp = take(static_cast<size_t>(fr.rows_in) * c.d);
    L.xs = take(static_cast<size_t>(fr.rows_in) * (c.d / 128) * sizeof(float));
    L.act = take(static_cast<size_t>(fr.rows_out) * c.I);
    L.act_s = take(static_cast<size_t>(fr.rows_out) * (c.I / 128) * sizeof(float));
    L.y = take(static_cast<size_t>(fr.rows_out) * c.d * 2);
  } else {
    L.xp = take(TK * c.d * es);
    L.act = take(R * c.I * es);
    L.y = take(R * c.d * es);
  }
  L.total = off;
  return L;
}

// Pre-normed forward: the forward's workspace, then the normalised tokens
// (the shared experts' input), the weighted centroids w * e_i and inv_rms.
struct PrenormLayout {
  size_t xs, ew, inv, total;
};
int centroid_dtype(const moe_cfg_t& c) { return c.wgt_dtype == MOE_E4M3 ? MOE_BF16 : c.wgt_dtype; }
PrenormLayout prenorm_layout(const moe_cfg_t& c) {
  PrenormLayout L{};
  L.xs = forward_layout(c).total;
  L.ew = L.xs + align_up(static_cast<size_t>(c.T) * c.d * esize(c.act_dtype), 256);
  L.inv = L.ew + align_up(static_cast<size_t>(c.E) * c.d * esize(centroid_dtype(c)), 256);
  L.total = L.inv + align_up(static_cast<size_t>(c.T) * sizeof(float), 256);
  return L;
}
size_t prenorm_ws(const moe_cfg_t& c) { return prenorm_layout(c).total; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_ptrs(const moe_cfg_t& c, std::initializer_list<const void*> dtype_ptrs,
                        std::initializer_list<const void*> other_ptrs) {
  for (const void* p : dtype_ptrs) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (c.act_dtype == MOE_BF16 && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  for (const void* p : other_ptrs)
    if (!p) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return MOE_OK;
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename P>
P* at(void* base, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(base) + off);
}

// ---------------------------------------------------------------- step bodies (no checks)

// row_scale [T] (optional): each token's logits are multiplied by it (the
// layer behind its RMSNorm, routed from the raw tokens; two-kernel router).
moe_status_t do_route(const moe_cfg_t& c, const void* x, const void* centroids,
                      const float* bias, int32_t* idx, float* gates, void* ws,
                      cudaStream_t st, float* scores = nullptr,
                      const float* row_scale = nullptr) {
  if (c.act_dtype == MOE_BF16) {
    // E <= 256: one fused kernel, logits reduced on chip
    FusedRouterPlan fp{};
    if (!row_scale && fused_router_plan(c.T, c.d, c.E, &fp))
      return launch_router_fused(fp, x, centroids, bias, c.T, c.d, c.E, c.K, c.score_func,
                                 c.normalize, c.n_groups, c.topk_groups, idx, gates, scores, 0.f,
                                 nullptr, device_status_word(), kWaitTimeoutNs, st);
    // otherwise the split-K router GEMM into fp32 partials, then the top-K kernel
    const RouterPlan p = router_plan(c);
    float* partial = static_cast<float*>(ws);
    GemmMaps maps{};
    if (!make_gemm_maps(&maps, centroids, c.E, nullptr, 0, 128, x, c.T, nullptr, 0, c.d,
                        kTokBox0Single))
      return MOE_ERR_CUDA;
    GemmArgs a{};
    a.G = 1;
    a.E = 1;
    a.m_blocks = p.eb;
    a.a_rows_per_group = 0;
    a.a1_off = 128;
    a.k_blocks = p.k_blocks;
    a.k_splits = p.splits;
    a.k_per_split = p.kps;
    a.router_T = c.T;
    a.router_bs = p.bs;
    a.router_nb = p.nb;
    a.out_ld = c.E;
    a.out_cols = c.E;
    a.out_split_stride = static_cast<long long>(c.T) * c.E;
    a.out = partial;
    a.status = device_status_word();
    a.timeout_ns = kWaitTimeoutNs;
    const int tiles = p.nb * p.eb * p.splits;
    const int grid = tiles < num_sms() ? tiles : num_sms();
    moe_status_t s = launch_gemm_tc(GM_ROUTER, maps, a, grid, st);
    if (s != MOE_OK) return s;
    return launch_topk(partial, p.splits, a.out_split_stride, bias, c.T, c.E, c.K, c.score_func,
                       c.normalize, c.n_groups, c.topk_groups, idx, gates, st, scores,
                       row_scale);
  }
  float* logits = static_cast<float*>(ws);
  moe_status_t s = launch_logits_f32(static_cast<const float*>(x),
                                     static_cast<const float*>(centroids), c.T, c.d, c.E, logits,
                                     st);
  if (s != MOE_OK) return s;
  return launch_topk(logits, 1, 0, bias, c.T, c.E, c.K, c.score_func, c.normalize, c.n_groups,
                     c.topk_groups, idx, gates, st, scores, row_scale);
}

// w8 (an FP8 layer's e4m3 weights and block scales) replaces w13..ws2: the
// same bf16 GEMMs with the weights dequantised in shared memory.
// h (training forward, bf16 weights only): the gate/up GEMM writes the
// pre-activations h [R, 2I] and act is formed from them.
moe_status_t do_experts(const moe_cfg_t& c, const void* xp, const void* x,
                        const int32_t* offsets, const void* w13, const void* w2,
                        const void* ws13, const void* ws2, void* act, void* y, void* ws,
                        cudaStream_t st, const moe_fp8_weights_t* w8 = nullptr,
                        void* h = nullptr) {
  if (c.act_dtype != MOE_BF16) {
    return launch_experts_f32(static_cast<const float*>(xp), static_cast<const float*>(x),
                              offsets, static_cast<const float*>(w13),
                              static_cast<const float*>(w2), static_cast<const float*>(ws13),
                              static_cast<const float*>(ws2), static_cast<float*>(act),
                              static_cast<float*>(y), c.T, c.K, c.E, c.S, c.d, c.I, st);
  }
  const int G = c.E + c.S;
  int32_t* tab = static_cast<int32_t*>(ws);
  int32_t* rows = tab;
  int32_t* brow = rows + (G + 1);
  int32_t* orow = brow + (G + 1);
  int32_t* bs = orow + (G + 1);
  int32_t* bstart = bs + (G + 1);
  // W8 tiles keep both accumulators and two weight slots in TMEM: <= 192 tokens.
  // Small batches (decode: every group holds at most T rows) use token blocks
  // of <= 64 and the kernels' deeper ring for streaming weights.
  const bool small = !w8 && c.T <= 512;
  const GroupLayout lay{0, c.T * c.K, c.T, w8 ? 192 : small ? 64 : 256};
  moe_status_t s = launch_build_groups(offsets, nullptr, c.T, c.E, c.S, lay, rows, brow, orow, bs,
                                       bstart, st);
  if (s != MOE_OK) return s;
  const long long TK = static_cast<long long>(c.T) * c.K;
  const long long R = TK + static_cast<long long>(c.S) * c.T;
  const int grid = num_sms();

  // gate/up + SwiGLU: A = W13 rows, B = dispatched rows (routed) or tokens (shared)
  const uint64_t r13 = static_cast<uint64_t>(c.E) * 2 * c.I, rs13 = static_cast<uint64_t>(c.S) * 2 * c.I;
  const uint64_t r2 = static_cast<uint64_t>(c.E) * c.d, rs2 = static_cast<uint64_t>(c.S) * c.d;
  // W8: e4m3 weight maps replace the bf16 ones (the token maps are the same)
  auto w8_maps = [&](GemmMaps* m, const void* a0, uint64_t n0, const void* a1, uint64_t n1,
                     uint64_t k) {
    if (!make_tmap_e4m3(&m->a[0], a0, n0, k)) return false;
    if (a1) return make_tmap_e4m3(&m->a[1], a1, n1, k);
    m->a[1] = m->a[0];
    return true;
  };
  if (w8) {
    w13 = w8->w13;
    w2 = w8->w2;
    ws13 = w8->ws13;
    ws2 = w8->ws2;
  }
  GemmMaps m1;
  if (!make_gemm_maps(&m1, w13, r13, c.S > 0 ? ws13 : nullptr, rs13, 128, xp, TK, x, c.T, c.d,
                      kTokBox0Pair) ||
      (w8 && !w8_maps(&m1, w13, r13, c.S > 0 ? ws13 : nullptr, rs13, c.d)))
    return MOE_ERR_CUDA;
  GemmArgs a{};
  a.gt = GroupTable{rows, brow, orow, bs, bstart};
  a.G = G;
  a.E = c.E;
  a.m_blocks = ceil_div(c.I, 256);   // 256 gate rows and their up rows per CTA pair
  a.a_rows_per_group = 2 * c.I;
  a.a1_off = c.I;
  a.k_blocks = c.d / 64;
  a.k_splits = 1;
  a.k_per_split = a.k_blocks;
  a.out_ld = c.I;
  a.out_cols = c.I;
  a.out = act;
  a.tile_counter = bstart + G + 1;
  a.status = device_status_word();
  a.timeout_ns = kWaitTimeoutNs;
  if (w8) {
    a.w_scale[0] = w8->w13_scale;
    a.w_scale[1] = c.S > 0 ? w8->ws13_scale : w8->w13_scale;
    a.scale_kb = c.d / 128;
  }
  if (h) {
    a.out = h;
    a.out_ld = 2 * c.I;
    s = launch_gemm_tc(GM_GATEUP_H, m1, a, grid, st, false, small);
    if (s != MOE_OK) return s;
    s = launch_swiglu_fwd(h, act, R, c.I, st);
  } else {
    s = launch_gemm_tc(GM_GATEUP, m1, a, grid, st, w8 != nullptr, small);
  }
  if (s != MOE_OK) return s;

  // down: A = W2 rows (two 128-row boxes), B = activations
  GemmMaps m2;
  if (!make_gemm_maps(&m2, w2, r2, c.S > 0 ? ws2 : nullptr, rs2, 128, act, R, nullptr, 0, c.I,
                      kTokBox0Pair) ||
      (w8 && !w8_maps(&m2, w2, r2, c.S > 0 ? ws2 : nullptr, rs2, c.I)))
    return MOE_ERR_CUDA;
  GemmArgs b = a;
  b.gt = GroupTable{rows, orow, orow, bs, bstart};
  b.m_blocks = ceil_div(c.d, 512);   // 512 rows of W2 per CTA pair
  b.a_rows_per_group = c.d;
  b.a1_off = 256;
  b.k_blocks = c.I / 64;
  b.k_per_split = b.k_blocks;
  b.out_ld = c.d;
  b.out_cols = c.d;
  b.out = y;
  b.tile_counter = bstart + G + 2;
  if (w8) {
    b.w_scale[0] = w8->w2_scale;
    b.w_scale[1] = c.S > 0 ? w8->ws2_scale : w8->w2_scale;
    b.scale_kb = c.I / 128;
  }
  return launch_gemm_tc(GM_DOWN, m2, b, grid, st, w8 != nullptr, small);
}

moe_status_t do_experts_fp8(const moe_cfg_t& c, const void* xq, const float* xs,
                            const int32_t* offsets, const int32_t* counts,
                            const moe_fp8_weights_t& w, void* act, float* act_s, void* y,
                            void* ws, cudaStream_t st) {
  const int G = c.E + c.S;
  const Fp8Rows fr = fp8_rows(c);
  int32_t* tab = static_cast<int32_t*>(ws);
  int32_t* rows = tab;
  int32_t* brow = rows + (G + 1);
  int32_t* orow = brow + (G + 1);
  int32_t* bs = orow + (G + 1);
  int32_t* bstart = bs + (G + 1);
  const GroupLayout lay{static_cast<int>(fr.P), static_cast<int>(fr.P), static_cast<int>(fr.Tp),
                        kFp8TileTokens};
  moe_status_t s = launch_build_groups(offsets, counts, c.T, c.E, c.S, lay, rows, brow, orow, bs,
                                       bstart, st);
  if (s != MOE_OK) return s;
  const bool sh = c.S > 0;

  // gate/up + SwiGLU + e4m3 quantisation of act (1 x 128 along I)
  Fp8GemmMaps m1;
  if (!make_fp8_maps(&m1, w.w13, static_cast<uint64_t>(c.E) * 2 * c.I, sh ? w.ws13 : nullptr,
                     static_cast<uint64_t>(c.S) * 2 * c.I, 64, xq, fr.rows_in, xs, c.d))
    return MOE_ERR_CUDA;
  Fp8GemmArgs a{};
  a.gt = GroupTable{rows, brow, orow, bs, bstart};
  a.G = G;
  a.E = c.E;
  a.m_blocks = c.I / 128;
  a.a_rows_per_group = 2 * c.I;
  a.a1_off = c.I;
  a.k_blocks = c.d / 128;
  a.w_scale[0] = w.w13_scale;
  a.w_scale[1] = sh ? w.ws13_scale : w.w13_scale;
  a.out_ld = c.I;
  a.out_cols = c.I;
  a.out = act;
  a.out_scale = act_s;
  a.out_scale_ld = fr.rows_out;
  a.status = device_status_word();
  a.timeout_ns = kWaitTimeoutNs;
  if ((s = launch_fp8_gemm(GM_GATEUP, m1, a, st)) != MOE_OK) return s;

  // down: A = W2 blocks, B = quantised activations
  Fp8GemmMaps m2;
  if (!make_fp8_maps(&m2, w.w2, static_cast<uint64_t>(c.E) * c.d, sh ? w.ws2 : nullptr,
                     static_cast<uint64_t>(c.S) * c.d, 128, act, fr.rows_out, act_s, c.I))
    return MOE_ERR_CUDA;
  Fp8GemmArgs b = a;
  b.gt = GroupTable{rows, orow, orow, bs, bstart};
  b.m_blocks = ceil_div(c.d, 256);
  b.a_rows_per_group = c.d;
  b.a1_off = 0;
  b.k_blocks = c.I / 128;
  b.w_scale[0] = w.w2_scale;
  b.w_scale[1] = sh ? w.ws2_scale : w.w2_scale;
  b.out_ld = c.d;
  b.out_cols = c.d;
  b.out = y;
  b.out_scale = nullptr;
  b.out_scale_ld = 0;
  return launch_fp8_gemm(GM_DOWN, m2, b, st);
}

// ---------------------------------------------------------------- training

size_t forward_train_ws(const moe_cfg_t& c) {
  return align_up(route_ws(c), 256) + align_up(dispatch_ws(c), 256) +
         align_up(experts_ws(c), 256);
}

// Backward workspace: the padded row layout (see backward.cu), the input-
// gradient GEMMs' group table, and the intermediate gradients.
struct BackwardLayout {
  size_t tab, dg, dlk, dlrow, dl, dxr, part, dy, dact, dh, dxp, total;
  long long rows_max;
  int max_blocks;
};

BackwardLayout backward_layout(const moe_cfg_t& c) {
  BackwardLayout L{};
  const size_t TK = static_cast<size_t>(c.T) * c.K;
  const int G = c.E + c.S;
  L.rows_max = static_cast<long long>(TK) + 15LL * c.E +
               static_cast<long long>(c.S) * round_up(c.T, 16);
  L.max_blocks = static_cast<int>(TK / 256) + c.E + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return o;
  };
  L.tab = take((static_cast<size_t>(c.E) + 1 + 5 * (static_cast<size_t>(G) + 1) + 4) *
               sizeof(int32_t));
  L.dg = take(TK * sizeof(float));
  const bool sm = c.score_func == MOE_SCORE_SOFTMAX;
  L.dlk = take(sm ? 0 : TK * sizeof(float));
  L.dlrow = take(sm ? 0 : TK * sizeof(float));
  L.dl = take(sm ? static_cast<size_t>(c.T) * c.E * sizeof(float) : 0);
  L.dxr = take(sm ? static_cast<size_t>(c.T) * c.d * sizeof(float) : 0);
  L.part = take((sm ? static_cast<size_t>(ceil_div(c.T, 256)) * c.E
                    : static_cast<size_t>(L.max_blocks) * kDcentSub) *
                c.d * sizeof(float));
  const size_t R = static_cast<size_t>(L.rows_max);
  L.dy = take(R * c.d * 2);
  L.dact = take(R * c.I * 2);
  L.dh = take(R * 2 * c.I * 2);
  L.dxp = take(R * c.d * 2);
  L.total = off;
  return L;
}

bool is_bf16(const moe_cfg_t& c) {
  return c.act_dtype == MOE_BF16 && c.wgt_dtype == MOE_BF16;
}

moe_status_t do_forward_train(const moe_cfg_t& c, const void* x, const void* centroids,
                              const float* bias, const void* w13, const void* w2,
                              const void* ws13, const void* ws2, const moe_train_state_t& t,
                              void* out, void* ws, cudaStream_t st) {
  const size_t o_disp = align_up(route_ws(c), 256);
  const size_t o_exp = o_disp + align_up(dispatch_ws(c), 256);
  moe_status_t s;
  if ((s = do_route(c, x, centroids, bias, t.idx, t.gates, ws, st, t.scores)) != MOE_OK) return s;
  if ((s = launch_dispatch(x, static_cast<size_t>(c.d) * 2, t.idx, c.T, c.K, c.E, t.counts,
                           t.offsets, t.xp, t.perm_tok, t.pos, at<int32_t>(ws, o_disp), st)) !=
      MOE_OK)
    return s;
  if ((s = do_experts(c, t.xp, x, t.offsets, w13, w2, ws13, ws2, t.act, t.y, at<void>(ws, o_exp),
                      st, nullptr, t.h)) != MOE_OK)
    return s;
  return launch_combine(c.act_dtype, t.y, t.gates, t.pos, x, out, c.T, c.K, c.S, c.d,
                        static_cast<long long>(c.T) * c.K, c.T, c.add_residual, st);
}

// Weight operand of an input-gradient GEMM: the group's [K, M] matrix read
// MN-major in boxes of 64 rows x 64 columns; token operand as the forward's.
bool make_dgrad_maps(GemmMaps* m, const void* a0, uint64_t a0_rows, const void* a1,
                     uint64_t a1_rows, uint64_t a_cols, const void* b, uint64_t b_rows,
                     uint64_t b_cols) {
  if (!make_tmap_bf16(&m->a[0], a0, a0_rows, a_cols, 64)) return false;
  if (a1) {
    if (!make_tmap_bf16(&m->a[1], a1, a1_rows, a_cols, 64)) return false;
  } else {
    m->a[1] = m->a[0];
  }
  for (int i = 0; i < kTokBoxes; ++i) {
    if (!make_tmap_bf16(&m->b[0][i], b, b_rows, b_cols, kTokBox0Pair << i)) return false;
    m->b[1][i] = m->b[0][i];
  }
  return true;
}

moe_status_t do_backward(const moe_cfg_t& c, const void* dout, const void* x,
                         const void* centroids, const void* w13, const void* w2,
                         const void* ws13, const void* ws2, const moe_train_state_t& t,
                         const moe_grads_t& gr, void* ws, cudaStream_t st) {
  const BackwardLayout L = backward_layout(c);
  const int G = c.E + c.S;
  int32_t* poff = at<int32_t>(ws, L.tab);
  int32_t* rows = poff + (c.E + 1);
  int32_t* brow = rows + (G + 1);
  int32_t* orow = brow + (G + 1);
  int32_t* bs = orow + (G + 1);
  int32_t* bstart = bs + (G + 1);
  int32_t* counters = bstart + (G + 1);
  float* dg = at<float>(ws, L.dg);
  void* dy = at<void>(ws, L.dy);
  void* dact = at<void>(ws, L.dact);
  void* dh = at<void>(ws, L.dh);
  void* dxp = at<void>(ws, L.dxp);
  const bool sm = c.score_func == MOE_SCORE_SOFTMAX;
  const long long TK = static_cast<long long>(c.T) * c.K;
  const long long R = TK + static_cast<long long>(c.S) * c.T;
  const bool sh = c.S > 0;
  moe_status_t s;
  if ((s = launch_build_bwd_groups(t.counts, c.T, c.E, c.S, poff, rows, brow, orow, bs, bstart,
                                   counters, st)) != MOE_OK)
    return s;
  if ((s = launch_combine_bwd(dout, t.y, t.gates, t.idx, t.perm_tok, t.counts, t.offsets, poff,
                              c.T, c.K, c.E, c.S, c.d, L.rows_max, dy, dg, st)) != MOE_OK)
    return s;
  if ((s = launch_router_bwd(dg, t.gates, t.idx, t.scores, t.pos, c.T, c.E, c.K, c.score_func,
                             c.normalize, at<float>(ws, L.dlk), at<float>(ws, L.dlrow),
                             at<float>(ws, L.dl), st)) != MOE_OK)
    return s;
  const int grid = num_sms();
  GemmArgs a{};
  a.gt = GroupTable{rows, brow, orow, bs, bstart};
  a.G = G;
  a.E = c.E;
  a.k_splits = 1;
  a.a1_off = 256;
  a.status = device_status_word();
  a.timeout_ns = kWaitTimeoutNs;
  // da = dy W2: W2 of each group as [d rows (K), I columns (M)]
  GemmMaps m1;
  if (!make_dgrad_maps(&m1, w2, static_cast<uint64_t>(c.E) * c.d, sh ? ws2 : nullptr,
                       static_cast<uint64_t>(c.S) * c.d, c.I, dy, L.rows_max, c.d))
    return MOE_ERR_CUDA;
  a.m_blocks = ceil_div(c.I, 512);
  a.a_rows_per_group = c.d;
  a.k_blocks = c.d / 64;
  a.k_per_split = a.k_blocks;
  a.out_ld = c.I;
  a.out_cols = c.I;
  a.out = dact;
  a.tile_counter = counters + 0;
  if ((s = launch_gemm_tc(GM_DGRAD, m1, a, grid, st, false, false, "gemm_dgrad_down")) != MOE_OK)
    return s;
  if ((s = launch_swiglu_bwd(dact, t.h, t.counts, t.offsets, poff, c.T, c.K, c.E, c.S, c.I,
                             L.rows_max, dh, st)) != MOE_OK)
    return s;
  // du = dh W13: W13 of each group as [2I rows (K), d columns (M)]
  GemmMaps m2;
  if (!make_dgrad_maps(&m2, w13, static_cast<uint64_t>(c.E) * 2 * c.I, sh ? ws13 : nullptr,
                       static_cast<uint64_t>(c.S) * 2 * c.I, c.d, dh, L.rows_max, 2 * c.I))
    return MOE_ERR_CUDA;
  a.m_blocks = ceil_div(c.d, 512);
  a.a_rows_per_group = 2 * c.I;
  a.k_blocks = 2 * c.I / 64;
  a.k_per_split = a.k_blocks;
  a.out_ld = c.d;
  a.out_cols = c.d;
  a.out = dxp;
  a.tile_counter = counters + 1;
  if ((s = launch_gemm_tc(GM_DGRAD, m2, a, grid, st, false, false, "gemm_dgrad_gateup")) !=
      MOE_OK)
    return s;
  if (sm && (s = launch_router_dx_dense(at<float>(ws, L.dl), centroids, c.T, c.E, c.d,
                                        at<float>(ws, L.dxr), st)) != MOE_OK)
    return s;
  if ((s = launch_dx(dxp, t.pos, t.idx, t.offsets, poff, sm ? nullptr : at<float>(ws, L.dlk),
                     centroids, sm ? at<float>(ws, L.dxr) : nullptr, dout, gr.dx, c.T, c.K, c.E,
                     c.S, c.d, c.add_residual, st)) != MOE_OK)
    return s;
  s = sm ? launch_dcent_dense(at<float>(ws, L.dl), x, c.T, c.E, c.d, at<float>(ws, L.part),
                              gr.dcentroids, st)
         : launch_dcent_sparse(at<float>(ws, L.dlrow), t.xp, t.counts, t.offsets, bs, bstart,
                               c.E, c.d, L.max_blocks, at<float>(ws, L.part), gr.dcentroids, st);
  if (s != MOE_OK) return s;
  // dW2 = dy^T act (M = d, N = I); dW13 = dh^T u (M = 2I, N = d)
  WgradArgs w{};
  w.counts = t.counts;
  w.offsets = t.offsets;
  w.poff = poff;
  w.E = c.E;
  w.S = c.S;
  w.T = c.T;
  w.T16 = round_up(c.T, 16);
  w.status = device_status_word();
  w.timeout_ns = kWaitTimeoutNs;
  WgradMaps wm;
  if (!make_tmap_bf16(&wm.a, dy, L.rows_max, c.d, 64) ||
      !make_tmap_bf16(&wm.b[0], t.act, R, c.I, 64))
    return MOE_ERR_CUDA;
  wm.b[1] = wm.b[0];
  w.b_sh0 = static_cast<int>(TK);
  w.b_shs = c.T;
  w.M = c.d;
  w.N = c.I;
  w.m_blocks = ceil_div(c.d, 256);
  w.n_blocks = ceil_div(c.I, 256);
  w.out_gstride = static_cast<long long>(c.d) * c.I;
  w.out_routed = gr.dw2;
  w.out_shared = sh ? gr.dws2 : gr.dw2;
  w.tile_counter = counters + 2;
  if ((s = launch_wgrad(wm, w, st, "gemm_wgrad_down")) != MOE_OK) return s;
  if (!make_tmap_bf16(&wm.a, dh, L.rows_max, 2 * c.I, 64) ||
      !make_tmap_bf16(&wm.b[0], t.xp, TK, c.d, 64) ||
      !make_tmap_bf16(&wm.b[1], x, c.T, c.d, 64))
    return MOE_ERR_CUDA;
  w.b_sh0 = 0;
  w.b_shs = 0;
  w.M = 2 * c.I;
  w.N = c.d;
  w.m_blocks = ceil_div(2 * c.I, 256);
  w.n_blocks = ceil_div(c.d, 256);
  w.out_gstride = static_cast<long long>(2 * c.I) * c.d;
  w.out_routed = gr.dw13;
  w.out_shared = sh ? gr.dws13 : gr.dw13;
  w.tile_counter = counters + 3;
  return launch_wgrad(wm, w, st, "gemm_wgrad_gateup");
}

moe_status_t check_fp8_weights(const moe_cfg_t& c, const moe_fp8_weights_t* w) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (!w->w13 || !w->w2 || !w->w13_scale || !w->w2_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w->w13) || !aligned16(w->w2)) return MOE_ERR_INVALID_ARG;
  if (c.S > 0 && (!w->ws13 || !w->ws2 || !w->ws13_scale || !w->ws2_scale ||
                  !aligned16(w->ws13) || !aligned16(w->ws2)))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

long long combine_shared0(const moe_cfg_t& c) {
  return is_fp8(c) ? fp8_rows(c).P : static_cast<long long>(c.T) * c.K;
}
long long combine_shared_stride(const moe_cfg_t& c) {
  return is_fp8(c) ? fp8_rows(c).Tp : c.T;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_check_cfg(const moe_cfg_t* cfg) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  const moe_cfg_t& c = *cfg;
  if (c.T < 0 || c.d < 1 || c.E < 1 || c.E > kMaxE || c.K < 1 || c.K > kMaxK || c.K > c.E ||
      c.S < 0 || c.S > kMaxS || c.I < 1)
    return MOE_ERR_INVALID_ARG;
  if (c.score_func != MOE_SCORE_SIGMOID && c.score_func != MOE_SCORE_SOFTMAX)
    return MOE_ERR_INVALID_ARG;
  if ((c.normalize != 0 && c.normalize != 1) || (c.add_residual != 0 && c.add_residual != 1))
    return MOE_ERR_INVALID_ARG;
  if (c.n_groups == 0) {
    if (c.topk_groups != 0) return MOE_ERR_INVALID_ARG;
  } else {
    // node-limited routing: equal groups of a power-of-two size below 32 or a
    // multiple of 32 experts, at most 32 groups, enough experts for K
    if (c.n_groups < 1 || c.n_groups > 32 || c.E % c.n_groups != 0) return MOE_ERR_INVALID_ARG;
    const int gs = c.E / c.n_groups;
    if (!(gs % 32 == 0 || (gs < 32 && (gs & (gs - 1)) == 0))) return MOE_ERR_INVALID_ARG;
    if (c.topk_groups < 1 || c.topk_groups > c.n_groups || c.K > c.topk_groups * gs)
      return MOE_ERR_INVALID_ARG;
  }
  if (c.act_dtype < MOE_F32 || c.act_dtype > MOE_E4M3 || c.wgt_dtype < MOE_F32 ||
      c.wgt_dtype > MOE_E4M3)
    return MOE_ERR_INVALID_ARG;
  const bool fp8 = c.act_dtype == MOE_BF16 && c.wgt_dtype == MOE_E4M3;
  if ((c.act_dtype != c.wgt_dtype && !fp8) || c.act_dtype == MOE_E4M3) return MOE_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(c.T) * c.K + static_cast<long long>(c.S) * c.T +
                         4LL * c.E + 4LL * (c.S + 1);
  if (rows >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  if (c.act_dtype == MOE_BF16 && (c.d % 128 != 0 || c.I % 128 != 0)) return MOE_ERR_INVALID_ARG;
  // FP8 GEMMs keep a tile's weight scales in shared memory: at most 64 K blocks
  if (fp8 && (c.d > 8192 || c.I > 8192)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

size_t moe_workspace_size(const moe_cfg_t* cfg, int32_t which) {
  if (moe_check_cfg(cfg) != MOE_OK) return 0;
  const moe_cfg_t& c = *cfg;
  switch (which) {
    case MOE_WS_ROUTE: return route_ws(c);
    case MOE_WS_DISPATCH: return dispatch_ws(c);
    case MOE_WS_EXPERTS: return experts_ws(c);
    case MOE_WS_FORWARD: return forward_layout(c).total;
    case MOE_WS_FORWARD_PRENORM: return prenorm_ws(c);
    case MOE_WS_FORWARD_W8A16: return is_fp8(c) ? forward_layout(bf16_layout(c)).total : 0;
    case MOE_WS_FORWARD_TRAIN: return is_bf16(c) ? forward_train_ws(c) : 0;
    case MOE_WS_BACKWARD: return is_bf16(c) ? backward_layout(c).total : 0;
    default: return 0;
  }
}

moe_status_t moe_route(const moe_cfg_t* cfg, const void* x, const void* centroids,
                       const float* bias, int32_t* idx, float* gates, void* ws, size_t ws_bytes,
                       void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (c.T == 0) return MOE_OK;
  if ((s = check_ptrs(c, {x, centroids}, {bias, idx, gates})) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, route_ws(c))) != MOE_OK) return s;
  return do_route(c, x, centroids, bias, idx, gates, ws, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_dispatch(const moe_cfg_t* cfg, const void* x, const int32_t* idx,
                          int32_t* counts, int32_t* offsets, void* xp, int32_t* perm_tok,
                          int32_t* pos, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (is_fp8(c)) return MOE_ERR_UNSUPPORTED;   // FP8 layers: the *_fp8 entry points
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (c.T > 0) {
    if ((s = check_ptrs(c, {x, xp}, {idx, perm_tok, pos})) != MOE_OK) return s;
  }
  if ((s = check_ws(ws, ws_bytes, dispatch_ws(c))) != MOE_OK) return s;
  return launch_dispatch(x, static_cast<size_t>(c.d) * esize(c.act_dtype), idx, c.T, c.K, c.E,
                         counts, offsets, xp, perm_tok, pos, static_cast<int32_t*>(ws),
                         static_cast<cudaStream_t>(stream));
}

moe_status_t moe_experts(const moe_cfg_t* cfg, const void* xp, const void* x,
                         const int32_t* offsets, const void* w13, const void* w2,
                         const void* ws13, const void* ws2, void* act, void* y, void* ws,
                         size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (is_fp8(c)) return MOE_ERR_UNSUPPORTED;   // FP8 layers: the *_fp8 entry points
  if (c.T == 0) return MOE_OK;
  if ((s = check_ptrs(c, {xp, x, w13, w2, act, y}, {offsets})) != MOE_OK) return s;
  if (c.S > 0 && (s = check_ptrs(c, {ws13, ws2}, {})) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, experts_ws(c))) != MOE_OK) return s;
  return do_experts(c, xp, x, offsets, w13, w2, ws13, ws2, act, y, ws,
                    static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- moe_experts_static
// The expert FFNs for callers that cannot allocate device memory: the group
// table that moe_experts keeps in the caller's workspace lives here in a
// module-scope device array instead.  Capacity: E + S <= kStaticMaxGroups
// groups (5 int32 arrays of kStaticMaxGroups + 1 entries and the two GEMMs'
// tile counters, about 22 KB), which
// every device that loads this library keeps until the process exits.  The
// array's address is looked up once per device (cudaGetSymbolAddress) on that
// device's first call.  All calls share the one array and keep the last
// call's table; every entry a call reads is first written by that call, so
// nothing needs clearing, but two calls that overlap on the GPU (different
// streams, no ordering) race on the table.
} // extern "C"

namespace {
constexpr int kStaticMaxGroups = kMaxE + kMaxS;
}  // namespace

static __device__ __align__(256) int32_t g_static_group_table[5 * (kStaticMaxGroups + 1) + 2];

namespace {
int32_t* static_group_table() {
  static int32_t* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev < 64 && cached[dev]) return cached[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_group_table) != cudaSuccess) return nullptr;
  if (dev < 64) cached[dev] = static_cast<int32_t*>(p);
  return static_cast<int32_t*>(p);
}
}  // namespace

extern "C" {

moe_status_t moe_experts_static(const moe_cfg_t* cfg, const void* xp, const void* x,
                                const int32_t* offsets, const void* w13, const void* w2,
                                const void* ws13, const void* ws2, void* act, void* y,
                                void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (is_fp8(c)) return MOE_ERR_UNSUPPORTED;   // FP8 layers: the *_fp8 entry points
  if (c.E + c.S > kStaticMaxGroups) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if ((s = check_ptrs(c, {xp, x, w13, w2, act, y}, {offsets})) != MOE_OK) return s;
  if (c.S > 0 && (s = check_ptrs(c, {ws13, ws2}, {})) != MOE_OK) return s;
  int32_t* table = static_group_table();
  if (!table) return MOE_ERR_CUDA;
  return do_experts(c, xp, x, offsets, w13, w2, ws13, ws2, act, y, table,
                    static_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine(const moe_cfg_t* cfg, const void* y, const float* gates,
                         const int32_t* pos, const void* x, void* out, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (c.T == 0) return MOE_OK;
  if ((s = check_ptrs(c, {y, out}, {gates, pos})) != MOE_OK) return s;
  if (c.add_residual && (s = check_ptrs(c, {x}, {})) != MOE_OK) return s;
  return launch_combine(c.act_dtype, y, gates, pos, x, out, c.T, c.K, c.S, c.d,
                        combine_shared0(c), combine_shared_stride(c), c.add_residual,
                        static_cast<cudaStream_t>(stream));
}

moe_status_t moe_update_bias(const moe_cfg_t* cfg, const int32_t* counts, float* bias,
                             float* load_stats, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!counts || !bias) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;  // no load observed: nothing to balance
  return launch_update_bias(counts, bias, load_stats, c.E, c.T, c.K, c.gamma,
                            static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// The layer on tokens xin (router and experts) with residual xres.  Arguments
// checked by the caller; T > 0.
moe_status_t do_forward(const moe_cfg_t& c, const void* xin, const void* xres,
                        const void* centroids, const float* bias, const void* w13,
                        const void* w2, const void* ws13, const void* ws2, int32_t* idx,
                        float* gates, int32_t* counts, void* out, void* ws, cudaStream_t st) {
  const ForwardLayout L = forward_layout(c);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* pos = at<int32_t>(ws, L.pos);
  void* xp = at<void>(ws, L.xp);
  void* act = at<void>(ws, L.act);
  void* y = at<void>(ws, L.y);
  moe_status_t s;
  if ((s = do_route(c, xin, centroids, bias, idx, gates, at<void>(ws, L.route), st)) != MOE_OK)
    return s;
  if ((s = launch_dispatch(xin, static_cast<size_t>(c.d) * esize(c.act_dtype), idx, c.T, c.K,
                           c.E, counts, offsets, xp, perm, pos, at<int32_t>(ws, L.dispatch),
                           st)) != MOE_OK)
    return s;
  if ((s = do_experts(c, xp, xin, offsets, w13, w2, ws13, ws2, act, y, at<void>(ws, L.experts),
                      st)) != MOE_OK)
    return s;
  return launch_combine(c.act_dtype, y, gates, pos, xres, out, c.T, c.K, c.S, c.d,
                        static_cast<long long>(c.T) * c.K, c.T, c.add_residual, st);
}

moe_status_t do_forward_fp8(const moe_cfg_t& c, const void* xin, const void* xres,
                            const void* centroids, const float* bias,
                            const moe_fp8_weights_t* w, int32_t* idx, float* gates,
                            int32_t* counts, void* out, void* ws, cudaStream_t st) {
  const ForwardLayout L = forward_layout(c);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* pos = at<int32_t>(ws, L.pos);
  const Fp8Rows fr = fp8_rows(c);
  moe_status_t s;
  if ((s = do_route(c, xin, centroids, bias, idx, gates, at<void>(ws, L.route), st)) != MOE_OK)
    return s;
  if ((s = launch_dispatch_index(idx, c.T, c.K, c.E, 4, counts, offsets, perm, pos,
                                 at<int32_t>(ws, L.dispatch), st)) != MOE_OK)
    return s;
  if ((s = launch_scatter_quant(xin, c.T, c.K, c.d, pos, c.S > 0 ? static_cast<int>(fr.P) : -1,
                                at<void>(ws, L.xp), at<float>(ws, L.xs), fr.rows_in, st)) !=
      MOE_OK)
    return s;
  if ((s = do_experts_fp8(c, at<void>(ws, L.xp), at<float>(ws, L.xs), offsets, counts, *w,
                          at<void>(ws, L.act), at<float>(ws, L.act_s), at<void>(ws, L.y),
                          at<void>(ws, L.experts), st)) != MOE_OK)
    return s;
  return launch_combine(c.act_dtype, at<void>(ws, L.y), gates, pos, xres, out, c.T, c.K, c.S,
                        c.d, fr.P, fr.Tp, c.add_residual, st);
}

// Router of the layer behind its RMSNorm (V3 walk-through, section 4.1):
// the logit (x * inv_rms * w) . e_i is computed as inv_rms * (x . (w * e_i))
// from the raw tokens and the weighted centroids ew = w * e (folded here).
// Fused router (bf16, E <= 256): inv_rms comes from the router kernel and the
// normalised tokens are formed later by the dispatch (*fused = true).
// Otherwise the RMSNorm kernel writes xn and inv_rms, and the two-kernel
// router scales its logits by inv_rms.
moe_status_t do_route_prenorm(const moe_cfg_t& c, const void* x, const float* norm_w, float eps,
                              const void* centroids, const float* bias, int32_t* idx,
                              float* gates, const PrenormLayout& P, void* ws, cudaStream_t st,
                              bool* fused) {
  void* ew = at<void>(ws, P.ew);
  float* inv = at<float>(ws, P.inv);
  moe_status_t s;
  if ((s = launch_fold_centroids(centroid_dtype(c), centroids, norm_w, c.E, c.d, ew, st)) !=
      MOE_OK)
    return s;
  FusedRouterPlan fp{};
  *fused = c.act_dtype == MOE_BF16 && fused_router_plan(c.T, c.d, c.E, &fp);
  if (*fused)
    return launch_router_fused(fp, x, ew, bias, c.T, c.d, c.E, c.K, c.score_func, c.normalize,
                               c.n_groups, c.topk_groups, idx, gates, nullptr, eps, inv,
                               device_status_word(), kWaitTimeoutNs, st);
  if ((s = launch_rmsnorm(c.act_dtype, x, norm_w, eps, c.T, c.d, at<void>(ws, P.xs), inv, st)) !=
      MOE_OK)
    return s;
  return do_route(c, x, ew, bias, idx, gates, at<void>(ws, forward_layout(c).route), st, nullptr,
                  inv);
}

// The layer behind its RMSNorm, bf16 or fp32 experts: the experts read the
// normalised tokens (rounded once to the activation type), the residual is x.
moe_status_t do_forward_prenorm(const moe_cfg_t& c, const void* x, const float* norm_w, float eps,
                                const void* centroids, const float* bias, const void* w13,
                                const void* w2, const void* ws13, const void* ws2, int32_t* idx,
                                float* gates, int32_t* counts, void* out, void* ws,
                                cudaStream_t st) {
  const ForwardLayout L = forward_layout(c);
  const PrenormLayout P = prenorm_layout(c);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* pos = at<int32_t>(ws, L.pos);
  void* xp = at<void>(ws, L.xp);
  void* xs = at<void>(ws, P.xs);
  moe_status_t s;
  bool fused = false;
  if ((s = do_route_prenorm(c, x, norm_w, eps, centroids, bias, idx, gates, P, ws, st, &fused)) !=
      MOE_OK)
    return s;
  if (fused) {
    // one read of each token row: normalised, rounded and written to its K
    // rows and its shared-expert row
    if ((s = launch_dispatch_index(idx, c.T, c.K, c.E, 1, counts, offsets, perm, pos,
                                   at<int32_t>(ws, L.dispatch), st)) != MOE_OK)
      return s;
    if ((s = launch_scatter_norm(x, at<float>(ws, P.inv), norm_w, c.T, c.K, c.d, pos, xp,
                                 c.S > 0 ? xs : nullptr, st)) != MOE_OK)
      return s;
  } else if ((s = launch_dispatch(xs, static_cast<size_t>(c.d) * esize(c.act_dtype), idx, c.T,
                                  c.K, c.E, counts, offsets, xp, perm, pos,
                                  at<int32_t>(ws, L.dispatch), st)) != MOE_OK) {
    return s;
  }
  if ((s = do_experts(c, xp, xs, offsets, w13, w2, ws13, ws2, at<void>(ws, L.act),
                      at<void>(ws, L.y), at<void>(ws, L.experts), st)) != MOE_OK)
    return s;
  return launch_combine(c.act_dtype, at<void>(ws, L.y), gates, pos, x, out, c.T, c.K, c.S, c.d,
                        static_cast<long long>(c.T) * c.K, c.T, c.add_residual, st);
}

// The FP8 layer behind its RMSNorm: the dispatch quantises the normalised
// tokens (bf16-rounded, then 1 x 128 e4m3 tiles) in its single read of x.
moe_status_t do_forward_fp8_prenorm(const moe_cfg_t& c, const void* x, const float* norm_w,
                                    float eps, const void* centroids, const float* bias,
                                    const moe_fp8_weights_t* w, int32_t* idx, float* gates,
                                    int32_t* counts, void* out, void* ws, cudaStream_t st) {
  const ForwardLayout L = forward_layout(c);
  const PrenormLayout P = prenorm_layout(c);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* pos = at<int32_t>(ws, L.pos);
  const Fp8Rows fr = fp8_rows(c);
  moe_status_t s;
  bool fused = false;
  if ((s = do_route_prenorm(c, x, norm_w, eps, centroids, bias, idx, gates, P, ws, st, &fused)) !=
      MOE_OK)
    return s;
  if ((s = launch_dispatch_index(idx, c.T, c.K, c.E, 4, counts, offsets, perm, pos,
                                 at<int32_t>(ws, L.dispatch), st)) != MOE_OK)
    return s;
  const int shared_row = c.S > 0 ? static_cast<int>(fr.P) : -1;
  if (fused)
    s = launch_scatter_quant_norm(x, at<float>(ws, P.inv), norm_w, c.T, c.K, c.d, pos, shared_row,
                                  at<void>(ws, L.xp), at<float>(ws, L.xs), fr.rows_in, st);
  else
    s = launch_scatter_quant(at<void>(ws, P.xs), c.T, c.K, c.d, pos, shared_row,
                             at<void>(ws, L.xp), at<float>(ws, L.xs), fr.rows_in, st);
  if (s != MOE_OK) return s;
  if ((s = do_experts_fp8(c, at<void>(ws, L.xp), at<float>(ws, L.xs), offsets, counts, *w,
                          at<void>(ws, L.act), at<float>(ws, L.act_s), at<void>(ws, L.y),
                          at<void>(ws, L.experts), st)) != MOE_OK)
    return s;
  return launch_combine(c.act_dtype, at<void>(ws, L.y), gates, pos, x, out, c.T, c.K, c.S, c.d,
                        fr.P, fr.Tp, c.add_residual, st);
}

moe_status_t forward_empty(const moe_cfg_t& c, int32_t* counts, cudaStream_t st) {
  TraceScope tr(st, "forward_empty");
  cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, st);
  return launch_status();
}

bool valid_eps(float eps) { return eps > 0.f && eps < 1e30f; }

}  // namespace

extern "C" {

moe_status_t moe_forward(const moe_cfg_t* cfg, const void* x, const void* centroids,
                         const float* bias, const void* w13, const void* w2, const void* ws13,
                         const void* ws2, int32_t* idx, float* gates, int32_t* counts, void* out,
                         void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (is_fp8(c)) return MOE_ERR_UNSUPPORTED;   // FP8 layers: the *_fp8 entry points
  if (!counts) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return forward_empty(c, counts, st);
  if ((s = check_ptrs(c, {x, centroids, w13, w2, out}, {bias, idx, gates})) != MOE_OK) return s;
  if (c.S > 0 && (s = check_ptrs(c, {ws13, ws2}, {})) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, forward_layout(c).total)) != MOE_OK) return s;
  return do_forward(c, x, x, centroids, bias, w13, w2, ws13, ws2, idx, gates, counts, out, ws,
                    st);
}

moe_status_t moe_rmsnorm(const moe_cfg_t* cfg, const void* x, const float* norm_w, float eps,
                         void* xn, float* inv_rms, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!valid_eps(eps)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if ((s = check_ptrs(c, {x, xn, norm_w}, {})) != MOE_OK) return s;
  return launch_rmsnorm(c.act_dtype, x, norm_w, eps, c.T, c.d, xn, inv_rms,
                        static_cast<cudaStream_t>(stream));
}

moe_status_t moe_forward_prenorm(const moe_cfg_t* cfg, const void* x, const float* norm_w,
                                 float eps, const void* centroids, const float* bias,
                                 const void* w13, const void* w2, const void* ws13,
                                 const void* ws2, int32_t* idx, float* gates, int32_t* counts,
                                 void* out, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (is_fp8(c)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !valid_eps(eps)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return forward_empty(c, counts, st);
  if ((s = check_ptrs(c, {x, norm_w, centroids, w13, w2, out}, {bias, idx, gates})) != MOE_OK)
    return s;
  if (c.S > 0 && (s = check_ptrs(c, {ws13, ws2}, {})) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, prenorm_ws(c))) != MOE_OK) return s;
  return do_forward_prenorm(c, x, norm_w, eps, centroids, bias, w13, w2, ws13, ws2, idx, gates,
                            counts, out, ws, st);
}

moe_status_t moe_forward_fp8_prenorm(const moe_cfg_t* cfg, const void* x, const float* norm_w,
                                     float eps, const void* centroids, const float* bias,
                                     const moe_fp8_weights_t* w, int32_t* idx, float* gates,
                                     int32_t* counts, void* out, void* ws, size_t ws_bytes,
                                     void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!is_fp8(c)) return MOE_ERR_INVALID_ARG;
  if (!counts || !valid_eps(eps)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return forward_empty(c, counts, st);
  if ((s = check_ptrs(c, {x, norm_w, centroids, out}, {bias, idx, gates})) != MOE_OK) return s;
  if ((s = check_fp8_weights(c, w)) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, prenorm_ws(c))) != MOE_OK) return s;
  return do_forward_fp8_prenorm(c, x, norm_w, eps, centroids, bias, w, idx, gates, counts, out,
                                ws, st);
}

moe_status_t moe_experts_w8a16(const moe_cfg_t* cfg, const void* xp, const void* x,
                               const int32_t* offsets, const moe_fp8_weights_t* w, void* act,
                               void* y, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!is_fp8(c)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if ((s = check_ptrs(c, {xp, x, act, y}, {offsets})) != MOE_OK) return s;
  if ((s = check_fp8_weights(c, w)) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, experts_ws(c))) != MOE_OK) return s;
  return do_experts(bf16_layout(c), xp, x, offsets, nullptr, nullptr, nullptr, nullptr, act, y,
                    ws, static_cast<cudaStream_t>(stream), w);
}

moe_status_t moe_forward_w8a16(const moe_cfg_t* cfg, const void* x, const void* centroids,
                               const float* bias, const moe_fp8_weights_t* w, int32_t* idx,
                               float* gates, int32_t* counts, void* out, void* ws,
                               size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!is_fp8(*cfg)) return MOE_ERR_INVALID_ARG;
  const moe_cfg_t c = bf16_layout(*cfg);
  if (!counts) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return forward_empty(c, counts, st);
  if ((s = check_ptrs(c, {x, centroids, out}, {bias, idx, gates})) != MOE_OK) return s;
  if ((s = check_fp8_weights(*cfg, w)) != MOE_OK) return s;
  const ForwardLayout L = forward_layout(c);
  if ((s = check_ws(ws, ws_bytes, L.total)) != MOE_OK) return s;
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* pos = at<int32_t>(ws, L.pos);
  void* xp = at<void>(ws, L.xp);
  void* act = at<void>(ws, L.act);
  void* y = at<void>(ws, L.y);
  if ((s = do_route(c, x, centroids, bias, idx, gates, at<void>(ws, L.route), st)) != MOE_OK)
    return s;
  if ((s = launch_dispatch(x, static_cast<size_t>(c.d) * 2, idx, c.T, c.K, c.E, counts, offsets,
                           xp, at<int32_t>(ws, L.perm), pos, at<int32_t>(ws, L.dispatch), st)) !=
      MOE_OK)
    return s;
  if ((s = do_experts(c, xp, x, offsets, nullptr, nullptr, nullptr, nullptr, act, y,
                      at<void>(ws, L.experts), st, w)) != MOE_OK)
    return s;
  return launch_combine(c.act_dtype, y, gates, pos, x, out, c.T, c.K, c.S, c.d,
                        static_cast<long long>(c.T) * c.K, c.T, c.add_residual, st);
}

moe_status_t moe_fp8_rows(const moe_cfg_t* cfg, int64_t* rows_in, int64_t* rows_out,
                          int64_t* shared_row) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!is_fp8(*cfg)) return MOE_ERR_INVALID_ARG;
  const Fp8Rows r = fp8_rows(*cfg);
  if (rows_in) *rows_in = r.rows_in;
  if (rows_out) *rows_out = r.rows_out;
  if (shared_row) *shared_row = r.P;
  return MOE_OK;
}

moe_status_t moe_dispatch_fp8(const moe_cfg_t* cfg, const void* x, const int32_t* idx,
                              int32_t* counts, int32_t* offsets, void* xq, float* xq_scale,
                              int32_t* perm_tok, int32_t* pos, void* ws, size_t ws_bytes,
                              void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!is_fp8(c)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (c.T > 0) {
    if ((s = check_ptrs(c, {x, xq}, {idx, perm_tok, pos, xq_scale})) != MOE_OK) return s;
  }
  if ((s = check_ws(ws, ws_bytes, dispatch_ws(c))) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = launch_dispatch_index(idx, c.T, c.K, c.E, 4, counts, offsets, perm_tok, pos,
                                 static_cast<int32_t*>(ws), st)) != MOE_OK)
    return s;
  const Fp8Rows fr = fp8_rows(c);
  return launch_scatter_quant(x, c.T, c.K, c.d, pos, c.S > 0 ? static_cast<int>(fr.P) : -1, xq,
                              xq_scale, fr.rows_in, st);
}

moe_status_t moe_experts_fp8(const moe_cfg_t* cfg, const void* xq, const float* xq_scale,
                             const int32_t* offsets, const int32_t* counts,
                             const moe_fp8_weights_t* w, void* act, float* act_scale, void* y,
                             void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!is_fp8(c)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if ((s = check_ptrs(c, {xq, act, y}, {xq_scale, offsets, counts, act_scale})) != MOE_OK)
    return s;
  if ((s = check_fp8_weights(c, w)) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, experts_ws(c))) != MOE_OK) return s;
  return do_experts_fp8(c, xq, xq_scale, offsets, counts, *w, act, act_scale, y, ws,
                        static_cast<cudaStream_t>(stream));
}

moe_status_t moe_forward_fp8(const moe_cfg_t* cfg, const void* x, const void* centroids,
                             const float* bias, const moe_fp8_weights_t* w, int32_t* idx,
                             float* gates, int32_t* counts, void* out, void* ws,
                             size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!is_fp8(c)) return MOE_ERR_INVALID_ARG;
  if (!counts) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return forward_empty(c, counts, st);
  if ((s = check_ptrs(c, {x, centroids, out}, {bias, idx, gates})) != MOE_OK) return s;
  if ((s = check_fp8_weights(c, w)) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, forward_layout(c).total)) != MOE_OK) return s;
  return do_forward_fp8(c, x, x, centroids, bias, w, idx, gates, counts, out, ws, st);
}

moe_status_t moe_forward_train(const moe_cfg_t* cfg, const void* x, const void* centroids,
                               const float* bias, const void* w13, const void* w2,
                               const void* ws13, const void* ws2, const moe_train_state_t* st,
                               void* out, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!is_bf16(c)) return MOE_ERR_UNSUPPORTED;
  if (!st || !st->counts) return MOE_ERR_INVALID_ARG;
  cudaStream_t sm = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return forward_empty(c, st->counts, sm);
  if ((s = check_ptrs(c, {x, centroids, w13, w2, out, st->xp, st->h, st->act, st->y},
                      {bias, st->idx, st->gates, st->scores, st->offsets, st->perm_tok,
                       st->pos})) != MOE_OK)
    return s;
  if (c.S > 0 && (s = check_ptrs(c, {ws13, ws2}, {})) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, forward_train_ws(c))) != MOE_OK) return s;
  return do_forward_train(c, x, centroids, bias, w13, w2, ws13, ws2, *st, out, ws, sm);
}

moe_status_t moe_backward(const moe_cfg_t* cfg, const void* dout, const void* x,
                          const void* centroids, const void* w13, const void* w2,
                          const void* ws13, const void* ws2, const moe_train_state_t* st,
                          const moe_grads_t* grads, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = moe_check_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_cfg_t& c = *cfg;
  if (!is_bf16(c)) return MOE_ERR_UNSUPPORTED;
  if (!st || !grads) return MOE_ERR_INVALID_ARG;
  if ((s = check_ptrs(c, {grads->dw13, grads->dw2}, {grads->dcentroids})) != MOE_OK) return s;
  if (c.S > 0 && (s = check_ptrs(c, {grads->dws13, grads->dws2, ws13, ws2}, {})) != MOE_OK)
    return s;
  cudaStream_t sm = static_cast<cudaStream_t>(stream);
  const size_t E = static_cast<size_t>(c.E), S = static_cast<size_t>(c.S);
  const size_t wsz = static_cast<size_t>(2) * c.I * c.d * 2;   // bytes of one expert's W13
  if (c.T == 0) {   // no tokens: every gradient is zero
    TraceScope tr(sm, "backward_empty");
    cudaMemsetAsync(grads->dcentroids, 0, E * c.d * sizeof(float), sm);
    cudaMemsetAsync(grads->dw13, 0, E * wsz, sm);
    cudaMemsetAsync(grads->dw2, 0, E * wsz / 2, sm);
    if (S > 0) {
      cudaMemsetAsync(grads->dws13, 0, S * wsz, sm);
      cudaMemsetAsync(grads->dws2, 0, S * wsz / 2, sm);
    }
    return launch_status();
  }
  if ((s = check_ptrs(c, {dout, x, centroids, w13, w2, grads->dx, st->xp, st->h, st->act, st->y},
                      {st->idx, st->gates, st->scores, st->counts, st->offsets, st->perm_tok,
                       st->pos})) != MOE_OK)
    return s;
  if ((s = check_ws(ws, ws_bytes, backward_layout(c).total)) != MOE_OK) return s;
  return do_backward(c, dout, x, centroids, w13, w2, ws13, ws2, *st, *grads, ws, sm);
}

moe_status_t moe_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
  return launch_wait_timeout_selftest(limit_ns, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_get_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_moe_status_word, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_moe_status_word, &zero, sizeof(zero)) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (v & ERRBIT_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
  if (v & ERRBIT_BOUNDS) return MOE_ERR_DEVICE_BOUNDS;
  return MOE_OK;
}

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_BOUNDS: return "device index out of bounds";
    default: return "unknown status";
  }
}

moe_status_t moe_trace_enable(int32_t on) {
  g_trace.on = on != 0;
  return MOE_OK;
}

moe_status_t moe_trace_read(moe_kernel_time_t* out, int32_t max, int32_t* n) {
  std::vector<moe_kernel_time_t> agg;
  moe_status_t st = MOE_OK;
  for (TraceRec& r : g_trace.recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.ev1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.ev0, r.ev1) != cudaSuccess)
      st = MOE_ERR_CUDA;
    size_t i = 0;
    for (; i < agg.size(); ++i)
      if (strncmp(agg[i].name, r.name, sizeof(agg[i].name)) == 0) break;
    if (i == agg.size()) {
      moe_kernel_time_t k{};
      strncpy(k.name, r.name, sizeof(k.name) - 1);
      agg.push_back(k);
    }
    agg[i].launches += 1;
    agg[i].total_ms += ms;
    g_trace.pool.push_back(r.ev0);
    g_trace.pool.push_back(r.ev1);
  }
  g_trace.recs.clear();
  if (n) *n = static_cast<int32_t>(agg.size());
  if (out)
    for (int32_t i = 0; i < max && i < static_cast<int32_t>(agg.size()); ++i) out[i] = agg[i];
  return st;
}

const char* moe_version(void) { return "moe-b300 0.1 (sm_103a)"; }

}  // extern "C"
