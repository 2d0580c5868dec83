// Shared host/device helpers of the MoE library (internal).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Device error word of the current device (set by bounded waits, read and
// cleared by moe_get_status).
enum : unsigned { ERRBIT_TIMEOUT = 1u, ERRBIT_BOUNDS = 2u };

unsigned* device_status_word();   // address of this device's error word

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxS = 64;

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int round_up(int a, int b) { return ceil_div(a, b) * b; }
__host__ __device__ inline size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

// ---------------------------------------------------------------- tracing
// Every launch goes through trace_begin/trace_end; when tracing is off they
// are two branch instructions.
void trace_begin(cudaStream_t s, const char* name);
void trace_end(cudaStream_t s);

struct TraceScope {
  cudaStream_t s;
  TraceScope(cudaStream_t st, const char* name) : s(st) { trace_begin(s, name); }
  ~TraceScope() { trace_end(s); }
};

inline moe_status_t launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- element IO
template <typename T> struct Elem;
template <> struct Elem<float> {
  __device__ static float ld(const float* p) { return *p; }
  __device__ static void st(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
  __device__ static float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

}  // namespace moe
