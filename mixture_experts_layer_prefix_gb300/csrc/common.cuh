// common.cuh -- device helpers shared by the libmoe kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- errors
// Kernels report device-side errors through a per-device error word whose
// address the host passes in; the first error wins.
__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Host side: address of this device's error word (api.cu).
int* device_error_word();

// Caller-supplied row indices of one token's k routed pairs (lane j < k holds
// pair j's): a pair whose row is outside [0, R), or (when E > 0) whose expert
// is outside [0, E), sets MOE_ERR_DEVICE_INDEX and is skipped by the caller.
// Returns the warp-uniform mask of usable pairs (bit j).
__device__ __forceinline__ unsigned usable_pairs(int row, int e, int lane, int k, long R, int E, int* err) {
  const bool bad = lane < k && (row < 0 || row >= R || (E > 0 && (e < 0 || e >= E)));
  const unsigned badm = __ballot_sync(0xffffffffu, bad);
  if (badm && lane == 0) set_error(err, MOE_ERR_DEVICE_INDEX);
  return ~badm;
}

// Host side: count one kernel launch (api.cu).
void count_launch(int n = 1);

// Host side: when the launch-timing recorder is armed (moe_timing_arm),
// record a CUDA event on `st` just before the launch named `name` (api.cu).
void mark_launch(cudaStream_t st, const char* name);

// Names of the grouped GEMM kinds, for the launch-timing recorder.
__host__ __forceinline__ const char* gemm_kind_name(int kind, bool mx) {
  static const char* bf[] = {"gemm1_swiglu", "gemm2", "gemm2_dgrad_swiglu_bwd", "gemm1_dgrad",
                             "gemm2_wgrad", "gemm1_wgrad", "router_gemm"};
  static const char* q[] = {"mx_gemm1_swiglu", "mx_gemm2", "mx_gemm2_dgrad_swiglu_bwd", "mx_gemm1_dgrad",
                            "mx_gemm2_wgrad", "mx_gemm1_wgrad", "mx_router_gemm"};
  return (kind >= 0 && kind < 7) ? (mx ? q[kind] : bf[kind]) : "gemm";
}

// ---------------------------------------------------- 16-byte vector I/O
// Load/store 16 bytes of T as floats: 8 bf16 or 4 fp32 elements.
template <typename T> struct Vec16;

template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const float* p, float* v) {
    float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ __forceinline__ static void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* v) {
    uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// SiLU and the logistic function through CUDA's fast exp and division
// (relative error ~1e-6 over the range that matters, far below the bf16
// rounding of every value they feed); for z below about -88, exp(-z) is +inf
// and both return (-)0.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }
__device__ __forceinline__ float sigmoid_f(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace moe

// ------------------------------------------------------------ host macros
#define MOE_CUDA_TRY(expr)                              \
  do {                                                  \
    cudaError_t e_ = (expr);                            \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;         \
  } while (0)

#define MOE_LAUNCH_CHECK() MOE_CUDA_TRY(cudaGetLastError())

// Prefix of every kernel launch: counts it and, when the launch-timing
// recorder is armed, marks it on its stream, e.g.
//   MOE_COUNTED_AS("permute", st) kern<<<g, b, s, st>>>(args);
#define MOE_COUNTED_AS(name, st) ::moe::count_launch(), ::moe::mark_launch((st), (name)),
