// gdn_common.cuh -- device helpers shared by the Gated DeltaNet kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// ------------------------------------------------------------------ activation dtypes

template <typename T> struct Act;

template <> struct Act<float> {
  // 4 consecutive values (16-byte aligned address)
  static __device__ __forceinline__ float4 ldg4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
  }
  // the same from shared memory
  static __device__ __forceinline__ float4 lds4(const float* p) {
    return *reinterpret_cast<const float4*>(p);
  }
  static __device__ __forceinline__ void store4(float* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
  }
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ float ldg(const float* p) { return __ldg(p); }
  static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
  static __device__ __forceinline__ float cvt(float v) { return v; }
};

template <> struct Act<__nv_bfloat16> {
  // 4 consecutive values (8-byte aligned address)
  static __device__ __forceinline__ float4 ldg4(const __nv_bfloat16* p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  }
  static __device__ __forceinline__ float4 lds4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  }
  static __device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
  }
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ float ldg(const __nv_bfloat16* p) {
    return __bfloat162float(__ldg(p));
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
  }
  static __device__ __forceinline__ __nv_bfloat16 cvt(float v) { return __float2bfloat16_rn(v); }
};

// ------------------------------------------------------------------ scalar math
// Plain calls of the CUDA math library (expf, log1pf); nothing here restates their internals.

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }
// softplus(x) = log(1 + e^x) in a form that does not overflow for large x.
__device__ __forceinline__ float softplusf_(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

// Hot-loop variants built on the approximate CUDA intrinsics __expf / __fdividef (relative error
// ~1e-6 here).  Used only for per-element work inside the prefill; every per-chunk decay scalar
// keeps the exact expf because its error would compound across chunks.
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }
__device__ __forceinline__ float exp_fast(float x) { return __expf(x); }

// g = -exp(A_log) * softplus(a + dt_bias);  beta = sigmoid(b)
__device__ __forceinline__ void gates(float A_log, float dt_bias, float a, float b, float& g,
                                      float& beta) {
  g = -expf(A_log) * softplusf_(a + dt_bias);
  beta = sigmoidf_(b);
}

// ------------------------------------------------------------------ launch order

// For a kernel launched as a programmatic dependent of the previous kernel in the stream: waits
// until that kernel has completed and its writes are visible, then lets the next kernel be placed
// on the SMs as they free up (it waits the same way).  A no-op for an ordinary launch.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ------------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void set_status(int32_t* status, int bit) {
  if (status) atomicOr(status, bit);
}

// Runtime dims passed by value to every kernel.
struct KDims {
  int Hk, Hv, dk, dv, K, r, cqkv;
  float q_scale, l2_eps, norm_eps;
};

}  // namespace gdn
