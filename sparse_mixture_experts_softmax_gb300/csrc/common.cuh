// Device helpers shared by the MoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

typedef __nv_bfloat16 bf16;

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vectors: 4 floats or 8 bf16.
template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  float v[4];
  __device__ __forceinline__ void load(const float* p) {
    float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ __forceinline__ void store(float* p) const {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __device__ __forceinline__ float get(int i) const { return v[i]; }
  __device__ __forceinline__ void set(int i, float f) { v[i] = f; }
};
template <> struct Vec<bf16> {
  static constexpr int N = 8;
  __nv_bfloat162 v[4];
  __device__ __forceinline__ void load(const bf16* p) {
    uint4 q = *reinterpret_cast<const uint4*>(p);
    v[0] = *reinterpret_cast<__nv_bfloat162*>(&q.x);
    v[1] = *reinterpret_cast<__nv_bfloat162*>(&q.y);
    v[2] = *reinterpret_cast<__nv_bfloat162*>(&q.z);
    v[3] = *reinterpret_cast<__nv_bfloat162*>(&q.w);
  }
  __device__ __forceinline__ void store(bf16* p) const {
    uint4 q;
    q.x = *reinterpret_cast<const uint32_t*>(&v[0]);
    q.y = *reinterpret_cast<const uint32_t*>(&v[1]);
    q.z = *reinterpret_cast<const uint32_t*>(&v[2]);
    q.w = *reinterpret_cast<const uint32_t*>(&v[3]);
    *reinterpret_cast<uint4*>(p) = q;
  }
  __device__ __forceinline__ float get(int i) const {
    return (i & 1) ? __high2float(v[i >> 1]) : __low2float(v[i >> 1]);
  }
  __device__ __forceinline__ void set(int i, float f) {
    bf16 b = __float2bfloat16_rn(f);
    if (i & 1) v[i >> 1].y = b; else v[i >> 1].x = b;
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Programmatic dependent launch.  Every kernel of the library is launched
// allowed to start before its predecessor in the stream has finished (so its
// launch and its on-chip set-up overlap the predecessor's tail); it waits for
// the predecessor's completion and memory before its first global access.
// The short kernels then let their successor be launched at once; the GEMMs
// do not (pdl_wait): a successor launched at their start would hold SM
// resources for the whole GEMM while it waits, and the GEMM steps measured
// slower that way.  Their blocks count as triggered when they exit.  A kernel
// launched without the attribute passes these instructions at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
  pdl_wait();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Routing indices before use.  A release build trusts the dispatch that
// wrote them: a slot s >= 0 is used, -1 (an assignment dropped by the expert
// capacity) is skipped; an expert id outside [0, E) is skipped.  A MOE_DEBUG
// build checks every index against its range before it is dereferenced: a
// slot outside [-1, R) or an expert id outside [0, E) is skipped and
// MOE_ERR_INVALID_ARG (1) is recorded in the status word (never a trap).
#ifdef MOE_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
constexpr int DEV_STATUS_INVALID_INDEX = 1;
__device__ __forceinline__ void debug_flag(int* status) {
  if (status != nullptr) atomicCAS(status, 0, DEV_STATUS_INVALID_INDEX);
}
__device__ __forceinline__ bool use_slot(int s, long long R, int* status) {
  if (!kDebugChecks) return s >= 0;
  if (s == -1) return false;
  if (s < 0 || (long long)s >= R) {
    debug_flag(status);
    return false;
  }
  return true;
}
__device__ __forceinline__ bool valid_expert(int e, int E, int* status) {
  if ((unsigned)e < (unsigned)E) return true;
  if (kDebugChecks) debug_flag(status);
  return false;
}

// Activations (course Part 1) and their derivatives.  CUDA's own tanhf/expf
// are called; nothing of their implementation is restated.
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float gelu_tanh_f(float h) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  return 0.5f * h * (1.0f + tanhf(c * (h + a * h * h * h)));
}
__device__ __forceinline__ float gelu_tanh_grad_f(float h) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  float t = tanhf(c * (h + a * h * h * h));
  return 0.5f * (1.0f + t) + 0.5f * h * (1.0f - t * t) * c * (1.0f + 3.0f * a * h * h);
}
__device__ __forceinline__ float silu_f(float h) { return h * sigmoidf_(h); }
__device__ __forceinline__ float silu_grad_f(float h) {
  float s = sigmoidf_(h);
  return s * (1.0f + h * (1.0f - s));
}

}  // namespace moe
