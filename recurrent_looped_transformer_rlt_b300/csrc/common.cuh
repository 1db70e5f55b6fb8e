// Common device helpers for the RLT kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

namespace rlt {

using bf16 = __nv_bfloat16;

// Storage-type conversions.  bf16 rounding is round-to-nearest-even
// (__float2bfloat16_rn), the only rounding the bf16 configurations use.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }
// Round an fp32 value through the storage type (identity for fp32).
template <typename T> __device__ __forceinline__ float round_st(float x) { return to_f32(from_f32<T>(x)); }
// Four consecutive values rounded to the storage type and written with one
// store (p aligned to 4 elements: 8 bytes for bf16, 16 for fp32).
template <typename T> __device__ __forceinline__ void store4_st(T* p, float4 v);
template <> __device__ __forceinline__ void store4_st<float>(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
template <> __device__ __forceinline__ void store4_st<bf16>(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<unsigned*>(&a);
  u.y = *reinterpret_cast<unsigned*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

template <typename T> __device__ __forceinline__ T nan_of();
template <> __device__ __forceinline__ float nan_of<float>() { return __int_as_float(0x7fc00000); }
template <> __device__ __forceinline__ bf16 nan_of<bf16>() { return __ushort_as_bfloat16((unsigned short)0x7fc0); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Sum over each half-warp (lanes 0-15 and 16-31 separately), butterfly
// order.  Each half-warp synchronises only its own 16 lanes, so a caller may
// have one half of a warp take a different path than the other (each half
// must be converged in itself).  1-D blocks: the half is bit 4 of the thread
// index.
__device__ __forceinline__ float half_warp_sum(float v) {
  const unsigned mask = (threadIdx.x & 16) ? 0xffff0000u : 0x0000ffffu;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(mask, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Device status flag (first word of the workspace).  The first error wins.
__device__ __forceinline__ void set_error(int* flag, int code) { atomicCAS(flag, 0, code); }

// Status codes mirrored from rlt.h for device code.
constexpr int kErrTimeout = -5;
constexpr int kErrBounds = -6;

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + __expf(-x)); }

// Step context read by the per-step kernels so that one captured step can be
// replayed: pos = position consumed by this step (0-based), step = index of
// the step inside the current call.
struct StepCtx {
  int pos;
  int step;
};

// Host-side set-up that CUDA keeps per device (a kernel's dynamic shared
// memory limit, occupancy): computed once for each device the process uses,
// under a lock, on the calling thread's current device.  get() returns the
// stored value (compute() must return non-zero), or -1 for a device index
// outside the table.
struct PerDevice {
  static constexpr int kMaxDevices = 128;
  std::mutex mu;
  int val[kMaxDevices] = {};
  template <class F>
  int get(F&& compute) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    std::lock_guard<std::mutex> lk(mu);
    if (val[dev] == 0) val[dev] = compute();
    return val[dev];
  }
};

}  // namespace rlt
