// common.cuh -- device helpers shared by the selective-scan kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;

// Decay products below this bound end the backward reconstruction of a segment's initial state:
// the omitted remainder is at most kCarryEps * |state| at the stopping point.
constexpr float kCarryEps = 1.4901161193847656e-08f;  // 2^-26

// 2^x with the SFU approximation (denormal results flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// e^z - 1 without cancellation for small |z|: a Taylor polynomial of degree 6 for |z| < 1/8 (remainder
// below 1e-10 relative there), else expz - 1 where expz is an approximation of e^z.
__device__ __forceinline__ float expm1_small(float z, float expz) {
  float p = fmaf(z, 1.0f / 720.0f, 1.0f / 120.0f);
  p = fmaf(z, p, 1.0f / 24.0f);
  p = fmaf(z, p, 1.0f / 6.0f);
  p = fmaf(z, p, 0.5f);
  p = fmaf(z, p, 1.0f);
  p *= z;
  return fabsf(z) < 0.125f ? p : expz - 1.0f;
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  __device__ __forceinline__ static float load(const void* p, int64_t i) {
    return __ldg(static_cast<const float*>(p) + i);
  }
  __device__ __forceinline__ static void store(void* p, int64_t i, float v) {
    static_cast<float*>(p)[i] = v;
  }
};
template <> struct Elem<__nv_bfloat16> {
  __device__ __forceinline__ static float load(const void* p, int64_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  }
  __device__ __forceinline__ static void store(void* p, int64_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
};

}  // namespace ssm
