// common.cuh -- device helpers shared by the selective-scan kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;

// Decay products below this bound end the backward reconstruction of a segment's initial state:
// the omitted remainder is at most kCarryEps * |state| at the stopping point.
constexpr float kCarryEps = 9.5367431640625e-07f;  // 2^-20

// 2^x with the SFU approximation (denormal results flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^w - 1 with no cancellation for small |w| (w = delta * A * log2(e)). For |w ln 2| < 1/32 the Taylor
// series to the cubic term (coefficients ln2^k / k!) is used: its remainder is below 4e-8 absolute, under the
// fp32 spacing of 1 + e, so the decay factor 1 + e stays exact to one rounding even when nothing decays for
// many steps. Above that bound a - 1, with a the SFU value of 2^w, has a relative error below 1e-5 and
// no accumulation problem (such entries forget within 32 steps).
__device__ __forceinline__ float exp2m1(float w, float a) {
  float q = fmaf(w, 0.05550410866482158f, 0.2402265069591007f);
  q = fmaf(w, q, 0.6931471805599453f);
  q *= w;
  return fabsf(w) < 0.04508422002825452f ? q : a - 1.0f;
}

// Reciprocal with the SFU approximation (relative error about one ulp; rcp(inf) = 0).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log(1 + u) for u in [0, 1] from the identity log(1 + u) = 2 artanh(s), s = u / (2 + u) <= 1/3, and the
// artanh series s + s^3/3 + ... + s^13/13 (the next term is below 5e-9 relative).
__device__ __forceinline__ float log1p_unit(float u) {
  const float s = u * rcp_approx(2.0f + u);
  const float t = s * s;
  float q = fmaf(t, 1.0f / 13.0f, 1.0f / 11.0f);
  q = fmaf(t, q, 1.0f / 9.0f);
  q = fmaf(t, q, 1.0f / 7.0f);
  q = fmaf(t, q, 1.0f / 5.0f);
  q = fmaf(t, q, 1.0f / 3.0f);
  q = fmaf(t, q, 1.0f);
  return 2.0f * s * q;
}

// softplus(v) = ln(1 + e^v) = max(v, 0) + log(1 + e^{-|v|}), with no overflow for large v.
__device__ __forceinline__ float softplus_f(float v) {
  return fmaxf(v, 0.0f) + log1p_unit(ex2(-fabsf(v) * kLog2e));
}

// SiLU(v) = v * sigma(v) = v / (1 + e^{-v}).
__device__ __forceinline__ float silu_f(float v) { return v * rcp_approx(1.0f + ex2(-v * kLog2e)); }

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
