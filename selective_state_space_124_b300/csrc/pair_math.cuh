// pair_math.cuh -- state entries two at a time (f32x2 arithmetic) for the structured decay A_n = (n + 1) A_0:
// every decay of a step follows from entry 0's by exact identities, so one SFU exp2 per (step, channel) serves
// all 16 entries.
#pragma once

#include "common.cuh"

namespace ssm {
namespace pairs {

__device__ __forceinline__ float2 bc(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// e_n = Abar_0^{n+1} - 1 for the first NP pairs (n < 2 NP) from e_0, by the exact identity
// e_{m+k+1} = e_m (1 + e_k) + e_k: no cancellation, and the relative error of e_n stays that of e_0.
template <int NP>
__device__ __forceinline__ void em1_tree(float e0, float2 (&e)[8]) {
  const float e1 = fmaf(e0, 1.0f + e0, e0);
  e[0] = make_float2(e0, e1);
  if (NP > 1) e[1] = fma2(e[0], bc(1.0f + e1), bc(e1));  // e2 e3
  if (NP > 2) {
    const float2 a3 = bc(1.0f + e[1].y), e3 = bc(e[1].y);
    e[2] = fma2(e[0], a3, e3);  // e4 e5
    e[3] = fma2(e[1], a3, e3);  // e6 e7
  }
  if (NP > 4) {
    const float2 a7 = bc(1.0f + e[3].y), e7 = bc(e[3].y);
#pragma unroll
    for (int k = 0; k < 4; ++k) e[4 + k] = fma2(e[k], a7, e7);
  }
}

// e_n for all 16 entries of one step: w = delta A_0 log2(e).
__device__ __forceinline__ void step_e16(float w, float2 (&e)[8]) { em1_tree<8>(exp2m1(w, ex2(w)), e); }

// P_n = p^{n+1} for the first NP pairs (a decay weight; relative error about (n + 1) times that of p).
template <int NP>
__device__ __forceinline__ void powers(float p, float2 (&P)[8]) {
  P[0] = make_float2(p, p * p);
  if (NP > 1) P[1] = mul2(P[0], bc(P[0].y));  // p^3 p^4
  if (NP > 2) {
    const float2 p4 = bc(P[1].y);
    P[2] = mul2(P[0], p4);
    P[3] = mul2(P[1], p4);
  }
  if (NP > 4) {
    const float2 p8 = bc(P[3].y);
#pragma unroll
    for (int k = 0; k < 4; ++k) P[4 + k] = mul2(P[k], p8);
  }
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Pairs still above the truncation weight, given the largest entry-0 weight pmax of the warp (entry n's
// weight is pmax^{n+1}, decreasing in n): 8, 4, 2 or 1 leading pairs, or 0 once entry 0 is below it too.
__device__ __forceinline__ int live_pairs(float pmax) {
  if (!(pmax >= kCarryEps)) return 0;
  const float p2 = pmax * pmax, p3 = p2 * pmax, p5 = p3 * p2, p9 = p5 * p2 * p2;
  return p9 >= kCarryEps ? 8 : p5 >= kCarryEps ? 4 : p3 >= kCarryEps ? 2 : 1;
}

}  // namespace pairs
}  // namespace ssm
