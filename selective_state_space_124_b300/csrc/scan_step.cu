// scan_step.cu -- one recurrent decode step ("Understanding Mamba" s3.2 / s10.1): for every (b, d) the
// N-entry state is read, advanced by Eq. (3) with this token's delta, B, C, written back in place, and
// y_t = C_t . h_t is produced. One thread per channel; the state row (N floats) is contiguous, so a warp
// reads and writes 32 consecutive rows.
#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

struct StepParams {
  float* state;
  const void* x;
  const void* delta;
  const float* A_log;
  const void* B;
  const void* C;
  void* y;
  int64_t batch, D, N;
};

template <int NP, bool ZOH, typename T, bool VEC>
__global__ void __launch_bounds__(256) scan_step_kernel(StepParams p) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= p.batch * p.D) return;
  const int N = static_cast<int>(p.N);
  const int64_t b = i / p.D, d = i % p.D;
  const float xv = Elem<T>::load(p.x, i);
  const float dt = Elem<T>::load(p.delta, i);
  float h[NP];
  float* srow = p.state + i * N;
  if (VEC) {
#pragma unroll
    for (int q = 0; q < NP / 4; ++q) {
      float4 v = reinterpret_cast<const float4*>(srow)[q];
      h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int n = 0; n < NP; ++n) h[n] = (n < N) ? srow[n] : 0.0f;
  }
  float yv = 0.0f;
#pragma unroll
  for (int n = 0; n < NP; ++n) {
    if (!VEC && n >= N) break;
    const float A = -ex2(__ldg(p.A_log + d * N + n) * kLog2e);
    const float w = dt * A * kLog2e;
    const float e = exp2m1(w, ex2(w));  // Abar - 1
    const float bn = Elem<T>::load(p.B, b * N + n);
    const float cn = Elem<T>::load(p.C, b * N + n);
    float bx;
    if (ZOH) {
      bx = (A == 0.0f ? dt : e / A) * bn * xv;
    } else {
      bx = dt * bn * xv;
    }
    h[n] = fmaf(e, h[n], h[n]) + bx;
    yv = fmaf(cn, h[n], yv);
  }
  if (VEC) {
#pragma unroll
    for (int q = 0; q < NP / 4; ++q)
      reinterpret_cast<float4*>(srow)[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
  } else {
#pragma unroll
    for (int n = 0; n < NP; ++n)
      if (n < N) srow[n] = h[n];
  }
  Elem<T>::store(p.y, i, yv);
}

template <int NP, bool ZOH, typename T, bool VEC>
cudaError_t go(const StepParams& sp, cudaStream_t s) {
  const int64_t n = sp.batch * sp.D;
  scan_step_kernel<NP, ZOH, T, VEC><<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(sp);
  return cudaGetLastError();
}

template <bool ZOH, typename T>
cudaError_t pick(const StepParams& sp, cudaStream_t s) {
  const bool aligned = (reinterpret_cast<uintptr_t>(sp.state) & 15) == 0;
  if (sp.N == 16 && aligned) return go<16, ZOH, T, true>(sp, s);
  if (sp.N == 8 && aligned) return go<8, ZOH, T, true>(sp, s);
  if (sp.N == 4 && aligned) return go<4, ZOH, T, true>(sp, s);
  if (sp.N <= 4) return go<4, ZOH, T, false>(sp, s);
  if (sp.N <= 8) return go<8, ZOH, T, false>(sp, s);
  return go<16, ZOH, T, false>(sp, s);
}

}  // namespace

cudaError_t launch_step(const StepArgs& a) {
  StepParams sp{a.state, a.x, a.delta, a.A_log, a.B, a.C, a.y, a.batch, a.D, a.N};
  if (a.disc == 1)
    return a.dtype == 1 ? pick<true, __nv_bfloat16>(sp, a.stream) : pick<true, float>(sp, a.stream);
  return a.dtype == 1 ? pick<false, __nv_bfloat16>(sp, a.stream) : pick<false, float>(sp, a.stream);
}

}  // namespace ssm
