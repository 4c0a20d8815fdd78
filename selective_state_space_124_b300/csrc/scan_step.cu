// scan_step.cu -- one recurrent decode step ("Understanding Mamba" s3.2 / s10.1): for every (b, d) the
// N-entry state is read, advanced by Eq. (3) with this token's delta, B, C, written back in place, and
// y_t = C_t . h_t is produced.
//
// N = 16 with 16-byte-aligned rows (the common case): four lanes per channel, each owning four state
// entries, so every load and store of state, A_log, B and C is one coalesced 16-byte access per lane (a warp
// moves 512 contiguous bytes of state per instruction). The read-out sums the four lanes' partial dot products
// with two shuffles. A persistent grid walks the (batch, channel) quads. Other shapes: one thread per
// channel.
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
  // optional layer pieces (see ssm_scan_step_ex); warp-uniform branches on the pointers / flag
  const float* delta_bias;  // [D] or null
  int softplus;
  const float* D_skip;      // [D] or null
  const void* z;            // [batch, D] or null
};

__device__ __forceinline__ float step_delta(const StepParams& p, float raw, int64_t d) {
  const float v = p.delta_bias ? raw + __ldg(p.delta_bias + d) : raw;
  return p.softplus ? softplus_f(v) : v;
}

template <typename T>
__device__ __forceinline__ float step_output(const StepParams& p, float y, float x, int64_t ch, int64_t d) {
  if (p.D_skip) y = fmaf(__ldg(p.D_skip + d), x, y);
  if (p.z) y *= silu_f(Elem<T>::load(p.z, ch));
  return y;
}

// ---- N = 16: four lanes per channel ---------------------------------------------------------------------
template <typename T> struct Vec4;
template <> struct Vec4<float> {
  __device__ __forceinline__ static float4 load(const void* p, int64_t i) {  // elements i .. i+3
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i));
  }
};
template <> struct Vec4<__nv_bfloat16> {
  __device__ __forceinline__ static float4 load(const void* p, int64_t i) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p) + i));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
  }
};

// One state entry: dl = delta * log2(e), u = delta * x (Euler) or x (ZOH).
template <bool ZOH>
__device__ __forceinline__ float step_entry(float& h, float alog, float dl, float dt, float u, float bn, float cn) {
  const float a2 = alog * kLog2e;
  const float ea = ex2(a2);             // exp(A_log) = -A
  const float w = -ea * dl;             // delta * A * log2(e)
  const float e = exp2m1(w, ex2(w));    // Abar - 1
  float bx;
  if (ZOH) {  // (Abar - 1) / A = -e / exp(A_log); where A is 0 in fp32, its limit delta
    const float coef = ea == 0.0f ? dt : -e * ex2(-a2);
    bx = coef * bn * u;
  } else {
    bx = u * bn;
  }
  h = fmaf(e, h, h) + bx;
  return cn * h;
}

struct QuadIn {  // one lane's share of a channel: four state entries and their inputs
  float4 h, al, bb, cc;
  float xv, dt;
};

template <bool FUSED, typename T>
__device__ __forceinline__ void quad_load(const StepParams& p, int64_t ch, int q, QuadIn& v) {
  // batch * D < 2^31 is checked on the host: a 32-bit division is a short sequence, a 64-bit one is not
  const uint32_t b32 = static_cast<uint32_t>(ch) / static_cast<uint32_t>(p.D);
  const int64_t b = b32, d = ch - b * p.D;
  v.h = reinterpret_cast<const float4*>(p.state + ch * 16)[q];
  v.al = __ldg(reinterpret_cast<const float4*>(p.A_log + d * 16) + q);
  v.bb = Vec4<T>::load(p.B, b * 16 + 4 * q);
  v.cc = Vec4<T>::load(p.C, b * 16 + 4 * q);
  v.xv = Elem<T>::load(p.x, ch);
  v.dt = Elem<T>::load(p.delta, ch);
  if (FUSED) v.dt = step_delta(p, v.dt, d);
}

template <bool ZOH>
__device__ __forceinline__ float quad_step(QuadIn& v) {
  const float dl = v.dt * kLog2e, u = ZOH ? v.xv : v.dt * v.xv;
  float yv = step_entry<ZOH>(v.h.x, v.al.x, dl, v.dt, u, v.bb.x, v.cc.x);
  yv += step_entry<ZOH>(v.h.y, v.al.y, dl, v.dt, u, v.bb.y, v.cc.y);
  yv += step_entry<ZOH>(v.h.z, v.al.z, dl, v.dt, u, v.bb.z, v.cc.z);
  yv += step_entry<ZOH>(v.h.w, v.al.w, dl, v.dt, u, v.bb.w, v.cc.w);
  return yv;
}

// Persistent grid over the (channel, quad) items; each trip handles two items, both loaded before either is
// computed, so that every lane keeps two state rows' worth of loads in flight. FUSED = any of the optional
// layer pieces is present; without them the kernel carries none of their loads or branches.
template <bool ZOH, bool FUSED, typename T>
__global__ void __launch_bounds__(256) scan_step_quad_kernel(StepParams p, int64_t quads) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t span = 2 * stride;
  const int64_t bound = quads + (span - quads % span) % span;  // same trip count for every lane of a warp
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < bound; i0 += span) {
    const int64_t i1 = i0 + stride;
    const bool live0 = i0 < quads, live1 = i1 < quads;
    const int q = static_cast<int>(i0 & 3);  // stride is a multiple of 4: both items use entries 4q .. 4q+3
    QuadIn v0, v1;
    if (live0) quad_load<FUSED, T>(p, i0 >> 2, q, v0);
    if (live1) quad_load<FUSED, T>(p, i1 >> 2, q, v1);
    float y0 = 0.0f, y1 = 0.0f;
    if (live0) {
      y0 = quad_step<ZOH>(v0);
      reinterpret_cast<float4*>(p.state + (i0 >> 2) * 16)[q] = v0.h;
    }
    if (live1) {
      y1 = quad_step<ZOH>(v1);
      reinterpret_cast<float4*>(p.state + (i1 >> 2) * 16)[q] = v1.h;
    }
    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
    if (FUSED) {
      const int64_t c0 = i0 >> 2, c1 = i1 >> 2;
      if (live0 && q == 0) y0 = step_output<T>(p, y0, v0.xv, c0, static_cast<uint32_t>(c0) % static_cast<uint32_t>(p.D));
      if (live1 && q == 0) y1 = step_output<T>(p, y1, v1.xv, c1, static_cast<uint32_t>(c1) % static_cast<uint32_t>(p.D));
    }
    if (live0 && q == 0) Elem<T>::store(p.y, i0 >> 2, y0);
    if (live1 && q == 0) Elem<T>::store(p.y, i1 >> 2, y1);
  }
}

template <int NP, bool ZOH, typename T, bool VEC>
__global__ void __launch_bounds__(256) scan_step_kernel(StepParams p) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= p.batch * p.D) return;
  const int N = static_cast<int>(p.N);
  const int64_t b = i / p.D, d = i % p.D;
  const float xv = Elem<T>::load(p.x, i);
  const float dt = step_delta(p, Elem<T>::load(p.delta, i), d);
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
  Elem<T>::store(p.y, i, step_output<T>(p, yv, xv, i, d));
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
  const uintptr_t bc_align = sizeof(T) == 2 ? 7 : 15;
  if (sp.N == 16 && aligned && sp.batch * sp.D < (int64_t(1) << 31) && (reinterpret_cast<uintptr_t>(sp.A_log) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(sp.B) & bc_align) == 0 && (reinterpret_cast<uintptr_t>(sp.C) & bc_align) == 0) {
    const int64_t quads = sp.batch * sp.D * 4;
    int64_t blocks = (quads + 255) / 256;
    // 8 blocks of 256 threads per SM, each looping over items; at about 60 registers a thread 4 are resident at
    // a time (a one-wave grid of 4 per SM measured the same)
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    blocks = (blocks + 1) / 2;                                   // two items per lane per trip
    if (blocks > cap) blocks = cap;
    if (sp.delta_bias || sp.softplus || sp.D_skip || sp.z)
      scan_step_quad_kernel<ZOH, true, T><<<static_cast<unsigned>(blocks), 256, 0, s>>>(sp, quads);
    else
      scan_step_quad_kernel<ZOH, false, T><<<static_cast<unsigned>(blocks), 256, 0, s>>>(sp, quads);
    return cudaGetLastError();
  }
  if (sp.N == 16 && aligned) return go<16, ZOH, T, true>(sp, s);
  if (sp.N == 8 && aligned) return go<8, ZOH, T, true>(sp, s);
  if (sp.N == 4 && aligned) return go<4, ZOH, T, true>(sp, s);
  if (sp.N <= 4) return go<4, ZOH, T, false>(sp, s);
  if (sp.N <= 8) return go<8, ZOH, T, false>(sp, s);
  return go<16, ZOH, T, false>(sp, s);
}

}  // namespace

cudaError_t launch_step(const StepArgs& a) {
  StepParams sp{a.state, a.x, a.delta, a.A_log, a.B, a.C, a.y, a.batch, a.D, a.N,
                a.delta_bias, a.softplus, a.D_skip, a.z};
  if (a.disc == 1)
    return a.dtype == 1 ? pick<true, __nv_bfloat16>(sp, a.stream) : pick<true, float>(sp, a.stream);
  return a.dtype == 1 ? pick<false, __nv_bfloat16>(sp, a.stream) : pick<false, float>(sp, a.stream);
}

}  // namespace ssm
