// scan_fwd_tma.cu -- the prefill scan for N = 16 and 16-byte-aligned rows: TMA-staged, one independent
// pipeline per warp, persistent over an even split of the (channel group, time) work.
//
// Layout of the work. A warp owns 32 consecutive channels of one batch element (one lane per channel, the
// 16 state entries in registers as 8 float pairs). The rows (batch b, channel group g) have their time
// axes laid end to end, and that line is cut into equal contiguous ranges, one per warp of the grid: every
// warp gets the same number of (channel, step) elements whatever the batch / length mix. Warps never wait
// on one another: each has its own shared-memory rings, its own mbarriers, and issues its own TMA copies
// (lane 0), so one warp's carry warm-up never stalls another.
//
// Carry without communication. A range that starts at t0 > 0 rebuilds the state entering t0 by walking
// the preceding steps backwards and summing prod_{k>j} Abar_k * Bbar_j x_j ("Mathematical Prerequisites
// for Mamba" s6, the unrolled sum of the recurrence), to t = 0 (exact) or until the decay product of an
// entry falls below 2^-20 for every lane of the warp: the omitted remainder of that entry is then at most
// 2^-20 (under 1e-6) of its state at that point, about the rounding noise a long fp32 recurrence carries
// anyway. For the S4D-structured A (A_n = (n + 1) A_0) the entries decay at
// rates 1..16 x A_0, so the walk drops state pairs as they die (8 -> 4 -> 2 -> 1 pairs active): the
// warm-up costs about a quarter of a full walk.
//
// Data movement. Per warp, a forward ring of NSF stages holds [TS steps x 32 channels] tiles of x and
// delta (and of the gate input z when the layer's gate is fused) and [TS x 16] tiles of B and C; a warm-up
// ring of NSW stages holds the x, delta, B tiles the backward walk reads. Both rings are filled by cp.async.bulk.tensor (TMA) with mbarrier completion;
// the forward ring is primed when a range starts, so its copies overlap the warm-up. B and C are read
// as shared-memory broadcasts (bf16 tiles are widened to fp32 once per stage by the warp; for the
// structured ZOH update the warp also divides B by n + 1 there, once per stage). y is stored straight to global memory (a warp writes 32 consecutive
// channels of one step). Every wait is bounded (%globaltimer): a wait that runs out sets a device
// status word that ssm_check_device() reports as SSM_ERR_TIMEOUT.
//
// Arithmetic (per step t, channel d, entry n; two entries per instruction with f32x2 FMA):
//  * structured channels (A_n = (n + 1) A_0 within 4 ulp, checked per warp): one SFU exp2 per (t, d),
//    e_n = Abar_n - 1 = Abar_0^{n+1} - 1 for all n by e_{m+k+1} = e_m (1 + e_k) + e_k from an e_0
//    computed without cancellation, so the decay h + e h is exact to one rounding even where nothing
//    decays for many steps.
//      Euler: h_n <- (h_n + e_n h_n) + (delta x) B_n                     (two FMAs)
//      ZOH:   h_n <- h_n + e_n (h_n + q_n), q_n = (B_n / (n+1)) (x / A_0)  (two FMAs; = Abar h + (Abar-1)/A B x)
//  * other channels: e_n = 2^{delta A_n log2 e} - 1 per entry, h_n <- (h_n + e_n h_n) + Bbar x.
//  * y = sum_n C_n h_n.
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace ssm {

__device__ int g_device_status = 0;  // nonzero: a bounded wait ran out (read by ssm_check_device)

namespace {

constexpr unsigned long long kWaitNs = kDefaultWaitNs;  // 2 s: the bound on the drains before a warp exits
constexpr float kDeadLog2 = -20.0f;                      // log2 of the decay bound that ends a warm-up

template <typename T, int CPL, int TS, int NSF, int TSW, int NSW>
struct alignas(128) WarpRing {
  static constexpr int CW = 32 * CPL;  // channels per warp
  T fx[NSF][TS * CW];   // forward ring: x, delta tiles [TS][CW]
  T fd[NSF][TS * CW];
  T fB[NSF][TS * 16];   // B, C tiles [TS][16]
  T fC[NSF][TS * 16];
  T wx[NSW][TSW * CW];  // warm-up ring: x, delta, B tiles of TSW steps
  T wd[NSW][TSW * CW];
  T wB[NSW][TSW * 16];
  static constexpr int kConvRows = sizeof(T) == 2 ? TS : 1;  // only bf16 inputs need the widened C
  float Bf[TS * 16];         // B of the stage being consumed as fp32 (bf16 inputs; structured ZOH: / (n + 1))
  float Cf[kConvRows * 16];  // C of the stage being consumed, widened to fp32 (bf16 inputs)
  unsigned long long fbar[NSF];
  unsigned long long wbar[NSW];
};

struct TmaParams {
  const float* A_log;
  const float* h0;
  void* y;
  float* final_state;
  int64_t L, D;
  int64_t G;        // channel groups (of 32 * CPL channels) per batch element
  int64_t total;    // batch * G * L
  int64_t nwarps;   // warps taking part
  // fused layer pieces (see ssm_scan_fwd_ex). Kept after the fields above: placed before them, the long
  // fp32 ZOH scan measured 4% slower with the same registers and instruction mix.
  const float* delta_bias;  // [D] or null
  const float* D_skip;      // [D] or null
  const void* z;            // [batch, L, D] or null
  unsigned long long wait_ns;  // bound on one consumer wait (ssm_set_wait_limit_ns)
};

// ---- PTX wrappers -----------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(unsigned long long* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(unsigned long long* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(unsigned long long* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test(unsigned long long* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait by every lane of the warp; the outcome is warp-uniform. One non-blocking probe, then
// blocking probes until limit_ns have passed. false: the phase did not complete in time (the device
// status word is set). Consumers pass the launch's limit (ssm_set_wait_limit_ns); the drains before a
// warp exits pass kWaitNs.
__device__ __forceinline__ bool mbar_wait(unsigned long long* b, uint32_t parity, unsigned long long limit_ns) {
  bool ok = mbar_test(b, parity);
  if (!ok) {
    const unsigned long long t0 = gtimer();
    while (gtimer() - t0 < limit_ns) {
      if ((ok = mbar_try(b, parity))) break;
    }
  }
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) atomicExch(&g_device_status, 4);
  return ok;
}
__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, int c0, int c1, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(su32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float2 bc2(float v) { return make_float2(v, v); }

template <typename T> __device__ __forceinline__ float tof(T v);
template <> __device__ __forceinline__ float tof<float>(float v) { return v; }
template <> __device__ __forceinline__ float tof<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Streaming (evict-first) store of one output, predicated inside the instruction so that a guarded
// store adds no branch: the steps of an unrolled tile stay one basic block the scheduler can interleave.
// No "memory" clobber: y is written only, never read by the kernel.
__device__ __forceinline__ void store_y(float* p, float v, bool pred) {
  asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q st.global.cs.f32 [%0], %1;\n}\n"
               ::"l"(p), "f"(v), "r"(static_cast<int>(pred)));
}
__device__ __forceinline__ void store_y(float* p, float v) { asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v)); }
__device__ __forceinline__ void store_y(__nv_bfloat16* p, float v) {
  const unsigned short bits = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  asm volatile("st.global.cs.b16 [%0], %1;" ::"l"(p), "h"(bits));
}
__device__ __forceinline__ void store_y(__nv_bfloat16* p, float v, bool pred) {
  const unsigned short bits = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q st.global.cs.b16 [%0], %1;\n}\n"
               ::"l"(p), "h"(bits), "r"(static_cast<int>(pred)));
}

// Pair k of a 16-entry B row (entries 2k, 2k+1) as fp32.
__device__ __forceinline__ float2 ld_pair(const float* row, int k) { return reinterpret_cast<const float2*>(row)[k]; }
__device__ __forceinline__ float2 ld_pair(const __nv_bfloat16* row, int k) {
  return __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(row)[k]);
}

// e_n = Abar_0^{n+1} - 1 for the first NP pairs (n < 2 NP) from e_0, by the exact identity
// e_{m+k+1} = e_m (1 + e_k) + e_k. Relative errors stay those of e_0 (no amplification with n).
template <int NP>
__device__ __forceinline__ void em1_tree(float e0, float2 (&e)[8]) {
  const float e1 = fmaf(e0, 1.0f + e0, e0);
  e[0] = make_float2(e0, e1);
  if (NP > 1) e[1] = __ffma2_rn(e[0], bc2(1.0f + e1), bc2(e1));  // e2 e3
  if (NP > 2) {
    const float2 a3 = bc2(1.0f + e[1].y), e3 = bc2(e[1].y);
    e[2] = __ffma2_rn(e[0], a3, e3);  // e4 e5
    e[3] = __ffma2_rn(e[1], a3, e3);  // e6 e7
  }
  if (NP > 4) {
    const float2 a7 = bc2(1.0f + e[3].y), e7 = bc2(e[3].y);
    e[4] = __ffma2_rn(e[0], a7, e7);
    e[5] = __ffma2_rn(e[1], a7, e7);
    e[6] = __ffma2_rn(e[2], a7, e7);
    e[7] = __ffma2_rn(e[3], a7, e7);
  }
}

// P_n = p^{n+1} for the first NP pairs (a decay weight; relative error about (n + 1) times that of p).
template <int NP>
__device__ __forceinline__ void powers(float p, float2 (&P)[8]) {
  P[0] = make_float2(p, p * p);
  if (NP > 1) P[1] = __fmul2_rn(P[0], bc2(P[0].y));  // p^3 p^4
  if (NP > 2) {
    const float2 p4 = bc2(P[1].y);
    P[2] = __fmul2_rn(P[0], p4);
    P[3] = __fmul2_rn(P[1], p4);
  }
  if (NP > 4) {
    const float2 p8 = bc2(P[3].y);
    P[4] = __fmul2_rn(P[0], p8);
    P[5] = __fmul2_rn(P[1], p8);
    P[6] = __fmul2_rn(P[2], p8);
    P[7] = __fmul2_rn(P[3], p8);
  }
}

struct ChanGen {  // per-channel constants of the generic (unstructured A) path
  float A2[16], invA[16];  // A log2(e); 1/A (0 where A == 0)
  float A2max;             // the slowest decay rate, max_n A2[n] (<= 0)
};

// Generic terms of one forward step for pair k: e = Abar - 1 and the input term Bbar x.
// ZOH uses (Abar - 1) / A * B x, or delta * B * x where A == 0 (its limit).
template <bool ZOH>
__device__ __forceinline__ void gen_pair(const ChanGen& g, int k, float dv, float xv, float2 bb, float2& e,
                                         float2& bx) {
  const float w0 = dv * g.A2[2 * k], w1 = dv * g.A2[2 * k + 1];
  e = make_float2(exp2m1(w0, ex2(w0)), exp2m1(w1, ex2(w1)));
  if (ZOH) {
    const float c0 = g.invA[2 * k] == 0.0f ? dv : e.x * g.invA[2 * k];
    const float c1 = g.invA[2 * k + 1] == 0.0f ? dv : e.y * g.invA[2 * k + 1];
    bx = __fmul2_rn(make_float2(c0, c1), __fmul2_rn(bb, bc2(xv)));
  } else {
    bx = __fmul2_rn(bc2(dv * xv), bb);
  }
}

// ---- fused layer pieces --------------------------------------------------------------------------------
// DX: how the scan reads delta. 0: as given; 2: softplus(delta + bias[d]) ("Understanding Mamba" Eq. (6)).
// EPI: 0: y as read out; 1: y + D[d] x (Eq. (1)/(3) feedthrough); 2: (y + D[d] x) * SiLU(z) (Eq. (9) gate).
template <int DX>
__device__ __forceinline__ float delta_in(float raw, float bias) {
  if (DX == 2) return softplus_f(raw + bias);
  if (DX == 1) return raw + bias;
  return raw;
}
template <int EPI>
__device__ __forceinline__ float epilogue(float y, float x, float dskip, float z) {
  if (EPI == 0) return y;
  const float v = fmaf(dskip, x, y);
  return EPI == 2 ? v * silu_f(z) : v;
}

// ---- backward warm-up over one staged tile (rows i = n-1 .. 0 of the tile, i.e. steps hi-1 .. lo) -------
// Structured A, NP pairs active. W[c] is log2 of the decay of entry 0 of channel c over the steps after the
// current one (running sum of delta * A_0 log2 e); P[c] holds the matching decay weights of the active pairs.
template <int NP, bool ZOH, int CPL, int DX, typename T>
__device__ __forceinline__ void warm_s4d_step(const T* xs, const T* ds, const T* Bs, int i, int lane,
                                              const float (&A2_0)[CPL], const float (&invA0)[CPL],
                                              const float (&dbias)[CPL], float (&W)[CPL], float2 (&P)[CPL][8],
                                              float2 (&h)[CPL][8]) {
  constexpr int CW = 32 * CPL;
  const T* Brow = Bs + i * 16;
  float2 bp[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) bp[k] = ld_pair(Brow, k);
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const float xv = tof<T>(xs[i * CW + c * 32 + lane]);
    const float dv = delta_in<DX>(tof<T>(ds[i * CW + c * 32 + lane]), dbias[c]);
    const float w = dv * A2_0[c];
    if (ZOH) {
      // contribution P_n (Abar_n - 1) / A_n B_n x = (P_n e_n) B_n (x / A_0) / (n + 1); the 1/(n+1) is applied
      // once when the walk ends.
      float2 e[8];
      em1_tree<NP>(exp2m1(w, ex2(w)), e);
      const float2 xi = bc2(xv * invA0[c]);
#pragma unroll
      for (int k = 0; k < NP; ++k)
        h[c][k] = __ffma2_rn(__fmul2_rn(P[c][k], e[k]), __fmul2_rn(bp[k], xi), h[c][k]);
    } else {
      const float2 u = bc2(dv * xv);
#pragma unroll
      for (int k = 0; k < NP; ++k) h[c][k] = __ffma2_rn(P[c][k], __fmul2_rn(bp[k], u), h[c][k]);
    }
    W[c] += w;
    powers<NP>(ex2(W[c]), P[c]);
  }
}

template <int NP, bool ZOH, int CPL, int TS, int DX, typename T>
__device__ __forceinline__ void warm_s4d(const T* xs, const T* ds, const T* Bs, int n, int lane,
                                         const float (&A2_0)[CPL], const float (&invA0)[CPL],
                                         const float (&dbias)[CPL], float (&W)[CPL], float2 (&P)[CPL][8],
                                         float2 (&h)[CPL][8]) {
  if (n == TS) {
#pragma unroll
    for (int i = TS - 1; i >= 0; --i)
      warm_s4d_step<NP, ZOH, CPL, DX>(xs, ds, Bs, i, lane, A2_0, invA0, dbias, W, P, h);
  } else {
#pragma unroll 1
    for (int i = n - 1; i >= 0; --i)
      warm_s4d_step<NP, ZOH, CPL, DX>(xs, ds, Bs, i, lane, A2_0, invA0, dbias, W, P, h);
  }
}

// Generic A, all pairs. S[c] is the running sum of delta over the steps after the current one.
template <bool ZOH, int CPL, int DX, typename T>
__device__ __forceinline__ void warm_gen(const T* xs, const T* ds, const T* Bs, int n, int lane,
                                         const ChanGen (&g)[CPL], const float (&dbias)[CPL], float (&S)[CPL],
                                         float2 (&P)[CPL][8], float2 (&h)[CPL][8]) {
  constexpr int CW = 32 * CPL;
#pragma unroll 1
  for (int i = n - 1; i >= 0; --i) {
    const T* Brow = Bs + i * 16;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const float xv = tof<T>(xs[i * CW + c * 32 + lane]);
      const float dv = delta_in<DX>(tof<T>(ds[i * CW + c * 32 + lane]), dbias[c]);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float2 e, bx;
        gen_pair<ZOH>(g[c], k, dv, xv, ld_pair(Brow, k), e, bx);
        h[c][k] = __ffma2_rn(P[c][k], bx, h[c][k]);
      }
      S[c] += dv;
#pragma unroll
      for (int k = 0; k < 8; ++k) P[c][k] = make_float2(ex2(g[c].A2[2 * k] * S[c]), ex2(g[c].A2[2 * k + 1] * S[c]));
    }
  }
}

// ---- one forward step (structured A) for the CPL channels of a lane, from fp32 B / C rows in shared memory -
// Split in two: the per-step decay factors e and input scalar s depend only on x and delta (fwd_prep), the
// recurrence and read-out (fwd_core) on the carried state. A stage computes step i+1's fwd_prep before step
// i's fwd_core, so the scheduler always has the next step's independent decay tree to interleave with the
// current step's dependent update chain.
template <bool ZOH, int CPL>
__device__ __forceinline__ void fwd_prep(const float (&xv)[CPL], const float (&dv)[CPL], const float (&A2_0)[CPL],
                                         const float (&invA0)[CPL], float2 (&e)[CPL][8], float2 (&s)[CPL]) {
  // dv is the delta the recurrence uses (already through delta_in)
#pragma unroll
  for (int c = 0; c < CPL; ++c) {  // s: x / A_0 (ZOH) or delta * x (Euler)
    const float w = dv[c] * A2_0[c];
    em1_tree<8>(exp2m1(w, ex2(w)), e[c]);
    s[c] = bc2(ZOH ? xv[c] * invA0[c] : dv[c] * xv[c]);
  }
}

template <bool ZOH, int CPL>
__device__ __forceinline__ void fwd_core(const float2 (&e)[CPL][8], const float2 (&s)[CPL], const float* Brow,
                                         const float* Crow, float2 (&h)[CPL][8], float (&y)[CPL]) {
  const float4* Bq = reinterpret_cast<const float4*>(Brow);
  const float4* Cq = reinterpret_cast<const float4*>(Crow);
  float2 ya[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) ya[c] = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 bb = Bq[q], cc = Cq[q];
    const float2 b0 = make_float2(bb.x, bb.y), b1 = make_float2(bb.z, bb.w);  // ZOH: already B_n / (n + 1)
    const float2 c0 = make_float2(cc.x, cc.y), c1 = make_float2(cc.z, cc.w);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      float2& h0 = h[c][2 * q];
      float2& h1 = h[c][2 * q + 1];
      if (ZOH) {  // h <- Abar h + (Abar - 1) q  ==  h + e (h + q),  q = (B / (n+1)) (x / A_0)
        h0 = __ffma2_rn(e[c][2 * q], __ffma2_rn(b0, s[c], h0), h0);
        h1 = __ffma2_rn(e[c][2 * q + 1], __ffma2_rn(b1, s[c], h1), h1);
      } else {    // h <- Abar h + (delta x) B  ==  (h + e h) + u B
        h0 = __ffma2_rn(s[c], b0, __ffma2_rn(e[c][2 * q], h0, h0));
        h1 = __ffma2_rn(s[c], b1, __ffma2_rn(e[c][2 * q + 1], h1, h1));
      }
      ya[c] = __ffma2_rn(c0, h0, ya[c]);
      ya[c] = __ffma2_rn(c1, h1, ya[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < CPL; ++c) y[c] = ya[c].x + ya[c].y;
}

template <bool ZOH, int CPL>
__device__ __forceinline__ void fwd_s4d(const float (&xv)[CPL], const float (&dv)[CPL], const float* Brow,
                                        const float* Crow, const float (&A2_0)[CPL], const float (&invA0)[CPL],
                                        float2 (&h)[CPL][8], float (&y)[CPL]) {
  float2 e[CPL][8];
  float2 s[CPL];
  fwd_prep<ZOH, CPL>(xv, dv, A2_0, invA0, e, s);
  fwd_core<ZOH, CPL>(e, s, Brow, Crow, h, y);
}

template <bool ZOH>
__device__ __forceinline__ float fwd_gen(float xv, float dv, const float* Brow, const float* Crow, const ChanGen& g,
                                         float2 (&h)[8]) {
  float2 ya = make_float2(0.0f, 0.0f), yb = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 bb = reinterpret_cast<const float2*>(Brow)[k];
    const float2 cc = reinterpret_cast<const float2*>(Crow)[k];
    float2 e, bx;
    gen_pair<ZOH>(g, k, dv, xv, bb, e, bx);
    h[k] = __fadd2_rn(__ffma2_rn(e, h[k], h[k]), bx);
    if (k & 1) yb = __ffma2_rn(cc, h[k], yb);
    else ya = __ffma2_rn(cc, h[k], ya);
  }
  return (ya.x + ya.y) + (yb.x + yb.y);
}

// Shared state of one warp's pipelines.
struct WarpPipe {
  uint32_t cseq;        // forward stages consumed
  uint32_t wiss, wcon;  // warm-up stages issued / consumed (over the warp's lifetime)
};

// Start of a warm-up walk into t0 > 0: wait for the copies a previous walk left in flight, then issue the
// first NSW tiles (before the caller's global loads of A_log, so their latency overlaps). Returns the number
// of tiles issued (all lanes), or -1 if a wait ran out.
template <typename T, int CPL, int TS, int NSF, int TSW, int NSW>
__device__ __forceinline__ int warm_prologue(WarpRing<T, CPL, TS, NSF, TSW, NSW>& r, const CUtensorMap* mx,
                                             const CUtensorMap* md, const CUtensorMap* mB, int lane, int64_t trow0,
                                             int col, int64_t t0, WarpPipe& wp) {
  constexpr int CW = 32 * CPL;
  constexpr uint32_t kWarmBytes = (2u * TSW * CW + TSW * 16) * sizeof(T);
  while (wp.wcon < wp.wiss) {
    if (!mbar_wait(&r.wbar[wp.wcon % NSW], (wp.wcon / NSW) & 1u, kWaitNs)) return -1;
    ++wp.wcon;
  }
  int kiss = 0;
#pragma unroll 1
  for (int i = 0; i < NSW; ++i) {
    const int64_t thi = t0 - static_cast<int64_t>(kiss) * TSW;
    if (thi <= 0) break;
    const int64_t tlo = thi - TSW > 0 ? thi - TSW : 0;
    if (lane == 0) {
      const int slot = static_cast<int>(wp.wiss % NSW);
      const int trow = static_cast<int>(trow0 + tlo);
      mbar_arrive_tx(&r.wbar[slot], kWarmBytes);
      tma_load(r.wx[slot], mx, col, trow, &r.wbar[slot]);
      tma_load(r.wd[slot], md, col, trow, &r.wbar[slot]);
      tma_load(r.wB[slot], mB, 0, trow, &r.wbar[slot]);
    }
    ++kiss;
    ++wp.wiss;
  }
  __syncwarp();
  return kiss;
}

// One piece of a warp's range: row (batch b, channel group), steps [t0, t1). Warm-up (t0 > 0), forward with
// y stores, final state (t1 == L). S4D selects the structured-A arithmetic at compile time, so the two
// paths do not hold each other's per-channel constants in registers. Returns false if a wait ran out.
template <bool S4D, typename T, bool ZOH, int CPL, int TS, int NSF, int TSW, int NSW, int DX, int EPI,
          typename IssueFwd>
__device__ __forceinline__ bool run_piece(WarpRing<T, CPL, TS, NSF, TSW, NSW>& r, const TmaParams& p,
                                          const CUtensorMap* mx, const CUtensorMap* md, const CUtensorMap* mB,
                                          int lane, int64_t row, int64_t t0, int64_t t1, WarpPipe& wp,
                                          IssueFwd& issue_fwd, int kiss0, const T* zr) {
  constexpr int CW = 32 * CPL;
  // With the gate, z comes through the forward ring like x and delta (zr: this warp's NSF stages of [TS][CW]
  // tiles): read from global memory inside the steps, each step waited for its own load.
  constexpr bool kZs = EPI == 2;
  constexpr bool kConv = sizeof(T) == 2;  // bf16: consumers read B and C from the widened Bf / Cf
  constexpr uint32_t kWarmBytes = (2u * TSW * CW + TSW * 16) * sizeof(T);
  const int64_t L = p.L;
  const int64_t b = row / p.G;
  const int64_t d0 = (row % p.G) * CW + lane;  // channel c of this lane is d0 + 32 c
  bool act[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) act[c] = d0 + 32 * c < p.D;
  const bool full = (row % p.G) * CW + CW <= p.D;  // every channel of the warp exists

  // ---- per-channel constants ----
  float dbias[CPL], dskip[CPL];  // fused pieces: delta bias, feedthrough D (0 where not given)
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const int64_t d = d0 + 32 * c;
    dbias[c] = (DX != 0 && act[c] && p.delta_bias) ? __ldg(p.delta_bias + d) : 0.0f;
    dskip[c] = (EPI != 0 && act[c] && p.D_skip) ? __ldg(p.D_skip + d) : 0.0f;
  }
  float A2_0[CPL], invA0[CPL];  // structured: A_0 log2(e), 1 / A_0
  ChanGen g[S4D ? 1 : CPL];     // generic: every entry's rate
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const int64_t d = d0 + 32 * c;
    if constexpr (S4D) {
      const float A0 = act[c] ? -expf(__ldg(p.A_log + d * 16)) : -1.0f;
      A2_0[c] = A0 * kLog2e;
      invA0[c] = 1.0f / A0;
    } else {
      ChanGen& gc = g[S4D ? 0 : c];
      gc.A2max = -3.0e38f;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const float A = act[c] ? -expf(__ldg(p.A_log + d * 16 + n)) : -static_cast<float>(n + 1);
        gc.A2[n] = A * kLog2e;
        gc.invA[n] = A == 0.0f ? 0.0f : 1.0f / A;
        gc.A2max = fmaxf(gc.A2max, gc.A2[n]);
      }
    }
  }

  float2 h[CPL][8];
#pragma unroll
  for (int c = 0; c < CPL; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) h[c][k] = make_float2(0.0f, 0.0f);
  const float* h0row[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) h0row[c] = (p.h0 && act[c]) ? p.h0 + (b * p.D + d0 + 32 * c) * 16 : nullptr;

  if (t0 == 0) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      if (h0row[c]) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 v = reinterpret_cast<const float4*>(h0row[c])[k];
          h[c][2 * k] = make_float2(v.x, v.y);
          h[c][2 * k + 1] = make_float2(v.z, v.w);
        }
      }
    }
  } else {
    // ---- state entering t0: backward walk over warm-up tiles (the first NSW were issued by the caller) ----
    int kiss = kiss0;  // warm-up tiles issued for this walk (tile k covers [max(t0 - (k+1) TSW, 0), t0 - k TSW))
    const int col = static_cast<int>((row % p.G) * CW);
    auto issue_warm = [&]() {
      const int64_t thi = t0 - static_cast<int64_t>(kiss) * TSW;
      if (thi <= 0) return;
      const int64_t tlo = thi - TSW > 0 ? thi - TSW : 0;
      const int slot = static_cast<int>(wp.wiss % NSW);
      const int trow = static_cast<int>(b * L + tlo);
      if (lane == 0) {
        mbar_arrive_tx(&r.wbar[slot], kWarmBytes);
        tma_load(r.wx[slot], mx, col, trow, &r.wbar[slot]);
        tma_load(r.wd[slot], md, col, trow, &r.wbar[slot]);
        tma_load(r.wB[slot], mB, 0, trow, &r.wbar[slot]);
      }
      ++kiss;  // every lane keeps the counters (warp-uniform)
      ++wp.wiss;
    };

    float2 P[CPL][8];
    float W[CPL];  // structured: log2 decay of entry 0 over the steps walked; generic: sum of delta
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      W[c] = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) P[c][k] = make_float2(1.0f, 1.0f);
    }
    int np = 8;  // structured: state pairs still accumulating
    for (int k = 0;; ++k) {
      const int64_t thi = t0 - static_cast<int64_t>(k) * TSW;
      const int64_t tlo = thi - TSW > 0 ? thi - TSW : 0;
      const int n = static_cast<int>(thi - tlo);
      const int slot = static_cast<int>(wp.wcon % NSW);
      if (!mbar_wait(&r.wbar[slot], (wp.wcon / NSW) & 1u, p.wait_ns)) return false;
      const T* xs = r.wx[slot];
      const T* ds = r.wd[slot];
      const T* Bs = r.wB[slot];
      if constexpr (S4D) {
        if (np == 8) warm_s4d<8, ZOH, CPL, TSW, DX>(xs, ds, Bs, n, lane, A2_0, invA0, dbias, W, P, h);
        else if (np == 4) warm_s4d<4, ZOH, CPL, TSW, DX>(xs, ds, Bs, n, lane, A2_0, invA0, dbias, W, P, h);
        else if (np == 2) warm_s4d<2, ZOH, CPL, TSW, DX>(xs, ds, Bs, n, lane, A2_0, invA0, dbias, W, P, h);
        else warm_s4d<1, ZOH, CPL, TSW, DX>(xs, ds, Bs, n, lane, A2_0, invA0, dbias, W, P, h);
      } else {
        warm_gen<ZOH, CPL, DX>(xs, ds, Bs, n, lane, g, dbias, W, P, h);
      }
      ++wp.wcon;
      // Pair k holds entries 2k, 2k+1 whose log2 decay is (2k+1) W, (2k+2) W (structured). A pair is
      // dropped once its slower entry has decayed below 2^-20 on every active channel; dropping is final.
      float wl = -3.0e38f;
#pragma unroll
      for (int c = 0; c < CPL; ++c)
        if (act[c]) wl = fmaxf(wl, S4D ? W[c] : W[c] * g[S4D ? 0 : c].A2max);
      const float wmax = warp_max(wl);
      const bool at_start = (tlo == 0);
      bool done;
      if (S4D) {
        // pair k is live while (2k+1) * wmax > kDeadLog2 (monotone in k); np shrinks to the smallest of
        // 8, 4, 2, 1, 0 that keeps every live pair.
        int live = 0;
        if (wmax > kDeadLog2 / 15.0f) live = 8;
        else if (wmax > kDeadLog2 / 13.0f) live = 7;
        else if (wmax > kDeadLog2 / 11.0f) live = 6;
        else if (wmax > kDeadLog2 / 9.0f) live = 5;
        else if (wmax > kDeadLog2 / 7.0f) live = 4;
        else if (wmax > kDeadLog2 / 5.0f) live = 3;
        else if (wmax > kDeadLog2 / 3.0f) live = 2;
        else if (wmax > kDeadLog2) live = 1;
        const int want = live > 4 ? 8 : live > 2 ? 4 : live;  // 8, 4, 2, 1 or 0
        if (want < np) np = want;
        done = at_start || np == 0;
      } else {
        done = at_start || wmax <= kDeadLog2;
      }
      if (done) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          if (ZOH && S4D) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              h[c][q] = __fmul2_rn(h[c][q], make_float2(1.0f / static_cast<float>(2 * q + 1),
                                                        1.0f / static_cast<float>(2 * q + 2)));
          }
          if (at_start && h0row[c]) {
            // plus (decay over [0, t0)) * h0 for the entries still live (dropped ones decayed below 2^-20)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 v = reinterpret_cast<const float4*>(h0row[c])[q];
              if (!S4D || 2 * q < np) h[c][2 * q] = __ffma2_rn(P[c][2 * q], make_float2(v.x, v.y), h[c][2 * q]);
              if (!S4D || 2 * q + 1 < np)
                h[c][2 * q + 1] = __ffma2_rn(P[c][2 * q + 1], make_float2(v.z, v.w), h[c][2 * q + 1]);
            }
          }
        }
        break;
      }
      __syncwarp();
      issue_warm();
    }
  }

  // ---- forward over [t0, t1) ----
  for (int64_t tb = t0; tb < t1; tb += TS) {
    const int n = static_cast<int>((t1 - tb) < TS ? (t1 - tb) : TS);
    const int slot = static_cast<int>(wp.cseq % NSF);
    if (!mbar_wait(&r.fbar[slot], (wp.cseq / NSF) & 1u, p.wait_ns)) return false;
    const T* xs = r.fx[slot];
    const T* ds = r.fd[slot];
    constexpr bool kScaleB = ZOH && S4D;  // the structured ZOH update takes B_n / (n + 1)
    if constexpr (kConv || kScaleB) {     // this stage's B (and for bf16 inputs C) as fp32, once per stage
      if constexpr (sizeof(T) == 4) {
        float4 v = reinterpret_cast<const float4*>(r.fB[slot])[lane];  // entries 4 lane .. 4 lane + 3
        const int n0 = (4 * lane) & 15;
        v.x *= 1.0f / static_cast<float>(n0 + 1);
        v.y *= 1.0f / static_cast<float>(n0 + 2);
        v.z *= 1.0f / static_cast<float>(n0 + 3);
        v.w *= 1.0f / static_cast<float>(n0 + 4);
        reinterpret_cast<float4*>(r.Bf)[lane] = v;
      } else {
#pragma unroll
        for (int j = 0; j < TS * 16 / 32; ++j) {
          const int i = lane + 32 * j;
          float bv = tof<T>(r.fB[slot][i]);
          if (kScaleB) bv *= 1.0f / static_cast<float>((i & 15) + 1);
          r.Bf[i] = bv;
          r.Cf[i] = tof<T>(r.fC[slot][i]);
        }
      }
      __syncwarp();
    }
    const float* Bs = (kConv || kScaleB) ? r.Bf : reinterpret_cast<const float*>(r.fB[slot]);
    const float* Cs = kConv ? r.Cf : reinterpret_cast<const float*>(r.fC[slot]);
    T* yp = static_cast<T*>(p.y) + (b * L + tb) * p.D + d0;  // channel c at yp + 32 c
    const T* zp = EPI == 2 ? static_cast<const T*>(p.z) + (b * L + tb) * p.D + d0 : nullptr;  // gate input
    if constexpr (S4D) {
      auto one = [&](auto all_active, int i) {
        float xv[CPL], dv[CPL], yv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          xv[c] = tof<T>(xs[i * CW + c * 32 + lane]);
          dv[c] = tof<T>(ds[i * CW + c * 32 + lane]);
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) dv[c] = delta_in<DX>(dv[c], dbias[c]);
        fwd_s4d<ZOH, CPL>(xv, dv, Bs + i * 16, Cs + i * 16, A2_0, invA0, h, yv);
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float zv = 0.0f;
          if constexpr (kZs) zv = tof<T>(zr[slot * TS * CW + i * CW + c * 32 + lane]);
          else if (EPI == 2 && act[c]) zv = tof<T>(zp[static_cast<int64_t>(i) * p.D + 32 * c]);
          yv[c] = epilogue<EPI>(yv[c], xv[c], dskip[c], zv);
          if constexpr (decltype(all_active)::value) store_y(yp + 32 * c, yv[c]);
          else store_y(yp + 32 * c, yv[c], act[c]);
        }
        yp += p.D;
      };
      // fp32 inputs (8-warp shape, registers to spare): step i+1's decay tree is computed before step i's
      // update, 8% faster on the long ZOH workload. bf16 inputs run 12 warps capped at 168 registers, where
      // the extra live values cost more than they gain.
      constexpr bool kPipe = sizeof(T) == 4;
      if (kPipe && n == TS && full) {
        float2 e[CPL][8], s2[CPL];
        float zt[EPI == 2 ? TS : 1][CPL];  // gate inputs of the stage, from its ring tile
        if constexpr (EPI == 2) {
#pragma unroll
          for (int i = 0; i < TS; ++i)
#pragma unroll
            for (int c = 0; c < CPL; ++c) zt[i][c] = tof<T>(zr[slot * TS * CW + i * CW + c * 32 + lane]);
        }
        auto prep = [&](int i, float2 (&ee)[CPL][8], float2 (&ss)[CPL]) {
          float xv[CPL], dv[CPL];
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            xv[c] = tof<T>(xs[i * CW + c * 32 + lane]);
            dv[c] = delta_in<DX>(tof<T>(ds[i * CW + c * 32 + lane]), dbias[c]);
          }
          fwd_prep<ZOH, CPL>(xv, dv, A2_0, invA0, ee, ss);
        };
        prep(0, e, s2);
#pragma unroll
        for (int i = 0; i < TS; ++i) {
          float2 en[CPL][8], sn[CPL];
          if (i + 1 < TS) prep(i + 1, en, sn);
          float yv[CPL];
          fwd_core<ZOH, CPL>(e, s2, Bs + i * 16, Cs + i * 16, h, yv);
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            if constexpr (EPI != 0)  // x of this step re-read from the stage for the feedthrough
              yv[c] = epilogue<EPI>(yv[c], tof<T>(xs[i * CW + c * 32 + lane]), dskip[c], EPI == 2 ? zt[i][c] : 0.0f);
            store_y(yp + 32 * c, yv[c]);
          }
          yp += p.D;
          if (i + 1 < TS) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
              s2[c] = sn[c];
#pragma unroll
              for (int k = 0; k < 8; ++k) e[c][k] = en[c][k];
            }
          }
        }
      } else if (n == TS && full) {
#pragma unroll
        for (int i = 0; i < TS; ++i) one(std::true_type{}, i);
      } else if (n == TS) {
#pragma unroll
        for (int i = 0; i < TS; ++i) one(std::false_type{}, i);
      } else {
#pragma unroll 1
        for (int i = 0; i < n; ++i) one(std::false_type{}, i);
      }
    } else {
#pragma unroll 1
      for (int i = 0; i < n; ++i) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const float xv = tof<T>(xs[i * CW + c * 32 + lane]);
          const float yv = fwd_gen<ZOH>(xv, delta_in<DX>(tof<T>(ds[i * CW + c * 32 + lane]), dbias[c]),
                                        Bs + i * 16, Cs + i * 16, g[S4D ? 0 : c], h[c]);
          float zv = 0.0f;
          if constexpr (kZs) zv = tof<T>(zr[slot * TS * CW + i * CW + c * 32 + lane]);
          else if (EPI == 2 && act[c]) zv = tof<T>(zp[static_cast<int64_t>(i) * p.D + 32 * c]);
          store_y(yp + 32 * c, epilogue<EPI>(yv, xv, dskip[c], zv), act[c]);
        }
        yp += p.D;
      }
    }
    __syncwarp();
    ++wp.cseq;
    issue_fwd();
  }
  if (t1 == L && p.final_state) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      if (!act[c]) continue;
      float4* fs = reinterpret_cast<float4*>(p.final_state + (b * p.D + d0 + 32 * c) * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        fs[q] = make_float4(h[c][2 * q].x, h[c][2 * q].y, h[c][2 * q + 1].x, h[c][2 * q + 1].y);
    }
  }
  return true;
}

// Register budget: the fp32 shape runs 8 warps (up to 255 registers a thread), the bf16 shape 12 (up to
// 170). Within the fp32 budget the compiler's schedule of the step loop depends on the register count it
// settles on; a cap of 240 measured fastest on the long ZOH workload (caps from 200 to 255 spread the
// launch time over about 7%).
template <typename T, bool ZOH, int CPL, int NW, int TS, int NSF, int TSW, int NSW, int DX, int EPI>
__global__ void __maxnreg__(sizeof(T) == 4 ? 240 : 168)
scan_fwd_tma_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap md,
                    const __grid_constant__ CUtensorMap mB, const __grid_constant__ CUtensorMap mC,
                    const __grid_constant__ CUtensorMap mxw, const __grid_constant__ CUtensorMap mdw,
                    const __grid_constant__ CUtensorMap mBw, const __grid_constant__ CUtensorMap mz,
                    TmaParams p) {
  using R = WarpRing<T, CPL, TS, NSF, TSW, NSW>;
  constexpr int CW = R::CW;
  constexpr int NZ = EPI == 2 ? NSF : 0;  // gate-input stages in the forward ring
  constexpr uint32_t kFwdBytes = (2u * TS * CW + 2u * TS * 16 + (NZ > 0 ? TS * CW : 0u)) * sizeof(T);

  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t pad = (128u - (su32(smem_raw) & 127u)) & 127u;
  R& r = reinterpret_cast<R*>(smem_raw + pad)[warp];
  T* zr = reinterpret_cast<T*>(smem_raw + pad + NW * sizeof(R)) + warp * (NZ * TS * CW);  // after the rings
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * NW + warp;
  if (wid >= p.nwarps) return;

  if (threadIdx.x == 0) {  // bring the copy descriptors into the descriptor cache before their first use
    const CUtensorMap* maps[8] = {&mx, &md, &mB, &mC, &mxw, &mdw, &mBw, &mz};
#pragma unroll
    for (int i = 0; i < 8; ++i) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(maps[i])) : "memory");
  }
  if (lane == 0) {
    for (int i = 0; i < NSF; ++i) mbar_init(&r.fbar[i], 1);
    for (int i = 0; i < NSW; ++i) mbar_init(&r.wbar[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  __syncwarp();

  const int64_t lo0 = static_cast<int64_t>(static_cast<__int128>(wid) * p.total / p.nwarps);
  const int64_t hi0 = static_cast<int64_t>(static_cast<__int128>(wid + 1) * p.total / p.nwarps);
  const int64_t L = p.L;

  // Forward stages, in the order the consumer takes them: the range [lo0, hi0) cut at row ends and every
  // TS steps, issued NSF ahead of consumption. Every lane advances the cursor and the counters (so that they
  // stay warp-uniform for the warp-wide waits); lane 0 issues the copies. The cursor advances without
  // divisions (64-bit division is a long software sequence).
  int64_t ipos = lo0;   // first step of the next forward stage to issue
  uint32_t iseq = 0;    // forward stages issued
  int64_t it = lo0 % L, ib = (lo0 / L) / p.G, ig = (lo0 / L) % p.G;  // its step, batch, channel group
  auto issue_fwd = [&]() {
    if (ipos >= hi0) return;
    const int64_t room = (L - it) < (hi0 - ipos) ? (L - it) : (hi0 - ipos);
    const int64_t n = room < TS ? room : TS;
    const int slot = static_cast<int>(iseq % NSF);
    const int trow = static_cast<int>(ib * L + it);
    const int col = static_cast<int>(ig * CW);
    if (lane == 0) {
      mbar_arrive_tx(&r.fbar[slot], kFwdBytes);
      tma_load(r.fx[slot], &mx, col, trow, &r.fbar[slot]);
      tma_load(r.fd[slot], &md, col, trow, &r.fbar[slot]);
      tma_load(r.fB[slot], &mB, 0, trow, &r.fbar[slot]);
      tma_load(r.fC[slot], &mC, 0, trow, &r.fbar[slot]);
      if constexpr (NZ > 0) tma_load(zr + slot * TS * CW, &mz, col, trow, &r.fbar[slot]);
    }
    ipos += n;
    it += n;
    if (it == L) {
      it = 0;
      if (++ig == p.G) {
        ig = 0;
        ++ib;
      }
    }
    ++iseq;
  };
  WarpPipe wp{0u, 0u, 0u};
  bool primed = false;
  int64_t lo = lo0;
  while (lo < hi0) {
    const int64_t row = lo / L, t0 = lo % L;
    const int64_t t1 = (hi0 - lo < L - t0) ? t0 + (hi0 - lo) : L;
    lo += t1 - t0;
    // This piece's A_log rows are loaded into registers before any bulk copy is issued, so that these small
    // loads enter the memory system ahead of the warps' first tiles (behind them they wait microseconds).
    const int64_t d0 = (row % p.G) * CW + lane;
    float Alog[CPL][16];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int64_t d = d0 + 32 * c;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = d < p.D ? __ldg(reinterpret_cast<const float4*>(p.A_log + d * 16) + q)
                                 : make_float4(0.0f, 0.6931472f, 1.0986123f, 1.3862944f);
        Alog[c][4 * q] = v.x;
        Alog[c][4 * q + 1] = v.y;
        Alog[c][4 * q + 2] = v.z;
        Alog[c][4 * q + 3] = v.w;
      }
    }
    int kiss0 = 0;
    if (t0 > 0) {  // the walk's first tiles go out before the forward ring is primed: they are needed first
      kiss0 = warm_prologue(r, &mxw, &mdw, &mBw, lane, (row / p.G) * L, static_cast<int>((row % p.G) * CW), t0, wp);
      if (kiss0 < 0) break;
    }
    if (!primed) {
      for (int i = 0; i < NSF; ++i) issue_fwd();
      primed = true;
    }
    // S4D structure check (warp-uniform): A[d, n] = (n + 1) A[d, 0] for every channel of the warp.
    bool ok = true;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      if (d0 + 32 * c < p.D) {
        const float A0 = -expf(Alog[c][0]);
        bool okc = A0 < -1e-30f && A0 > -3.0e38f;
#pragma unroll
        for (int n = 1; n < 16; ++n) {
          const float A = -expf(Alog[c][n]);
          okc = okc && fabsf(A - static_cast<float>(n + 1) * A0) <= 4.8e-7f * fabsf(A);
        }
        ok = ok && okc;
      }
    }
    const bool alive = __all_sync(0xffffffffu, ok)
                           ? run_piece<true, T, ZOH, CPL, TS, NSF, TSW, NSW, DX, EPI>(r, p, &mxw, &mdw, &mBw, lane, row, t0, t1, wp, issue_fwd, kiss0, zr)
                           : run_piece<false, T, ZOH, CPL, TS, NSF, TSW, NSW, DX, EPI>(r, p, &mxw, &mdw, &mBw, lane, row, t0, t1, wp, issue_fwd, kiss0, zr);
    if (!alive) break;
  }

  // No copy may still be writing this warp's shared memory when the CTA exits.
  while (wp.cseq < iseq) {
    if (!mbar_wait(&r.fbar[wp.cseq % NSF], (wp.cseq / NSF) & 1u, kWaitNs)) break;
    ++wp.cseq;
  }
  while (wp.wcon < wp.wiss) {
    if (!mbar_wait(&r.wbar[wp.wcon % NSW], (wp.wcon / NSW) & 1u, kWaitNs)) break;
    ++wp.wcon;
  }
}

// ---- host side ------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, bool bf16, uint64_t inner, uint64_t rows, uint32_t box_inner,
              uint32_t box_rows) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  const uint64_t es = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * es};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, bool ZOH, int CPL, int NW, int TS, int NSF, int TSW, int NSW, int DX, int EPI>
cudaError_t launch_cfg(const FwdArgs& a) {
  constexpr int CW = 32 * CPL;
  const bool bf16 = sizeof(T) == 2;
  CUtensorMap mx, md, mB, mC, mxw, mdw, mBw, mz;  // forward tiles (TS rows), warm-up tiles (TSW rows), gate
  const uint64_t rows = static_cast<uint64_t>(a.batch * a.L);
  if (!make_map(&mx, a.x, bf16, a.D, rows, CW, TS) || !make_map(&md, a.delta, bf16, a.D, rows, CW, TS) ||
      !make_map(&mB, a.B, bf16, 16, rows, 16, TS) || !make_map(&mC, a.C, bf16, 16, rows, 16, TS) ||
      !make_map(&mxw, a.x, bf16, a.D, rows, CW, TSW) || !make_map(&mdw, a.delta, bf16, a.D, rows, CW, TSW) ||
      !make_map(&mBw, a.B, bf16, 16, rows, 16, TSW))
    return cudaErrorInvalidValue;
  constexpr int NZ = EPI == 2 ? NSF : 0;
  if (NZ > 0) {
    if (!make_map(&mz, a.z, bf16, a.D, rows, CW, TS)) return cudaErrorInvalidValue;
  } else {
    mz = mx;  // not read
  }
  TmaParams p;
  p.A_log = a.A_log;
  p.h0 = a.h0;
  p.delta_bias = a.delta_bias;
  p.D_skip = a.D_skip;
  p.z = a.z;
  p.y = a.y;
  p.final_state = a.final_state;
  p.L = a.L;
  p.D = a.D;
  p.G = (a.D + CW - 1) / CW;
  p.total = a.batch * p.G * a.L;
  p.wait_ns = wait_limit_ns();
  const size_t smem = sizeof(WarpRing<T, CPL, TS, NSF, TSW, NSW>) * NW + NW * NZ * TS * CW * sizeof(T) + 128;
  auto kern = scan_fwd_tma_kernel<T, ZOH, CPL, NW, TS, NSF, TSW, NSW, DX, EPI>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!attr_set[dev & 63]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev & 63] = true;
  }
  // one CTA per SM; every warp's range at least a few stages long
  int64_t nwarps = static_cast<int64_t>(sm_count()) * NW;
  const int64_t min_steps = 4 * TS;
  const int64_t cap = (p.total + min_steps - 1) / min_steps;
  if (nwarps > cap) nwarps = cap;
  if (nwarps < 1) nwarps = 1;
  p.nwarps = nwarps;
  const int64_t nctas = (nwarps + NW - 1) / NW;
  kern<<<static_cast<unsigned>(nctas), NW * 32, smem, a.stream>>>(mx, md, mB, mC, mxw, mdw, mBw, mz, p);
  return cudaGetLastError();
}

// Kernel shapes: channels per lane, warps per CTA, forward stage steps and stages, warm-up tile steps and
// stages. fp32 inputs: 8 warps (2 per SM sub-partition) with deeper rings; bf16 inputs (half the bytes per
// element, so smaller rings suffice): 12 warps, whose extra latency hiding is worth 12% there.
struct ShapeF32 { static constexpr int CPL = 2, NW = 8, TS = 8, NSF = 3, TSW = 8, NSW = 2; };
// fp32 with the gate: the z tiles take the room of half the warm-up ring (4-step warm-up tiles)
struct ShapeF32Gate { static constexpr int CPL = 2, NW = 8, TS = 8, NSF = 3, TSW = 4, NSW = 2; };
struct ShapeBF16 { static constexpr int CPL = 2, NW = 12, TS = 8, NSF = 2, TSW = 4, NSW = 2; };

template <typename T, bool ZOH, typename S, int DX, int EPI>
cudaError_t launch_fused(const FwdArgs& a) {
  return launch_cfg<T, ZOH, S::CPL, S::NW, S::TS, S::NSF, S::TSW, S::NSW, DX, EPI>(a);
}

// The plain scan, and softplus(delta + bias) with the feedthrough alone or with the gate (the layer's usual
// combinations); other combinations go to the general kernel.
template <typename T, bool ZOH, typename S>
cudaError_t launch_shape(const FwdArgs& a) {
  const int dx = a.softplus ? 2 : 0;
  const int epi = a.z ? 2 : (a.D_skip || a.softplus) ? 1 : 0;
  if (dx == 0 && epi == 0) return launch_fused<T, ZOH, S, 0, 0>(a);
  if (dx == 2 && epi == 1) return launch_fused<T, ZOH, S, 2, 1>(a);
  if (dx == 2 && epi == 2) return launch_fused<T, ZOH, S, 2, 2>(a);
  return cudaErrorNotSupported;  // tma_path_ok() keeps other combinations away
}

}  // namespace

bool tma_path_ok(const FwdArgs& a) {
  if (a.N != 16) return false;
  // fused combinations this kernel is built for: none, or softplus(delta + bias) with the feedthrough
  // (D_skip or none) and optionally the gate
  const bool plain = !a.softplus && !a.delta_bias && !a.D_skip && !a.z;
  if (!plain && !a.softplus) return false;
  const int es = a.dtype == 1 ? 2 : 4;
  if ((a.D * es) % 16 != 0) return false;
  const void* ptrs[] = {a.x, a.delta, a.B, a.C};
  for (const void* q : ptrs)
    if (reinterpret_cast<uintptr_t>(q) % 16 != 0) return false;
  if (a.final_state && reinterpret_cast<uintptr_t>(a.final_state) % 16 != 0) return false;
  if (a.h0 && reinterpret_cast<uintptr_t>(a.h0) % 16 != 0) return false;
  if (reinterpret_cast<uintptr_t>(a.A_log) % 16 != 0) return false;  // rows read as float4
  if (a.z && reinterpret_cast<uintptr_t>(a.z) % 16 != 0) return false;  // bf16 gate inputs are copied as tiles
  if (a.batch * a.L > (int64_t(1) << 30)) return false;  // TMA row coordinates are 32-bit
  if (encoder() == nullptr) return false;
  return true;
}

cudaError_t launch_fwd_tma(const FwdArgs& a) {
  if (a.dtype == 1)
    return a.disc == 1 ? launch_shape<__nv_bfloat16, true, ShapeBF16>(a)
                       : launch_shape<__nv_bfloat16, false, ShapeBF16>(a);
  if (a.z)
    return a.disc == 1 ? launch_shape<float, true, ShapeF32Gate>(a) : launch_shape<float, false, ShapeF32Gate>(a);
  return a.disc == 1 ? launch_shape<float, true, ShapeF32>(a) : launch_shape<float, false, ShapeF32>(a);
}

int read_and_clear_device_status() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) {
    int z = 0;
    cudaMemcpyToSymbol(g_device_status, &z, sizeof(int));
  }
  return v;
}

}  // namespace ssm
