// scan_fwd_tma.cu -- the prefill scan for aligned shapes with N = 16: TMA-staged, warp-specialised,
// persistent over an even split of the (channel tile, time) work.
//
// Layout of the work. A CTA owns DT = 32 * NW consecutive channels of one batch element at a time (one
// lane of one consumer warp per channel) and a contiguous range of time steps; the rows' time axes are laid
// end to end and cut into equal ranges, one per CTA, so every SM gets the same number of (channel, step)
// elements whatever the batch / length mix. A range that starts at t0 > 0 rebuilds the state entering t0
// by walking the preceding steps backwards ("Mathematical Prerequisites for Mamba" s6: h(t0-1) is the sum
// over j of prod_{k>j} Abar_k * Bbar_j x_j) until every decay product is below kCarryEps (or t = 0, where
// the sum is exact), then runs the recurrence of "Understanding Mamba" Eq. (3) forward. No CTA waits on
// another and no scratch memory is used.
//
// Data movement. One issue warp streams [TS rows x DT channels] tiles of x and delta and [TS x 16] tiles
// of B and C into a ring of NS shared-memory stages with cp.async.bulk.tensor (TMA), completion tracked by
// mbarriers; one staging warp widens B and C to fp32 (and pre-scales B for the ZOH form below) once per
// stage for all channels; NW consumer warps keep their channel's 16 state entries in registers, read x /
// delta (one word per lane, conflict free) and B / C (broadcast) from shared memory, and store y straight
// to global memory (32 consecutive channels per warp store). Every mbarrier wait is bounded.
//
// Arithmetic (per step t, channel d, state entry n; packed two entries at a time with f32x2 FMA):
//  * S4D-structured channels (A[d, n] = (n + 1) A[d, 0], checked per warp): one SFU exp2 per (t, d) and
//    e_n = Abar_n - 1 = Abar_0^{n+1} - 1 for all n by the exact recurrence e_{m+k+1} = e_m (1 + e_k) + e_k
//    from an e_0 with no cancellation (one FMA per entry; errors do not grow with n).
//      Euler: h_n = Abar_n h_n + (delta x) B_n  ==  (h_n + e_n h_n) + u B_n, two FMAs
//      ZOH:   with q_n = B_n x / A_n = (B_n / (n+1)) (x / A_0):
//             h_n = h_n + e_n (h_n + q_n), i.e. the ZOH step Abar h + (Abar - 1) q, two FMAs.
//    The backward warm-up keeps each decay product P_n as its own running product P_n (1 + e_n).
//  * other channels: e_n = 2^{delta A_n log2 e} - 1 per entry (SFU exp2, Taylor series where |delta A_n| is
//    small), h_n = (h_n + e_n h_n) + Bbar x; about twice the FP32 work of the structured path.
//    y = sum_n C_n h_n.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

#ifndef SSM_TMA_CFG
#define SSM_TMA_CFG 0
#endif

namespace ssm {

__device__ int g_device_status = 0;  // nonzero: a bounded wait ran out (read by ssm_check_device)

namespace {

constexpr int kWarm = 0, kFwd = 1, kEnd = 2;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s bound on any single mbarrier wait

struct Tag {
  int kind, t_start, t_lo, t_hi;
};

template <typename T, int NW, int TS, int NS>
struct Smem {
  static constexpr int DT = NW * 32;
  T x[NS][TS * DT];
  T dl[NS][TS * DT];
  T Braw[NS][TS * 16];
  T Craw[NS][TS * 16];
  float Bf[NS][TS * 16];
  float Cf[NS][TS * 16];
  float Bp[NS][TS * 16];
  Tag tag[NS];
  unsigned long long full[NS], ready[NS], empty[NS];
  int done_count;
  int abort;
};

struct TmaParams {
  const float* A_log;
  const float* h0;
  void* y;
  float* final_state;
  int64_t batch, L, D;
  int64_t tiles;   // ceil(D / DT)
  int64_t total;   // batch * tiles * L
  int64_t nctas;
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
__device__ __forceinline__ void mbar_arrive(unsigned long long* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
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
// Bounded wait: false (and the device status set) if the phase does not complete within kWaitNs.
__device__ __forceinline__ bool mbar_wait(unsigned long long* b, uint32_t parity, volatile int* abort) {
  if (mbar_try(b, parity)) return true;
  const unsigned long long t0 = gtimer();
  while (true) {
    if (mbar_try(b, parity)) return true;
    if (*abort) return false;
    if (gtimer() - t0 > kWaitNs) {
      atomicExch(&g_device_status, 4);
      *abort = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, int c0, int c1, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(su32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(su32(bar))
      : "memory");
}

__device__ __forceinline__ float2 bc2(float v) { return make_float2(v, v); }

template <typename T> __device__ __forceinline__ float tof(T v);
template <> __device__ __forceinline__ float tof<float>(float v) { return v; }
template <> __device__ __forceinline__ float tof<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// e_n = Abar_0^{n+1} - 1 for n = 0..15 (eight pairs) from e_0, by the exact identity
// e_{m+k+1} = e_m (1 + e_k) + e_k. Relative errors stay those of e_0 (no amplification with n), so the
// decay factor 1 + e_n is as accurate as one rounding even where nothing decays for many steps.
__device__ __forceinline__ void em1_tree(float e0, float2 (&e)[8]) {
  const float e1 = fmaf(e0, 1.0f + e0, e0);
  e[0] = make_float2(e0, e1);
  e[1] = __ffma2_rn(e[0], bc2(1.0f + e1), bc2(e1));        // e2 e3
  const float2 a3 = bc2(1.0f + e[1].y), e3 = bc2(e[1].y);
  e[2] = __ffma2_rn(e[0], a3, e3);                           // e4 e5
  e[3] = __ffma2_rn(e[1], a3, e3);                           // e6 e7
  const float2 a7 = bc2(1.0f + e[3].y), e7 = bc2(e[3].y);
  e[4] = __ffma2_rn(e[0], a7, e7);
  e[5] = __ffma2_rn(e[1], a7, e7);
  e[6] = __ffma2_rn(e[2], a7, e7);
  e[7] = __ffma2_rn(e[3], a7, e7);
}

struct ChanGen {  // per-channel constants of the generic path
  float A2[16], invA[16];  // A log2(e); 1/A (0 where A == 0)
};

// Generic (unstructured A) terms of one step for state pair k: e = Abar - 1 and the input term Bbar x.
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

template <typename T, int NW, int TS, int NS, bool ZOH, int MINB>
__global__ void __launch_bounds__((NW + 2) * 32, MINB)
scan_fwd_tma_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap md,
                    const __grid_constant__ CUtensorMap mB, const __grid_constant__ CUtensorMap mC, TmaParams p) {
  using S = Smem<T, NW, TS, NS>;
  constexpr int DT = S::DT;
  extern __shared__ unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &s.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.ready[i], 32);
      mbar_init(&s.empty[i], NW);
    }
    s.done_count = 0;
    s.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  const int64_t lo0 = static_cast<int64_t>(static_cast<__int128>(blockIdx.x) * p.total / p.nctas);
  const int64_t hi0 = static_cast<int64_t>(static_cast<__int128>(blockIdx.x + 1) * p.total / p.nctas);
  constexpr uint32_t kStageBytes = 2u * TS * DT * sizeof(T) + 2u * TS * 16 * sizeof(T);

  if (warp == NW) {
    // ================= issue warp: TMA loads in stage order =================
    if (lane != 0) return;
    int64_t seq = 0;
    int warm_index = 0;
    auto issue = [&](int kind, int64_t b, int t_start, int t_lo, int t_hi, int d0) -> bool {
      const int slot = static_cast<int>(seq % NS);
      const uint32_t par = static_cast<uint32_t>((seq / NS) & 1) ^ 1u;
      if (!mbar_wait(&s.empty[slot], par, abort)) return false;
      s.tag[slot] = Tag{kind, t_start, t_lo, t_hi};
      if (kind == kEnd) {
        mbar_arrive(&s.full[slot]);
      } else {
        mbar_arrive_tx(&s.full[slot], kStageBytes);
        const int row = static_cast<int>(b * p.L) + t_start;
        tma_load(s.x[slot], &mx, d0, row, &s.full[slot]);
        tma_load(s.dl[slot], &md, d0, row, &s.full[slot]);
        tma_load(s.Braw[slot], &mB, 0, row, &s.full[slot]);
        tma_load(s.Craw[slot], &mC, 0, row, &s.full[slot]);
      }
      ++seq;
      return true;
    };
    int64_t lo = lo0;
    while (lo < hi0) {
      const int64_t row = lo / p.L, t0 = lo % p.L;
      const int64_t t1 = (hi0 - lo < p.L - t0) ? t0 + (hi0 - lo) : p.L;
      lo += t1 - t0;
      const int64_t b = row / p.tiles;
      const int d0 = static_cast<int>((row % p.tiles) * DT);
      if (t0 > 0) {
        ++warm_index;
        for (int k = 1;; ++k) {
          const int ts = static_cast<int>(t0) - k * TS;
          if (k > 1 && *reinterpret_cast<volatile int*>(&s.done_count) >= NW * warm_index) break;
          if (!issue(kWarm, b, ts, ts > 0 ? ts : 0, ts + TS, d0)) return;
          if (ts <= 0) break;
        }
      }
      for (int64_t t = t0; t < t1; t += TS)
        if (!issue(kFwd, b, static_cast<int>(t), static_cast<int>(t), static_cast<int>(t + TS < t1 ? t + TS : t1), d0))
          return;
    }
    issue(kEnd, 0, 0, 0, 0, 0);
    return;
  }

  if (warp == NW + 1) {
    // ================= staging warp: widen / pre-scale B and C once per stage =================
    int64_t seq = 0;
    while (true) {
      const int slot = static_cast<int>(seq % NS);
      const uint32_t par = static_cast<uint32_t>((seq / NS) & 1);
      if (!mbar_wait(&s.full[slot], par, abort)) return;
      const int kind = s.tag[slot].kind;
      if (kind != kEnd) {
#pragma unroll 4
        for (int i = lane; i < TS * 16; i += 32) {
          const float bv = tof<T>(s.Braw[slot][i]);
          s.Bf[slot][i] = bv;
          s.Cf[slot][i] = tof<T>(s.Craw[slot][i]);
          s.Bp[slot][i] = bv * (1.0f / static_cast<float>((i & 15) + 1));
        }
      }
      mbar_arrive(&s.ready[slot]);
      ++seq;
      if (kind == kEnd) return;
    }
  }

  // ================= consumer warps =================
  const int c = warp * 32 + lane;  // column of this lane inside the tile
  int64_t seq = 0;
  int64_t lo = lo0;
  while (lo < hi0) {
    const int64_t row = lo / p.L, t0 = lo % p.L;
    const int64_t t1 = (hi0 - lo < p.L - t0) ? t0 + (hi0 - lo) : p.L;
    lo += t1 - t0;
    const int64_t b = row / p.tiles;
    const int64_t d = (row % p.tiles) * DT + c;
    const bool act = d < p.D;

    // ---- channel constants; S4D structure check (warp-uniform) ----
    float Araw[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) Araw[n] = act ? -expf(__ldg(p.A_log + d * 16 + n)) : -static_cast<float>(n + 1);
    bool ok = Araw[0] < -1e-30f && Araw[0] > -3.0e38f;
#pragma unroll
    for (int n = 1; n < 16; ++n)
      ok = ok && fabsf(Araw[n] - static_cast<float>(n + 1) * Araw[0]) <= 4.8e-7f * fabsf(Araw[n]);
    const bool s4d = __all_sync(0xffffffffu, ok);
    const float A2_0 = Araw[0] * kLog2e, invA0 = 1.0f / Araw[0];
    ChanGen g;
    if (!s4d) {
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        g.A2[n] = Araw[n] * kLog2e;
        g.invA[n] = Araw[n] == 0.0f ? 0.0f : 1.0f / Araw[n];
      }
    }

    float2 h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = make_float2(0.0f, 0.0f);
    const float* h0row = p.h0 ? p.h0 + (b * p.D + d) * 16 : nullptr;

    // ---- state entering t0: backward accumulation over staged warm-up tiles ----
    bool pending_fwd = false;  // the first forward stage has been waited for already
    if (t0 == 0) {
      if (h0row && act) {
#pragma unroll
        for (int k = 0; k < 8; ++k) h[k] = make_float2(h0row[2 * k], h0row[2 * k + 1]);
      }
    } else {
      bool done = false;
      float2 Pg[8];  // prod of Abar_n over the steps after the current one
#pragma unroll
      for (int k = 0; k < 8; ++k) Pg[k] = make_float2(1.0f, 1.0f);
      while (true) {
        const int slot = static_cast<int>(seq % NS);
        const uint32_t par = static_cast<uint32_t>((seq / NS) & 1);
        if (!mbar_wait(&s.full[slot], par, abort) || !mbar_wait(&s.ready[slot], par, abort)) return;
        const Tag tg = s.tag[slot];
        if (tg.kind != kWarm) {
          pending_fwd = true;
          break;
        }
        if (!done) {
          const T* xs = s.x[slot];
          const T* ds = s.dl[slot];
          const float* Bs = s.Bf[slot];
          const float* Bps = s.Bp[slot];
          for (int t = tg.t_hi - 1; t >= tg.t_lo; --t) {
            const int r = t - tg.t_start;
            const float xv = tof<T>(xs[r * DT + c]);
            const float dv = act ? tof<T>(ds[r * DT + c]) : 0.0f;
            if (s4d) {
              const float w = dv * A2_0;
              float2 e[8];
              em1_tree(exp2m1(w, ex2(w)), e);
              if (ZOH) {
                const float4* Bq = reinterpret_cast<const float4*>(Bps + r * 16);
                const float2 xi = bc2(xv * invA0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float4 bb = Bq[q];
                  const float2 d0 = __fmul2_rn(Pg[2 * q], e[2 * q]);  // P (Abar - 1)
                  const float2 d1 = __fmul2_rn(Pg[2 * q + 1], e[2 * q + 1]);
                  h[2 * q] = __ffma2_rn(d0, __fmul2_rn(xi, make_float2(bb.x, bb.y)), h[2 * q]);
                  h[2 * q + 1] = __ffma2_rn(d1, __fmul2_rn(xi, make_float2(bb.z, bb.w)), h[2 * q + 1]);
                  Pg[2 * q] = __fadd2_rn(Pg[2 * q], d0);  // P Abar
                  Pg[2 * q + 1] = __fadd2_rn(Pg[2 * q + 1], d1);
                }
              } else {
                const float4* Bq = reinterpret_cast<const float4*>(Bs + r * 16);
                const float2 u = bc2(dv * xv);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float4 bb = Bq[q];
                  h[2 * q] = __ffma2_rn(Pg[2 * q], __fmul2_rn(u, make_float2(bb.x, bb.y)), h[2 * q]);
                  h[2 * q + 1] = __ffma2_rn(Pg[2 * q + 1], __fmul2_rn(u, make_float2(bb.z, bb.w)), h[2 * q + 1]);
                  Pg[2 * q] = __ffma2_rn(Pg[2 * q], e[2 * q], Pg[2 * q]);
                  Pg[2 * q + 1] = __ffma2_rn(Pg[2 * q + 1], e[2 * q + 1], Pg[2 * q + 1]);
                }
              }
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float2 bb = reinterpret_cast<const float2*>(Bs + r * 16)[k];
                float2 e, bx;
                gen_pair<ZOH>(g, k, dv, xv, bb, e, bx);
                h[k] = __ffma2_rn(Pg[k], bx, h[k]);
                Pg[k] = __ffma2_rn(Pg[k], e, Pg[k]);
              }
            }
          }
          // decay check; inactive lanes do not hold the warp back. Products above 1 (delta < 0) never
          // decay: only t = 0 ends such a walk.
          float pm = 0.0f;
#pragma unroll
          for (int k = 0; k < 8; ++k) pm = fmaxf(pm, fmaxf(fabsf(Pg[k].x), fabsf(Pg[k].y)));
          if (!act) pm = 0.0f;
          const bool reached_start = (tg.t_lo == 0);
          if (reached_start && h0row && act) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              h[k] = __ffma2_rn(Pg[k], make_float2(h0row[2 * k], h0row[2 * k + 1]), h[k]);
          }
          if (reached_start || !__any_sync(0xffffffffu, pm >= kCarryEps)) {
            done = true;
            if (lane == 0) atomicAdd(&s.done_count, 1);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[slot]);
        ++seq;
      }
    }

    // ---- forward over [t0, t1) ----
    for (int64_t tb = t0; tb < t1; tb += TS) {
      const int slot = static_cast<int>(seq % NS);
      if (!pending_fwd) {
        const uint32_t par = static_cast<uint32_t>((seq / NS) & 1);
        if (!mbar_wait(&s.full[slot], par, abort) || !mbar_wait(&s.ready[slot], par, abort)) return;
      }
      pending_fwd = false;
      const Tag tg = s.tag[slot];
      const T* xs = s.x[slot];
      const T* ds = s.dl[slot];
      const float* Bs = (ZOH && s4d) ? s.Bp[slot] : s.Bf[slot];
      const float* Cs = s.Cf[slot];
#pragma unroll 2
      for (int t = tg.t_lo; t < tg.t_hi; ++t) {
        const int r = t - tg.t_start;
        const float xv = tof<T>(xs[r * DT + c]);
        const float dv = tof<T>(ds[r * DT + c]);
        const float4* Bq = reinterpret_cast<const float4*>(Bs + r * 16);
        const float4* Cq = reinterpret_cast<const float4*>(Cs + r * 16);
        float2 ya = make_float2(0.0f, 0.0f), yb = make_float2(0.0f, 0.0f);
        if (s4d) {
          const float w = dv * A2_0;
          float2 e[8];
          em1_tree(exp2m1(w, ex2(w)), e);
          if (ZOH) {
            // h <- Abar h + (Abar - 1) q  ==  h + e (h + q),  q = (B / (n+1)) (x / A_0)
            const float2 xi = bc2(xv * invA0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 bb = Bq[q], cc = Cq[q];
              const float2 s0 = __ffma2_rn(make_float2(bb.x, bb.y), xi, h[2 * q]);
              h[2 * q] = __ffma2_rn(e[2 * q], s0, h[2 * q]);
              const float2 s1 = __ffma2_rn(make_float2(bb.z, bb.w), xi, h[2 * q + 1]);
              h[2 * q + 1] = __ffma2_rn(e[2 * q + 1], s1, h[2 * q + 1]);
              ya = __ffma2_rn(make_float2(cc.x, cc.y), h[2 * q], ya);
              yb = __ffma2_rn(make_float2(cc.z, cc.w), h[2 * q + 1], yb);
            }
          } else {
            // h <- Abar h + (delta x) B  ==  (h + e h) + u B
            const float2 u = bc2(dv * xv);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 bb = Bq[q], cc = Cq[q];
              const float2 t0v = __ffma2_rn(e[2 * q], h[2 * q], h[2 * q]);
              h[2 * q] = __ffma2_rn(u, make_float2(bb.x, bb.y), t0v);
              const float2 t1v = __ffma2_rn(e[2 * q + 1], h[2 * q + 1], h[2 * q + 1]);
              h[2 * q + 1] = __ffma2_rn(u, make_float2(bb.z, bb.w), t1v);
              ya = __ffma2_rn(make_float2(cc.x, cc.y), h[2 * q], ya);
              yb = __ffma2_rn(make_float2(cc.z, cc.w), h[2 * q + 1], yb);
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 bb = reinterpret_cast<const float2*>(Bs + r * 16)[k];
            const float2 cc = reinterpret_cast<const float2*>(Cs + r * 16)[k];
            float2 e, bx;
            gen_pair<ZOH>(g, k, dv, xv, bb, e, bx);
            h[k] = __fadd2_rn(__ffma2_rn(e, h[k], h[k]), bx);
            if (k & 1) yb = __ffma2_rn(cc, h[k], yb);
            else ya = __ffma2_rn(cc, h[k], ya);
          }
        }
        if (act) Elem<T>::store(p.y, (b * p.L + t) * p.D + d, (ya.x + ya.y) + (yb.x + yb.y));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[slot]);
      ++seq;
    }
    if (t1 == p.L && p.final_state && act) {
      float4* fs = reinterpret_cast<float4*>(p.final_state + (b * p.D + d) * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) fs[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
    }
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
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct LaunchCache {  // per device: opt-in shared memory set, resident CTAs per SM
  int per_sm = 0;
};

template <typename T, int NW, int TS, int NS, bool ZOH, int MINB>
cudaError_t launch_cfg(const FwdArgs& a) {
  constexpr int DT = NW * 32;
  const bool bf16 = sizeof(T) == 2;
  CUtensorMap mx, md, mB, mC;
  const uint64_t rows = static_cast<uint64_t>(a.batch * a.L);
  if (!make_map(&mx, a.x, bf16, a.D, rows, DT, TS) || !make_map(&md, a.delta, bf16, a.D, rows, DT, TS) ||
      !make_map(&mB, a.B, bf16, 16, rows, 16, TS) || !make_map(&mC, a.C, bf16, 16, rows, 16, TS))
    return cudaErrorInvalidValue;
  TmaParams p;
  p.A_log = a.A_log;
  p.h0 = a.h0;
  p.y = a.y;
  p.final_state = a.final_state;
  p.batch = a.batch;
  p.L = a.L;
  p.D = a.D;
  p.tiles = (a.D + DT - 1) / DT;
  p.total = a.batch * p.tiles * a.L;
  const size_t smem = sizeof(Smem<T, NW, TS, NS>) + 128;
  auto kern = scan_fwd_tma_kernel<T, NW, TS, NS, ZOH, MINB>;
  static LaunchCache cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  LaunchCache& lc = cache[dev & 63];
  if (lc.per_sm == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, (NW + 2) * 32, smem);
    if (e != cudaSuccess) return e;
    lc.per_sm = per_sm < 1 ? 1 : per_sm;
  }
  int64_t nctas = static_cast<int64_t>(sm_count()) * lc.per_sm;
  const int64_t min_steps = 4 * TS;  // keep every CTA's range at least a few stages long
  const int64_t cap = (p.total + min_steps - 1) / min_steps;
  if (nctas > cap) nctas = cap;
  if (nctas < 1) nctas = 1;
  p.nctas = nctas;
  kern<<<static_cast<unsigned>(nctas), (NW + 2) * 32, smem, a.stream>>>(mx, md, mB, mC, p);
  return cudaGetLastError();
}

// Kernel shape: consumer warps per CTA, rows per stage, stages, CTAs per SM the registers allow.
#if SSM_TMA_CFG == 1
constexpr int kNW = 4, kTS = 16, kNS = 4, kMinB = 2;
#elif SSM_TMA_CFG == 2
constexpr int kNW = 8, kTS = 16, kNS = 4, kMinB = 1;
#else
constexpr int kNW = 4, kTS = 32, kNS = 4, kMinB = 1;
#endif

}  // namespace

bool tma_path_ok(const FwdArgs& a) {
  if (a.N != 16) return false;
  const int es = a.dtype == 1 ? 2 : 4;
  if ((a.D * es) % 16 != 0) return false;
  const void* ptrs[] = {a.x, a.delta, a.B, a.C};
  for (const void* q : ptrs)
    if (reinterpret_cast<uintptr_t>(q) % 16 != 0) return false;
  if (a.final_state && reinterpret_cast<uintptr_t>(a.final_state) % 16 != 0) return false;
  if (a.batch * a.L > (int64_t(1) << 30)) return false;  // TMA row coordinates are 32-bit
  if (encoder() == nullptr) return false;
  return true;
}

cudaError_t launch_fwd_tma(const FwdArgs& a) {
  if (a.dtype == 1)
    return a.disc == 1 ? launch_cfg<__nv_bfloat16, kNW, kTS, kNS, true, kMinB>(a)
                       : launch_cfg<__nv_bfloat16, kNW, kTS, kNS, false, kMinB>(a);
  return a.disc == 1 ? launch_cfg<float, kNW, kTS, kNS, true, kMinB>(a) : launch_cfg<float, kNW, kTS, kNS, false, kMinB>(a);
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
