// scan_fwd_simple.cu -- general-shape prefill scan (any D, any N in [1, 16], any alignment).
//
// Work layout: one lane per channel d, one warp per 32 consecutive channels of one batch element
// (a "row"). The rows' time axes are laid end to end and cut into equal contiguous pieces, one per warp
// of the grid, so every warp gets the same number of (row, t) steps whatever the shape.
//
// A piece that starts at t0 > 0 first rebuilds the state entering t0 with no communication: it walks the
// preceding steps backwards and accumulates
//     h(t0-1) = sum_j ( prod_{k=j+1..t0-1} Abar_k ) * Bbar_j x_j          ("Mathematical Prerequisites for
//                                                                          Mamba" s6, unrolled sum)
// stopping once every decay product is below kCarryEps (the rest is at most that fraction of the state
// there) or at t = 0, where the sum is exact (plus prod * h0 when an initial state is given). It then
// runs the recurrence of "Understanding Mamba" Eq. (3) forward over its own steps, writing y.
//
// Discretisation: e = Abar - 1 = 2^{delta A log2 e} - 1 (SFU exp2, a Taylor series where |delta A| is small,
// so the decay h + e h is exact to one rounding over arbitrarily long walks); Euler Bbar = delta B, ZOH
// Bbar = e / A B, delta B where A == 0.
#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int kWarps = 4;           // warps per CTA
constexpr int kMinPiece = 32;       // shortest piece worth a separate warp

struct SimpleParams {
  const void* x;
  const void* delta;
  const float* A_log;
  const void* B;
  const void* C;
  const float* h0;
  void* y;
  float* final_state;
  int64_t batch, L, D, N;
  int64_t groups;   // ceil(D / 32)
  int64_t total;    // batch * groups * L
  int64_t nwarps;   // warps taking part
  // optional layer pieces (see ssm_scan_fwd_ex); applied with warp-uniform branches
  const float* delta_bias;  // [D] or null: delta + bias[d]
  int softplus;             // delta = softplus(delta + bias[d])
  const float* D_skip;      // [D] or null: y + D[d] x
  const void* z;            // [batch, L, D] or null: y * SiLU(z)
};

__device__ __forceinline__ float delta_of(const SimpleParams& p, float raw, float bias) {
  const float v = raw + bias;
  return p.softplus ? softplus_f(v) : v;
}

template <int NP, bool ZOH>
struct Chan {
  float A2[NP];    // A * log2(e)
  float invA[NP];  // 1 / A (ZOH), 0 where A == 0
  bool zeroA[NP];
};

// e = Abar - 1 (no cancellation) and the input term Bbar x of one state entry.
template <int NP, bool ZOH>
__device__ __forceinline__ void step_terms(const Chan<NP, ZOH>& c, int n, float dt, float x, float b, float& e,
                                          float& bx) {
  const float w = dt * c.A2[n];
  e = exp2m1(w, ex2(w));
  if (ZOH) {
    const float coef = c.zeroA[n] ? dt : e * c.invA[n];
    bx = coef * b * x;
  } else {
    bx = dt * b * x;
  }
}

// Inputs are staged kKS steps at a time: each lane loads its channel's x and delta for the chunk's steps and
// its share of the chunk's B and C rows (contiguous in memory) into registers one chunk ahead, then stores
// them into this warp's shared memory, from which the steps read them. One global round trip then serves
// kKS steps instead of one. 16 steps for up to 8 state entries; 8 for 16, whose registers go to the state.
template <int NP>
constexpr int kKSof = NP == 16 ? 8 : 16;

template <int NP>
struct Stage {  // one chunk in flight: this lane's x and raw delta per step, its share of the B and C rows
  static constexpr int kKS = kKSof<NP>;
  float x[kKS], d[kKS], b[kKS * NP / 32], c[kKS * NP / 32];
};

// Per-warp shared memory (floats): xs, ds [kKS][32] (delta already through delta_of), Bs, Cs [kKS][N].
template <int NP>
constexpr int kStageFloats = 2 * kKSof<NP> * 32 + 2 * kKSof<NP> * NP;

// Steps [s, s + n) of row (b, channel group) for channel d; the C rows only when WC.
template <int NP, typename T, bool WC>
__device__ __forceinline__ void stage_load(const SimpleParams& p, int64_t b, int64_t d, bool act, int lane,
                                           int64_t s, int n, Stage<NP>& st) {
  constexpr int kKS = kKSof<NP>;
  const int N = static_cast<int>(p.N);
#pragma unroll
  for (int k = 0; k < kKS; ++k) {
    const bool ok = act && k < n;
    const int64_t xi = (b * p.L + s + k) * p.D + d;
    st.x[k] = ok ? Elem<T>::load(p.x, xi) : 0.0f;
    st.d[k] = ok ? Elem<T>::load(p.delta, xi) : 0.0f;
  }
  const int64_t bi = (b * p.L + s) * N;
  const int cnt = n * N;
#pragma unroll
  for (int m = 0; m < kKS * NP / 32; ++m) {
    const int i = lane + 32 * m;
    st.b[m] = i < cnt ? Elem<T>::load(p.B, bi + i) : 0.0f;
    if (WC) st.c[m] = i < cnt ? Elem<T>::load(p.C, bi + i) : 0.0f;
  }
}

template <int NP, bool WC>
__device__ __forceinline__ void stage_store(const SimpleParams& p, const Stage<NP>& st, bool act, float dbias,
                                            int lane, float* xs, float* ds, float* Bs, float* Cs) {
  constexpr int kKS = kKSof<NP>;
#pragma unroll
  for (int k = 0; k < kKS; ++k) {
    xs[k * 32 + lane] = st.x[k];
    ds[k * 32 + lane] = act ? delta_of(p, st.d[k], dbias) : 0.0f;
  }
#pragma unroll
  for (int m = 0; m < kKS * NP / 32; ++m) {
    Bs[lane + 32 * m] = st.b[m];
    if (WC) Cs[lane + 32 * m] = st.c[m];
  }
}

template <int NP, bool ZOH, typename T>
__global__ void __launch_bounds__(kWarps * 32) scan_fwd_simple_kernel(SimpleParams p) {
  constexpr int kKS = kKSof<NP>;
  __shared__ float smem[kWarps * kStageFloats<NP>];
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (gw >= p.nwarps) return;  // whole warp leaves together
  float* xs = smem + (threadIdx.x >> 5) * kStageFloats<NP>;
  float* ds = xs + kKS * 32;
  float* Bs = ds + kKS * 32;  // [kKS][N]
  float* Cs = Bs + kKS * NP;
  int64_t lo = static_cast<int64_t>(static_cast<__int128>(gw) * p.total / p.nwarps);
  const int64_t hi = static_cast<int64_t>(static_cast<__int128>(gw + 1) * p.total / p.nwarps);
  const int N = static_cast<int>(p.N);
  while (lo < hi) {
    const int64_t row = lo / p.L;
    const int64_t t0 = lo % p.L;
    const int64_t t1 = (hi - lo < p.L - t0) ? t0 + (hi - lo) : p.L;
    lo += t1 - t0;
    const int64_t b = row / p.groups;
    const int64_t d = (row % p.groups) * 32 + lane;
    const bool act = d < p.D;
    const float dbias = (act && p.delta_bias) ? __ldg(p.delta_bias + d) : 0.0f;
    const float dskip = (act && p.D_skip) ? __ldg(p.D_skip + d) : 0.0f;

    Chan<NP, ZOH> c;
#pragma unroll
    for (int n = 0; n < NP; ++n) {
      float A = -1.0f;
      if (act && n < N) A = -expf(__ldg(p.A_log + d * N + n));
      c.A2[n] = A * kLog2e;
      c.zeroA[n] = (A == 0.0f);
      c.invA[n] = c.zeroA[n] ? 0.0f : 1.0f / A;
    }
    const float* h0row = p.h0 ? p.h0 + (b * p.D + d) * N : nullptr;
    Stage<NP> st;

    // ---- state entering t0 -------------------------------------------------------------------
    float h[NP];
#pragma unroll
    for (int n = 0; n < NP; ++n) h[n] = 0.0f;
    if (t0 == 0) {
      if (h0row && act) {
#pragma unroll
        for (int n = 0; n < NP; ++n)
          if (n < N) h[n] = h0row[n];
      }
    } else {
      // chunks [cs, ce) from t0 backwards; steps taken from ce - 1 down to cs
      float P[NP];
#pragma unroll
      for (int n = 0; n < NP; ++n) P[n] = 1.0f;
      int64_t ce = t0;
      int64_t cs = ce > kKS ? ce - kKS : 0;
      int64_t steps = 0;
      bool done = false;
      stage_load<NP, T, false>(p, b, d, act, lane, cs, static_cast<int>(ce - cs), st);
      while (!done) {
        __syncwarp();
        stage_store<NP, false>(p, st, act, dbias, lane, xs, ds, Bs, Cs);
        __syncwarp();
        const int cn = static_cast<int>(ce - cs);
        const int64_t cs2 = cs > kKS ? cs - kKS : 0;
        if (cs > 0) stage_load<NP, T, false>(p, b, d, act, lane, cs2, static_cast<int>(cs - cs2), st);
#pragma unroll 1
        for (int k = cn - 1; k >= 0; --k) {
          const float xv = xs[k * 32 + lane];
          const float dt = ds[k * 32 + lane];
#pragma unroll
          for (int n = 0; n < NP; ++n) {
            const float bn = (n < N) ? Bs[k * N + n] : 0.0f;
            float e, bx;
            step_terms<NP, ZOH>(c, n, dt, xv, bn, e, bx);
            h[n] = fmaf(P[n], bx, h[n]);
            P[n] = fmaf(P[n], e, P[n]);
          }
          ++steps;
          if (cs + k == 0) {
            if (h0row && act) {
#pragma unroll
              for (int n = 0; n < NP; ++n)
                if (n < N) h[n] = fmaf(P[n], h0row[n], h[n]);
            }
            done = true;
            break;
          }
          if ((steps & 7) == 0) {
            float pm = 0.0f;
#pragma unroll
            for (int n = 0; n < NP; ++n) pm = fmaxf(pm, fabsf(P[n]));
            if (!act) pm = 0.0f;
            if (!__any_sync(0xffffffffu, pm >= kCarryEps)) {
              done = true;
              break;
            }
          }
        }
        ce = cs;
        cs = cs2;
      }
    }

    // ---- forward over [t0, t1), in chunks ------------------------------------------------------
    stage_load<NP, T, true>(p, b, d, act, lane, t0, static_cast<int>(t1 - t0 < kKS ? t1 - t0 : kKS), st);
    for (int64_t cs = t0; cs < t1; cs += kKS) {
      const int cn = static_cast<int>(t1 - cs < kKS ? t1 - cs : kKS);
      __syncwarp();
      stage_store<NP, true>(p, st, act, dbias, lane, xs, ds, Bs, Cs);
      __syncwarp();
      const int64_t cs2 = cs + kKS;
      if (cs2 < t1) stage_load<NP, T, true>(p, b, d, act, lane, cs2, static_cast<int>(t1 - cs2 < kKS ? t1 - cs2 : kKS), st);
#pragma unroll 1
      for (int k = 0; k < cn; ++k) {
        const float xv = xs[k * 32 + lane];
        const float dt = ds[k * 32 + lane];
        float yv = 0.0f;
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          const float bn = (n < N) ? Bs[k * N + n] : 0.0f;
          const float cn_ = (n < N) ? Cs[k * N + n] : 0.0f;
          float e, bx;
          step_terms<NP, ZOH>(c, n, dt, xv, bn, e, bx);
          h[n] = fmaf(e, h[n], h[n]) + bx;
          yv = fmaf(cn_, h[n], yv);
        }
        if (act) {
          const int64_t xi = (b * p.L + cs + k) * p.D + d;
          if (p.D_skip) yv = fmaf(dskip, xv, yv);
          if (p.z) yv *= silu_f(Elem<T>::load(p.z, xi));
          Elem<T>::store(p.y, xi, yv);
        }
      }
    }
    if (t1 == p.L && p.final_state && act) {
      float* fs = p.final_state + (b * p.D + d) * N;
#pragma unroll
      for (int n = 0; n < NP; ++n)
        if (n < N) fs[n] = h[n];
    }
  }
}

// Warps for a launch: one per piece of at least kMinPiece steps, at most as many as are resident at once.
template <int NP, bool ZOH, typename T>
cudaError_t launch_np(SimpleParams sp, cudaStream_t s) {
  static int per_sm[64] = {0};  // resident CTAs per SM, per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int& k = per_sm[dev & 63];
  if (k == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, scan_fwd_simple_kernel<NP, ZOH, T>, kWarps * 32, 0);
    if (e != cudaSuccess) return e;
    if (k < 1) k = 1;
  }
  const int64_t rows = sp.batch * sp.groups;
  const int64_t want = static_cast<int64_t>(sm_count()) * k * kWarps;
  int64_t nw = rows * ((sp.L + kMinPiece - 1) / kMinPiece);
  if (nw > want) nw = want;
  if (nw < 1) nw = 1;
  sp.nwarps = nw;
  const int64_t blocks = (nw + kWarps - 1) / kWarps;
  scan_fwd_simple_kernel<NP, ZOH, T><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(sp);
  return cudaGetLastError();
}

template <bool ZOH, typename T>
cudaError_t launch_disc(const SimpleParams& sp, cudaStream_t s) {
  if (sp.N <= 4) return launch_np<4, ZOH, T>(sp, s);
  if (sp.N <= 8) return launch_np<8, ZOH, T>(sp, s);
  return launch_np<16, ZOH, T>(sp, s);
}

__global__ void init_state_kernel(const float* h0, float* out, int64_t n) {
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) out[i] = h0 ? h0[i] : 0.0f;
}

}  // namespace

cudaError_t launch_fwd_simple(const FwdArgs& a) {
  SimpleParams sp;
  sp.x = a.x; sp.delta = a.delta; sp.A_log = a.A_log; sp.B = a.B; sp.C = a.C; sp.h0 = a.h0;
  sp.y = a.y; sp.final_state = a.final_state;
  sp.delta_bias = a.delta_bias; sp.softplus = a.softplus; sp.D_skip = a.D_skip; sp.z = a.z;
  sp.batch = a.batch; sp.L = a.L; sp.D = a.D; sp.N = a.N;
  sp.groups = (a.D + 31) / 32;
  sp.total = a.batch * sp.groups * a.L;
  if (a.disc == 1)
    return a.dtype == 1 ? launch_disc<true, __nv_bfloat16>(sp, a.stream) : launch_disc<true, float>(sp, a.stream);
  return a.dtype == 1 ? launch_disc<false, __nv_bfloat16>(sp, a.stream) : launch_disc<false, float>(sp, a.stream);
}

cudaError_t launch_init_state(const FwdArgs& a) {
  const int64_t n = a.batch * a.D * a.N;
  if (n == 0 || a.final_state == nullptr) return cudaSuccess;
  init_state_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, a.stream>>>(a.h0, a.final_state, n);
  return cudaGetLastError();
}

}  // namespace ssm
