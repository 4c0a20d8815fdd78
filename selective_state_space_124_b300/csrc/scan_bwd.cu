// scan_bwd.cu -- backward pass of the prefill scan: gradients of
//     J = sum dy * y + sum dfinal * final_state
// with respect to x, delta, A_log, B, C and h0, with the states recomputed rather than stored ("State Space
// Models & Mamba" chapter, the paragraph on the fused kernel: the backward pass recomputes h_t instead of
// keeping it). The gradient formulas are the chain rule of the forward recurrence h_t = Abar_t h_{t-1} +
// Bbar_t x_t, y_t = C_t . h_t, run backwards through the adjoint lambda_t = dJ/dh_t:
//     lambda_t = C_t dy_t + Abar_{t+1} lambda_{t+1}                 (lambda_{L-1} adds dfinal)
//     dx_t = sum_n lambda Bbar,   dC_t,n = dy_t h_t,   dB_t,n = lambda x (Bbar / B)
//     ddelta_t = sum_n lambda h_{t-1} A Abar + lambda x dBbar/ddelta,   dA_n = sum_t lambda h_{t-1} delta Abar
//                + lambda x dBbar/dA,   dA_log = dA * A,   dh0 = Abar_0 lambda_0
// with dBbar/ddelta = B (Euler) or Abar B (ZOH) and, for ZOH, dBbar/dA = B delta^2 f(delta A),
// f(w) = (w e^w - (e^w - 1)) / w^2 (limit 1/2 at A = 0, the same continuous extension as Bbar there).
//
// Work layout: the forward kernels' split. One lane per channel, one warp per 32 consecutive channels of
// one batch element (a row); the rows' time axes are laid end to end and cut into equal contiguous
// pieces, one per warp. A piece [t0, t1) of a row:
//   1. rebuilds h(t0-1) by the backward warm-up walk of the forward kernels (exact at t = 0);
//   2. runs forward over [t0, t1), saving h at the end of every aligned chunk of kChunk steps that is
//      followed by another chunk of the piece into the workspace (global memory; the only scratch);
//   3. rebuilds mu = Abar_{t1} lambda_{t1} (the adjoint flowing into h_{t1-1} from later steps) by walking
//      forward from t1: mu = sum_{j >= t1} (prod_{k=t1..j} Abar_k) (C_j dy_j + [j = L-1] dfinal), stopping
//      once every decay product is below kCarryEps or at j = L - 1, where it is exact;
//   4. walks the chunks backwards: recomputes the chunk's states from its saved start into shared memory
//      (each lane its own column, so no lane reads another's and no barrier is needed), then steps back
//      through the chunk accumulating the gradients.
// Two implementations of a piece: bwd_piece_s4d where every channel of the warp has the structured decay
// A_n = (n + 1) A_0 at N = 16 (paired f32x2 arithmetic, one decay tree per step, pair-dropping walks), and
// bwd_piece for any A and N <= 16.
// dB and dC sum over channels: each warp reduces its 32 lanes' terms (a shared-memory transpose in the
// structured path, a shuffle reduce-scatter in the generic one) and adds the result into the outputs with one
// atomic add per (step, entry) per warp; dA_log sums over the batch and the time axis: one atomic add per
// entry per piece. A zeroing kernel clears the three first; this kernel is launched as its programmatic
// dependent and waits for it only before its first atomic add.
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "pair_math.cuh"

namespace ssm {
namespace {

constexpr int kBwdWarps = 8;       // warps per CTA
constexpr int kChunk = 8;          // steps per recomputed chunk (shared-memory rows per warp: kChunk + 2)
constexpr int kMinBwdPiece = 128;  // shortest piece worth a separate warp (each piece runs two warm-ups)
constexpr float kLn2 = 0.6931471805599453f;

struct BwdParams {
  const void* x;
  const void* delta;
  const float* A_log;
  const void* B;
  const void* C;
  const float* h0;
  const void* dy;
  const float* dfinal;
  void* dx;
  void* ddelta;
  float* dA_log;
  float* dB;
  float* dC;
  float* dh0;
  float* ws;        // [batch, nck, N, D] chunk-end states
  int64_t batch, L, D, N;
  int64_t nck;      // chunks per row that are followed by another: ceil(L / kChunk) - 1
  int64_t groups;   // ceil(D / 32)
  int64_t total;    // batch * groups * L
  int64_t nwarps;
  int vec;          // fp32 with D % 4 == 0 and 16-byte-aligned x, delta, dy, B, C: chunks load as float4 tiles
};

// f(w) = (w e^w - (e^w - 1)) / w^2 = sum_{m >= 2} (m - 1) w^(m-2) / m!: the Taylor series up to w^6 where the
// difference would cancel (|w| < 1/4; the next term is below 2e-9 there), the difference itself elsewhere
// (a = e^w, e = e^w - 1 computed without cancellation).
__device__ __forceinline__ float zoh_dA_factor(float w, float a, float e) {
  if (fabsf(w) < 0.25f) {
    float q = fmaf(w, 1.0f / 5760.0f, 1.0f / 840.0f);
    q = fmaf(w, q, 1.0f / 144.0f);
    q = fmaf(w, q, 1.0f / 30.0f);
    q = fmaf(w, q, 1.0f / 8.0f);
    q = fmaf(w, q, 1.0f / 3.0f);
    return fmaf(w, q, 0.5f);
  }
  return (w * a - e) / (w * w);
}

// floats of shared memory per warp: kChunk + 2 rows of NP x 32 states, then a chunk's x, delta and dy columns
// and its B and C rows
template <int NP>
constexpr int kBwdWarpFloats = (kChunk + 2) * NP * 32 + 3 * kChunk * 32 + 2 * kChunk * 16;

template <int NP, bool ZOH>
struct BwdChan {
  float A2[NP];    // A * log2(e)
  float invA[NP];  // 1 / A (ZOH), 0 where A == 0
};

// e_n = Abar_n - 1 of every entry at one step, for the generic path: one SFU exp2 (and the cancellation-free
// series) per entry. (The structured path below derives all 16 from e_0 with the decay tree.)
template <int NP, bool ZOH>
__device__ __forceinline__ void step_e(const BwdChan<NP, ZOH>& c, float dt, float (&e)[NP]) {
#pragma unroll
  for (int n = 0; n < NP; ++n) {
    const float w = dt * c.A2[n];
    e[n] = exp2m1(w, ex2(w));
  }
}

// Bbar / B of entry n: delta (Euler), e_n / A_n (ZOH; delta where A_n == 0).
template <int NP, bool ZOH>
__device__ __forceinline__ float bfac(const BwdChan<NP, ZOH>& c, int n, float dt, float e) {
  if (ZOH) return c.A2[n] == 0.0f ? dt : e * c.invA[n];
  return dt;
}

// Sum over the warp of 32 values per lane (v[j], j < 32); lane l returns the total of v[l]. Recursive
// halving: at each level a lane keeps the half of its values selected by one bit of its index and adds
// the partner's copy of that half (16 + 8 + 4 + 2 + 1 shuffles).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = up ? v[j] : v[j + w];
      const float keep = up ? v[j + w] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// One chunk of at most kChunk consecutive steps [s, s + n) of a row, staged in this warp's shared memory for
// the arithmetic: each lane's x, delta and dy in its own column (xs, ds, gs: [kChunk][32]), the shared B and C
// rows in bs, cs ([kChunk][16]). All loads of a chunk are issued before any is stored, so a chunk costs one
// memory round trip rather than one per step, and the step loops can stay rolled (small code) while still
// indexing the chunk's steps.
template <typename T, bool WX, bool WG, bool WB, bool WC>
__device__ __forceinline__ void load_chunk(const BwdParams& p, int64_t b, int64_t d, bool act, int lane, int64_t s,
                                           int n, float* xs, float* ds, float* gs, float* bs, float* cs) {
  const int64_t base = (b * p.L + s) * p.D + d;
  const int N = static_cast<int>(p.N);
  const int64_t bc = (b * p.L + s) * p.N;
  float xv[kChunk], dv[kChunk], gv[kChunk], bv[kChunk * 16 / 32], cv[kChunk * 16 / 32];
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    const bool ok = act && i < n;
    if (WX) xv[i] = ok ? Elem<T>::load(p.x, base + static_cast<int64_t>(i) * p.D) : 0.0f;
    dv[i] = ok ? Elem<T>::load(p.delta, base + static_cast<int64_t>(i) * p.D) : 0.0f;
    if (WG) gv[i] = ok ? Elem<T>::load(p.dy, base + static_cast<int64_t>(i) * p.D) : 0.0f;
  }
#pragma unroll
  for (int m = 0; m < kChunk * 16 / 32; ++m) {
    const int k = lane + 32 * m, i = k >> 4, nn = k & 15;
    const bool ok = i < n && nn < N;
    if (WB) bv[m] = ok ? Elem<T>::load(p.B, bc + static_cast<int64_t>(i) * N + nn) : 0.0f;
    if (WC) cv[m] = ok ? Elem<T>::load(p.C, bc + static_cast<int64_t>(i) * N + nn) : 0.0f;
  }
  __syncwarp();  // every lane has finished reading the previous chunk
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    if (WX) xs[i * 32 + lane] = xv[i];
    ds[i * 32 + lane] = dv[i];
    if (WG) gs[i * 32 + lane] = gv[i];
  }
#pragma unroll
  for (int m = 0; m < kChunk * 16 / 32; ++m) {
    if (WB) bs[lane + 32 * m] = bv[m];
    if (WC) cs[lane + 32 * m] = cv[m];
  }
  __syncwarp();
}

// One piece [t0, t1) of a row, any A (see the file comment for the four phases).
template <int NP, bool ZOH, typename T>
__device__ __forceinline__ void bwd_piece(const BwdParams& p, const BwdChan<NP, ZOH>& c, float* hs, float* xs,
                                          float* ds, float* gs, float* bs, float* cs, int lane, int64_t row,
                                          int64_t t0, int64_t t1) {
  auto hrow = [&](int r, int n) -> float& { return hs[(r * NP + n) * 32 + lane]; };
  constexpr int kStart = kChunk + 1;
  const int N = static_cast<int>(p.N);
  const int64_t L = p.L, D = p.D;
  const int64_t b = row / p.groups;
  const int64_t d = (row % p.groups) * 32 + lane;
  const bool act = d < D;
  // ---- 1. h(t0 - 1): walk back from t0 - 1 one chunk at a time ------------------------------------------
  float h[NP];
#pragma unroll
  for (int n = 0; n < NP; ++n) h[n] = 0.0f;
  const float* h0row = p.h0 ? p.h0 + (b * D + d) * N : nullptr;
  if (t0 > 0) {
    float P[NP];
#pragma unroll
    for (int n = 0; n < NP; ++n) P[n] = 1.0f;
    for (int64_t j = t0; j > 0;) {  // chunk [s, j)
      const int64_t s = j > kChunk ? j - kChunk : 0;
      const int cn = static_cast<int>(j - s);
      load_chunk<T, true, false, true, false>(p, b, d, act, lane, s, cn, xs, ds, gs, bs, cs);
#pragma unroll 1
      for (int i = cn - 1; i >= 0; --i) {
        const float xv = xs[i * 32 + lane], dt = ds[i * 32 + lane];
        float ev[NP];
        step_e<NP, ZOH>(c, dt, ev);
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          h[n] = fmaf(P[n], bfac(c, n, dt, ev[n]) * bs[i * 16 + n] * xv, h[n]);
          P[n] = fmaf(P[n], ev[n], P[n]);
        }
      }
      j = s;
      float pm = 0.0f;
#pragma unroll
      for (int n = 0; n < NP; ++n) pm = fmaxf(pm, fabsf(P[n]));
      if (!act) pm = 0.0f;
      if (j > 0 && !__any_sync(0xffffffffu, pm >= kCarryEps)) break;
      if (j == 0 && h0row && act) {  // the walk reached t = 0: exact, plus the decayed initial state
#pragma unroll
        for (int n = 0; n < NP; ++n)
          if (n < N) h[n] = fmaf(P[n], h0row[n], h[n]);
      }
    }
  } else if (h0row && act) {
#pragma unroll
    for (int n = 0; n < NP; ++n)
      if (n < N) h[n] = h0row[n];
  }
#pragma unroll
  for (int n = 0; n < NP; ++n) hrow(kStart, n) = h[n];

  // ---- 2. forward over the piece in aligned chunks, saving the state at each chunk end followed by another
  for (int64_t ck = t0 / kChunk; ck * kChunk < t1; ++ck) {
    const int64_t s = ck * kChunk > t0 ? ck * kChunk : t0;
    const int64_t e_ = (ck + 1) * kChunk < t1 ? (ck + 1) * kChunk : t1;
    const int cn = static_cast<int>(e_ - s);
    load_chunk<T, true, false, true, false>(p, b, d, act, lane, s, cn, xs, ds, gs, bs, cs);
#pragma unroll 1
    for (int i = 0; i < cn; ++i) {
      const float xv = xs[i * 32 + lane], dt = ds[i * 32 + lane];
      float ev[NP];
      step_e<NP, ZOH>(c, dt, ev);
#pragma unroll
      for (int n = 0; n < NP; ++n) h[n] = fmaf(ev[n], h[n], h[n]) + bfac(c, n, dt, ev[n]) * bs[i * 16 + n] * xv;
    }
    if (e_ == (ck + 1) * kChunk && e_ < t1 && act) {  // chunk ck ends inside the piece
      float* w = p.ws + ((b * p.nck + ck) * N) * D + d;
#pragma unroll
      for (int n = 0; n < NP; ++n)
        if (n < N) w[static_cast<int64_t>(n) * D] = h[n];
    }
  }

  // ---- 3. the adjoint entering from the right of the piece: walk forward from t1 one chunk at a time ----
  float mu[NP];
#pragma unroll
  for (int n = 0; n < NP; ++n) mu[n] = 0.0f;
  const float* dfrow = p.dfinal ? p.dfinal + (b * D + d) * N : nullptr;
  if (t1 == L) {
    if (dfrow && act) {
#pragma unroll
      for (int n = 0; n < NP; ++n)
        if (n < N) mu[n] = dfrow[n];
    }
  } else {
    float P[NP];
#pragma unroll
    for (int n = 0; n < NP; ++n) P[n] = 1.0f;
    for (int64_t j = t1; j < L;) {  // chunk [j, e_)
      const int64_t e_ = j + kChunk < L ? j + kChunk : L;
      const int cn = static_cast<int>(e_ - j);
      load_chunk<T, false, true, false, true>(p, b, d, act, lane, j, cn, xs, ds, gs, bs, cs);
#pragma unroll 1
      for (int i = 0; i < cn; ++i) {
        const float dt = ds[i * 32 + lane], g = gs[i * 32 + lane];
        float ev[NP];
        step_e<NP, ZOH>(c, dt, ev);
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          P[n] = fmaf(P[n], ev[n], P[n]);
          mu[n] = fmaf(P[n], cs[i * 16 + n] * g, mu[n]);
        }
      }
      j = e_;
      if (j == L) {  // exact: add the final-state gradient, decayed through every step after t1 - 1
        if (dfrow && act) {
#pragma unroll
          for (int n = 0; n < NP; ++n)
            if (n < N) mu[n] = fmaf(P[n], dfrow[n], mu[n]);
        }
        break;
      }
      float pm = 0.0f;
#pragma unroll
      for (int n = 0; n < NP; ++n) pm = fmaxf(pm, fabsf(P[n]));
      if (!act) pm = 0.0f;
      if (!__any_sync(0xffffffffu, pm >= kCarryEps)) break;
    }
  }

  // ---- 4. chunks backwards ----------------------------------------------------------------------------
  // dB, dC and dA_log are zeroed by the launch before this kernel, which may still be running (programmatic
  // dependent launch): wait for it before the first atomic add. A no-op once it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float dA[NP];
#pragma unroll
  for (int n = 0; n < NP; ++n) dA[n] = 0.0f;
  for (int64_t ck = (t1 - 1) / kChunk; ck >= t0 / kChunk; --ck) {
    const int64_t s = ck * kChunk > t0 ? ck * kChunk : t0;
    const int64_t e_ = (ck + 1) * kChunk < t1 ? (ck + 1) * kChunk : t1;
    const int cn = static_cast<int>(e_ - s);
    load_chunk<T, true, true, true, true>(p, b, d, act, lane, s, cn, xs, ds, gs, bs, cs);
    if (s == t0) {
#pragma unroll
      for (int n = 0; n < NP; ++n) h[n] = hrow(kStart, n);
    } else {  // s = ck * kChunk > t0: chunk ck - 1 ends inside the piece; step 2 saved its state
      const float* w = p.ws + ((b * p.nck + ck - 1) * N) * D + d;
#pragma unroll
      for (int n = 0; n < NP; ++n) h[n] = (act && n < N) ? w[static_cast<int64_t>(n) * D] : 0.0f;
    }
#pragma unroll
    for (int n = 0; n < NP; ++n) hrow(0, n) = h[n];
#pragma unroll 1
    for (int i = 0; i < cn; ++i) {
      const float xv = xs[i * 32 + lane], dt = ds[i * 32 + lane];
      float ev[NP];
      step_e<NP, ZOH>(c, dt, ev);
#pragma unroll
      for (int n = 0; n < NP; ++n) {
        h[n] = fmaf(ev[n], h[n], h[n]) + bfac(c, n, dt, ev[n]) * bs[i * 16 + n] * xv;
        hrow(i + 1, n) = h[n];
      }
    }
#pragma unroll 1
    for (int i = cn - 1; i >= 0; --i) {
      const int64_t t = s + i;
      const float xv = xs[i * 32 + lane], dt = ds[i * 32 + lane], g = gs[i * 32 + lane];
      float gx = 0.0f, gdt = 0.0f;
      float ev[NP];
      step_e<NP, ZOH>(c, dt, ev);
      float v[32];  // this lane's terms of dB (v[n]) and dC (v[16 + n]) at step t
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        v[n] = 0.0f;
        v[16 + n] = 0.0f;
      }
#pragma unroll
      for (int n = 0; n < NP; ++n) {
        const float bn = bs[i * 16 + n], cn_ = cs[i * 16 + n];
        const float e = ev[n], a = 1.0f + e, bf = bfac(c, n, dt, e);
        const float An = c.A2[n] * kLn2;
        const float lam = fmaf(cn_, g, mu[n]);
        const float gb = lam * xv;           // dJ/dBbar
        const float ga = lam * hrow(i, n);   // dJ/dAbar = lambda h_{t-1}
        v[16 + n] = g * hrow(i + 1, n);      // dC term: dy h_t
        v[n] = gb * bf;                      // dB term
        gx = fmaf(lam * bf, bn, gx);
        gdt = fmaf(ga * An, a, gdt);
        dA[n] = fmaf(ga * dt, a, dA[n]);
        if (ZOH) {
          gdt = fmaf(gb * a, bn, gdt);
          dA[n] = fmaf(gb * bn, dt * dt * zoh_dA_factor(dt * An, a, e), dA[n]);
        } else {
          gdt = fmaf(gb, bn, gdt);
        }
        mu[n] = a * lam;
      }
      if (act) {
        const int64_t xi = (b * L + t) * D + d;
        Elem<T>::store(p.dx, xi, gx);
        Elem<T>::store(p.ddelta, xi, gdt);
      }
      const float tot = warp_reduce_scatter32(v, lane);  // lane l: total of v[l] over the warp
      const int n_out = lane & 15;
      if (n_out < N) atomicAdd((lane < 16 ? p.dB : p.dC) + (b * L + t) * N + n_out, tot);
    }
  }
  if (act) {
    if (t0 == 0 && p.dh0) {
      float* out = p.dh0 + (b * D + d) * N;
#pragma unroll
      for (int n = 0; n < NP; ++n)
        if (n < N) out[n] = mu[n];
    }
#pragma unroll
    for (int n = 0; n < NP; ++n)
      if (n < N) atomicAdd(p.dA_log + d * N + n, dA[n] * c.A2[n] * kLn2);
  }
}

// ---- structured A (N = 16, A_n = (n + 1) A_0 on every channel of the warp) ------------------------------
// The same four phases, two state entries per f32x2 instruction, with the per-step algebra cut down:
//   * one decay tree e_0 -> e_1 .. e_15 per step (exact identity, one SFU exp2);
//   * the decayed previous state u_n = Abar_n h_{t-1,n} is formed once and serves both dA_n (sum of
//     delta lambda u) and ddelta's decay term (sum of A_n lambda u);
//   * Euler: dx and ddelta's input term share sigma = sum_n lambda_n B_n (dx = delta sigma, + x sigma);
//   * the walks drop state pairs once their weight is below the truncation bound on every lane (entry n
//     decays (n + 1) times as fast as entry 0);
//   * dB and dC, sums over the warp's channels, go through a transposition tile in shared memory (each lane
//     writes its 32 terms as a row, reads a column and adds it up) instead of a shuffle tree;
//   * the next chunk's inputs are loaded into registers while the current chunk is computed.
// Per-warp shared memory (floats): hs [kChunk][8 pairs][32 lanes] float2, the state before each step of the
// chunk being differentiated; hst [8][32] float2, the state entering the piece; xs, ds, gs [kChunk][32];
// bs, cs [kChunk][16]; red [32][32], the transposition tile.
constexpr int kS4dWarpFloats = kChunk * 512 + 512 + 3 * kChunk * 32 + 2 * kChunk * 16 + 1024;

// 2k + 1 and 2k + 2: entry n's decay rate is (n + 1) times entry 0's
__constant__ float2 kPairN1[8] = {{1.f, 2.f},   {3.f, 4.f},   {5.f, 6.f},   {7.f, 8.f},
                                  {9.f, 10.f},  {11.f, 12.f}, {13.f, 14.f}, {15.f, 16.f}};
__constant__ float2 kPairInvN1[8] = {{1.f, 1.f / 2.f},         {1.f / 3.f, 1.f / 4.f},   {1.f / 5.f, 1.f / 6.f},
                                     {1.f / 7.f, 1.f / 8.f},   {1.f / 9.f, 1.f / 10.f},  {1.f / 11.f, 1.f / 12.f},
                                     {1.f / 13.f, 1.f / 14.f}, {1.f / 15.f, 1.f / 16.f}};

// A chunk's inputs held in registers between their load and their store to shared memory, so that the loads
// of the next chunk are in flight while the current one is computed. Two layouts: each lane's own channel for
// the chunk's steps (x[i] = step i), or, when p.vec is set, the warp's [kChunk x 32] tiles read as float4s
// (lane l holds columns 4 (l % 8) .. + 3 of rows l / 8 and l / 8 + 4 in x[0..3] and x[4..7]; B, C: float4 l of
// the chunk's [kChunk x 16] rows). Both land in shared memory in the same [step][lane] layout.
struct ChunkRegs {
  float x[kChunk], d[kChunk], g[kChunk], b[kChunk * 16 / 32], c[kChunk * 16 / 32];
};

__device__ __forceinline__ float4 ld4(const float* p, bool ok) {
  return ok ? __ldg(reinterpret_cast<const float4*>(p)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}
__device__ __forceinline__ void put4(float* dst, float4 v) { dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w; }
__device__ __forceinline__ float4 get4(const float* src) { return make_float4(src[0], src[1], src[2], src[3]); }

template <typename T, bool WX, bool WG, bool WB, bool WC>
__device__ __forceinline__ void chunk_load(const BwdParams& p, int64_t b, int64_t d, bool act, int lane, int64_t s,
                                           int n, ChunkRegs& r) {
  static_assert(kChunk == 8, "the float4 tile layout covers 8 steps");
  if (sizeof(T) == 4 && p.vec) {
    const int q = lane & 7, r0 = lane >> 3;
    const int64_t col = d - lane + 4 * q;  // first channel of this lane's float4
    const bool cok = col < p.D;            // D % 4 == 0: a float4 is wholly inside or wholly past the row
    const int64_t o0 = (b * p.L + s + r0) * p.D + col, o1 = o0 + 4 * p.D;
    const bool ok0 = cok && r0 < n, ok1 = cok && r0 + 4 < n;
    if (WX) { put4(r.x, ld4(static_cast<const float*>(p.x) + o0, ok0)); put4(r.x + 4, ld4(static_cast<const float*>(p.x) + o1, ok1)); }
    put4(r.d, ld4(static_cast<const float*>(p.delta) + o0, ok0));
    put4(r.d + 4, ld4(static_cast<const float*>(p.delta) + o1, ok1));
    if (WG) { put4(r.g, ld4(static_cast<const float*>(p.dy) + o0, ok0)); put4(r.g + 4, ld4(static_cast<const float*>(p.dy) + o1, ok1)); }
    const int64_t bc = (b * p.L + s) * 16 + 4 * lane;
    const bool bok = (lane >> 2) < n;
    if (WB) put4(r.b, ld4(static_cast<const float*>(p.B) + bc, bok));
    if (WC) put4(r.c, ld4(static_cast<const float*>(p.C) + bc, bok));
    return;
  }
  const int64_t base = (b * p.L + s) * p.D + d;
  const int64_t bc = (b * p.L + s) * 16;
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    const bool ok = act && i < n;
    if (WX) r.x[i] = ok ? Elem<T>::load(p.x, base + static_cast<int64_t>(i) * p.D) : 0.0f;
    r.d[i] = ok ? Elem<T>::load(p.delta, base + static_cast<int64_t>(i) * p.D) : 0.0f;
    if (WG) r.g[i] = ok ? Elem<T>::load(p.dy, base + static_cast<int64_t>(i) * p.D) : 0.0f;
  }
#pragma unroll
  for (int m = 0; m < kChunk * 16 / 32; ++m) {
    const int k = lane + 32 * m;
    const bool ok = (k >> 4) < n;
    if (WB) r.b[m] = ok ? Elem<T>::load(p.B, bc + k) : 0.0f;
    if (WC) r.c[m] = ok ? Elem<T>::load(p.C, bc + k) : 0.0f;
  }
}

template <bool WX, bool WG, bool WB, bool WC>
__device__ __forceinline__ void chunk_store(const BwdParams& p, const ChunkRegs& r, int lane, float* xs, float* ds,
                                            float* gs, float* bs, float* cs) {
  __syncwarp();  // every lane has finished reading the previous chunk
  if (p.vec) {
    const int o0 = (lane >> 3) * 32 + 4 * (lane & 7), o1 = o0 + 4 * 32;
    if (WX) { *reinterpret_cast<float4*>(xs + o0) = get4(r.x); *reinterpret_cast<float4*>(xs + o1) = get4(r.x + 4); }
    *reinterpret_cast<float4*>(ds + o0) = get4(r.d);
    *reinterpret_cast<float4*>(ds + o1) = get4(r.d + 4);
    if (WG) { *reinterpret_cast<float4*>(gs + o0) = get4(r.g); *reinterpret_cast<float4*>(gs + o1) = get4(r.g + 4); }
    if (WB) *reinterpret_cast<float4*>(bs + 4 * lane) = get4(r.b);
    if (WC) *reinterpret_cast<float4*>(cs + 4 * lane) = get4(r.c);
  } else {
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      if (WX) xs[i * 32 + lane] = r.x[i];
      ds[i * 32 + lane] = r.d[i];
      if (WG) gs[i * 32 + lane] = r.g[i];
    }
#pragma unroll
    for (int m = 0; m < kChunk * 16 / 32; ++m) {
      if (WB) bs[lane + 32 * m] = r.b[m];
      if (WC) cs[lane + 32 * m] = r.c[m];
    }
  }
  __syncwarp();
}

// Phase 1 over one staged chunk, steps cn - 1 .. 0, with the first ACT pairs live. W: log2 of entry 0's decay
// over the steps after the current one; P: the live pairs' weights. ZOH accumulates P e B x / A_0; the 1/(n+1)
// of Bbar is applied once when the walk ends.
template <int ACT, bool ZOH>
__device__ __forceinline__ void s4d_walk_back(const float* xs, const float* ds, const float* bs, int cn, int lane,
                                              float A2_0, float invA0, float& W, float2 (&P)[8], float2 (&h)[8]) {
  using namespace pairs;
#pragma unroll 1
  for (int i = cn - 1; i >= 0; --i) {
    const float xv = xs[i * 32 + lane], dv = ds[i * 32 + lane];
    const float2* brow = reinterpret_cast<const float2*>(bs + i * 16);
    const float w = dv * A2_0;
    if (ZOH) {
      float2 e[8];
      em1_tree<ACT>(exp2m1(w, ex2(w)), e);
      const float2 xi = bc(xv * invA0);
#pragma unroll
      for (int k = 0; k < ACT; ++k) h[k] = fma2(mul2(P[k], e[k]), mul2(brow[k], xi), h[k]);
    } else {
      const float2 u = bc(dv * xv);
#pragma unroll
      for (int k = 0; k < ACT; ++k) h[k] = fma2(P[k], mul2(brow[k], u), h[k]);
    }
    W += w;
    powers<ACT>(ex2(W), P);
  }
}

// Phase 3 over one staged chunk, steps 0 .. cn - 1: mu_n += (decay of entry n from t1 through the step)
// C_n dy. W: log2 of entry 0's decay from t1 through the current step.
template <int ACT>
__device__ __forceinline__ void s4d_walk_fwd(const float* ds, const float* gs, const float* cs, int cn, int lane,
                                             float A2_0, float& W, float2 (&P)[8], float2 (&mu)[8]) {
  using namespace pairs;
#pragma unroll 1
  for (int i = 0; i < cn; ++i) {
    W = fmaf(ds[i * 32 + lane], A2_0, W);
    powers<ACT>(ex2(W), P);
    const float2 g = bc(gs[i * 32 + lane]);
    const float2* crow = reinterpret_cast<const float2*>(cs + i * 16);
#pragma unroll
    for (int k = 0; k < ACT; ++k) mu[k] = fma2(P[k], mul2(crow[k], g), mu[k]);
  }
}

// One forward step of the structured recurrence on all 16 entries (the forward kernels' update):
// Euler h + e h + (delta x) B; ZOH h + e (h + (x / A_0) B / (n + 1)).
template <bool ZOH>
__device__ __forceinline__ void s4d_fwd_step(float xv, float dv, const float* brow_f, float A2_0, float invA0,
                                             float2 (&h)[8]) {
  using namespace pairs;
  const float2* brow = reinterpret_cast<const float2*>(brow_f);
  float2 e[8];
  step_e16(dv * A2_0, e);
  if (ZOH) {
    const float2 s = bc(xv * invA0);
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = fma2(e[k], fma2(mul2(brow[k], kPairInvN1[k]), s, h[k]), h[k]);
  } else {
    const float2 s = bc(dv * xv);
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = fma2(s, brow[k], fma2(e[k], h[k], h[k]));
  }
}

// f(w) = (w e^w - (e^w - 1)) / w^2 for a pair (ZOH dBbar/dA = B delta^2 f(delta A)): its Taylor series where
// the difference would cancel (|w| < 1/4), the difference itself elsewhere; a = e^w, e = e^w - 1.
__device__ __forceinline__ float2 zoh_f2(float2 w, float2 a, float2 e) {
  using namespace pairs;
  float2 q = fma2(w, bc(1.0f / 5760.0f), bc(1.0f / 840.0f));
  q = fma2(w, q, bc(1.0f / 144.0f));
  q = fma2(w, q, bc(1.0f / 30.0f));
  q = fma2(w, q, bc(1.0f / 8.0f));
  q = fma2(w, q, bc(1.0f / 3.0f));
  q = fma2(w, q, bc(0.5f));
  const float2 num = fma2(w, a, make_float2(-e.x, -e.y));
  const float2 w2 = mul2(w, w);
  return make_float2(fabsf(w.x) < 0.25f ? q.x : num.x * rcp_approx(w2.x),
                     fabsf(w.y) < 0.25f ? q.y : num.y * rcp_approx(w2.y));
}

template <bool ZOH, typename T>
__device__ __forceinline__ void bwd_piece_s4d(const BwdParams& p, float A0, float* wsm, int lane, int64_t row,
                                              int64_t t0, int64_t t1) {
  using namespace pairs;
  float2* hs = reinterpret_cast<float2*>(wsm);             // [kChunk][8][32]
  float2* hst = hs + kChunk * 8 * 32;                       // [8][32]
  float* xs = reinterpret_cast<float*>(hst + 8 * 32);
  float* ds = xs + kChunk * 32;
  float* gs = ds + kChunk * 32;
  float* bs = gs + kChunk * 32;
  float* cs = bs + kChunk * 16;
  float* red = cs + kChunk * 16;                            // [32][32]
  const int64_t L = p.L, D = p.D;
  const int64_t b = row / p.groups;
  const int64_t d = (row % p.groups) * 32 + lane;
  const bool act = d < D;
  const float A2_0 = A0 * kLog2e, invA0 = 1.0f / A0;
  ChunkRegs nx;

  // ---- 1. h(t0 - 1) by the truncated backward walk ---------------------------------------------------
  float2 h[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) h[k] = make_float2(0.0f, 0.0f);
  const float* h0row = p.h0 ? p.h0 + (b * D + d) * 16 : nullptr;
  if (t0 > 0) {
    float W = 0.0f;
    float2 P[8];
    powers<8>(1.0f, P);
    int live = 8;
    int64_t j = t0;
    int64_t s = j > kChunk ? j - kChunk : 0;
    chunk_load<T, true, false, true, false>(p, b, d, act, lane, s, static_cast<int>(j - s), nx);
    while (true) {  // chunk [s, j)
      const int cn = static_cast<int>(j - s);
      chunk_store<true, false, true, false>(p, nx, lane, xs, ds, gs, bs, cs);
      const int64_t s2 = s > kChunk ? s - kChunk : 0;
      if (s > 0) chunk_load<T, true, false, true, false>(p, b, d, act, lane, s2, static_cast<int>(s - s2), nx);
      if (live == 8) s4d_walk_back<8, ZOH>(xs, ds, bs, cn, lane, A2_0, invA0, W, P, h);
      else if (live == 4) s4d_walk_back<4, ZOH>(xs, ds, bs, cn, lane, A2_0, invA0, W, P, h);
      else if (live == 2) s4d_walk_back<2, ZOH>(xs, ds, bs, cn, lane, A2_0, invA0, W, P, h);
      else s4d_walk_back<1, ZOH>(xs, ds, bs, cn, lane, A2_0, invA0, W, P, h);
      j = s;
      s = s2;
      if (j == 0) break;
      const int l2 = live_pairs(warp_max_f(act ? ex2(W) : 0.0f));
      if (l2 == 0) break;
      live = l2 < live ? l2 : live;  // a dropped pair's weights are no longer updated: never revive one
    }
    if (ZOH) {  // the walk summed P e B x / A_0: Bbar_n x = e_n B_n x / ((n + 1) A_0)
#pragma unroll
      for (int k = 0; k < 8; ++k) h[k] = mul2(h[k], kPairInvN1[k]);
    }
    if (j == 0 && h0row && act) {  // the walk reached t = 0: add the initial state, decayed through t0 - 1
      powers<8>(ex2(W), P);
#pragma unroll
      for (int k = 0; k < 8; ++k) h[k] = fma2(P[k], make_float2(h0row[2 * k], h0row[2 * k + 1]), h[k]);
    }
  } else if (h0row && act) {
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = make_float2(h0row[2 * k], h0row[2 * k + 1]);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) hst[k * 32 + lane] = h[k];

  // ---- 2. forward over the piece in aligned chunks, saving the state at each chunk end followed by another
  {
    const int64_t ck0 = t0 / kChunk, ck1 = (t1 - 1) / kChunk;
    auto span = [&](int64_t ck, int64_t& s, int64_t& e) {
      s = ck * kChunk > t0 ? ck * kChunk : t0;
      e = (ck + 1) * kChunk < t1 ? (ck + 1) * kChunk : t1;
    };
    int64_t s, e;
    span(ck0, s, e);
    chunk_load<T, true, false, true, false>(p, b, d, act, lane, s, static_cast<int>(e - s), nx);
    for (int64_t ck = ck0; ck <= ck1; ++ck) {
      span(ck, s, e);
      chunk_store<true, false, true, false>(p, nx, lane, xs, ds, gs, bs, cs);
      if (ck < ck1) {
        int64_t s2, e2;
        span(ck + 1, s2, e2);
        chunk_load<T, true, false, true, false>(p, b, d, act, lane, s2, static_cast<int>(e2 - s2), nx);
      }
      const int cn = static_cast<int>(e - s);
#pragma unroll 1
      for (int i = 0; i < cn; ++i) s4d_fwd_step<ZOH>(xs[i * 32 + lane], ds[i * 32 + lane], bs + i * 16, A2_0, invA0, h);
      if (ck < ck1 && act) {  // chunk ck ends inside the piece
        float* w = p.ws + ((b * p.nck + ck) * 16) * D + d;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          w[static_cast<int64_t>(2 * k) * D] = h[k].x;
          w[static_cast<int64_t>(2 * k + 1) * D] = h[k].y;
        }
      }
    }
  }

  // ---- 3. the adjoint entering from the right of the piece: forward walk from t1 ---------------------------
  float2 mu[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mu[k] = make_float2(0.0f, 0.0f);
  const float* dfrow = p.dfinal ? p.dfinal + (b * D + d) * 16 : nullptr;
  if (t1 == L) {
    if (dfrow && act) {
#pragma unroll
      for (int k = 0; k < 8; ++k) mu[k] = make_float2(dfrow[2 * k], dfrow[2 * k + 1]);
    }
  } else {
    float W = 0.0f;
    float2 P[8];
    powers<8>(1.0f, P);
    int live = 8;
    int64_t j = t1;
    int64_t e = j + kChunk < L ? j + kChunk : L;
    chunk_load<T, false, true, false, true>(p, b, d, act, lane, j, static_cast<int>(e - j), nx);
    while (true) {  // chunk [j, e)
      const int cn = static_cast<int>(e - j);
      chunk_store<false, true, false, true>(p, nx, lane, xs, ds, gs, bs, cs);
      const int64_t e2 = e + kChunk < L ? e + kChunk : L;
      if (e < L) chunk_load<T, false, true, false, true>(p, b, d, act, lane, e, static_cast<int>(e2 - e), nx);
      if (live == 8) s4d_walk_fwd<8>(ds, gs, cs, cn, lane, A2_0, W, P, mu);
      else if (live == 4) s4d_walk_fwd<4>(ds, gs, cs, cn, lane, A2_0, W, P, mu);
      else if (live == 2) s4d_walk_fwd<2>(ds, gs, cs, cn, lane, A2_0, W, P, mu);
      else s4d_walk_fwd<1>(ds, gs, cs, cn, lane, A2_0, W, P, mu);
      j = e;
      e = e2;
      if (j == L) {  // exact: the final-state gradient, decayed through every step after t1 - 1
        if (dfrow && act) {
          powers<8>(ex2(W), P);
#pragma unroll
          for (int k = 0; k < 8; ++k) mu[k] = fma2(P[k], make_float2(dfrow[2 * k], dfrow[2 * k + 1]), mu[k]);
        }
        break;
      }
      const int l2 = live_pairs(warp_max_f(act ? ex2(W) : 0.0f));
      if (l2 == 0) break;
      live = l2 < live ? l2 : live;
    }
  }

  // ---- 4. chunks backwards ----------------------------------------------------------------------------
  // dB, dC and dA_log are zeroed by the launch before this kernel, which may still be running (programmatic
  // dependent launch): wait for it before the first atomic add. A no-op once it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float2 dA[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) dA[k] = make_float2(0.0f, 0.0f);
  const int64_t ck0 = t0 / kChunk, ck1 = (t1 - 1) / kChunk;
  auto span = [&](int64_t ck, int64_t& s, int64_t& e) {
    s = ck * kChunk > t0 ? ck * kChunk : t0;
    e = (ck + 1) * kChunk < t1 ? (ck + 1) * kChunk : t1;
  };
  // the saved state entering chunk ck (> ck0): the end state of chunk ck - 1
  auto ws_load = [&](int64_t ck, float2 (&hn)[8]) {
    const float* w = p.ws + ((b * p.nck + ck - 1) * 16) * D + d;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      hn[k] = act ? make_float2(w[static_cast<int64_t>(2 * k) * D], w[static_cast<int64_t>(2 * k + 1) * D])
                  : make_float2(0.0f, 0.0f);
  };
  float2 hn[8];
  {
    int64_t s, e;
    span(ck1, s, e);
    chunk_load<T, true, true, true, true>(p, b, d, act, lane, s, static_cast<int>(e - s), nx);
    if (ck1 > ck0) ws_load(ck1, hn);
  }
  const int sw = lane & 7;
  for (int64_t ck = ck1; ck >= ck0; --ck) {
    int64_t s, e;
    span(ck, s, e);
    const int cn = static_cast<int>(e - s);
    chunk_store<true, true, true, true>(p, nx, lane, xs, ds, gs, bs, cs);
    if (ck > ck0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) h[k] = hn[k];
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) h[k] = hst[k * 32 + lane];
    }
    if (ck > ck0) {  // the previous chunk's inputs and entering state, in flight during this chunk
      int64_t s2, e2;
      span(ck - 1, s2, e2);
      chunk_load<T, true, true, true, true>(p, b, d, act, lane, s2, static_cast<int>(e2 - s2), nx);
      if (ck - 1 > ck0) ws_load(ck - 1, hn);
    }
    // recompute the chunk's states: hs row i = the state before step i
#pragma unroll 1
    for (int i = 0; i < cn; ++i) {
#pragma unroll
      for (int k = 0; k < 8; ++k) hs[(i * 8 + k) * 32 + lane] = h[k];
      s4d_fwd_step<ZOH>(xs[i * 32 + lane], ds[i * 32 + lane], bs + i * 16, A2_0, invA0, h);
    }
    // h now holds the state after the chunk's last step
#pragma unroll 1
    for (int i = cn - 1; i >= 0; --i) {
      const int64_t t = s + i;
      const float xv = xs[i * 32 + lane], dv = ds[i * 32 + lane], g = gs[i * 32 + lane];
      const float2* brow = reinterpret_cast<const float2*>(bs + i * 16);
      const float2* crow = reinterpret_cast<const float2*>(cs + i * 16);
      float2 e[8];
      step_e16(dv * A2_0, e);
      const float2 gg = bc(g), dd = bc(dv);
      float2 gd = make_float2(0.0f, 0.0f);  // sum_n (n + 1) lambda_n u_n (times A_0 below)
      float2 sg = make_float2(0.0f, 0.0f);  // sum_n lambda_n B_n
      float2 se = make_float2(0.0f, 0.0f);  // ZOH: sum_n lambda_n e_n B_n
      float2 sq = make_float2(0.0f, 0.0f);  // ZOH: sum_n lambda_n e_n B_n / (n + 1)
      float2 v[16];                         // this lane's dB terms (pairs 0..7) and dC terms (pairs 8..15)
      const float2 dxv = bc(dv * xv), xq = bc(xv * invA0);
      const float2 zq = bc(xv * dv * dv);   // ZOH: x delta^2
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 hp = hs[(i * 8 + k) * 32 + lane];  // h_{t-1}
        const float2 lam = fma2(crow[k], gg, mu[k]);
        const float2 lu = mul2(lam, fma2(e[k], hp, hp));  // lambda Abar h_{t-1}
        dA[k] = fma2(lu, dd, dA[k]);
        gd = fma2(lu, kPairN1[k], gd);
        sg = fma2(lam, brow[k], sg);
        v[8 + k] = mul2(gg, h[k]);  // dC: dy h_t
        if (ZOH) {
          const float2 le = mul2(lam, e[k]);
          se = fma2(le, brow[k], se);
          sq = fma2(le, mul2(brow[k], kPairInvN1[k]), sq);
          v[k] = mul2(le, mul2(xq, kPairInvN1[k]));  // dB: lambda x e_n / A_n
          const float2 w = mul2(kPairN1[k], bc(dv * A0));
          dA[k] = fma2(mul2(mul2(lam, brow[k]), zq), zoh_f2(w, add2(e[k], bc(1.0f)), e[k]), dA[k]);
        } else {
          v[k] = mul2(lam, dxv);  // dB: lambda delta x
        }
        mu[k] = fma2(e[k], lam, lam);
        h[k] = hp;
      }
      const float sgs = sg.x + sg.y;
      float gx, gdt;
      if (ZOH) {
        gx = (sq.x + sq.y) * invA0;
        gdt = fmaf(gd.x + gd.y, A0, xv * (sgs + se.x + se.y));
      } else {
        gx = dv * sgs;
        gdt = fmaf(gd.x + gd.y, A0, xv * sgs);
      }
      if (act) {
        const int64_t xi = (b * L + t) * D + d;
        Elem<T>::store(p.dx, xi, gx);
        Elem<T>::store(p.ddelta, xi, gdt);
      }
      // dB, dC: lane l writes its 32 terms as row l of the tile (16-byte pieces XOR-swizzled by l mod 8), then
      // sums column l (term l of every lane)
      float4* rrow = reinterpret_cast<float4*>(red + lane * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) rrow[q ^ sw] = make_float4(v[2 * q].x, v[2 * q].y, v[2 * q + 1].x, v[2 * q + 1].y);
      __syncwarp();
      float2 acc[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) acc[a] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int r = 0; r < 32; r += 2) {
        const int c0 = (((lane >> 2) ^ (r & 7)) << 2) | (lane & 3);
        const int c1 = (((lane >> 2) ^ ((r + 1) & 7)) << 2) | (lane & 3);
        acc[(r >> 1) & 3] = add2(acc[(r >> 1) & 3], make_float2(red[r * 32 + c0], red[(r + 1) * 32 + c1]));
      }
      __syncwarp();
      const float2 a01 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
      atomicAdd((lane < 16 ? p.dB : p.dC) + (b * L + t) * 16 + (lane & 15), a01.x + a01.y);
    }
  }
  if (act) {
    if (t0 == 0 && p.dh0) {
      float* out = p.dh0 + (b * D + d) * 16;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        out[2 * k] = mu[k].x;
        out[2 * k + 1] = mu[k].y;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // dA_log_n = dA_n A_n, A_n = (n + 1) A_0
      const float2 g = mul2(dA[k], mul2(kPairN1[k], bc(A0)));
      atomicAdd(p.dA_log + d * 16 + 2 * k, g.x);
      atomicAdd(p.dA_log + d * 16 + 2 * k + 1, g.y);
    }
  }
}

// floats of shared memory per warp: the generic layout, or the structured one where N = 16 may take it
template <int NP>
constexpr int kBwdSmemFloats = NP == 16 && kS4dWarpFloats > kBwdWarpFloats<NP> ? kS4dWarpFloats : kBwdWarpFloats<NP>;

template <int NP, bool ZOH, typename T>
__global__ void __launch_bounds__(kBwdWarps * 32, 1) scan_bwd_kernel(BwdParams p) {
  extern __shared__ float smem_bwd[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kBwdWarps + wid;
  if (gw >= p.nwarps) return;  // whole warp leaves together
  // this warp's shared memory: rows of states hs[(r * NP + n) * 32 + lane] (r = 0 the chunk's initial state,
  // r = 1 + i after step i of the chunk, r = kChunk + 1 the piece's initial state), then the staged chunk
  float* hs = smem_bwd + static_cast<size_t>(wid) * kBwdSmemFloats<NP>;
  float* xs = hs + (kChunk + 2) * NP * 32;
  float* ds = xs + kChunk * 32;
  float* gs = ds + kChunk * 32;
  float* bs = gs + kChunk * 32;
  float* cs = bs + kChunk * 16;

  int64_t lo = static_cast<int64_t>(static_cast<__int128>(gw) * p.total / p.nwarps);
  const int64_t hi = static_cast<int64_t>(static_cast<__int128>(gw + 1) * p.total / p.nwarps);
  const int N = static_cast<int>(p.N);
  const int64_t L = p.L, D = p.D;
  while (lo < hi) {
    const int64_t row = lo / L;
    const int64_t t0 = lo % L;
    const int64_t t1 = (hi - lo < L - t0) ? t0 + (hi - lo) : L;
    lo += t1 - t0;
    const int64_t d = (row % p.groups) * 32 + lane;
    const bool act = d < D;

    BwdChan<NP, ZOH> c;
    bool s4d = NP == 16 && N == 16;  // A[d, n] = (n + 1) A[d, 0] on every channel of the warp
#pragma unroll
    for (int n = 0; n < NP; ++n) {
      float A = -1.0f;
      if (act && n < N) A = -expf(__ldg(p.A_log + d * N + n));
      c.A2[n] = A * kLog2e;
      c.invA[n] = A == 0.0f ? 0.0f : 1.0f / A;
    }
    if (act) {
      const float A0 = c.A2[0] / kLog2e;
      s4d = s4d && A0 < -1e-30f && A0 > -3.0e38f;
#pragma unroll
      for (int n = 1; n < NP; ++n) {
        const float A = -expf(__ldg(p.A_log + d * N + (n < N ? n : 0)));
        s4d = s4d && fabsf(A - static_cast<float>(n + 1) * A0) <= 4.8e-7f * fabsf(A);
      }
    }
    if constexpr (NP == 16) {
      if (__all_sync(0xffffffffu, s4d)) {
        bwd_piece_s4d<ZOH, T>(p, act ? -expf(__ldg(p.A_log + d * N)) : -1.0f, hs, lane, row, t0, t1);
        continue;
      }
    }
    bwd_piece<NP, ZOH, T>(p, c, hs, xs, ds, gs, bs, cs, lane, row, t0, t1);
  }
}

template <int NP, bool ZOH, typename T>
cudaError_t launch_bwd_np(const BwdParams& bp, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(kBwdWarps) * kBwdSmemFloats<NP> * sizeof(float);
  auto kern = scan_bwd_kernel<NP, ZOH, T>;
  static bool attr_set[64] = {false};  // per device, once per instantiation
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!attr_set[dev & 63]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev & 63] = true;
  }
  const int64_t blocks = (bp.nwarps + kBwdWarps - 1) / kBwdWarps;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kBwdWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, kern, bp)) != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool ZOH, typename T>
cudaError_t launch_bwd_disc(const BwdParams& bp, cudaStream_t s) {
  if (bp.N <= 4) return launch_bwd_np<4, ZOH, T>(bp, s);
  if (bp.N <= 8) return launch_bwd_np<8, ZOH, T>(bp, s);
  return launch_bwd_np<16, ZOH, T>(bp, s);
}

// Zero dA_log, dB and dC (the atomic sums) in one launch; the backward kernel after it may start at once and
// waits for this grid only before its first atomic add.
__global__ void bwd_zero_kernel(float* a, int64_t na, float* b, int64_t nb, float* c, int64_t nc) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < na + nb + nc; i += stride) {
    if (i < na) a[i] = 0.0f;
    else if (i < na + nb) b[i - na] = 0.0f;
    else c[i - na - nb] = 0.0f;
  }
}

// dh0 = dfinal (or 0) when there are no steps.
__global__ void copy_or_zero_kernel(const float* src, float* dst, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = src ? src[i] : 0.0f;
}

}  // namespace

// ---- built-in scratch for ssm_scan_bwd_noalloc ----------------------------------------------------------
// A fixed array in the library's own device memory, for callers that cannot allocate a workspace. Every
// device that loads the library holds it until the process exits; every call of ssm_scan_bwd_noalloc on a
// device uses the same array.
static __device__ __align__(256) unsigned char g_bwd_scratch[kBwdNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {nullptr};
}  // namespace

cudaError_t bwd_noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    // the array's name is only a host-side stand-in: its device address comes from the runtime, once per
    // device, with that device current
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t bwd_workspace_bytes(int64_t batch, int64_t L, int64_t D, int64_t N) {
  const int64_t nck = L > 0 ? (L + kChunk - 1) / kChunk - 1 : 0;
  return static_cast<size_t>(batch) * static_cast<size_t>(nck) * static_cast<size_t>(N) * static_cast<size_t>(D) *
         sizeof(float);
}

cudaError_t launch_bwd(const BwdArgs& a) {
  cudaError_t e = cudaSuccess;
  const int64_t na = a.D * a.N, nbc = a.batch * a.L * a.N;
  if (na + 2 * nbc > 0) {
    const int64_t zb = (na + 2 * nbc + 255) / 256;
    const int64_t zcap = static_cast<int64_t>(sm_count()) * 4;
    bwd_zero_kernel<<<static_cast<unsigned>(zb < zcap ? zb : zcap), 256, 0, a.stream>>>(a.dA_log, na, a.dB, nbc,
                                                                                          a.dC, nbc);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.L == 0) {
    const int64_t n = a.batch * a.D * a.N;
    if (a.dh0 && n > 0) {
      copy_or_zero_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, a.stream>>>(a.dfinal, a.dh0, n);
      return cudaGetLastError();
    }
    return cudaSuccess;
  }
  BwdParams bp;
  bp.x = a.x; bp.delta = a.delta; bp.A_log = a.A_log; bp.B = a.B; bp.C = a.C; bp.h0 = a.h0;
  bp.dy = a.dy; bp.dfinal = a.dfinal;
  bp.dx = a.dx; bp.ddelta = a.ddelta; bp.dA_log = a.dA_log; bp.dB = a.dB; bp.dC = a.dC; bp.dh0 = a.dh0;
  bp.ws = a.workspace;
  bp.batch = a.batch; bp.L = a.L; bp.D = a.D; bp.N = a.N;
  bp.nck = (a.L + kChunk - 1) / kChunk - 1;
  bp.groups = (a.D + 31) / 32;
  const int64_t rows = a.batch * bp.groups;
  bp.total = rows * a.L;
  if (bp.total == 0) return cudaSuccess;  // no channels: the zeroed sums are the whole answer
  int64_t nw = rows * ((a.L + kMinBwdPiece - 1) / kMinBwdPiece);
  const int64_t want = static_cast<int64_t>(sm_count()) * kBwdWarps;
  if (nw > want) nw = want;
  if (nw < 1) nw = 1;
  bp.nwarps = nw;
  auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  bp.vec = a.dtype == 0 && a.N == 16 && a.D % 4 == 0 && a16(a.x) && a16(a.delta) && a16(a.dy) && a16(a.B) && a16(a.C);
  if (a.disc == 1)
    return a.dtype == 1 ? launch_bwd_disc<true, __nv_bfloat16>(bp, a.stream) : launch_bwd_disc<true, float>(bp, a.stream);
  return a.dtype == 1 ? launch_bwd_disc<false, __nv_bfloat16>(bp, a.stream) : launch_bwd_disc<false, float>(bp, a.stream);
}

}  // namespace ssm
