// ssd_fwd.cu -- Mamba-2 SSD layer: the scan with A = a I per head, in its chunked (dual) form.
//
// "State Space Models & Mamba" chapter, the Mamba-2 paragraph, and "Mathematical Prerequisites for Mamba"
// s7 and the paragraph after it: with a scalar decay per head the recurrence is multiplication by a
// 1-semiseparable matrix, so inside a chunk of Q steps the outputs are masked matrix products (tensor-core
// work) and the state is carried between chunks by the recurrence. For one head (state S [N, P]) and one
// chunk with s_i = sum_{k<=i} delta_k A (the log of the decay from the chunk start through step i),
// u_j = coef_j x_j (coef = delta (Euler) or (e^{delta A} - 1) / A (ZOH)):
//     y_i   = sum_{j<=i} e^{s_i - s_j} (C_i . B_j) u_j  +  e^{s_i} C_i S_prev               (intra + inter)
//     S_end = e^{s_last} S_prev + sum_j e^{s_last - s_j} B_j u_j^T
//
// Work layout: one CTA of 4 warps per (batch element, head, block of 16 head channels); the CTA walks its
// sequence chunk by chunk (Q = 64), keeping its [N, 16] slice of the state in registers (fp32) and a bf16
// copy in shared memory as an MMA operand. Per chunk, warp w owns rows 16w .. 16w+15:
//   G  = C B^T (its 16 rows, causal columns only), scaled by e^{s_i - s_j} coef_j and masked to j <= i,
//        kept in registers and reused directly as the A operand of
//   Y1 = G X,   Y2 = C S_prev (the C fragments of G reused),   y = Y1 + e^{s_i} Y2  -> bf16
//   S  = e^{s_last} S + B^T (w X),  w_j = e^{s_last - s_j} coef_j  (warp w: state rows N/4 w ..)
// Products use the warp-level bf16 tensor-core MMA (m16n8k16, fp32 accumulate); operands come from
// shared memory through ldmatrix. The next chunk's x, B, C tiles stream in with cp.async while the
// current one is computed.
//
// Segments (optional caller workspace, used when one CTA per sequence would leave SMs idle): each sequence
// is cut into runs of chunks that separate CTAs scan from a zero state, recording each run's end state and
// total log decay; ssd_fixup_kernel then carries the true state into every run and adds its contribution
// e^{cum_i} C_i . H to the outputs, one CTA per chunk.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int kQ = 64;       // chunk length (steps)
constexpr int kPB = 16;      // head channels per CTA
constexpr int kThreads = 128;

struct SsdParams {
  const __nv_bfloat16* x;  // [batch, L, H, P]
  const float* delta;      // [batch, L, H]
  const float* A_log;      // [H]
  const __nv_bfloat16* B;  // [batch, L, N]
  const __nv_bfloat16* C;
  const float* h0;         // [batch, H, P, N] or null
  __nv_bfloat16* y;        // [batch, L, H, P]
  float* final_state;      // [batch, H, P, N] or null
  int64_t batch, L, H, P;
  int pblocks;             // P / kPB
  // segments: each (batch element, head) sequence is cut into nseg runs of cps chunks, scanned by separate CTAs
  // from a zero state (segment 0 from h0); seg_state / seg_logdec receive each segment's end state and total
  // log decay for the fix-up pass. nseg == 1: one CTA walks the whole sequence and writes final_state itself.
  int nseg;
  int64_t cps;
  float* seg_state;        // [batch, H, nseg, P, N] or null (nseg == 1)
  float* seg_logdec;       // [batch, H, nseg]
};

// ---- PTX wrappers ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  // 16 bytes global -> shared; a row past the end of the sequence is zero-filled (nothing is read)
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// D += A B, m16n8k16, bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
               "{%8, %9}, {%0, %1, %2, %3};\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ---- shared-memory tiles -------------------------------------------------------------------------------
// B and C chunks: [kQ rows][N bf16], rows of N * 2 bytes in 16-byte pieces, piece index XOR (row & 7) so that
// the 8 rows an ldmatrix reads at one column fall in 8 different bank groups.
template <int N>
__device__ __forceinline__ uint32_t bc_off(int row, int piece) {
  return static_cast<uint32_t>(row * (N * 2) + ((piece ^ (row & 7)) << 4));
}
// 16-column tiles (x, scaled x, state copy): rows of 32 bytes (two pieces), piece XOR ((row >> 2) & 1).
__device__ __forceinline__ uint32_t p16_off(int row, int piece) {
  return static_cast<uint32_t>(row * 32 + ((piece ^ ((row >> 2) & 1)) << 4));
}

template <int N>
struct SsdSmem {
  alignas(128) __nv_bfloat16 Bt[2][kQ * N];
  alignas(128) __nv_bfloat16 Ct[2][kQ * N];
  alignas(128) __nv_bfloat16 Xt[2][kQ * kPB];
  alignas(128) __nv_bfloat16 Sb[N * kPB];   // bf16 copy of the state slice [N][16]
  float dt[2][kQ];
  // per warp (each warp forms its own copy, so no barrier separates them from their use):
  float s[kThreads / 32][kQ];               // log decay from the chunk start through step i
  float coef[kThreads / 32][kQ];
  float w[kThreads / 32][kQ];               // e^{s_last - s_j} coef_j
};

template <int N>
__device__ __forceinline__ void load_chunk(const SsdParams& p, SsdSmem<N>& sm, int buf, int64_t b, int64_t h,
                                           int p0, int64_t t0, int tid) {
  constexpr int kPieces = N * 2 / 16;  // 16-byte pieces per B / C row
  const int64_t L = p.L;
#pragma unroll
  for (int k = tid; k < kQ * kPieces; k += kThreads) {
    const int row = k / kPieces, piece = k % kPieces;
    const int64_t t = t0 + row;
    const bool ok = t < L;
    const int64_t src = ok ? (b * L + t) * N + piece * 8 : 0;
    cp_async16(reinterpret_cast<char*>(sm.Bt[buf]) + bc_off<N>(row, piece), p.B + src, ok);
    cp_async16(reinterpret_cast<char*>(sm.Ct[buf]) + bc_off<N>(row, piece), p.C + src, ok);
  }
  {
    const int row = tid >> 1, piece = tid & 1;  // kQ rows x 2 pieces = 128 = kThreads
    const int64_t t = t0 + row;
    const bool ok = t < L;
    const int64_t src = ok ? ((b * L + t) * p.H + h) * p.P + p0 + piece * 8 : 0;
    cp_async16(reinterpret_cast<char*>(sm.Xt[buf]) + p16_off(row, piece), p.x + src, ok);
  }
  cp_async_commit();
}

template <int N, bool ZOH>
__global__ void __launch_bounds__(kThreads) ssd_fwd_kernel(SsdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SsdSmem<N>& sm = *reinterpret_cast<SsdSmem<N>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p0 = (blockIdx.x % p.pblocks) * kPB;
  const int seg = static_cast<int>((blockIdx.x / p.pblocks) % p.nseg);
  const int64_t bh = blockIdx.x / p.pblocks / p.nseg;
  const int64_t b = bh / p.H, h = bh % p.H;
  const int64_t L = p.L;
  const float A = -ex2(__ldg(p.A_log + h) * kLog2e);
  const float A2 = A * kLog2e;
  constexpr int kNW = N / 4;  // state rows per warp in the update
  constexpr int kMT = kNW / 16;

  // state slice in accumulator layout: S[n][p] for n = warp * kNW + mt * 16 + lane / 4 (+ 8), p = nt * 8 +
  // 2 * (lane % 4) (+ 1)
  float st[kMT][2][4];
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int n = warp * kNW + mt * 16 + (lane >> 2) + ((r & 2) ? 8 : 0);
        const int pp = p0 + nt * 8 + 2 * (lane & 3) + (r & 1);
        st[mt][nt][r] = (p.h0 && seg == 0) ? p.h0[((b * p.H + h) * p.P + pp) * N + n] : 0.0f;
      }
  auto write_state_copy = [&]() {
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int n = warp * kNW + mt * 16 + (lane >> 2) + hr * 8;
          const int col = nt * 8 + 2 * (lane & 3);
          *reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(sm.Sb) + p16_off(n, col >> 3) + (col & 7) * 2) =
              pack_bf16(st[mt][nt][2 * hr], st[mt][nt][2 * hr + 1]);
        }
  };
  write_state_copy();

  const int64_t nchunks_all = (L + kQ - 1) / kQ;
  const int64_t cbeg = seg * p.cps;
  const int64_t nchunks = cbeg + p.cps < nchunks_all ? cbeg + p.cps : nchunks_all;  // this segment's end chunk
  if (cbeg < nchunks) load_chunk<N>(p, sm, 0, b, h, p0, cbeg * kQ, tid);
  float dt_next = (tid < kQ && cbeg * kQ + tid < L) ? p.delta[(b * L + cbeg * kQ + tid) * p.H + h] : 0.0f;
  if (tid < kQ) sm.dt[0][tid] = dt_next;
  float logdec = 0.0f;  // the segment's total log decay (sum of delta A)

  for (int64_t c = cbeg; c < nchunks; ++c) {
    const int buf = static_cast<int>((c - cbeg) & 1);
    const int64_t t0 = c * kQ;
    if (c + 1 < nchunks) {  // the other buffer's last readers finished before the previous chunk's barrier
      load_chunk<N>(p, sm, buf ^ 1, b, h, p0, t0 + kQ, tid);
      const int64_t t = t0 + kQ + tid;
      dt_next = (tid < kQ && t < L) ? p.delta[(b * L + t) * p.H + h] : 0.0f;
      cp_async_wait_prev();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();  // chunk c's tiles, dt and the state copy are visible to every warp

    // ---- running log decay, input coefficients and state-update weights (every warp its own copy) -----
    float* const sw = sm.s[warp];
    float* const cw = sm.coef[warp];
    float* const ww = sm.w[warp];
    {
      const float d0 = sm.dt[buf][2 * lane], d1 = sm.dt[buf][2 * lane + 1];
      float v0 = d0 * A, v1 = v0 + d1 * A;  // inclusive sums within the lane's pair
      float inc = v1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      float before = __shfl_up_sync(0xffffffffu, inc, 1);  // sum over earlier lanes' pairs
      if (lane == 0) before = 0.0f;
      const float s0 = before + v0, s1 = before + v1;
      const float last = __shfl_sync(0xffffffffu, inc, 31);
      auto coef_of = [&](float d) {
        if (!ZOH) return d;
        const float w2 = d * A2;
        const float e = exp2m1(w2, ex2(w2));
        return A == 0.0f ? d : e / A;
      };
      const float c0 = coef_of(d0), c1 = coef_of(d1);
      sw[2 * lane] = s0;
      sw[2 * lane + 1] = s1;
      cw[2 * lane] = c0;
      cw[2 * lane + 1] = c1;
      ww[2 * lane] = ex2((last - s0) * kLog2e) * c0;
      ww[2 * lane + 1] = ex2((last - s1) * kLog2e) * c1;
    }
    __syncwarp();
    const float s_last = sw[kQ - 1];
    logdec += s_last;

    const uint32_t Cb = smem_u32(sm.Ct[buf]), Bb = smem_u32(sm.Bt[buf]), Xb = smem_u32(sm.Xt[buf]);
    const uint32_t Sbb = smem_u32(sm.Sb);
    const int mi = lane >> 3, r8 = lane & 7;  // ldmatrix: which 8x8 matrix this lane addresses, and its row

    // ---- G = C B^T for this warp's 16 rows (causal column tiles only) --------------------------------
    uint32_t ca[N / 16][4];  // C fragments (A operand), reused for Y2
#pragma unroll
    for (int kk = 0; kk < N / 16; ++kk) {
      const int row = warp * 16 + (mi & 1) * 8 + r8;
      ldsm_x4(Cb + bc_off<N>(row, kk * 2 + (mi >> 1)), ca[kk][0], ca[kk][1], ca[kk][2], ca[kk][3]);
    }
    float g[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) g[nt][r] = 0.0f;
#pragma unroll
    for (int np = 0; np < 4; ++np) {  // pairs of column tiles (16 columns j)
      if (np > warp) break;           // columns beyond this warp's rows are masked out anyway
#pragma unroll
      for (int kk = 0; kk < N / 16; ++kk) {
        uint32_t b0, b1, b2, b3;
        const int row = np * 16 + (mi >> 1) * 8 + r8;
        ldsm_x4(Bb + bc_off<N>(row, kk * 2 + (mi & 1)), b0, b1, b2, b3);
        mma_bf16(g[2 * np], ca[kk], b0, b1);
        mma_bf16(g[2 * np + 1], ca[kk], b2, b3);
      }
    }
    // mask and scale: G'[i][j] = G[i][j] e^{s_i - s_j} coef_j for j <= i, else 0
    const int i_lo = warp * 16 + (lane >> 2), i_hi = i_lo + 8;
    const float si_lo = sw[i_lo], si_hi = sw[i_hi];
    uint32_t ga[4][4];  // G' as the A operand of Y1 (k = j)
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      float v[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int j = (2 * np + q) * 8 + 2 * (lane & 3) + (r & 1);
          const int i = (r & 2) ? i_hi : i_lo;
          const float si = (r & 2) ? si_hi : si_lo;
          v[q][r] = (np <= warp && j <= i) ? g[2 * np + q][r] * ex2((si - sw[j]) * kLog2e) * cw[j] : 0.0f;
        }
      ga[np][0] = pack_bf16(v[0][0], v[0][1]);
      ga[np][1] = pack_bf16(v[0][2], v[0][3]);
      ga[np][2] = pack_bf16(v[1][0], v[1][1]);
      ga[np][3] = pack_bf16(v[1][2], v[1][3]);
    }
    // ---- Y1 = G' X, Y2 = C S_prev ----------------------------------------------------------------------
    float y1[2][4], y2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) y1[nt][r] = y2[nt][r] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (kk > warp) break;
      uint32_t b0, b1, b2, b3;
      const int row = kk * 16 + (mi & 1) * 8 + r8;
      ldsm_x4_t(Xb + p16_off(row, mi >> 1), b0, b1, b2, b3);
      mma_bf16(y1[0], ga[kk], b0, b1);
      mma_bf16(y1[1], ga[kk], b2, b3);
    }
#pragma unroll
    for (int kk = 0; kk < N / 16; ++kk) {
      uint32_t b0, b1, b2, b3;
      const int row = kk * 16 + (mi & 1) * 8 + r8;
      ldsm_x4_t(Sbb + p16_off(row, mi >> 1), b0, b1, b2, b3);
      mma_bf16(y2[0], ca[kk], b0, b1);
      mma_bf16(y2[1], ca[kk], b2, b3);
    }
    {
      const float e_lo = ex2(si_lo * kLog2e), e_hi = ex2(si_hi * kLog2e);
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = hr ? i_hi : i_lo;
        const int64_t t = t0 + i;
        if (t < L) {
          const float e = hr ? e_hi : e_lo;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int col = p0 + nt * 8 + 2 * (lane & 3);
            const float a0 = fmaf(e, y2[nt][2 * hr], y1[nt][2 * hr]);
            const float a1 = fmaf(e, y2[nt][2 * hr + 1], y1[nt][2 * hr + 1]);
            *reinterpret_cast<uint32_t*>(p.y + ((b * L + t) * p.H + h) * p.P + col) = pack_bf16(a0, a1);
          }
        }
      }
    }
    // ---- state update: S = e^{s_last} S + B^T (w x) ------------------------------------------------------
    {
      const float dec = ex2(s_last * kLog2e);
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) st[mt][nt][r] *= dec;
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk) {
        uint32_t b0, b1, b2, b3;
        const int xrow = kk * 16 + (mi & 1) * 8 + r8;
        ldsm_x4_t(Xb + p16_off(xrow, mi >> 1), b0, b1, b2, b3);
        {  // scale row k of x by w_k in registers: b0, b2 hold rows k0, k0 + 1; b1, b3 rows k0 + 8, k0 + 9
          const int k0 = kk * 16 + 2 * (lane & 3);
          const float2 wa = *reinterpret_cast<const float2*>(ww + k0);
          const float2 wb = *reinterpret_cast<const float2*>(ww + k0 + 8);
          auto scale = [](uint32_t v, float2 f) {
            const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&v);
            return pack_bf16(__low2float(x) * f.x, __high2float(x) * f.y);
          };
          b0 = scale(b0, wa);
          b2 = scale(b2, wa);
          b1 = scale(b1, wb);
          b3 = scale(b3, wb);
        }
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          // A = B^T: rows n (this warp's), k = j; the transposed load of B rows j gives it
          uint32_t a[4];
          const int brow = kk * 16 + (mi >> 1) * 8 + r8;
          const int npiece = (warp * kNW + mt * 16) / 8 + (mi & 1);
          ldsm_x4_t(Bb + bc_off<N>(brow, npiece), a[0], a[1], a[2], a[3]);
          mma_bf16(st[mt][0], a, b0, b1);
          mma_bf16(st[mt][1], a, b2, b3);
        }
      }
    }
    __syncthreads();  // every warp is done with this chunk's tiles and the old state copy
    write_state_copy();
    if (tid < kQ) sm.dt[buf ^ 1][tid] = dt_next;
  }
  float* const out = p.nseg > 1 ? p.seg_state + (bh * p.nseg + seg) * p.P * N
                                 : (p.final_state ? p.final_state + bh * p.P * N : nullptr);
  if (out) {
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int n = warp * kNW + mt * 16 + (lane >> 2) + ((r & 2) ? 8 : 0);
          const int pp = p0 + nt * 8 + 2 * (lane & 3) + (r & 1);
          out[static_cast<int64_t>(pp) * N + n] = st[mt][nt][r];
        }
  }
  if (p.nseg > 1 && p0 == 0 && tid == 0) p.seg_logdec[bh * p.nseg + seg] = logdec;
}

// Fix-up of segments 1 .. nseg-1 (one CTA per batch element, head, segment, chunk of the segment and 16-channel
// block, so every chunk is corrected in parallel). The state
// entering segment s is H_s = E_{s-1} + e^{D_{s-1}} H_{s-1}, H_1 = E_0 (E_u, D_u: segment u's end state from a
// zero start and its total log decay; segment 0 started from h0). Its contribution to every output of the
// segment is e^{cum_i} C_i . H_s, cum_i the log decay from the segment start through step i: a product with the
// C rows, added to the y the first pass wrote. The last segment's first-chunk CTA also writes the final state
// E_last + e^{D_last} H_last.
template <int N>
struct FixSmem {
  alignas(128) __nv_bfloat16 Ct[kQ * N];
  alignas(128) __nv_bfloat16 Sb[N * kPB];
  float dt[kQ];
  float cum[kQ];
  float part[kThreads / 32];
};

template <int N>
__global__ void __launch_bounds__(kThreads) ssd_fixup_kernel(SsdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  FixSmem<N>& sm = *reinterpret_cast<FixSmem<N>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p0 = (blockIdx.x % p.pblocks) * kPB;
  const int64_t ci = (blockIdx.x / p.pblocks) % p.cps;  // chunk within the segment
  const int seg = 1 + static_cast<int>((blockIdx.x / p.pblocks / p.cps) % (p.nseg - 1));
  const int64_t bh = blockIdx.x / p.pblocks / p.cps / (p.nseg - 1);
  const int64_t b = bh / p.H, h = bh % p.H;
  const int64_t L = p.L;
  const int64_t c = seg * p.cps + ci;
  if (c * kQ >= L) return;  // the last segment can be shorter (whole CTA leaves together)
  const float A = -ex2(__ldg(p.A_log + h) * kLog2e);
  constexpr int kPieces = N * 2 / 16;
  constexpr int kNW = N / 4;
  constexpr int kMT = kNW / 16;

  // H_seg for this CTA's [N, 16] slice, element (n, pp) in the accumulator layout of the first pass
  float hs[kMT][2][4];
  const float* E = p.seg_state + bh * p.nseg * p.P * N;
  const float* Dl = p.seg_logdec + bh * p.nseg;
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int n = warp * kNW + mt * 16 + (lane >> 2) + ((r & 2) ? 8 : 0);
        const int64_t pn = static_cast<int64_t>(p0 + nt * 8 + 2 * (lane & 3) + (r & 1)) * N + n;
        float v = E[pn];  // H_1 = E_0
        for (int u = 1; u < seg; ++u) v = fmaf(ex2(Dl[u] * kLog2e), v, E[u * p.P * N + pn]);
        hs[mt][nt][r] = v;
        if (seg == p.nseg - 1 && ci == 0 && p.final_state)
          p.final_state[bh * p.P * N + pn] = fmaf(ex2(Dl[seg] * kLog2e), v, E[seg * p.P * N + pn]);
        // bf16 copy as the MMA operand: written below
      }
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int n = warp * kNW + mt * 16 + (lane >> 2) + hr * 8;
        const int col = nt * 8 + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(sm.Sb) + p16_off(n, col >> 3) + (col & 7) * 2) =
            pack_bf16(hs[mt][nt][2 * hr], hs[mt][nt][2 * hr + 1]);
      }

  const int mi = lane >> 3, r8 = lane & 7;
  const int64_t t0 = c * kQ;
#pragma unroll
  for (int k = tid; k < kQ * kPieces; k += kThreads) {
    const int row = k / kPieces, piece = k % kPieces;
    const bool ok = t0 + row < L;
    cp_async16(reinterpret_cast<char*>(sm.Ct) + bc_off<N>(row, piece), p.C + (ok ? (b * L + t0 + row) * N + piece * 8 : 0),
               ok);
  }
  cp_async_commit();
  if (tid < kQ) sm.dt[tid] = (t0 + tid < L) ? p.delta[(b * L + t0 + tid) * p.H + h] : 0.0f;
  // log decay from the segment start to this chunk's start: A times the sum of delta over those steps
  float acc = 0.0f;
  for (int64_t t = seg * p.cps * kQ + tid; t < t0; t += kThreads) acc += p.delta[(b * L + t) * p.H + h];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) sm.part[warp] = acc;
  cp_async_wait_all();
  __syncthreads();  // C tile, dt, partial sums and the state copy are visible
  {
    if (warp == 0) {  // cum_i = off + running sum of delta A through step i
      float off = 0.0f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) off += sm.part[w];
      off *= A;
      const float v0 = sm.dt[2 * lane] * A, v1 = v0 + sm.dt[2 * lane + 1] * A;
      float inc = v1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      float before = __shfl_up_sync(0xffffffffu, inc, 1);
      if (lane == 0) before = 0.0f;
      sm.cum[2 * lane] = off + before + v0;
      sm.cum[2 * lane + 1] = off + before + v1;
    }
    __syncthreads();
    const uint32_t Cb = smem_u32(sm.Ct), Sbb = smem_u32(sm.Sb);
    float y2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) y2[nt][r] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < N / 16; ++kk) {
      uint32_t a[4], b0, b1, b2, b3;
      ldsm_x4(Cb + bc_off<N>(warp * 16 + (mi & 1) * 8 + r8, kk * 2 + (mi >> 1)), a[0], a[1], a[2], a[3]);
      ldsm_x4_t(Sbb + p16_off(kk * 16 + (mi & 1) * 8 + r8, mi >> 1), b0, b1, b2, b3);
      mma_bf16(y2[0], a, b0, b1);
      mma_bf16(y2[1], a, b2, b3);
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = warp * 16 + (lane >> 2) + hr * 8;
      const int64_t t = t0 + i;
      if (t < L) {
        const float e = ex2(sm.cum[i] * kLog2e);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t* yp = reinterpret_cast<uint32_t*>(p.y + ((b * L + t) * p.H + h) * p.P + p0 + nt * 8 + 2 * (lane & 3));
          const uint32_t old = *yp;
          const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&old);
          *yp = pack_bf16(fmaf(e, y2[nt][2 * hr], __low2float(v)), fmaf(e, y2[nt][2 * hr + 1], __high2float(v)));
        }
      }
    }
  }
}

// Opt a kernel in to its dynamic shared memory once per device. Keyed by the kernel itself (every kernel
// here has the same type, so a type parameter would share one flag between them).
template <auto Kern>
cudaError_t smem_attr_once(size_t smem) {
  static bool attr_set[64] = {false};
  auto kern = Kern;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!attr_set[dev & 63]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev & 63] = true;
  }
  return cudaSuccess;
}

template <int N, bool ZOH>
cudaError_t launch_ssd_n(const SsdParams& sp, cudaStream_t s) {
  auto kern = ssd_fwd_kernel<N, ZOH>;
  cudaError_t e = smem_attr_once<ssd_fwd_kernel<N, ZOH>>(sizeof(SsdSmem<N>));
  if (e != cudaSuccess) return e;
  const int64_t blocks = sp.batch * sp.H * sp.pblocks * sp.nseg;
  kern<<<static_cast<unsigned>(blocks), kThreads, sizeof(SsdSmem<N>), s>>>(sp);
  if ((e = cudaGetLastError()) != cudaSuccess || sp.nseg == 1) return e;
  auto fix = ssd_fixup_kernel<N>;
  if ((e = smem_attr_once<ssd_fixup_kernel<N>>(sizeof(FixSmem<N>))) != cudaSuccess) return e;
  const int64_t fblocks = sp.batch * sp.H * sp.pblocks * (sp.nseg - 1) * sp.cps;
  fix<<<static_cast<unsigned>(fblocks), kThreads, sizeof(FixSmem<N>), s>>>(sp);
  return cudaGetLastError();
}

// Segments per sequence: only when one CTA per sequence would leave SMs idle (fewer CTAs than SMs), then
// enough for one CTA per SM, segments of at least 4 chunks, at most 16. With 192 CTAs on 148 SMs, two
// segments per sequence measured slower (111 us against 84 us): the per-chunk work of the resident CTAs
// already shares each SM, so splitting only pays where SMs would otherwise sit idle.
void ssd_segments(int64_t batch, int64_t L, int64_t H, int64_t P, int* nseg, int64_t* cps) {
  const int64_t nchunks = (L + kQ - 1) / kQ;
  const int64_t ctas = batch * H * (P / kPB);
  const int64_t sms = sm_count();
  int64_t s = (ctas > 0 && ctas < sms) ? (sms + ctas - 1) / ctas : 1;
  const int64_t by_len = nchunks / 4;
  if (s > by_len) s = by_len;
  if (s > 16) s = 16;
  if (s < 1) s = 1;
  const int64_t c = (nchunks + s - 1) / s;  // chunks per segment; no segment is left empty
  *cps = c > 0 ? c : 1;
  *nseg = static_cast<int>(c > 0 ? (nchunks + c - 1) / c : 1);
}

}  // namespace

bool ssd_shape_ok(int64_t P, int64_t N) { return (N == 64 || N == 128) && P > 0 && P % kPB == 0; }

size_t ssd_segment_bytes(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N) {
  int nseg = 1;
  int64_t cps = 1;
  ssd_segments(batch, L, H, P, &nseg, &cps);
  if (nseg <= 1) return 0;
  return static_cast<size_t>(batch * H * nseg) * static_cast<size_t>(P * N + 1) * sizeof(float);
}

size_t ssd_workspace_bytes(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N) {
  const size_t tc = ssd_tc_workspace_bytes(batch, L, H, P, N);
  if (tc > 0) return tc;  // the tensor-core path takes this shape
  return ssd_segment_bytes(batch, L, H, P, N);
}

cudaError_t launch_ssd(const SsdArgs& a) {
  if (ssd_tc_ok(a)) return launch_ssd_tc(a);
  SsdParams sp;
  sp.x = static_cast<const __nv_bfloat16*>(a.x);
  sp.delta = a.delta;
  sp.A_log = a.A_log;
  sp.B = static_cast<const __nv_bfloat16*>(a.B);
  sp.C = static_cast<const __nv_bfloat16*>(a.C);
  sp.h0 = a.h0;
  sp.y = static_cast<__nv_bfloat16*>(a.y);
  sp.final_state = a.final_state;
  sp.batch = a.batch; sp.L = a.L; sp.H = a.H; sp.P = a.P;
  sp.pblocks = static_cast<int>(a.P / kPB);
  sp.nseg = 1;
  sp.cps = (a.L + kQ - 1) / kQ;
  sp.seg_state = nullptr;
  sp.seg_logdec = nullptr;
  const size_t need = ssd_segment_bytes(a.batch, a.L, a.H, a.P, a.N);
  if (need > 0 && a.workspace && a.workspace_bytes >= need) {  // without it, one CTA walks each sequence
    ssd_segments(a.batch, a.L, a.H, a.P, &sp.nseg, &sp.cps);
    if (a.batch * a.H * sp.pblocks * sp.nseg * sp.cps > INT32_MAX) {  // grid too large: one CTA per sequence
      sp.nseg = 1;
      sp.cps = (a.L + kQ - 1) / kQ;
    }
    if (sp.nseg > 1) {
      sp.seg_state = static_cast<float*>(a.workspace);
      sp.seg_logdec = sp.seg_state + a.batch * a.H * sp.nseg * a.P * a.N;
    }
  }
  if (a.N == 64) return a.disc == 1 ? launch_ssd_n<64, true>(sp, a.stream) : launch_ssd_n<64, false>(sp, a.stream);
  return a.disc == 1 ? launch_ssd_n<128, true>(sp, a.stream) : launch_ssd_n<128, false>(sp, a.stream);
}

}  // namespace ssm
