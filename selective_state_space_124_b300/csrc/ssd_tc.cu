// ssd_tc.cu -- Mamba-2 SSD layer on the fifth-generation tensor cores: tcgen05 MMAs with TMEM accumulators,
// operands staged by TMA, chunks processed in parallel.
//
// "State Space Models & Mamba" chapter, the Mamba-2 paragraph, and "Mathematical Prerequisites for Mamba" s7:
// with one scalar decay per head the recurrence is multiplication by a 1-semiseparable matrix, so inside a
// chunk the work is masked matrix products and the recurrence only carries a state from chunk to chunk. For
// one head (state S [P, N]) and chunk c of Q = 128 steps, with s_i = sum_{k<=i} delta_k A (the log decay from
// the chunk start through step i) and coef_j = delta_j (Euler) or (e^{delta_j A} - 1) / A (ZOH):
//     E_c[p][n]  = sum_j e^{s_last - s_j} coef_j x_j[p] B_j[n]           (the chunk's state, from a zero start)
//     S_{c+1}    = e^{s_last} S_c + E_c,  S_0 = h0                        (the state entering each chunk)
//     y_i[p]     = sum_{j<=i} (C_i . B_j) e^{s_i - s_j} coef_j x_j[p]  +  e^{s_i} sum_n C_i[n] S_c[p][n]
// Three launches:
//   1. ssd_chunk_state_kernel: one CTA per (batch element, chunk, group of head pairs). Per head pair, E for
//      both heads is one MMA chain: M = 128 rows (head, p), N = state size, K = the chunk's 128 steps, A = the
//      x tile scaled by e^{s_last - s_j} coef_j (read in its natural layout, MN-major), B = the chunk's B tile
//      (natural layout, MN-major). E goes to the workspace in bf16 (the precision of the operands it is formed
//      from; it is the largest intermediate, and half the bytes cut the traffic of launches 1 and 2).
//   2. ssd_state_pass_kernel: the recurrence between chunks in fp32, elementwise over (b, h, p, n); writes every
//      S_c in bf16 (the operand of launch 3) and the final state in fp32.
//   3. ssd_output_kernel: one CTA per (batch element, chunk, group of heads). G = C B^T (M = N = 128, K = state
//      size) is formed once and shared by the group's heads; per head the mask-and-decay of G is written to
//      shared memory in bf16 (A operand), and two MMA chains give D1 = (G o L) X (B = the x tile, MN-major) and
//      D2 = C S_c (B = S_c, K-major); the epilogue writes y = D1 + e^{s_i} D2 in bf16.
// Tiles use the 128-byte swizzle throughout (TMA writes them that way; the MMA descriptors read them that way).
// Steps past the sequence end read zeros (3-D tensor maps per batch element) and take delta = 0, so a last
// partial chunk needs no special case. Every mbarrier wait is bounded (2 s); a wait that runs out sets this
// file's status word, reported by ssm_check_device() as SSM_ERR_TIMEOUT.
#include <cstddef>

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

__device__ int g_ssd_status = 0;  // nonzero: a bounded wait of these kernels ran out

namespace {

constexpr int kTQ = 128;  // chunk length (steps): the M of every product
constexpr int kTP = 64;   // head dimension of this path
constexpr int kTT = 256;  // threads per CTA: warp w reads TMEM lanes (tile rows) 32 (w % 4) .. +31 and takes
                          // column half w / 4 of them
constexpr int kPairsPerCta = 1;  // launch 1: head pairs per CTA
// launch 3: heads per CTA. 3 where the grid fits the resident CTAs about once (Mamba-2-130M: 2, 4, 6 and 8
// measured slower); 6 where it would take several waves (Mamba-2-2.7B: 4% faster than 3), so that the per-CTA
// setup (TMEM allocation, C and B tiles, G) is shared by more heads.
constexpr int kHeadsFew = 3, kHeadsMany = 6;
constexpr unsigned long long kTcWaitNs = 2000000000ull;

// ---- PTX wrappers ----------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t s32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mb_init(unsigned long long* b) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s32(b)) : "memory");
}
__device__ __forceinline__ void mb_expect(unsigned long long* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s32(b)), "r"(bytes) : "memory");
}
// Programmatic dependent launch: the next kernel of the layer may be scheduled from here on (its CTAs wait in
// pdl_wait() until this grid has completed and its writes are visible); and the wait itself. Both are no-ops
// for a kernel launched without the programmatic-serialisation attribute.
__device__ __forceinline__ void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Bounded wait for phase `parity` of an mbarrier (every calling thread waits; no warp-wide agreement needed).
__device__ __forceinline__ bool mb_wait(unsigned long long* b, uint32_t parity) {
  uint32_t ok = 0;
  const unsigned long long t0 = gtime();
  while (true) {
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(s32(b)), "r"(parity)
                 : "memory");
    if (ok) return true;
    if (gtime() - t0 > kTcWaitNs) {
      atomicExch(&g_ssd_status, 4);
      return false;
    }
  }
}
__device__ __forceinline__ void tma3(void* dst, const CUtensorMap* m, int c0, int c1, int c2, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(s32(dst)), "l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(s32(bar))
      : "memory");
}
__device__ __forceinline__ void tma2(void* dst, const CUtensorMap* m, int c0, int c1, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(s32(dst)), "l"(m), "r"(c0), "r"(c1), "r"(s32(bar))
      : "memory");
}
// Bulk tensor store of a shared-memory box to global memory, tracked by the issuing thread's bulk group.
__device__ __forceinline__ void tma_store2(const CUtensorMap* m, int c0, int c1, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(m), "r"(c0), "r"(c1), "r"(s32(src))
               : "memory");
}
__device__ __forceinline__ void tma_store3(const CUtensorMap* m, int c0, int c1, int c2, const void* src) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
               ::"l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(s32(src))
               : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's committed bulk stores have read their shared-memory sources.
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void tma_store_drain() {
  tma_store_commit();
  tma_store_wait_read();
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// TMEM allocation by one whole warp; the base address is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s32(dst)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Shared-memory matrix descriptor for a 128-byte-swizzled tile. K-major tiles: rows of 128 bytes (64 bf16 along
// K), 8-row groups 1024 bytes apart (sbo); MN-major tiles: rows along K, 64-element MN column blocks lbo bytes
// apart, 8-row K groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version of this architecture
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}
// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator, M x N, A / B MN-major flags.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// D (TMEM) = A B (+ D if accumulate), issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(static_cast<uint32_t>(acc))
      : "memory");
}
__device__ __forceinline__ void mma_commit(unsigned long long* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s32(bar)) : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32 (w % 4) .. + 31), without
// waiting: the registers are valid after tmem_wait().
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

struct TcParams {
  const float* delta;   // [batch, L, H]
  const float* A_log;   // [H]
  const float* h0;      // [batch, H, 64, N] or null
  __nv_bfloat16* y;     // [batch, L, H, 64]
  float* final_state;   // [batch, H, 64, N] or null
  __nv_bfloat16* E;     // workspace: [batch, nc, H, 64, N] bf16 chunk states
  __nv_bfloat16* S;     // workspace: [batch, nc, H, 64, N] bf16 states entering each chunk
  float* slast;         // workspace: [batch, nc, H] total log decay of each chunk
  int64_t batch, L, H, nc;
};

// Per-step log decay s (inclusive running sum of delta A over the chunk) and input coefficient, one warp for one
// head: lane l takes steps 4 l .. 4 l + 3. Steps past L take delta = 0.
// The deltas of steps 4 lane .. 4 lane + 3 of chunk c for head h (0 past L). Loaded before a CTA issues its bulk
// copies, so that these small loads do not queue behind them.
__device__ __forceinline__ void load_deltas(const TcParams& p, int64_t b, int64_t c, int64_t h, int lane, float (&d)[4],
                                            float& alog) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t t = c * kTQ + 4 * lane + k;
    d[k] = t < p.L ? __ldg(p.delta + (b * p.L + t) * p.H + h) : 0.0f;
  }
  alog = __ldg(p.A_log + h);
}

template <bool ZOH>
__device__ __forceinline__ void chunk_decays(const float (&dv)[4], float alog, int lane, float (&s)[4], float (&cf)[4],
                                             float& s_last) {
  const float A = -ex2(alog * kLog2e);
  const float A2 = A * kLog2e;
  float a[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float d = dv[k];
    a[k] = d * A;
    if (ZOH) {
      const float w = d * A2;
      cf[k] = A == 0.0f ? d : exp2m1(w, ex2(w)) / A;
    } else {
      cf[k] = d;
    }
  }
  const float l0 = a[0], l1 = l0 + a[1], l2 = l1 + a[2], l3 = l2 + a[3];
  float inc = l3;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  const float before = inc - l3;
  s[0] = before + l0;
  s[1] = before + l1;
  s[2] = before + l2;
  s[3] = before + l3;
  s_last = __shfl_sync(0xffffffffu, inc, 31);
}

// ---- launch 1: chunk states ------------------------------------------------------------------------------
template <int N>
struct ChunkSmem {
  alignas(1024) unsigned char Bt[N * 256];          // B tile [128 steps][N]: N / 64 blocks of [128][128 B]
  alignas(1024) unsigned char Xt[2 * kTQ * 128];    // x tile of a head pair [128 steps][2 x 64]: 2 blocks
  float w[2][kTQ];                                  // e^{s_last - s_j} coef_j of the pair's heads
  unsigned long long barB, barX, barM;
  uint32_t tmem;
};

template <int N, bool ZOH>
__global__ void __launch_bounds__(kTT) ssd_chunk_state_kernel(const __grid_constant__ CUtensorMap mX,
                                                              const __grid_constant__ CUtensorMap mB,
                                                              const __grid_constant__ CUtensorMap mE, TcParams p) {
  // E leaves through shared memory: the B tile (free once the MMA is done) holds the pair's [2 heads][N / 64
  // column blocks][64 rows][64 bf16] boxes, which bulk tensor stores write to the workspace. E is rounded to
  // bf16 there, like the tensor-core operands it is formed from (the x tile scaled by its decay weights). The
  // B tile is loaded once per CTA, so this needs one head pair per CTA.
  static_assert(kPairsPerCta == 1, "the E staging reuses the B tile");
  static_assert(N * 256 >= 2 * kTP * N * 2, "the B tile must hold the pair's E in bf16");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  ChunkSmem<N>& sm = *reinterpret_cast<ChunkSmem<N>*>(smem_raw + ((1024u - (s32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t npairs = (p.H + 1) / 2;
  const int64_t groups = (npairs + kPairsPerCta - 1) / kPairsPerCta;
  const int64_t g = blockIdx.x % groups, c = (blockIdx.x / groups) % p.nc, b = blockIdx.x / groups / p.nc;
  pdl_allow_next();  // the state pass reads E and slast only after this grid completes (pdl_wait)

  if (tid == 0) {
    mb_init(&sm.barB);
    mb_init(&sm.barX);
    mb_init(&sm.barM);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(&sm.tmem, 128);
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  const uint32_t tmem = sm.tmem;
  // Outstanding asynchronous work (thread 0's view): the phase each barrier still owes, or -1.
  int pendB = -1, pendX = -1, pendM = -1;
  float dv[4] = {0.0f, 0.0f, 0.0f, 0.0f}, alog = 0.0f;  // warps 0, 1: the first pair's deltas (loaded first)
  if (warp < 2 && 2 * g * kPairsPerCta + warp < p.H) load_deltas(p, b, c, 2 * g * kPairsPerCta + warp, lane, dv, alog);
  if (tid == 0) {
    mb_expect(&sm.barB, N * 256);
#pragma unroll
    for (int kb = 0; kb < N / 64; ++kb)
      tma3(sm.Bt + kb * kTQ * 128, &mB, kb * 64, static_cast<int>(c * kTQ), static_cast<int>(b), &sm.barB);
    pendB = 0;
  }
  bool ok = true;
  uint32_t phase = 0;
  for (int q = 0; q < kPairsPerCta; ++q) {
    const int64_t h0 = 2 * (g * kPairsPerCta + q);
    if (h0 >= p.H) break;  // uniform over the CTA
    if (tid == 0) {        // the pair's x tile: heads h0, h0 + 1 (a missing second head reads zeros)
      mb_expect(&sm.barX, 2 * kTQ * 128);
      tma3(sm.Xt, &mX, static_cast<int>(h0 * kTP), static_cast<int>(c * kTQ), static_cast<int>(b), &sm.barX);
      tma3(sm.Xt + kTQ * 128, &mX, static_cast<int>((h0 + 1) * kTP), static_cast<int>(c * kTQ), static_cast<int>(b),
           &sm.barX);
      pendX = static_cast<int>(phase);
    }
    if (warp < 2) {  // warp 0: head h0, warp 1: head h0 + 1
      const int64_t h = h0 + warp;
      if (h < p.H) {
        if (q > 0) load_deltas(p, b, c, h, lane, dv, alog);
        float s[4], cf[4], s_last;
        chunk_decays<ZOH>(dv, alog, lane, s, cf, s_last);
#pragma unroll
        for (int k = 0; k < 4; ++k) sm.w[warp][4 * lane + k] = ex2((s_last - s[k]) * kLog2e) * cf[k];
        if (lane == 0) p.slast[(b * p.nc + c) * p.H + h] = s_last;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) sm.w[warp][4 * lane + k] = 0.0f;
      }
    }
    __syncthreads();
    bool okx = mb_wait(&sm.barX, phase);
    if (okx) {
      if (tid == 0) pendX = -1;
      // scale row j of each head's block by that head's w_j (a row of a block is one step: the swizzle only
      // permutes its 16-byte pieces)
      for (int idx = tid; idx < 2 * kTQ * 8; idx += kTT) {
        const int blk = idx / (kTQ * 8), row = (idx / 8) % kTQ, piece = idx % 8;
        uint4* ptr = reinterpret_cast<uint4*>(sm.Xt + blk * kTQ * 128 + row * 128 + piece * 16);
        const uint4 v = *ptr;
        const float f = sm.w[blk][row];
        auto scale2 = [f](uint32_t u) {
          const __nv_bfloat162 x2 = *reinterpret_cast<const __nv_bfloat162*>(&u);
          return bf2(__low2float(x2) * f, __high2float(x2) * f);
        };
        *ptr = make_uint4(scale2(v.x), scale2(v.y), scale2(v.z), scale2(v.w));
      }
    }
    if (q == 0 && okx) {
      okx = mb_wait(&sm.barB, 0);
      if (okx && tid == 0) pendB = -1;
    }
    fence_async_smem();
    tc_before_sync();
    ok = __syncthreads_and(okx) != 0;
    tc_after_sync();
    if (!ok) break;
    if (tid == 0) {
      constexpr uint32_t idesc = mma_idesc(128, N, 1, 1);
#pragma unroll
      for (int ks = 0; ks < kTQ / 16; ++ks) {
        const uint64_t ad = sw128_desc(s32(sm.Xt) + ks * 2048, kTQ * 128, 1024);
        const uint64_t bd = sw128_desc(s32(sm.Bt) + ks * 2048, kTQ * 128, 1024);
        mma_bf16(tmem, ad, bd, idesc, ks > 0);
      }
      mma_commit(&sm.barM);
      pendM = static_cast<int>(phase);
    }
    bool okm = mb_wait(&sm.barM, phase);
    tc_after_sync();
    ok = __syncthreads_and(okm) != 0;
    if (!ok) break;
    if (tid == 0) pendM = -1;
    {
      // row m of D is head h0 + m / 64, channel p = m % 64: its N entries of E go to the staging boxes as bf16,
      // rows of 128 bytes whose 16-byte pieces are XOR-swizzled by the row (the tensor map's 128-byte swizzle;
      // the 32 lanes' rows then fill all banks)
      const int m = (warp & 3) * 32 + lane;
      const int hh = m >> 6, r = m & 63;
      uint32_t v[N / 32][16];  // this thread's N / 2 columns: all loads, then one wait
#pragma unroll
      for (int k = 0; k < N / 32; ++k)
        tmem_ld16_async(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + (warp >> 2) * (N / 2) + 16 * k, v[k]);
      tmem_wait();
      unsigned char* stage = sm.Bt;
#pragma unroll
      for (int k = 0; k < N / 32; ++k) {
        const int col = (warp >> 2) * (N / 2) + 16 * k;  // 16 columns: a quarter of column block col / 64
        unsigned char* row = stage + ((hh * (N / 64) + col / 64) * 64 + r) * 128;
        const int piece = (col & 63) >> 3;  // two 16-byte pieces: columns col .. col + 7, col + 8 .. col + 15
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pk[e] = bf2(__uint_as_float(v[k][2 * e]), __uint_as_float(v[k][2 * e + 1]));
        *reinterpret_cast<uint4*>(row + ((piece ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(row + (((piece + 1) ^ (r & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        for (int q2 = 0; q2 < 2; ++q2) {
          const int64_t h = h0 + q2;
          if (h >= p.H) break;
          const int erow = static_cast<int>(((b * p.nc + c) * p.H + h) * kTP);
#pragma unroll
          for (int cb = 0; cb < N / 64; ++cb) tma_store2(&mE, cb * 64, erow, stage + (q2 * (N / 64) + cb) * 64 * 128);
        }
        tma_store_drain();  // the staging tiles are read before they are reused or the CTA exits
      }
    }
    phase ^= 1u;
    tc_before_sync();
    __syncthreads();  // the x tile and the accumulator are free for the next pair
    tc_after_sync();
  }
  if (tid == 0) {  // after a wait ran out: let the copies and MMAs still in flight finish before leaving
    if (pendB >= 0) mb_wait(&sm.barB, static_cast<uint32_t>(pendB));
    if (pendX >= 0) mb_wait(&sm.barX, static_cast<uint32_t>(pendX));
    if (pendM >= 0) mb_wait(&sm.barM, static_cast<uint32_t>(pendM));
  }
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  if (warp == 0) tmem_free(tmem, 128);
}

// ---- launch 2: the recurrence between chunks ---------------------------------------------------------------
// One thread per (b, h, p, 4 consecutive n).
template <int N>
__global__ void __launch_bounds__(256, 2) ssd_state_pass_kernel(TcParams p) {
  pdl_wait();  // E and slast of launch 1
  const int64_t total = p.batch * p.H * kTP * (N / 4);
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t n4 = i % (N / 4), pp = (i / (N / 4)) % kTP, h = (i / (N / 4) / kTP) % p.H, b = i / (N / 4) / kTP / p.H;
  const int64_t row = (b * p.H + h) * kTP + pp;  // (b, h, p) of h0 / final_state
  float4 s = p.h0 ? *reinterpret_cast<const float4*>(p.h0 + row * N + 4 * n4) : make_float4(0.f, 0.f, 0.f, 0.f);
  // (b, c, h, p) rows of E / S and (b, c, h) entries of slast step by H * 64 rows and H entries per chunk
  const __nv_bfloat16* ep = p.E + ((b * p.nc * p.H + h) * kTP + pp) * N + 4 * n4;
  __nv_bfloat16* sp = p.S + ((b * p.nc * p.H + h) * kTP + pp) * N + 4 * n4;
  const float* dp = p.slast + b * p.nc * p.H + h;
  const int64_t estep = p.H * kTP * N;
  // chunks whose E (kept packed until used) and decay are loaded together, ahead of the dependent updates:
  // 16 at up to 128 registers measured 8% faster on a 64-chunk sequence than 8 at 64 registers
  constexpr int kAhead = 16;
  for (int64_t c0 = 0; c0 < p.nc; c0 += kAhead) {
    const int n = p.nc - c0 < kAhead ? static_cast<int>(p.nc - c0) : kAhead;
    uint2 e[kAhead];  // four bf16 each, widened where they are used
    float dl[kAhead];
#pragma unroll
    for (int k = 0; k < kAhead; ++k) {
      if (k < n) {
        e[k] = *reinterpret_cast<const uint2*>(ep + k * estep);
        dl[k] = dp[k * p.H];
      }
    }
#pragma unroll
    for (int k = 0; k < kAhead; ++k) {
      if (k < n) {
        uint2 packed;
        packed.x = bf2(s.x, s.y);
        packed.y = bf2(s.z, s.w);
        *reinterpret_cast<uint2*>(sp + k * estep) = packed;
        const float dec = ex2(dl[k] * kLog2e);
        s = make_float4(fmaf(dec, s.x, __uint_as_float(e[k].x << 16)),
                        fmaf(dec, s.y, __uint_as_float(e[k].x & 0xffff0000u)),
                        fmaf(dec, s.z, __uint_as_float(e[k].y << 16)),
                        fmaf(dec, s.w, __uint_as_float(e[k].y & 0xffff0000u)));
      }
    }
    ep += kAhead * estep;
    sp += kAhead * estep;
    dp += kAhead * p.H;
  }
  if (p.final_state) *reinterpret_cast<float4*>(p.final_state + row * N + 4 * n4) = s;
}

// ---- launch 3: outputs -----------------------------------------------------------------------------------
template <int N, int HPC>
struct OutSmem {
  alignas(1024) unsigned char Ct[N * 256];            // C tile [128 steps][N] (K-major A operand)
  alignas(1024) unsigned char BM[kTQ * 256];          // B tile [128][N] for G, then the masked G tile [128][128]
  alignas(1024) unsigned char Xt[kTQ * 128];          // x tile of one head [128 steps][64] (MN-major B operand)
  alignas(1024) unsigned char St[kTP * N * 2];        // S_c of one head [64 p][N] (K-major B operand)
  float s[HPC][kTQ];                                  // log2 of the decay from the chunk start through step i
  float cf[HPC][kTQ];                                 // input coefficient of step j
  unsigned long long barCB, barXS, barG, barM;
  uint32_t tmem;
};

template <int N, bool ZOH, int HPC>
__global__ void __launch_bounds__(kTT) ssd_output_kernel(const __grid_constant__ CUtensorMap mX,
                                                         const __grid_constant__ CUtensorMap mB,
                                                         const __grid_constant__ CUtensorMap mC,
                                                         const __grid_constant__ CUtensorMap mS,
                                                         const __grid_constant__ CUtensorMap mY, TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  static_assert(HPC <= kTT / 32, "one warp loads each head's deltas");
  OutSmem<N, HPC>& sm = *reinterpret_cast<OutSmem<N, HPC>*>(smem_raw + ((1024u - (s32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t groups = (p.H + HPC - 1) / HPC;
  const int64_t g = blockIdx.x % groups, c = (blockIdx.x / groups) % p.nc, b = blockIdx.x / groups / p.nc;
  const int64_t hbase = g * HPC;
  const int nh = static_cast<int>(p.H - hbase < HPC ? p.H - hbase : HPC);
  constexpr uint32_t kXSBytes = kTQ * 128 + kTP * N * 2;

  if (tid == 0) {
    mb_init(&sm.barCB);
    mb_init(&sm.barXS);
    mb_init(&sm.barG);
    mb_init(&sm.barM);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(&sm.tmem, 256);
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  const uint32_t tmem = sm.tmem;  // columns 0 .. 127: G; 128 .. 191: D1; 192 .. 255: D2
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const int half = warp >> 2;  // which half of the columns this warp takes
  // Outstanding asynchronous work (thread 0's view): the phase each barrier still owes, or -1.
  int pendCB = -1, pendXS = -1, pendG = -1, pendM = -1;
  float dv[4] = {0.0f, 0.0f, 0.0f, 0.0f}, alog = 0.0f;  // warp w < nh: deltas of head hbase + w (loaded first)
  if (warp < nh) load_deltas(p, b, c, hbase + warp, lane, dv, alog);
  auto issue_xs = [&](int64_t h, uint32_t ph) {  // x tile and S_c of head h (thread 0)
    mb_expect(&sm.barXS, kXSBytes);
    tma3(sm.Xt, &mX, static_cast<int>(h * kTP), static_cast<int>(c * kTQ), static_cast<int>(b), &sm.barXS);
    const int srow = static_cast<int>(((b * p.nc + c) * p.H + h) * kTP);
#pragma unroll
    for (int kb = 0; kb < N / 64; ++kb) tma2(sm.St + kb * kTP * 128, &mS, kb * 64, srow, &sm.barXS);
    pendXS = static_cast<int>(ph);
  };
  if (tid == 0) {
    mb_expect(&sm.barCB, 2 * N * 256);
#pragma unroll
    for (int kb = 0; kb < N / 64; ++kb) {
      tma3(sm.Ct + kb * kTQ * 128, &mC, kb * 64, static_cast<int>(c * kTQ), static_cast<int>(b), &sm.barCB);
      tma3(sm.BM + kb * kTQ * 128, &mB, kb * 64, static_cast<int>(c * kTQ), static_cast<int>(b), &sm.barCB);
    }
    pendCB = 0;
    pdl_wait();  // S_c of launch 2 (the C and B tiles above are the layer's inputs)
    issue_xs(hbase, 0);
  }
  if (warp < nh) {  // warp w: decays of head hbase + w
    float s[4], cf[4], s_last;
    chunk_decays<ZOH>(dv, alog, lane, s, cf, s_last);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      sm.s[warp][4 * lane + k] = s[k] * kLog2e;
      sm.cf[warp][4 * lane + k] = cf[k];
    }
  }
  bool ok = mb_wait(&sm.barCB, 0);
  ok = __syncthreads_and(ok) != 0;
  if (ok && tid == 0) {  // G = C B^T: M = 128 (i), N = 128 (j), K = state size
    pendCB = -1;
    tc_after_sync();
    constexpr uint32_t idesc = mma_idesc(128, 128, 0, 0);
#pragma unroll
    for (int ks = 0; ks < N / 16; ++ks) {
      const uint32_t off = (ks / 4) * kTQ * 128 + (ks % 4) * 32;
      mma_bf16(tmem, sw128_desc(s32(sm.Ct) + off, 16, 1024), sw128_desc(s32(sm.BM) + off, 16, 1024), idesc, ks > 0);
    }
    mma_commit(&sm.barG);
    pendG = 0;
  }
  if (ok) {
    ok = mb_wait(&sm.barG, 0);
    tc_after_sync();
    ok = __syncthreads_and(ok) != 0;
    if (ok && tid == 0) pendG = -1;
  }
  const int i = (warp & 3) * 32 + lane;  // this thread's row: step i of the chunk, TMEM lane i
  uint32_t phase = 0;
  for (int q = 0; q < nh && ok; ++q) {
    const int64_t h = hbase + q;
    // ---- masked, decayed G of head h -> bf16 A operand [i][j] in BM (K-major, 128-byte swizzle) ----
    // This thread: row i, columns j of its half (64 .. ); j > i is masked to zero without touching G.
    {
      const float si = sm.s[q][i];
      const float4* s4 = reinterpret_cast<const float4*>(sm.s[q]);
      const float4* c4 = reinterpret_cast<const float4*>(sm.cf[q]);
      uint32_t graw[4][16];  // G[i][j] for this thread's 64 columns, four loads and one wait
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) tmem_ld16_async(tmem + lane_base + half * 64 + 16 * g4, graw[g4]);
      tmem_wait();
      if (q > 0) {  // BM still holds the previous head's y tile until its bulk store has read it
        if (tid == 0) tma_store_wait_read();
        __syncthreads();
      }
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        const int j0 = half * 64 + 16 * g4;
        uint32_t pk[8];
        if (j0 > i) {  // the whole group lies above the diagonal
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = 0u;
        } else {
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 sj = s4[j0 / 4 + e4], cj = c4[j0 / 4 + e4];
            const int j = j0 + 4 * e4;
            const float m0 = j <= i ? __uint_as_float(graw[g4][4 * e4]) * ex2(si - sj.x) * cj.x : 0.0f;
            const float m1 = j + 1 <= i ? __uint_as_float(graw[g4][4 * e4 + 1]) * ex2(si - sj.y) * cj.y : 0.0f;
            const float m2 = j + 2 <= i ? __uint_as_float(graw[g4][4 * e4 + 2]) * ex2(si - sj.z) * cj.z : 0.0f;
            const float m3 = j + 3 <= i ? __uint_as_float(graw[g4][4 * e4 + 3]) * ex2(si - sj.w) * cj.w : 0.0f;
            pk[2 * e4] = bf2(m0, m1);
            pk[2 * e4 + 1] = bf2(m2, m3);
          }
        }
        unsigned char* rowp = sm.BM + (j0 >> 6) * kTQ * 128 + i * 128;
        const int piece = (j0 & 63) >> 3;  // two 16-byte pieces: j0 .. j0 + 7, j0 + 8 .. j0 + 15
        *reinterpret_cast<uint4*>(rowp + ((piece ^ (i & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(rowp + (((piece + 1) ^ (i & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    fence_async_smem();
    bool okq = mb_wait(&sm.barXS, phase);
    tc_before_sync();
    ok = __syncthreads_and(okq) != 0;
    tc_after_sync();
    if (!ok) break;
    if (tid == 0) {
      pendXS = -1;
      // D1 = (masked G) X: A = BM (K-major, K = j), B = x tile (MN-major, N = p)
      constexpr uint32_t id1 = mma_idesc(128, kTP, 0, 1);
#pragma unroll
      for (int ks = 0; ks < kTQ / 16; ++ks)
        mma_bf16(tmem + 128, sw128_desc(s32(sm.BM) + (ks / 4) * kTQ * 128 + (ks % 4) * 32, 16, 1024),
                 sw128_desc(s32(sm.Xt) + ks * 2048, kTQ * 128, 1024), id1, ks > 0);
      // D2 = C S_c: A = C tile (K-major, K = n), B = S_c (K-major rows p, K = n)
      constexpr uint32_t id2 = mma_idesc(128, kTP, 0, 0);
#pragma unroll
      for (int ks = 0; ks < N / 16; ++ks)
        mma_bf16(tmem + 192, sw128_desc(s32(sm.Ct) + (ks / 4) * kTQ * 128 + (ks % 4) * 32, 16, 1024),
                 sw128_desc(s32(sm.St) + (ks / 4) * kTP * 128 + (ks % 4) * 32, 16, 1024), id2, ks > 0);
      mma_commit(&sm.barM);
      pendM = static_cast<int>(phase);
    }
    okq = mb_wait(&sm.barM, phase);
    tc_after_sync();
    ok = __syncthreads_and(okq) != 0;
    if (!ok) break;
    if (tid == 0) {
      pendM = -1;
      if (q + 1 < nh) issue_xs(h + 1, phase ^ 1u);  // the MMAs that read the x and S tiles are done
    }
    // ---- epilogue: y = D1 + e^{s_i} D2, staged in BM as the [128 steps][64] bf16 box of the y tensor map
    // (128-byte rows, 16-byte pieces XOR-swizzled by the row) and written by one bulk tensor store, which
    // leaves out the steps past L ----
    {
      const float e = ex2(sm.s[q][i]);
      uint32_t d1[2][16], d2[2][16];  // this thread's 32 columns of D1 and D2: four loads, one wait
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        tmem_ld16_async(tmem + lane_base + 128 + half * (kTP / 2) + 16 * k, d1[k]);
        tmem_ld16_async(tmem + lane_base + 192 + half * (kTP / 2) + 16 * k, d2[k]);
      }
      tmem_wait();
      unsigned char* yrow = sm.BM + i * 128;
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int piece = (half * (kTP / 2) + 16 * k2) >> 3;  // columns 8 piece .. 8 piece + 15
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 16; k += 2)
          pk[k / 2] = bf2(fmaf(e, __uint_as_float(d2[k2][k]), __uint_as_float(d1[k2][k])),
                          fmaf(e, __uint_as_float(d2[k2][k + 1]), __uint_as_float(d1[k2][k + 1])));
        *reinterpret_cast<uint4*>(yrow + ((piece ^ (i & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(yrow + (((piece + 1) ^ (i & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      fence_async_smem();
    }
    phase ^= 1u;
    tc_before_sync();
    __syncthreads();  // the y tile is staged; the TMEM accumulators are free for the next head
    tc_after_sync();
    if (tid == 0) {
      tma_store3(&mY, static_cast<int>(h * kTP), static_cast<int>(c * kTQ), static_cast<int>(b), sm.BM);
      tma_store_commit();
    }
  }
  if (tid == 0) {  // after a wait ran out: let the copies and MMAs still in flight finish before leaving
    tma_store_wait_read();  // and the last y tile's store read its staging
    if (pendCB >= 0) mb_wait(&sm.barCB, static_cast<uint32_t>(pendCB));
    if (pendXS >= 0) mb_wait(&sm.barXS, static_cast<uint32_t>(pendXS));
    if (pendG >= 0) mb_wait(&sm.barG, static_cast<uint32_t>(pendG));
    if (pendM >= 0) mb_wait(&sm.barM, static_cast<uint32_t>(pendM));
  }
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  if (warp == 0) tmem_free(tmem, 256);
}

// ---- host side ----------------------------------------------------------------------------------------------
typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                             const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                             CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn tc_encoder() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  }
  return fn;
}

// bf16 tensor map with the 128-byte swizzle: dims / box innermost first, strides in bytes of dims 1 ...
bool bf16_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box) {
  EncodeFn enc = tc_encoder();
  if (!enc) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <auto Kern>
cudaError_t tc_smem_once(size_t smem) {
  static bool set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!set[dev & 63]) {
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    set[dev & 63] = true;
  }
  return cudaSuccess;
}

struct TcLayout {
  size_t e_off, s_off, d_off, bytes;
};
TcLayout tc_layout(int64_t batch, int64_t L, int64_t H, int64_t N) {
  const int64_t nc = (L + kTQ - 1) / kTQ;
  const size_t states = static_cast<size_t>(batch) * nc * H * kTP * N;
  TcLayout t;
  t.e_off = 0;
  t.s_off = ((states * 2 + 255) / 256) * 256;
  t.d_off = t.s_off + ((states * 2 + 255) / 256) * 256;
  t.bytes = t.d_off + static_cast<size_t>(batch) * nc * H * 4;
  return t;
}

template <int N, bool ZOH, int HPC>
cudaError_t launch_out(const SsdArgs& a, const TcParams& p, const CUtensorMap& mX, const CUtensorMap& mB,
                       const CUtensorMap& mC, const CUtensorMap& mS, const CUtensorMap& mY,
                       cudaLaunchAttribute* pdl) {
  const size_t smem3 = sizeof(OutSmem<N, HPC>) + 1024;
  cudaError_t e = tc_smem_once<ssd_output_kernel<N, ZOH, HPC>>(smem3);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg3 = {};
  cfg3.gridDim = dim3(static_cast<unsigned>(a.batch * p.nc * ((a.H + HPC - 1) / HPC)));
  cfg3.blockDim = dim3(kTT);
  cfg3.dynamicSmemBytes = smem3;
  cfg3.stream = a.stream;
  cfg3.attrs = pdl;
  cfg3.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg3, ssd_output_kernel<N, ZOH, HPC>, mX, mB, mC, mS, mY, p);
}

template <int N, bool ZOH>
cudaError_t launch_tc_n(const SsdArgs& a) {
  TcParams p;
  p.delta = a.delta;
  p.A_log = a.A_log;
  p.h0 = a.h0;
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.final_state = a.final_state;
  p.batch = a.batch;
  p.L = a.L;
  p.H = a.H;
  p.nc = (a.L + kTQ - 1) / kTQ;
  const TcLayout lay = tc_layout(a.batch, a.L, a.H, N);
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  p.E = reinterpret_cast<__nv_bfloat16*>(ws + lay.e_off);
  p.S = reinterpret_cast<__nv_bfloat16*>(ws + lay.s_off);
  p.slast = reinterpret_cast<float*>(ws + lay.d_off);

  CUtensorMap mX, mB, mC, mS, mE, mY;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.H * kTP), static_cast<cuuint64_t>(a.L),
                                static_cast<cuuint64_t>(a.batch)};
    const cuuint64_t str[2] = {static_cast<cuuint64_t>(a.H * kTP * 2), static_cast<cuuint64_t>(a.L * a.H * kTP * 2)};
    const cuuint32_t box[3] = {64, kTQ, 1};
    if (!bf16_map(&mX, a.x, 3, dims, str, box) || !bf16_map(&mY, a.y, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(a.L), static_cast<cuuint64_t>(a.batch)};
    const cuuint64_t str[2] = {static_cast<cuuint64_t>(N * 2), static_cast<cuuint64_t>(a.L * N * 2)};
    const cuuint32_t box[3] = {64, kTQ, 1};
    if (!bf16_map(&mB, a.B, 3, dims, str, box) || !bf16_map(&mC, a.C, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {  // S (read by launch 3) and E (written by launch 1): [rows (b, c, h, p)][N] bf16, boxes of 64 x 64
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(a.batch * p.nc * a.H * kTP)};
    const cuuint64_t str[1] = {static_cast<cuuint64_t>(N * 2)};
    const cuuint32_t box[2] = {64, kTP};
    if (!bf16_map(&mS, p.S, 2, dims, str, box) || !bf16_map(&mE, p.E, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  cudaError_t e;
  const size_t smem1 = sizeof(ChunkSmem<N>) + 1024;
  if ((e = tc_smem_once<ssd_chunk_state_kernel<N, ZOH>>(smem1)) != cudaSuccess) return e;
  const int64_t g1 = ((a.H + 1) / 2 + kPairsPerCta - 1) / kPairsPerCta;
  ssd_chunk_state_kernel<N, ZOH><<<static_cast<unsigned>(a.batch * p.nc * g1), kTT, smem1, a.stream>>>(mX, mB, mE, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t threads = a.batch * a.H * kTP * (N / 4);
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256));
  cfg2.blockDim = dim3(256);
  cfg2.stream = a.stream;
  cfg2.attrs = pdl;
  cfg2.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg2, ssd_state_pass_kernel<N>, p)) != cudaSuccess) return e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // launch 3: few heads per CTA unless that grid would need more than two rounds of the two CTAs an SM holds
  const int64_t few = a.batch * p.nc * ((a.H + kHeadsFew - 1) / kHeadsFew);
  if (few <= 4 * static_cast<int64_t>(sm_count()))
    e = launch_out<N, ZOH, kHeadsFew>(a, p, mX, mB, mC, mS, mY, pdl);
  else
    e = launch_out<N, ZOH, kHeadsMany>(a, p, mX, mB, mC, mS, mY, pdl);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool ssd_tc_ok(const SsdArgs& a) {
  if (a.P != kTP || (a.N != 64 && a.N != 128) || a.L <= 0 || a.batch <= 0 || a.H <= 0) return false;
  if (tc_encoder() == nullptr) return false;
  const int64_t nc = (a.L + kTQ - 1) / kTQ;
  const int64_t ctas = a.batch * nc * ((a.H + 1) / 2 + 1);
  if (ctas > INT32_MAX || a.batch * nc * a.H * kTP > INT32_MAX) return false;  // grid and TMA row coordinates
  if (reinterpret_cast<uintptr_t>(a.workspace) % 256 != 0) return false;
  if (a.h0 && reinterpret_cast<uintptr_t>(a.h0) % 16 != 0) return false;
  if (a.final_state && reinterpret_cast<uintptr_t>(a.final_state) % 16 != 0) return false;
  return a.workspace != nullptr && a.workspace_bytes >= ssd_tc_workspace_bytes(a.batch, a.L, a.H, a.P, a.N);
}

size_t ssd_tc_workspace_bytes(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N) {
  if (P != kTP || (N != 64 && N != 128) || L <= 0 || batch <= 0 || H <= 0) return 0;
  return tc_layout(batch, L, H, N).bytes;
}

cudaError_t launch_ssd_tc(const SsdArgs& a) {
  if (a.N == 64) return a.disc == 1 ? launch_tc_n<64, true>(a) : launch_tc_n<64, false>(a);
  return a.disc == 1 ? launch_tc_n<128, true>(a) : launch_tc_n<128, false>(a);
}

int read_and_clear_ssd_status() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_ssd_status, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) {
    int z = 0;
    cudaMemcpyToSymbol(g_ssd_status, &z, sizeof(int));
  }
  return v;
}

}  // namespace ssm
