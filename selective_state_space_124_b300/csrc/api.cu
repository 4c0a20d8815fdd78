// api.cu -- the C ABI declared in include/ssm_scan.h: argument checks, kernel choice, launch, status.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/ssm_scan.h"
#include "launch.h"

#include <atomic>
#include <mutex>

namespace ssm {

namespace {
thread_local char g_last_error[256] = "";
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};

ssm_status fail(ssm_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

ssm_status cuda_fail(cudaError_t e, const char* where) {
  return fail(SSM_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct Range {
  uintptr_t lo, hi;
};
Range range_of(const void* p, int64_t count, int64_t elem) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + static_cast<uintptr_t>(count) * static_cast<uintptr_t>(elem)};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

bool valid_enums(ssm_dtype dt, ssm_disc disc) {
  return (dt == SSM_DTYPE_F32 || dt == SSM_DTYPE_BF16) && (disc == SSM_DISC_EULER || disc == SSM_DISC_ZOH);
}

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    cached[dev] = v;
  }
  return cached[dev];
}

namespace {
// Library-owned copy streams and events of ssm_scan_fwd_host, one set per device, created on first use.
struct HostStreamSet {
  std::mutex mu;  // held while a call enqueues its work
  bool ready = false;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start, fin, ev_up[2], ev_comp[2], ev_down[2];
};
HostStreamSet g_host_sets[64];

cudaError_t host_set_init(HostStreamSet& h) {
  if (h.ready) return cudaSuccess;
  cudaError_t e;
  if ((e = cudaStreamCreateWithFlags(&h.up, cudaStreamNonBlocking)) != cudaSuccess) return e;
  if ((e = cudaStreamCreateWithFlags(&h.down, cudaStreamNonBlocking)) != cudaSuccess) return e;
  cudaEvent_t* evs[] = {&h.start, &h.fin, &h.ev_up[0], &h.ev_up[1], &h.ev_comp[0], &h.ev_comp[1],
                        &h.ev_down[0], &h.ev_down[1]};
  for (cudaEvent_t* ev : evs)
    if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
  h.ready = true;
  return cudaSuccess;
}

// Workspace of ssm_scan_fwd_host: A_log, two states, then two slots of (x, delta, B, C, y) for seg_L steps,
// every piece 256-byte aligned.
struct HostLayout {
  size_t a_log, st[2], x[2], d[2], b[2], c[2], y[2], bytes;
};
size_t align256(size_t v) { return (v + 255) / 256 * 256; }
HostLayout host_layout(int64_t batch, int64_t D, int64_t N, int64_t es, int64_t seg_L) {
  HostLayout l;
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t at = off;
    off += align256(n);
    return at;
  };
  const size_t sd = static_cast<size_t>(batch) * seg_L * D * es, sn = static_cast<size_t>(batch) * seg_L * N * es;
  l.a_log = take(static_cast<size_t>(D) * N * 4);
  for (int k = 0; k < 2; ++k) l.st[k] = take(static_cast<size_t>(batch) * D * N * 4);
  for (int k = 0; k < 2; ++k) {
    l.x[k] = take(sd);
    l.d[k] = take(sd);
    l.b[k] = take(sn);
    l.c[k] = take(sn);
    l.y[k] = take(sd);
  }
  l.bytes = off;
  return l;
}

// rows of `width` bytes: batch rows, `hpitch` apart on the host, packed on the device
cudaError_t copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, int64_t rows,
                      cudaMemcpyKind kind, cudaStream_t s) {
  if (width == 0 || rows == 0) return cudaSuccess;
  if (rows == 1) return cudaMemcpyAsync(dst, src, width, kind, s);
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, static_cast<size_t>(rows), kind, s);
}
}  // namespace

}  // namespace ssm

using namespace ssm;

extern "C" {

ssm_status ssm_scan_fwd(const void* x, const void* delta, const float* A_log, const void* B, const void* C,
                        const float* h0, void* y, float* final_state, int64_t batch, int64_t L, int64_t D,
                        int64_t N, ssm_dtype dtype, ssm_disc disc, void* stream) {
  return ssm_scan_fwd_ex(x, delta, A_log, B, C, h0, nullptr, 0, nullptr, nullptr, y, final_state, batch, L, D, N,
                         dtype, disc, stream);
}

ssm_status ssm_scan_fwd_ex(const void* x, const void* delta, const float* A_log, const void* B, const void* C,
                           const float* h0, const float* delta_bias, int delta_softplus, const float* D_skip,
                           const void* z, void* y, float* final_state, int64_t batch, int64_t L, int64_t D,
                           int64_t N, ssm_dtype dtype, ssm_disc disc, void* stream) {
  g_last_error[0] = '\0';
  if (!valid_enums(dtype, disc)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: bad dtype or disc");
  if (batch < 0 || L < 0 || D < 0 || N < 1)
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: sizes must be >= 0 and N >= 1");
  if (N > 16) return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_fwd: N = %lld > 16", (long long)N);
  int64_t bl, bld, bln, bd, bdn;
  if (!mul_ok(batch, L, &bl) || !mul_ok(bl, D, &bld) || !mul_ok(bl, N, &bln) || !mul_ok(batch, D, &bd) ||
      !mul_ok(bd, N, &bdn))
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: sizes overflow");
  const int64_t es = dtype == SSM_DTYPE_BF16 ? 2 : 4;
  if (bld > 0 && (!x || !delta || !y)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: null x/delta/y");
  if (bln > 0 && (!B || !C)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: null B/C");
  if (bld > 0 && !A_log) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: null A_log");
  const Range ry = range_of(y, bld, es);
  const Range rf = range_of(final_state, final_state ? bdn : 0, 4);
  const Range ins[] = {range_of(x, bld, es),        range_of(delta, bld, es),  range_of(A_log, D * N, 4),
                       range_of(B, bln, es),        range_of(C, bln, es),      range_of(h0, h0 ? bdn : 0, 4),
                       range_of(delta_bias, delta_bias ? D : 0, 4), range_of(D_skip, D_skip ? D : 0, 4),
                       range_of(z, z ? bld : 0, es)};
  for (const Range& r : ins)
    if (overlap(ry, r) || overlap(rf, r)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: outputs overlap inputs");
  if (overlap(ry, rf)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: y overlaps final_state");

  FwdArgs a{x, delta, A_log, B, C, h0, y, final_state, batch, L, D, N, static_cast<int>(dtype),
            static_cast<int>(disc), static_cast<cudaStream_t>(stream)};
  a.delta_bias = delta_bias;
  a.softplus = delta_softplus != 0;
  a.D_skip = D_skip;
  a.z = z;
  if (batch == 0 || D == 0) return SSM_OK;
  cudaError_t e = (L == 0) ? launch_init_state(a) : (tma_path_ok(a) ? launch_fwd_tma(a) : launch_fwd_simple(a));
  if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd launch");
  return SSM_OK;
}

size_t ssm_scan_fwd_host_workspace_size(int64_t batch, int64_t D, int64_t N, ssm_dtype dtype, int64_t seg_L) {
  if (batch < 0 || D < 0 || N < 1 || N > 16 || seg_L < 1 || !valid_enums(dtype, SSM_DISC_EULER)) return 0;
  int64_t t;
  if (!mul_ok(batch, seg_L, &t) || !mul_ok(t, D + N, &t) || !mul_ok(t, 64, &t)) return 0;
  return host_layout(batch, D, N, dtype == SSM_DTYPE_BF16 ? 2 : 4, seg_L).bytes;
}

ssm_status ssm_scan_fwd_host(const void* x, const void* delta, const float* A_log, const void* B, const void* C,
                             const float* h0, void* y, float* final_state, void* workspace, size_t workspace_bytes,
                             int64_t seg_L, int64_t batch, int64_t L, int64_t D, int64_t N, ssm_dtype dtype,
                             ssm_disc disc, void* stream) {
  g_last_error[0] = '\0';
  if (!valid_enums(dtype, disc)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: bad dtype or disc");
  if (batch < 0 || L < 0 || D < 0 || N < 1)
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: sizes must be >= 0 and N >= 1");
  if (N > 16) return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_fwd_host: N = %lld > 16", (long long)N);
  if (seg_L < 1) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: seg_L must be >= 1");
  int64_t bl, bld, bln, bd, bdn, tmp;
  if (!mul_ok(batch, L, &bl) || !mul_ok(bl, D, &bld) || !mul_ok(bl, N, &bln) || !mul_ok(batch, D, &bd) ||
      !mul_ok(bd, N, &bdn) || !mul_ok(batch, seg_L, &tmp) || !mul_ok(tmp, D + N, &tmp) || !mul_ok(tmp, 64, &tmp))
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: sizes overflow");
  const int64_t es = dtype == SSM_DTYPE_BF16 ? 2 : 4;
  if (bld > 0 && (!x || !delta || !y)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: null x/delta/y");
  if (bln > 0 && (!B || !C)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: null B/C");
  if (bld > 0 && !A_log) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: null A_log");
  const Range ry = range_of(y, bld, es);
  const Range rf = range_of(final_state, final_state ? bdn : 0, 4);
  const Range ins[] = {range_of(x, bld, es), range_of(delta, bld, es), range_of(A_log, D * N, 4),
                       range_of(B, bln, es), range_of(C, bln, es),     range_of(h0, h0 ? bdn : 0, 4)};
  for (const Range& r : ins)
    if (overlap(ry, r) || overlap(rf, r))
      return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: outputs overlap inputs");
  if (overlap(ry, rf)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: y overlaps final_state");
  if (batch == 0 || D == 0) return SSM_OK;
  if (L == 0) {  // no steps: the final state is the initial one
    if (final_state) {
      if (h0) std::memcpy(final_state, h0, static_cast<size_t>(bdn) * 4);
      else std::memset(final_state, 0, static_cast<size_t>(bdn) * 4);
    }
    return SSM_OK;
  }
  const HostLayout l = host_layout(batch, D, N, es, seg_L);
  if (!workspace || workspace_bytes < l.bytes)
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd_host: workspace of %zu bytes, %zu needed", workspace_bytes, l.bytes);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd_host");
  if (dev < 0 || dev >= 64) return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_fwd_host: device %d", dev);
  HostStreamSet& hs = g_host_sets[dev];
  std::lock_guard<std::mutex> lock(hs.mu);
  if ((e = host_set_init(hs)) != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd_host: streams");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
#define SSM_HOST_CK(expr)                                                      \
  do {                                                                         \
    if ((e = (expr)) != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd_host"); \
  } while (0)
  // everything after the work already on the caller's stream
  SSM_HOST_CK(cudaEventRecord(hs.start, cs));
  SSM_HOST_CK(cudaStreamWaitEvent(hs.up, hs.start, 0));
  SSM_HOST_CK(cudaStreamWaitEvent(hs.down, hs.start, 0));
  SSM_HOST_CK(cudaMemcpyAsync(w + l.a_log, A_log, static_cast<size_t>(D) * N * 4, h2d, hs.up));
  if (h0) SSM_HOST_CK(cudaMemcpyAsync(w + l.st[1], h0, static_cast<size_t>(bdn) * 4, h2d, hs.up));
  const int64_t nseg = (L + seg_L - 1) / seg_L;
  const size_t hrow_d = static_cast<size_t>(L) * D * es, hrow_n = static_cast<size_t>(L) * N * es;
  for (int64_t sg = 0; sg < nseg; ++sg) {
    const int k = static_cast<int>(sg & 1);
    const int64_t t0 = sg * seg_L, n = seg_L < L - t0 ? seg_L : L - t0;
    const size_t wd = static_cast<size_t>(n) * D * es, wn = static_cast<size_t>(n) * N * es;
    const size_t od = static_cast<size_t>(t0) * D * es, on = static_cast<size_t>(t0) * N * es;
    // slot k's inputs are free once the compute of segment sg - 2 is done
    if (sg >= 2) SSM_HOST_CK(cudaStreamWaitEvent(hs.up, hs.ev_comp[k], 0));
    SSM_HOST_CK(copy_rows(w + l.x[k], wd, static_cast<const char*>(x) + od, hrow_d, wd, batch, h2d, hs.up));
    SSM_HOST_CK(copy_rows(w + l.d[k], wd, static_cast<const char*>(delta) + od, hrow_d, wd, batch, h2d, hs.up));
    SSM_HOST_CK(copy_rows(w + l.b[k], wn, static_cast<const char*>(B) + on, hrow_n, wn, batch, h2d, hs.up));
    SSM_HOST_CK(copy_rows(w + l.c[k], wn, static_cast<const char*>(C) + on, hrow_n, wn, batch, h2d, hs.up));
    SSM_HOST_CK(cudaEventRecord(hs.ev_up[k], hs.up));
    SSM_HOST_CK(cudaStreamWaitEvent(cs, hs.ev_up[k], 0));
    // slot k's y is free once the copy-out of segment sg - 2 is done
    if (sg >= 2) SSM_HOST_CK(cudaStreamWaitEvent(cs, hs.ev_down[k], 0));
    const float* hin = sg == 0 ? (h0 ? reinterpret_cast<const float*>(w + l.st[1]) : nullptr)
                               : reinterpret_cast<const float*>(w + l.st[(sg - 1) & 1]);
    const ssm_status st = ssm_scan_fwd(w + l.x[k], w + l.d[k], reinterpret_cast<const float*>(w + l.a_log),
                                       w + l.b[k], w + l.c[k], hin, w + l.y[k],
                                       reinterpret_cast<float*>(w + l.st[k]), batch, n, D, N, dtype, disc, cs);
    if (st != SSM_OK) return st;
    SSM_HOST_CK(cudaEventRecord(hs.ev_comp[k], cs));
    SSM_HOST_CK(cudaStreamWaitEvent(hs.down, hs.ev_comp[k], 0));
    SSM_HOST_CK(copy_rows(static_cast<char*>(y) + od, hrow_d, w + l.y[k], wd, wd, batch, d2h, hs.down));
    SSM_HOST_CK(cudaEventRecord(hs.ev_down[k], hs.down));
  }
  if (final_state)
    SSM_HOST_CK(cudaMemcpyAsync(final_state, w + l.st[(nseg - 1) & 1], static_cast<size_t>(bdn) * 4, d2h, hs.down));
  // the caller's stream continues after the last copy-out (the last upload precedes the last compute)
  SSM_HOST_CK(cudaEventRecord(hs.fin, hs.down));
  SSM_HOST_CK(cudaStreamWaitEvent(cs, hs.fin, 0));
#undef SSM_HOST_CK
  return SSM_OK;
}

ssm_status ssm_scan_step(float* state, const void* x_t, const void* delta_t, const float* A_log,
                         const void* B_t, const void* C_t, void* y_t, int64_t batch, int64_t D, int64_t N,
                         ssm_dtype dtype, ssm_disc disc, void* stream) {
  return ssm_scan_step_ex(state, x_t, delta_t, A_log, B_t, C_t, nullptr, 0, nullptr, nullptr, y_t, batch, D, N, dtype,
                          disc, stream);
}

ssm_status ssm_scan_step_ex(float* state, const void* x_t, const void* delta_t, const float* A_log,
                            const void* B_t, const void* C_t, const float* delta_bias, int delta_softplus,
                            const float* D_skip, const void* z_t, void* y_t, int64_t batch, int64_t D, int64_t N,
                            ssm_dtype dtype, ssm_disc disc, void* stream) {
  g_last_error[0] = '\0';
  if (!valid_enums(dtype, disc)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_step: bad dtype or disc");
  if (batch < 0 || D < 0 || N < 1)
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_step: sizes must be >= 0 and N >= 1");
  if (N > 16) return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_step: N = %lld > 16", (long long)N);
  int64_t bd, bdn, bn;
  if (!mul_ok(batch, D, &bd) || !mul_ok(bd, N, &bdn) || !mul_ok(batch, N, &bn))
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_step: sizes overflow");
  if (bd == 0) return SSM_OK;
  if (!state || !x_t || !delta_t || !A_log || !B_t || !C_t || !y_t)
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_step: null pointer");
  const int64_t es = dtype == SSM_DTYPE_BF16 ? 2 : 4;
  const Range rs = range_of(state, bdn, 4), ry = range_of(y_t, bd, es);
  const Range ins[] = {range_of(x_t, bd, es), range_of(delta_t, bd, es), range_of(A_log, D * N, 4),
                       range_of(B_t, bn, es), range_of(C_t, bn, es), range_of(delta_bias, delta_bias ? D : 0, 4),
                       range_of(D_skip, D_skip ? D : 0, 4), range_of(z_t, z_t ? bd : 0, es)};
  for (const Range& r : ins)
    if (overlap(rs, r) || overlap(ry, r)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_step: outputs overlap inputs");
  if (overlap(rs, ry)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_step: y_t overlaps state");
  StepArgs a{state, x_t, delta_t, A_log, B_t, C_t, y_t, batch, D, N, static_cast<int>(dtype),
             static_cast<int>(disc), static_cast<cudaStream_t>(stream)};
  a.delta_bias = delta_bias;
  a.softplus = delta_softplus != 0;
  a.D_skip = D_skip;
  a.z = z_t;
  cudaError_t e = launch_step(a);
  if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_step launch");
  return SSM_OK;
}

size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t L, int64_t D, int64_t N) {
  int64_t bl = 0, bld = 0, bldn = 0;
  if (N < 1 || N > 16 || !mul_ok(batch, L, &bl) || !mul_ok(bl, D, &bld) || !mul_ok(bld, N, &bldn)) return 0;
  if (bldn > INT64_MAX / 4) return 0;
  return bwd_workspace_bytes(batch, L, D, N);
}

ssm_status ssm_scan_bwd(const void* x, const void* delta, const float* A_log, const void* B, const void* C,
                        const float* h0, const void* dy, const float* dfinal, void* dx, void* ddelta, float* dA_log,
                        float* dB, float* dC, float* dh0, void* workspace, size_t workspace_bytes, int64_t batch,
                        int64_t L, int64_t D, int64_t N, ssm_dtype dtype, ssm_disc disc, void* stream) {
  g_last_error[0] = '\0';
  if (!valid_enums(dtype, disc)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: bad dtype or disc");
  if (batch < 0 || L < 0 || D < 0 || N < 1)
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: bad sizes (batch %lld, L %lld, D %lld, N %lld)",
                static_cast<long long>(batch), static_cast<long long>(L), static_cast<long long>(D),
                static_cast<long long>(N));
  if (N > 16) return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_bwd: N = %lld > 16", static_cast<long long>(N));
  int64_t bl = 0, bld = 0, bln = 0, bdn = 0, dn = 0, bldn = 0;
  if (!mul_ok(batch, L, &bl) || !mul_ok(bl, D, &bld) || !mul_ok(bl, N, &bln) || !mul_ok(batch * D, N, &bdn) ||
      !mul_ok(D, N, &dn) || !mul_ok(bld, N, &bldn) || bldn > INT64_MAX / 4)
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: size overflow");
  const int64_t es = dtype == SSM_DTYPE_BF16 ? 2 : 4;
  if (bld > 0 && (!x || !delta || !dy || !dx || !ddelta))
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: null x, delta, dy, dx or ddelta");
  if (bln > 0 && (!B || !C || !dB || !dC)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: null B, C, dB or dC");
  if (dn > 0 && (!A_log || !dA_log)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: null A_log or dA_log");
  const size_t need = bwd_workspace_bytes(batch, L, D, N);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : static_cast<size_t>(0));
  const Range outs[] = {range_of(dx, bld, es), range_of(ddelta, bld, es), range_of(dA_log, dn, 4),
                        range_of(dB, bln, 4), range_of(dC, bln, 4), range_of(dh0, dh0 ? bdn : 0, 4),
                        range_of(workspace, static_cast<int64_t>(need), 1)};
  const Range ins[] = {range_of(x, bld, es), range_of(delta, bld, es), range_of(A_log, dn, 4), range_of(B, bln, es),
                       range_of(C, bln, es), range_of(h0, h0 ? bdn : 0, 4), range_of(dy, bld, es),
                       range_of(dfinal, dfinal ? bdn : 0, 4)};
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
    for (const Range& r : ins)
      if (overlap(outs[i], r)) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: outputs overlap inputs");
    for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
      if (overlap(outs[i], outs[j])) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_bwd: outputs overlap each other");
  }
  BwdArgs a{x, delta, A_log, B, C, h0, dy, dfinal, dx, ddelta, dA_log, dB, dC, dh0,
            static_cast<float*>(workspace), batch, L, D, N, static_cast<int>(dtype), static_cast<int>(disc),
            static_cast<cudaStream_t>(stream)};
  cudaError_t e = launch_bwd(a);
  if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_bwd launch");
  return SSM_OK;
}

ssm_status ssm_scan_bwd_noalloc(const void* x, const void* delta, const float* A_log, const void* B, const void* C,
                                const float* h0, const void* dy, const float* dfinal, void* dx, void* ddelta,
                                float* dA_log, float* dB, float* dC, float* dh0, int64_t batch, int64_t L, int64_t D,
                                int64_t N, ssm_dtype dtype, ssm_disc disc, void* stream) {
  g_last_error[0] = '\0';
  if (N >= 1 && N <= 16 && batch >= 0 && L >= 0 && D >= 0) {
    const size_t need = ssm_scan_bwd_workspace_size(batch, L, D, N);
    if (need > kBwdNoAllocScratchBytes)
      return fail(SSM_ERR_INVALID_ARG,
                  "ssm_scan_bwd_noalloc: these sizes need %zu bytes of scratch, the built-in scratch holds %zu "
                  "(call ssm_scan_bwd with a workspace instead)",
                  need, kBwdNoAllocScratchBytes);
  }
  void* scratch = nullptr;
  const cudaError_t e = bwd_noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_bwd_noalloc: scratch address");
  return ssm_scan_bwd(x, delta, A_log, B, C, h0, dy, dfinal, dx, ddelta, dA_log, dB, dC, dh0, scratch,
                      kBwdNoAllocScratchBytes, batch, L, D, N, dtype, disc, stream);
}

size_t ssm_ssd_fwd_workspace_size(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N) {
  int64_t bl = 0, blh = 0, blhp = 0;
  if (!ssd_shape_ok(P, N) || !mul_ok(batch, L, &bl) || !mul_ok(bl, H, &blh) || !mul_ok(blh, P, &blhp)) return 0;
  return ssd_workspace_bytes(batch, L, H, P, N);
}

ssm_status ssm_ssd_fwd(const void* x, const float* delta, const float* A_log, const void* B, const void* C,
                       const float* h0, void* y, float* final_state, void* workspace, size_t workspace_bytes,
                       int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N, ssm_dtype dtype, ssm_disc disc,
                       void* stream) {
  g_last_error[0] = '\0';
  if (!valid_enums(dtype, disc)) return fail(SSM_ERR_INVALID_ARG, "ssm_ssd_fwd: bad dtype or disc");
  if (batch < 0 || L < 0 || H < 0 || P < 1 || N < 1)
    return fail(SSM_ERR_INVALID_ARG, "ssm_ssd_fwd: bad sizes (batch %lld, L %lld, H %lld, P %lld, N %lld)",
                static_cast<long long>(batch), static_cast<long long>(L), static_cast<long long>(H),
                static_cast<long long>(P), static_cast<long long>(N));
  if (dtype != SSM_DTYPE_BF16) return fail(SSM_ERR_UNSUPPORTED, "ssm_ssd_fwd: x, B, C and y must be bf16");
  if (!ssd_shape_ok(P, N))
    return fail(SSM_ERR_UNSUPPORTED, "ssm_ssd_fwd: needs N = 64 or 128 and P a multiple of 16 (N %lld, P %lld)",
                static_cast<long long>(N), static_cast<long long>(P));
  int64_t bl = 0, blh = 0, blhp = 0, bln = 0, bh = 0, bhpn = 0;
  if (!mul_ok(batch, L, &bl) || !mul_ok(bl, H, &blh) || !mul_ok(blh, P, &blhp) || !mul_ok(bl, N, &bln) ||
      !mul_ok(batch, H, &bh) || !mul_ok(bh * P, N, &bhpn) || bh * (P / 16) > INT32_MAX)
    return fail(SSM_ERR_INVALID_ARG, "ssm_ssd_fwd: size overflow");
  if (blhp > 0 && (!x || !delta || !y)) return fail(SSM_ERR_INVALID_ARG, "ssm_ssd_fwd: null x, delta or y");
  if (bln > 0 && (!B || !C)) return fail(SSM_ERR_INVALID_ARG, "ssm_ssd_fwd: null B or C");
  if (H > 0 && !A_log) return fail(SSM_ERR_INVALID_ARG, "ssm_ssd_fwd: null A_log");
  const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(B) |
                        reinterpret_cast<uintptr_t>(C) | reinterpret_cast<uintptr_t>(y);
  if (mis & 15) return fail(SSM_ERR_UNSUPPORTED, "ssm_ssd_fwd: x, B, C and y must be 16-byte aligned");
  const Range ry = range_of(y, blhp, 2);
  const Range rf = range_of(final_state, final_state ? bhpn : 0, 4);
  const Range rw = range_of(workspace, workspace ? static_cast<int64_t>(workspace_bytes) : 0, 1);
  const Range ins[] = {range_of(x, blhp, 2), range_of(delta, blh, 4), range_of(A_log, H, 4), range_of(B, bln, 2),
                       range_of(C, bln, 2), range_of(h0, h0 ? bhpn : 0, 4)};
  for (const Range& r : ins)
    if (overlap(ry, r) || overlap(rf, r) || overlap(rw, r))
      return fail(SSM_ERR_INVALID_ARG, "ssm_ssd_fwd: outputs or workspace overlap inputs");
  if (overlap(ry, rf) || overlap(rw, ry) || overlap(rw, rf))
    return fail(SSM_ERR_INVALID_ARG, "ssm_ssd_fwd: y, final_state and workspace overlap");
  if (bh == 0) return SSM_OK;
  SsdArgs a{x, delta, A_log, B, C, h0, y, final_state, workspace, workspace_bytes, batch, L, H, P, N,
            static_cast<int>(disc), static_cast<cudaStream_t>(stream)};
  cudaError_t e = launch_ssd(a);
  if (e != cudaSuccess) return cuda_fail(e, "ssm_ssd_fwd launch");
  return SSM_OK;
}

ssm_status ssm_check_device(void* stream) {
  g_last_error[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ssm_check_device");
  const int st = read_and_clear_device_status(), st2 = read_and_clear_ssd_status();
  if (st < 0 || st2 < 0) return fail(SSM_ERR_CUDA, "ssm_check_device: cannot read the device status word");
  if (st != 0 || st2 != 0) return fail(SSM_ERR_TIMEOUT, "ssm_check_device: a kernel gave up a bounded wait");
  return SSM_OK;
}

uint64_t ssm_set_wait_limit_ns(uint64_t ns) { return g_wait_limit_ns.exchange(ns); }

const char* ssm_status_string(ssm_status s) {
  switch (s) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
    case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
  }
  return "SSM_ERR_UNKNOWN";
}

const char* ssm_last_error(void) { return g_last_error; }

int ssm_version(void) { return 100; }

}  // extern "C"
