// launch.h -- host-side launchers shared between the C ABI (api.cu) and the kernel files.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace ssm {

struct FwdArgs {
  const void* x;
  const void* delta;
  const float* A_log;
  const void* B;
  const void* C;
  const float* h0;
  void* y;
  float* final_state;
  int64_t batch, L, D, N;
  int dtype;  // 0 f32, 1 bf16
  int disc;   // 0 euler, 1 zoh
  cudaStream_t stream;
  // optional layer pieces (all off: the plain scan)
  const float* delta_bias = nullptr;  // [D]
  int softplus = 0;                   // delta = softplus(delta + bias)
  const float* D_skip = nullptr;      // [D]
  const void* z = nullptr;            // [batch, L, D] (dtype): y = (y + D x) * SiLU(z)
};

struct StepArgs {
  float* state;
  const void* x;
  const void* delta;
  const float* A_log;
  const void* B;
  const void* C;
  void* y;
  int64_t batch, D, N;
  int dtype;
  int disc;
  cudaStream_t stream;
  const float* delta_bias = nullptr;  // [D]
  int softplus = 0;
  const float* D_skip = nullptr;      // [D]
  const void* z = nullptr;            // [batch, D] (dtype)
};

struct BwdArgs {
  const void* x;
  const void* delta;
  const float* A_log;
  const void* B;
  const void* C;
  const float* h0;      // or null
  const void* dy;
  const float* dfinal;  // or null
  void* dx;
  void* ddelta;
  float* dA_log;
  float* dB;
  float* dC;
  float* dh0;           // or null
  float* workspace;     // bwd_workspace_bytes() bytes
  int64_t batch, L, D, N;
  int dtype;
  int disc;
  cudaStream_t stream;
};

struct SsdArgs {
  const void* x;        // [batch, L, H, P] bf16
  const float* delta;   // [batch, L, H]
  const float* A_log;   // [H]
  const void* B;        // [batch, L, N] bf16
  const void* C;
  const float* h0;      // [batch, H, P, N] or null
  void* y;              // [batch, L, H, P] bf16
  float* final_state;   // [batch, H, P, N] or null
  void* workspace;      // ssd_workspace_bytes() bytes (tensor-core path or segmented scan), or null
  size_t workspace_bytes;
  int64_t batch, L, H, P, N;
  int disc;
  cudaStream_t stream;
};

int sm_count();  // multiprocessors of the current device (cached per device)
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // default bound on one consumer wait of a kernel (2 s)
uint64_t wait_limit_ns();                           // the current bound (ssm_set_wait_limit_ns)

cudaError_t launch_fwd_simple(const FwdArgs& a);
bool tma_path_ok(const FwdArgs& a);       // N == 16, 16-byte aligned rows and pointers, 32-bit row coords
cudaError_t launch_fwd_tma(const FwdArgs& a);
int read_and_clear_device_status();       // nonzero if a kernel recorded a failed bounded wait
cudaError_t launch_init_state(const FwdArgs& a);  // final_state = h0 or 0 (used when L == 0)
cudaError_t launch_step(const StepArgs& a);
size_t bwd_workspace_bytes(int64_t batch, int64_t L, int64_t D, int64_t N);
constexpr size_t kBwdNoAllocScratchBytes = size_t(64) << 20;  // the built-in scratch of ssm_scan_bwd_noalloc
cudaError_t bwd_noalloc_scratch(void** out);                     // its device address on the current device
cudaError_t launch_bwd(const BwdArgs& a);
bool ssd_shape_ok(int64_t P, int64_t N);  // N in {64, 128}, P a multiple of 16
size_t ssd_workspace_bytes(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N);  // current device
cudaError_t launch_ssd(const SsdArgs& a);
// The tensor-core (tcgen05) SSD path: P = 64, N = 64 or 128, L > 0, with a workspace of
// ssd_tc_workspace_bytes() (chunk states and the states entering each chunk).
size_t ssd_tc_workspace_bytes(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N);
bool ssd_tc_ok(const SsdArgs& a);
cudaError_t launch_ssd_tc(const SsdArgs& a);
int read_and_clear_ssd_status();  // nonzero if a kernel of that path recorded a failed bounded wait

}  // namespace ssm
