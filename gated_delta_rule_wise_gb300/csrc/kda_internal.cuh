// kda_internal.cuh -- device helpers shared by the libkda kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// First 256 bytes of every kda_chunk_fwd workspace.
struct WorkspaceHeader {
  unsigned int err;    // 0 = fine, else a kda_status value
  unsigned int where;  // kernel-specific code of the wait that gave up
  unsigned int pad[62];
};
static_assert(sizeof(WorkspaceHeader) == 256, "header must stay 256 bytes");

// Record a device-side failure (first writer wins).
__device__ __forceinline__ void report_error(WorkspaceHeader *hdr, unsigned code,
                                             unsigned where) {
  if (hdr && atomicCAS(&hdr->err, 0u, code) == 0u) hdr->where = where;
}

template <typename T> struct Io;
template <> struct Io<float> {
  static __device__ __forceinline__ float ld(const float *p) { return *p; }
  static __device__ __forceinline__ void st(float *p, float x) { *p = x; }
};
template <> struct Io<__nv_bfloat16> {
  static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
  }
  static __device__ __forceinline__ void st(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
  }
};

// Per-step multiplicative decay a = exp(-exp(log_alpha)).
__device__ __forceinline__ float decay_of(float log_alpha) { return expf(-expf(log_alpha)); }
// log(a) = -exp(log_alpha): what the chunked form accumulates.
__device__ __forceinline__ float log_decay_of(float log_alpha) { return -expf(log_alpha); }

// Records caller-provided CUDA events around a call's kernel launches:
// mark() before launch i records events[i]; a final mark() after the last
// launch records events[launches].  No events: marks do nothing.
struct LaunchTimer {
  void *const *ev = nullptr;
  int n = 0;
  cudaStream_t s = nullptr;
  int next = 0;
  void mark() {
    if (ev && next < n) cudaEventRecord(static_cast<cudaEvent_t>(ev[next]), s);
    ++next;
  }
};

}  // namespace kda

// Host-side launchers, one per translation unit (C++ linkage, internal to libkda).
namespace kda {
kda_status launch_decode(const void *q, const void *k, const void *v, const float *beta,
                         const float *log_alpha, float *S, void *o, int N, int H, int dk,
                         int dv, kda_dtype dt, kda_alpha_mode am, cudaStream_t stream);
kda_status launch_chunk_ffma(const void *q, const void *k, const void *v, const float *beta,
                             const float *log_alpha, const float *h0, void *o, float *hT,
                             int B, int H, int T, int dk, int dv, int C, kda_dtype dt,
                             kda_alpha_mode am, WorkspaceHeader *hdr, cudaStream_t stream,
                             LaunchTimer &timer);
// Kernel launches a chunk call makes on each path, and their names.
int chunk_ffma_launches(int BH, int T, bool has_hT);
const char *chunk_ffma_kernel_name(int i);
int chunk_tc_launches(int BH, int T, bool has_hT);
const char *chunk_tc_kernel_name(int i);
bool chunk_tc_supported(int dk, int dv, int C, kda_dtype dt);
size_t chunk_tc_workspace_bytes(int B, int H, int T, int dk, int dv, int C);
kda_status launch_chunk_tc(const void *q, const void *k, const void *v, const float *beta,
                           const float *log_alpha, const float *h0, void *o, float *hT,
                           int B, int H, int T, int dk, int dv, int C, kda_alpha_mode am,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream,
                           LaunchTimer &timer);
kda_status launch_selftest_wait(WorkspaceHeader *hdr, unsigned spin_limit,
                                cudaStream_t stream);
}  // namespace kda
