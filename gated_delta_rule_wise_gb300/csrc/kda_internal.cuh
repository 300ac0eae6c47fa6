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

}  // namespace kda
