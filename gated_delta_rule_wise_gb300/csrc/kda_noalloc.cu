// kda_noalloc.cu -- kda_chunk_fwd for callers that cannot allocate device
// memory.
//
// Some callers have no way to provide a workspace: code that runs behind a
// plugin or host interface which hands it only its input and output buffers,
// or a serving loop that must not call cudaMalloc on its hot path because the
// call can synchronise the whole device and stall every stream.  For them
// this file holds the prefill's scratch (the per-chunk records that the prep
// kernel writes and the scan kernel reads, plus the device error word) in one
// fixed array that the library owns.  Every GPU that loads libkda keeps this
// array for the life of the process.
#include <mutex>

#include "kda_launch.cuh"

namespace {

// Fixed scratch for kda_chunk_fwd_noalloc: 64 MiB, including the 256-byte
// error header at its start.
constexpr size_t kNoallocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up once
// per device (the host-side name of the array is only a stand-in).
kda_status scratch_on_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                            const float *beta, const float *log_alpha,
                                            const float *h0, void *o, float *hT, int B, int H,
                                            int T, int dk, int dv, int C, kda_dtype dt,
                                            kda_alpha_mode am, kda_stream_t stream) {
  const size_t need = kda_chunk_fwd_workspace_size(B, H, T, dk, dv, C, dt, am);
  if (need == 0)  // invalid or unsupported: let the full check name which
    return kda_chunk_fwd(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, dt, am,
                         reinterpret_cast<void *>(256), 0, stream);
  if (need > kNoallocScratchBytes) return KDA_ERR_UNSUPPORTED;
  // every argument check of kda_chunk_fwd, made before anything is enqueued
  // (the scratch address stands in for the workspace: its only requirement,
  // 256-byte alignment, holds by declaration)
  const kda_status valid =
      kda::validate_chunk_fwd(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, dt, am,
                              reinterpret_cast<void *>(256), kNoallocScratchBytes, KDA_PATH_AUTO);
  if (valid != KDA_OK) return valid;
  void *scratch = nullptr;
  const kda_status st = scratch_on_current_device(&scratch);
  if (st != KDA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The error word must start at zero; the records are rewritten by every call.
  if (cudaMemsetAsync(scratch, 0, sizeof(kda::WorkspaceHeader), s) != cudaSuccess)
    return KDA_ERR_CUDA;
  return kda_chunk_fwd(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, dt, am, scratch,
                       kNoallocScratchBytes, stream);
}
