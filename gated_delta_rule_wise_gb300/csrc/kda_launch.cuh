// kda_launch.cuh -- host-side launchers of libkda's kernels (C++ linkage,
// internal to the library) and the launch timer used by kda_chunk_fwd_ex.
#pragma once

#include "kda_internal.cuh"

namespace kda {

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
// Launches of a tensor-path call: 2 (prep, scan), 1 for an empty sequence
// with a final state, 2 per segment when the call is pipelined.
int chunk_tc_launches(int BH, int T, bool has_hT, int dk, int rule, int scan);
// Segments of a call: 1, or G > 1 when the prep of each segment overlaps the
// scan of the one before (d = 128; scan = 3 requests it).
int chunk_tc_segments(int BH, int T, int dk, int rule, int scan);
// scan: 0 automatic, 1 the value-column split scan, 2 the one-CTA-per-head
// scan (d = 128 only; not for the normalised linear-attention rule), 3 the
// pipelined call (d = 128, same restriction).
bool chunk_tc_wide_scan(int BH, int dk, int rule, int scan);
const char *chunk_tc_kernel_name(int BH, int T, int dk, int scan, int i);
bool chunk_tc_supported(int dk, int dv, int C, kda_dtype dt);
size_t chunk_tc_workspace_bytes(int B, int H, int T, int dk, int dv, int C);
// rule: KDA_RULE_DELTA / KDA_RULE_LINEAR; maps: KDA_MAP_* bits (both other
// than 0 only for dk = dv = 128).
kda_status launch_chunk_tc(const void *q, const void *k, const void *v, const float *beta,
                           const float *log_alpha, const float *h0, void *o, float *hT,
                           int B, int H, int T, int dk, int dv, int C, kda_alpha_mode am,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream,
                           LaunchTimer &timer, int rule = 0, unsigned maps = 0, int scan = 0);
kda_status launch_selftest_wait(WorkspaceHeader *hdr, unsigned spin_limit,
                                cudaStream_t stream);
// Every check kda_chunk_fwd_ex makes before it launches anything (shapes,
// enums, pointers, alignment, workspace size); KDA_OK if a call with these
// arguments would launch.
kda_status validate_chunk_fwd(const void *q, const void *k, const void *v, const float *beta,
                              const float *log_alpha, const float *h0, const void *o,
                              const float *hT, int B, int H, int T, int dk, int dv, int C,
                              kda_dtype dt, kda_alpha_mode am, const void *workspace,
                              size_t ws_bytes, kda_path path);
}  // namespace kda
