// kda_api.cu -- the extern "C" boundary of libkda: argument checks, path
// choice, workspace layout and status reporting.  No kernel arithmetic here.
#include <stdint.h>

#include "kda_launch.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

inline bool is_pow2_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline bool valid_dtype(kda_dtype dt) { return dt == KDA_F32 || dt == KDA_BF16; }
inline bool valid_alpha(kda_alpha_mode am) {
  return am == KDA_ALPHA_NONE || am == KDA_ALPHA_SCALAR || am == KDA_ALPHA_CHANNEL;
}

// Shape / enum validation shared by the workspace query and the call.
kda_status check_chunk_shape(int B, int H, int T, int dk, int dv, int C, kda_dtype dt,
                             kda_alpha_mode am, kda_path path) {
  if (B < 0 || H < 0 || T < 0) return KDA_ERR_INVALID_ARG;
  if (!valid_dtype(dt) || !valid_alpha(am)) return KDA_ERR_INVALID_ARG;
  if (path != KDA_PATH_AUTO && path != KDA_PATH_CUDA_CORE && path != KDA_PATH_TENSOR &&
      path != KDA_PATH_TENSOR_SPLIT_SCAN && path != KDA_PATH_TENSOR_WIDE_SCAN &&
      path != KDA_PATH_TENSOR_PIPELINED)
    return KDA_ERR_INVALID_ARG;
  if (!is_pow2_dim(dk) || !is_pow2_dim(dv)) return KDA_ERR_UNSUPPORTED;
  if (C != 16 && C != 32 && C != 64) return KDA_ERR_UNSUPPORTED;
  if ((long long)B * H > 65535) return KDA_ERR_UNSUPPORTED;
  const bool tensor_only = path == KDA_PATH_TENSOR || path == KDA_PATH_TENSOR_SPLIT_SCAN ||
                           path == KDA_PATH_TENSOR_WIDE_SCAN || path == KDA_PATH_TENSOR_PIPELINED;
  if (tensor_only && !chunk_tc_supported(dk, dv, C, dt)) return KDA_ERR_UNSUPPORTED;
  if ((path == KDA_PATH_TENSOR_WIDE_SCAN || path == KDA_PATH_TENSOR_PIPELINED) && dk != 128)
    return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

bool use_tensor(int dk, int dv, int C, kda_dtype dt, kda_path path) {
  if (path == KDA_PATH_CUDA_CORE) return false;
  return chunk_tc_supported(dk, dv, C, dt);
}

// Scan choice handed to the tensor path: 0 automatic, 1 split, 2 wide,
// 3 pipelined.
int scan_choice(kda_path path) {
  switch (path) {
    case KDA_PATH_TENSOR_SPLIT_SCAN: return 1;
    case KDA_PATH_TENSOR_WIDE_SCAN: return 2;
    case KDA_PATH_TENSOR_PIPELINED: return 3;
    default: return 0;
  }
}

size_t workspace_bytes(int B, int H, int T, int dk, int dv, int C, kda_dtype dt,
                       kda_alpha_mode am, kda_path path) {
  if (check_chunk_shape(B, H, T, dk, dv, C, dt, am, path) != KDA_OK) return 0;
  size_t bytes = sizeof(WorkspaceHeader);
  if (use_tensor(dk, dv, C, dt, path)) bytes += chunk_tc_workspace_bytes(B, H, T, dk, dv, C);
  return bytes;
}

}  // namespace

kda_status validate_chunk_fwd(const void *q, const void *k, const void *v, const float *beta,
                              const float *log_alpha, const float *h0, const void *o,
                              const float *hT, int B, int H, int T, int dk, int dv, int C,
                              kda_dtype dt, kda_alpha_mode am, const void *workspace,
                              size_t ws_bytes, kda_path path) {
  kda_status st = check_chunk_shape(B, H, T, dk, dv, C, dt, am, path);
  if (st != KDA_OK) return st;
  const bool has_tokens = (long long)B * H * T > 0;
  if (has_tokens) {
    if (!q || !k || !v || !beta || !o) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(beta) || !aligned16(o))
      return KDA_ERR_INVALID_ARG;
  }
  if (am == KDA_ALPHA_NONE) {
    if (log_alpha) return KDA_ERR_INVALID_ARG;
  } else if (has_tokens && (!log_alpha || !aligned16(log_alpha))) {
    return KDA_ERR_INVALID_ARG;
  }
  if ((h0 && !aligned16(h0)) || (hT && !aligned16(hT))) return KDA_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace)) return KDA_ERR_INVALID_ARG;
  if (ws_bytes < workspace_bytes(B, H, T, dk, dv, C, dt, am, path)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

}  // namespace kda

using namespace kda;

extern "C" {

int kda_abi_version(void) { return KDA_ABI_VERSION; }

const char *kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported shape or mode";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA launch or runtime error";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: an on-device wait expired";
  }
  return "KDA status: unknown code";
}

size_t kda_chunk_fwd_workspace_size_ex(int B, int H, int T, int dk, int dv, int C, kda_dtype dt,
                                       kda_alpha_mode am, kda_path path) {
  return workspace_bytes(B, H, T, dk, dv, C, dt, am, path);
}

size_t kda_chunk_fwd_workspace_size(int B, int H, int T, int dk, int dv, int C, kda_dtype dt,
                                    kda_alpha_mode am) {
  return workspace_bytes(B, H, T, dk, dv, C, dt, am, KDA_PATH_AUTO);
}

int kda_chunk_fwd_launches(int B, int H, int T, int dk, int dv, int C, kda_dtype dt,
                           kda_alpha_mode am, kda_path path) {
  if (check_chunk_shape(B, H, T, dk, dv, C, dt, am, path) != KDA_OK) return -1;
  const int BH = B * H;
  // hT present is the worst case (an empty sequence still copies h0 -> hT)
  return use_tensor(dk, dv, C, dt, path) ? chunk_tc_launches(BH, T, true, dk, 0, scan_choice(path))
                                         : chunk_ffma_launches(BH, T, true);
}

const char *kda_chunk_fwd_kernel_name(int B, int H, int T, int dk, int dv, int C, kda_dtype dt,
                                      kda_alpha_mode am, kda_path path, int i) {
  if (check_chunk_shape(B, H, T, dk, dv, C, dt, am, path) != KDA_OK) return nullptr;
  if (i < 0 || i >= kda_chunk_fwd_launches(B, H, T, dk, dv, C, dt, am, path)) return nullptr;
  return use_tensor(dk, dv, C, dt, path) ? chunk_tc_kernel_name(B * H, T, dk, scan_choice(path), i)
                                         : chunk_ffma_kernel_name(i);
}

kda_status kda_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *beta,
                            const float *log_alpha, const float *h0, void *o, float *hT, int B,
                            int H, int T, int dk, int dv, int C, kda_dtype dt,
                            kda_alpha_mode am, void *workspace, size_t ws_bytes,
                            kda_stream_t stream, kda_path path, void *const *events,
                            int n_events) {
  kda_status st = validate_chunk_fwd(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, dt,
                                     am, workspace, ws_bytes, path);
  if (st != KDA_OK) return st;
  if (n_events < 0 || (n_events > 0 && !events)) return KDA_ERR_INVALID_ARG;
  const bool tensor = use_tensor(dk, dv, C, dt, path);
  const int launches = tensor ? chunk_tc_launches(B * H, T, hT != nullptr, dk, 0, scan_choice(path))
                              : chunk_ffma_launches(B * H, T, hT != nullptr);
  if (n_events > 0 && n_events < launches + 1) return KDA_ERR_INVALID_ARG;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  WorkspaceHeader *hdr = static_cast<WorkspaceHeader *>(workspace);
  if (launches == 0) return KDA_OK;
  LaunchTimer timer;
  timer.ev = events;
  timer.n = n_events;
  timer.s = s;
  if (tensor)
    return launch_chunk_tc(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, am,
                           workspace, ws_bytes, s, timer, 0, 0u, scan_choice(path));
  return launch_chunk_ffma(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, dt, am,
                           hdr, s, timer);
}

kda_status kda_chunk_fwd_rule(const void *q, const void *k, const void *v, const float *beta,
                              const float *log_alpha, const float *h0, void *o, float *hT, int B,
                              int H, int T, int dk, int dv, int C, kda_dtype dt,
                              kda_alpha_mode am, kda_rule rule, unsigned maps, void *workspace,
                              size_t ws_bytes, kda_stream_t stream) {
  const unsigned known = KDA_MAP_QK_SILU_NORM | KDA_MAP_BETA_SIGMOID | KDA_MAP_QK_ELU1;
  if (rule != KDA_RULE_DELTA && rule != KDA_RULE_LINEAR && rule != KDA_RULE_LINEAR_NORM)
    return KDA_ERR_INVALID_ARG;
  if ((maps & ~known) != 0u) return KDA_ERR_INVALID_ARG;
  if (rule != KDA_RULE_DELTA && (maps & KDA_MAP_BETA_SIGMOID)) return KDA_ERR_INVALID_ARG;
  if ((maps & KDA_MAP_QK_SILU_NORM) && (maps & KDA_MAP_QK_ELU1)) return KDA_ERR_INVALID_ARG;
  if (rule == KDA_RULE_DELTA && (maps & KDA_MAP_QK_ELU1)) return KDA_ERR_INVALID_ARG;
  if (rule == KDA_RULE_LINEAR_NORM && (h0 || hT)) return KDA_ERR_UNSUPPORTED;
  if (rule == KDA_RULE_DELTA && maps == 0u)
    return kda_chunk_fwd_ex(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, dt, am,
                            workspace, ws_bytes, stream, KDA_PATH_AUTO, nullptr, 0);
  // everything else: the d = 128 tensor path
  kda_status st = check_chunk_shape(B, H, T, dk, dv, C, dt, am, KDA_PATH_TENSOR);
  if (st != KDA_OK) return st;
  if (dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
  const bool has_tokens = (long long)B * H * T > 0;
  const bool need_beta = rule == KDA_RULE_DELTA;
  if (has_tokens) {
    if (!q || !k || !v || !o || (need_beta && !beta)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (beta && !aligned16(beta)))
      return KDA_ERR_INVALID_ARG;
  }
  if (am == KDA_ALPHA_NONE) {
    if (log_alpha) return KDA_ERR_INVALID_ARG;
  } else if (has_tokens && (!log_alpha || !aligned16(log_alpha))) {
    return KDA_ERR_INVALID_ARG;
  }
  if ((h0 && !aligned16(h0)) || (hT && !aligned16(hT))) return KDA_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace)) return KDA_ERR_INVALID_ARG;
  if (ws_bytes < workspace_bytes(B, H, T, dk, dv, C, dt, am, KDA_PATH_TENSOR))
    return KDA_ERR_INVALID_ARG;
  if (chunk_tc_launches(B * H, T, hT != nullptr, dk, (int)rule, 0) == 0) return KDA_OK;
  LaunchTimer timer;
  timer.s = reinterpret_cast<cudaStream_t>(stream);
  return launch_chunk_tc(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, am, workspace,
                         ws_bytes, timer.s, timer, (int)rule, maps);
}

kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const float *beta,
                         const float *log_alpha, const float *h0, void *o, float *hT, int B,
                         int H, int T, int dk, int dv, int C, kda_dtype dt, kda_alpha_mode am,
                         void *workspace, size_t ws_bytes, kda_stream_t stream) {
  return kda_chunk_fwd_ex(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, dt, am,
                          workspace, ws_bytes, stream, KDA_PATH_AUTO, nullptr, 0);
}

kda_status kda_chunk_fwd_status(void *workspace, kda_stream_t stream) {
  if (!workspace || !aligned256(workspace)) return KDA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
  WorkspaceHeader h;
  if (cudaMemcpy(&h, workspace, 2 * sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (h.err == 0) return KDA_OK;
  if (cudaMemset(workspace, 0, 2 * sizeof(unsigned)) != cudaSuccess) return KDA_ERR_CUDA;
  return h.err == KDA_ERR_TIMEOUT ? KDA_ERR_TIMEOUT : KDA_ERR_CUDA;
}

kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *beta,
                           const float *log_alpha, float *S_inout, void *o, int N, int H,
                           int dk, int dv, kda_dtype dt, kda_alpha_mode am,
                           kda_stream_t stream) {
  if (N < 0 || H < 0 || !valid_dtype(dt) || !valid_alpha(am)) return KDA_ERR_INVALID_ARG;
  if (!is_pow2_dim(dk) || !is_pow2_dim(dv)) return KDA_ERR_UNSUPPORTED;
  if ((long long)N * H == 0) return KDA_OK;
  if (!q || !k || !v || !beta || !S_inout || !o) return KDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(beta) ||
      !aligned16(S_inout) || !aligned16(o))
    return KDA_ERR_INVALID_ARG;
  if (am == KDA_ALPHA_NONE) {
    if (log_alpha) return KDA_ERR_INVALID_ARG;
  } else if (!log_alpha || !aligned16(log_alpha)) {
    return KDA_ERR_INVALID_ARG;
  }
  return launch_decode(q, k, v, beta, log_alpha, S_inout, o, N, H, dk, dv, dt, am,
                       reinterpret_cast<cudaStream_t>(stream));
}

kda_status kda_selftest_wait_timeout(void *workspace, size_t ws_bytes, unsigned spin_limit,
                                     kda_stream_t stream) {
  if (!workspace || !aligned256(workspace) || ws_bytes < sizeof(WorkspaceHeader))
    return KDA_ERR_INVALID_ARG;
  if (spin_limit < 1 || spin_limit > (1u << 20)) return KDA_ERR_INVALID_ARG;
  return launch_selftest_wait(static_cast<WorkspaceHeader *>(workspace), spin_limit,
                              reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
