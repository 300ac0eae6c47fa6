// kda_chunk_tc.cu -- tensor-core (tcgen05) chunked prefill: not built yet.
#include "kda_launch.cuh"

namespace kda {

bool chunk_tc_supported(int, int, int, kda_dtype) { return false; }
size_t chunk_tc_workspace_bytes(int, int, int, int, int, int) { return 0; }
kda_status launch_chunk_tc(const void *, const void *, const void *, const float *,
                           const float *, const float *, void *, float *, int, int, int, int,
                           int, int, kda_alpha_mode, void *, size_t, cudaStream_t,
                           LaunchTimer &) {
  return KDA_ERR_UNSUPPORTED;
}
int chunk_tc_launches(int, int, bool) { return 0; }
const char *chunk_tc_kernel_name(int) { return nullptr; }

}  // namespace kda
