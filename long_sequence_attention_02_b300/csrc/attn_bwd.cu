// Attention backward (placeholder until the tcgen05 backward lands).
#include "common.cuh"
#include "kernels.cuh"

namespace wan {

size_t attn_bwd_workspace_bytes(int B, int L, int H) {
  const size_t n = (size_t)B * L * H;
  return n * kHeadDim * 2 * 2 + n * kHeadDim * 4 + n * 4 + 1024;
}

int launch_attn_bwd(const void*, const void*, const void*, const void*, const float*, const void*, void*, void*,
                    void*, int, wan_grid_t, int, RopeTables, float, void*, const LaunchCommon&, cudaStream_t) {
  return WAN_ERR_UNSUPPORTED;
}

}  // namespace wan
