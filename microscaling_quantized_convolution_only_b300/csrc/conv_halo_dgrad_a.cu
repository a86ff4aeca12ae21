// conv_halo_dgrad_a.cu -- instantiations of the halo-reuse dgrad convolution
// (conv_halo.cuh) whose fused requantization writes format 0 or 4 (0: none).
#include "conv_halo.cuh"

namespace mq {

cudaError_t halo_dispatch_dgrad_04(int fa, int fb, int fr, const CUtensorMap &a, const CUtensorMap &b,
                                   const HaloConv &h, int grid, cudaStream_t st) {
  if (fr == 0) return hc_dispatch<OP_DGRAD, 0>(fa, fb, a, b, h, grid, st);
  return hc_dispatch<OP_DGRAD, 4>(fa, fb, a, b, h, grid, st);
}

}  // namespace mq
