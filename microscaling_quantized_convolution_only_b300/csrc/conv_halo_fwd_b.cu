// conv_halo_fwd_b.cu -- instantiations of the halo-reuse fwd convolution
// (conv_halo.cuh) whose fused requantization writes format 6 or 8 (0: none).
#include "conv_halo.cuh"

namespace mq {

cudaError_t halo_dispatch_fwd_68(int fa, int fb, int fr, const CUtensorMap &a, const CUtensorMap &b,
                                   const HaloConv &h, int grid, cudaStream_t st) {
  if (fr == 6) return hc_dispatch<OP_FWD, 6>(fa, fb, a, b, h, grid, st);
  return hc_dispatch<OP_FWD, 8>(fa, fb, a, b, h, grid, st);
}

}  // namespace mq
