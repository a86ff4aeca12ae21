// conv_halo_wide.cu -- instantiations of the wide form of the halo-reuse
// forward / data-gradient convolution (conv_halo.cuh): one operand format f
// for input and weights, requantized output in format f or none.
#include "conv_halo.cuh"

namespace mq {

namespace {

template <int OP, int F>
cudaError_t wide_fr(int fr, const CUtensorMap &a, const CUtensorMap &b, const HaloConv &h, int grid,
                    cudaStream_t st) {
  return fr ? hc_launch_wide<OP, F, F>(a, b, h, grid, st) : hc_launch_wide<OP, F, 0>(a, b, h, grid, st);
}

template <int OP>
cudaError_t wide_f(int f, int fr, const CUtensorMap &a, const CUtensorMap &b, const HaloConv &h, int grid,
                   cudaStream_t st) {
  switch (f) {
    case 4: return wide_fr<OP, 4>(fr, a, b, h, grid, st);
    case 6: return wide_fr<OP, 6>(fr, a, b, h, grid, st);
    default: return wide_fr<OP, 8>(fr, a, b, h, grid, st);
  }
}

}  // namespace

cudaError_t halo_dispatch_wide(int op, int f, int fr, const CUtensorMap &a, const CUtensorMap &b, const HaloConv &h,
                               int grid, cudaStream_t st) {
  if (fr != 0 && fr != f) return cudaErrorInvalidValue;
  return op == OP_FWD ? wide_f<OP_FWD>(f, fr, a, b, h, grid, st) : wide_f<OP_DGRAD>(f, fr, a, b, h, grid, st);
}

}  // namespace mq
