// bf16 instantiations of the mma.sync decode kernels.
#include "fd_kernel.cuh"

namespace fd {
cudaError_t launch_bf16_mma(const Params& p, int d, int G, int path, int mode, bool pdl, int grid,
                            cudaStream_t s) {
  return launch_typed_mma<__nv_bfloat16>(p, d, G, path, mode, pdl, grid, s);
}
}  // namespace fd
