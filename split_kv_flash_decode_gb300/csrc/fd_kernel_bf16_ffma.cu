// bf16 instantiations of the CUDA-core decode kernels.
#include "fd_kernel.cuh"

namespace fd {
cudaError_t launch_bf16_ffma(const Params& p, int d, int G, int mode, bool pdl, int grid,
                             cudaStream_t s) {
  return launch_typed_ffma<__nv_bfloat16>(p, d, G, mode, pdl, grid, s);
}
}  // namespace fd
