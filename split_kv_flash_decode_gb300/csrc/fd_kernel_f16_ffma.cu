// fp16 instantiations of the CUDA-core decode kernels.
#include "fd_kernel.cuh"

namespace fd {
cudaError_t launch_f16_ffma(const Params& p, int d, int G, int mode, bool pdl, int grid,
                            cudaStream_t s) {
  return launch_typed_ffma<__half>(p, d, G, mode, pdl, grid, s);
}
}  // namespace fd
