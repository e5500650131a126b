// fp16 instantiations of the mma.sync decode kernels (16-bit and E4M3 K/V).
#include "fd_kernel.cuh"

namespace fd {
cudaError_t launch_f16_mma(const Params& p, int d, int G, int path, int mode, bool pdl, int grid,
                           cudaStream_t s) {
  return launch_typed_mma<__half>(p, d, G, path, mode, pdl, grid, s);
}
}  // namespace fd
