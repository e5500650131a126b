// fp16 instantiations of the split-KV Flash Decode kernels.
#include "fd_kernel.cuh"

namespace fd {
cudaError_t launch_f16(const Params& p, int d, int G, int path, int mode, bool pdl, int grid,
                       cudaStream_t s) {
  return launch_typed<__half>(p, d, G, path, mode, pdl, grid, s);
}
}  // namespace fd
