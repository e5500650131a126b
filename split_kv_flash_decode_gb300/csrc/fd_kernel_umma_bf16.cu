// bf16 instantiations of the tcgen05 (fifth-generation tensor core) decode kernels.
#include "fd_kernel.cuh"

namespace fd {
cudaError_t launch_umma_bf16(const Params& p, int d, int G, int mode, bool pdl, int grid,
                         cudaStream_t s) {
  return launch_typed_umma<__nv_bfloat16>(p, d, G, mode, pdl, grid, s);
}
}  // namespace fd
