// bf16 instantiations of the small-M kernel (decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace w4a16 {
namespace decode {
cudaError_t launch_bf16(bool zp, int wpg, int nt, const CUtensorMap* maps, const Params& p,
                        int grid, size_t smem, cudaStream_t stream) {
    return launch_dtype<true>(zp, wpg, nt, maps, p, grid, smem, stream);
}
}  // namespace decode
}  // namespace w4a16
