// ra_fused_f32.cu -- fused ring all-reduce kernels, binary32 gradients.
#include "ra_fused_launch.cuh"

namespace ra {
cudaError_t launch_fused_f32(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    return fused_launch_dtype<F32>(L, ntiles, s);
}
}  // namespace ra
