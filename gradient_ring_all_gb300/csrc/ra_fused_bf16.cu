// ra_fused_bf16.cu -- fused ring all-reduce kernels, bf16 gradients with
// binary32 accumulation.
#include "ra_fused_launch.cuh"

namespace ra {
cudaError_t launch_fused_bf16(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    return fused_launch_dtype<BF16>(L, ntiles, s);
}
}  // namespace ra
