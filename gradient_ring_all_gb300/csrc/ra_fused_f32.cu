// ra_fused_f32.cu -- fused ring all-reduce kernels, binary32 gradients.
#include "ra_fused_launch.cuh"

namespace ra {
cudaError_t launch_fused_f32(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    return fused_launch_dtype<F32>(L, ntiles, s);
}

// A wait that cannot end: an mbarrier expecting 16 bytes that no copy will
// deliver.  The bounded wait gives up after limit_ns, records the error and
// returns -- the library's self-test of the timeout path.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, unsigned int *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_addr(&bar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], 16;" :: "r"(smem_addr(&bar)) : "memory");
    }
    __syncthreads();
    if (!mbar_wait_bounded(smem_addr(&bar), 0, limit_ns) && threadIdx.x == 0) atomicOr(err, 1u);
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned int *err, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, err);
    return cudaGetLastError();
}
}  // namespace ra
