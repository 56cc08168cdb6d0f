// Failure-detection self-test: the bounded barrier wait that every kernel's
// waits share, run against an mbarrier that nothing ever completes.  The wait
// gives up after kWaitLimitNs, records its site in this module's status word
// and the kernel returns; nothing faults and the context stays usable.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace selftest {

__device__ int g_status;

__global__ void wait_timeout_kernel(int site) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);   // one arrival completes phase 0; none is ever made
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(&bar, 0u, &g_status, site);
}

}  // namespace selftest

cudaError_t launch_wait_timeout(int site, cudaStream_t stream) {
    selftest::wait_timeout_kernel<<<1, 32, 0, stream>>>(site);
    return cudaGetLastError();
}

int take_status_selftest() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, selftest::g_status, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(selftest::g_status, &z, sizeof(int));
    return v;
}

}  // namespace w4a16
