// pa_selftest.cu -- a fault-free exercise of the kernels' failure path: one
// CTA waits on a shared-memory barrier that nothing completes, with the same
// bounded wait the decode kernel uses, gives up and records the expiry in a
// device status word that pa_device_status reads like the kernels' own.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_selftest_status;

__global__ void selftest_wait_kernel(uint32_t polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0u, polls)) atomicOr(&g_selftest_status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t polls, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(polls);
    return cudaGetLastError();
}

uint32_t selftest_status(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_selftest_status, sizeof(v));
    if (clear) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_selftest_status, &z, sizeof(z));
    }
    return v;
}

}  // namespace pa
