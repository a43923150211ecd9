// selftest.cu -- health check of the device-side failure detection: a bounded
// mbarrier wait that is never satisfied must give up, record
// RA_ERR_DEVICE_TIMEOUT in the status word and return, leaving the context
// usable.  The same wait primitive (ra::mbar_wait) guards every pipeline stage
// of the attention kernels.
#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {

static __device__ unsigned g_selftest_status[2];

namespace {

// One thread initialises an mbarrier that expects one arrival, never arrives,
// and waits for it for at most limit_ns.
__global__ void wait_timeout_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint32_t a = smem_u32(&bar);
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(a, 0)) {
        if (global_ns() - t0 > limit_ns) {
            atomicCAS(&g_selftest_status[0], 0u, kDevTimeout);
            atomicCAS(&g_selftest_status[1], 0u, 0x7F000000u);
            return;
        }
    }
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(unsigned long long limit_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 1, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

unsigned read_clear_status_selftest(unsigned* where) {
    unsigned h[2] = {0, 0};
    cudaMemcpyFromSymbol(h, g_selftest_status, sizeof h);
    if (h[0]) {
        const unsigned z[2] = {0, 0};
        cudaMemcpyToSymbol(g_selftest_status, z, sizeof z);
    }
    if (where) *where = h[1];
    return h[0];
}

}  // namespace ra
