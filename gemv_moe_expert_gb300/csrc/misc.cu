// misc.cu -- the device error word and the kernel that exercises the
// bounded-wait timeout path.
#include "device_common.cuh"

namespace gbmm {

// Set (never trapped on) by kernels whose bounded mbarrier wait ran out.
__device__ uint32_t g_device_error_word;

namespace {

__global__ void bounded_wait_test_kernel(uint32_t *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing ever arrives on this barrier: phase 0 never completes
        if (!mbar_wait_bounded(smem_addr(&bar), 0, limit_ns, nullptr))
            report_device_error(err, kKidBoundedWaitTest);
    }
}

}  // namespace

uint32_t *device_error_word() {
    static uint32_t *cached[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (cached[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_error_word) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<uint32_t *>(ptr);
    }
    return cached[dev];
}

int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cached[dev] == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 1;
    }
    return cached[dev];
}

cudaError_t launch_bounded_wait_test(uint32_t *err, uint64_t limit_ns, cudaStream_t s) {
    bounded_wait_test_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace gbmm
