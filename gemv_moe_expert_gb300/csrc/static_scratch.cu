// static_scratch.cu -- the GroupedPrefill expert-ID matmul for callers that
// cannot allocate device memory.
//
// The grouped route needs two scratch buffers (per-expert row counts and the
// per-expert lists of routed rows).  gbmm_matmul_id takes them from the
// caller.  Some callers have no way to provide them: a host that hands this
// library only the operands and outputs of each call and owns every other
// byte of device memory (a plugin slot in someone else's runtime), or a
// serving loop that must not call cudaMalloc once it is running, because an
// allocation can stall on a device-wide synchronisation.  For them,
// gbmm_matmul_id_static_scratch keeps the scratch in one fixed array that is
// part of this library's device image: it is reserved on every GPU that
// loads the library, for as long as the process lives, and nothing is
// allocated per call.
#include <cstdio>
#include <mutex>

#include "../../include/gbmm.h"
#include "kernel_params.h"

namespace gbmm {
int record_error(int status, const char *message);  // api.cu: sets gbmm_last_error()
}

namespace {

// counts: u32[GBMM_GROUPED_MAX_EXPERTS] at the start, routed rows after it
constexpr uint64_t kCountsBytes = static_cast<uint64_t>(GBMM_GROUPED_MAX_EXPERTS) * 4;
constexpr uint64_t kRoutedRowsBytes = GBMM_STATIC_SCRATCH_ROUTED_ROWS_BYTES;
constexpr uint64_t kScratchWords = (kCountsBytes + kRoutedRowsBytes) / 4;

static __device__ __align__(256) uint32_t g_static_scratch[kScratchWords];

std::mutex g_addr_mu;
uint32_t *g_addr[64] = {nullptr};

// Device address of g_static_scratch on the current device, looked up once
// per device.  In host code the array's name only stands for the device
// symbol; the kernels must be given the address the runtime reports.  The
// first lookup on a device also loads this part of the library there (lazy
// module loading), which reserves the array; the cached address is only
// valid while the device's primary context lives (not across a device reset).
gbmm_status scratch_address(uint32_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64)
        return static_cast<gbmm_status>(gbmm::record_error(
            GBMM_ERR_CUDA, "gbmm_matmul_id_static_scratch: no usable current device"));
    std::lock_guard<std::mutex> g(g_addr_mu);
    if (g_addr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            char msg[256];
            snprintf(msg, sizeof msg,
                     "gbmm_matmul_id_static_scratch: cannot resolve the static scratch on device %d: %s",
                     dev, cudaGetErrorString(e));
            return static_cast<gbmm_status>(gbmm::record_error(GBMM_ERR_CUDA, msg));
        }
        g_addr[dev] = static_cast<uint32_t *>(ptr);
    }
    *out = g_addr[dev];
    return GBMM_OK;
}

}  // namespace

extern "C" gbmm_status gbmm_matmul_id_static_scratch(const gbmm_matmul_id_params *p,
                                                     gbmm_dtype weight_dtype, const void *weights,
                                                     uint64_t weights_bytes, const float *input,
                                                     uint64_t input_bytes, const uint32_t *ids,
                                                     uint64_t ids_bytes, float *out,
                                                     uint64_t out_bytes, gbmm_stream stream,
                                                     gbmm_matmul_id_receipt *receipt) {
    if (p == nullptr)
        return static_cast<gbmm_status>(gbmm::record_error(
            GBMM_ERR_INVALID_ARGUMENT, "gbmm_matmul_id_static_scratch: params is null"));
    if (p->route != GBMM_ROUTE_GROUPED_PREFILL)
        return static_cast<gbmm_status>(gbmm::record_error(
            GBMM_ERR_INVALID_ARGUMENT,
            "gbmm_matmul_id_static_scratch: only the GroupedPrefill route uses scratch; "
            "call gbmm_matmul_id for the Direct route"));
    gbmm_matmul_id_capability_t cap;
    gbmm_status st = gbmm_matmul_id_capability(weight_dtype, p, &cap);
    if (st != GBMM_OK) return st;
    if (cap.expert_counts_bytes > kCountsBytes || cap.routed_rows_bytes > kRoutedRowsBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "gbmm_matmul_id_static_scratch: n_experts * m * 4 = %llu bytes of routed-row "
                 "scratch needed, the static scratch holds %llu (n_experts * m <= %llu); pass "
                 "caller-owned scratch to gbmm_matmul_id instead",
                 (unsigned long long)cap.routed_rows_bytes, (unsigned long long)kRoutedRowsBytes,
                 (unsigned long long)(kRoutedRowsBytes / 4));
        return static_cast<gbmm_status>(gbmm::record_error(GBMM_ERR_SCRATCH, msg));
    }

    uint32_t *base = nullptr;
    st = scratch_address(&base);
    if (st != GBMM_OK) return st;
    // Nothing in the array has to start at zero: the routing-map launch
    // rewrites every count and every list entry that the grouped launch reads.
    gbmm_matmul_id_scratch s;
    s.expert_counts = base;
    s.expert_counts_bytes = kCountsBytes;
    s.routed_rows = base + kCountsBytes / 4;
    s.routed_rows_bytes = kRoutedRowsBytes;
    s.max_experts = p->n_experts;
    s.max_tokens = p->m;
    return gbmm_matmul_id(p, weight_dtype, weights, weights_bytes, input, input_bytes, ids, ids_bytes,
                          out, out_bytes, &s, stream, receipt);
}

extern "C" gbmm_status gbmm_test_static_scratch_copy(void *dst, uint64_t bytes, gbmm_stream stream) {
    if (dst == nullptr || bytes > kScratchWords * 4)
        return static_cast<gbmm_status>(gbmm::record_error(
            GBMM_ERR_INVALID_ARGUMENT, "gbmm_test_static_scratch_copy: null destination or more bytes than the array"));
    uint32_t *base = nullptr;
    gbmm_status st = scratch_address(&base);
    if (st != GBMM_OK) return st;
    cudaError_t e = cudaMemcpyAsync(dst, base, bytes, cudaMemcpyDeviceToDevice,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return static_cast<gbmm_status>(gbmm::record_error(GBMM_ERR_CUDA, cudaGetErrorString(e)));
    return GBMM_OK;
}
