// gemv.cu -- matrix x vector kernels (m == 1 or n == 1) and the skinny "wide"
// path (2..15 rows of A against B stored [n, k]), plus the zero fill used
// when k == 0.
//
// Semantics: tract-metal 0.23.6, src/kernels/matmul/mlx_gemm/mod.rs,
// `dispatch_metal_mlx_gemv` (which operand is the matrix, its leading dim
// and transposition) and `dispatch_metal_mlx_gemv_wide` (c = a b^T for a few
// rows of a).  The Metal tile heuristics there are not used.
//
// Two orientations:
//   rowdot -- each output is a dot product along a contiguous matrix row.
//             One warp per output row: lanes read consecutive 16-byte
//             vectors (coalesced 512-byte warp requests, L1 bypassed since
//             every matrix byte is used once), accumulate in f32, then a
//             warp-shuffle reduction.  Up to 16 vectors share one pass over
//             the matrix (register tile of vector rows).
//   coldot -- the matrix is contiguous along the outputs.  A thread owns one
//             16-byte vector of consecutive outputs and walks the
//             contraction dim; 8 warps split k inside the CTA and, when the
//             output tiles alone cannot fill the GPU, a thread-block cluster
//             of up to 8 CTAs splits k further and reduces the partial sums
//             through distributed shared memory (no scratch, no atomics).
#include <cooperative_groups.h>

#include "device_common.cuh"

namespace cg = cooperative_groups;

namespace gbmm {

namespace {

constexpr int kRowdotThreads = 256;
constexpr int kRowdotUnroll = 8;  // 16-byte vectors in flight per lane per row

template <typename T, int NV>
__global__ void __launch_bounds__(kRowdotThreads)
gemv_rowdot_kernel(GemvParams p) {
    constexpr int V = Elem<T>::kVec;
    const int lane = threadIdx.x & 31;
    const int64_t warps_per_block = blockDim.x >> 5;
    const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * warps_per_block;
    const int nvec = p.nvec;

    for (int64_t bat = blockIdx.y; bat < p.batch; bat += gridDim.y) {
        const T *mat = static_cast<const T *>(p.mat) + bat * p.mat_bs;
        const T *vec = static_cast<const T *>(p.vec) + bat * p.vec_bs;
        T *out = static_cast<T *>(p.out) + bat * p.out_bs;

        for (int64_t row = gwarp; row < p.rows; row += nwarps) {
            float acc[NV];
#pragma unroll
            for (int r = 0; r < NV; ++r) acc[r] = 0.f;
            const T *mrow = mat + row * p.mat_rs;

            if (p.vec_ok) {
                // groups of kU 16-byte vectors per lane, all loads of a group issued
                // before any use (the last group is predicated, not split off)
                constexpr int kU = NV <= 2 ? 2 * kRowdotUnroll : kRowdotUnroll;
                const int64_t nch = p.k / V;
                for (int64_t c0 = 0; c0 < nch; c0 += 32 * kU) {
                    uint4 w[kU];
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int64_t c = c0 + u * 32 + lane;
                        w[u] = c < nch ? ld_stream16(mrow + c * V) : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int64_t c = c0 + u * 32 + lane;
                        if (c < nch) {
                            float wf[V];
                            unpack16<T>(w[u], wf);
#pragma unroll
                            for (int r = 0; r < NV; ++r) {
                                if (r < nvec) {
                                    float xf[V];
                                    unpack16<T>(ld_cached16(vec + r * p.vec_rr + c * V), xf);
#pragma unroll
                                    for (int i = 0; i < V; ++i) acc[r] = fmaf(wf[i], xf[i], acc[r]);
                                }
                            }
                        }
                    }
                }
                for (int64_t x = nch * V + lane; x < p.k; x += 32) {
                    const float wv = Elem<T>::to_f(mrow[x]);
#pragma unroll
                    for (int r = 0; r < NV; ++r)
                        if (r < nvec) acc[r] = fmaf(wv, Elem<T>::to_f(vec[r * p.vec_rr + x]), acc[r]);
                }
            } else {
                for (int64_t x = lane; x < p.k; x += 32) {
                    const float wv = Elem<T>::to_f(mrow[x * p.mat_ks]);
#pragma unroll
                    for (int r = 0; r < NV; ++r)
                        if (r < nvec)
                            acc[r] = fmaf(wv, Elem<T>::to_f(vec[r * p.vec_rr + x * p.vec_ks]), acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < NV; ++r) acc[r] = warp_sum(acc[r]);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < NV; ++r)
                    if (r < nvec) out[r * p.out_rr + row * p.out_os] = Elem<T>::from_f(acc[r]);
            }
        }
    }
}

constexpr int kColdotThreads = 256;  // 32 output vectors x 8 k-slices

template <typename T>
__global__ void __launch_bounds__(kColdotThreads)
gemv_coldot_kernel(GemvParams p, int ksplit) {
    constexpr int V = Elem<T>::kVec;
    constexpr int TILE = 32 * V;
    __shared__ float red[8][TILE];
    __shared__ float part[TILE];

    const int tx = threadIdx.x & 31;
    const int ty = threadIdx.x >> 5;
    const int64_t tile = blockIdx.x / ksplit;
    const int rank = blockIdx.x % ksplit;  // == rank in the cluster (cluster dims = ksplit)
    const int64_t o0 = tile * TILE + tx * V;
    // contraction range of this CTA
    const int64_t kper = (p.k + ksplit - 1) / ksplit;
    const int64_t kbeg = rank * kper;
    const int64_t kend = kbeg + kper < p.k ? kbeg + kper : p.k;

    for (int64_t bat = blockIdx.y; bat < p.batch; bat += gridDim.y) {
        const T *mat = static_cast<const T *>(p.mat) + bat * p.mat_bs;
        const T *vec = static_cast<const T *>(p.vec) + bat * p.vec_bs;
        T *out = static_cast<T *>(p.out) + bat * p.out_bs;

        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;

        if (p.vec_ok && o0 + V <= p.rows) {
            int64_t x = kbeg + ty;
            for (; x + 24 < kend; x += 32) {
                uint4 w[4];
                float v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    w[u] = ld_stream16(mat + (x + 8 * u) * p.mat_ks + o0);
                    v[u] = Elem<T>::to_f(vec[(x + 8 * u) * p.vec_ks]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float wf[V];
                    unpack16<T>(w[u], wf);
#pragma unroll
                    for (int i = 0; i < V; ++i) acc[i] = fmaf(wf[i], v[u], acc[i]);
                }
            }
            for (; x < kend; x += 8) {
                float wf[V];
                unpack16<T>(ld_stream16(mat + x * p.mat_ks + o0), wf);
                const float v = Elem<T>::to_f(vec[x * p.vec_ks]);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] = fmaf(wf[i], v, acc[i]);
            }
        } else {
            for (int64_t x = kbeg + ty; x < kend; x += 8) {
                const float v = Elem<T>::to_f(vec[x * p.vec_ks]);
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    const int64_t o = o0 + i;
                    if (o < p.rows) acc[i] = fmaf(Elem<T>::to_f(mat[x * p.mat_ks + o * p.mat_rs]), v, acc[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < V; ++i) red[ty][tx * V + i] = acc[i];
        __syncthreads();
        for (int c = threadIdx.x; c < TILE; c += blockDim.x) {
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) s += red[j][c];
            part[c] = s;
        }
        if (ksplit > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();  // every CTA's partial sums are visible cluster-wide
            if (rank == 0) {
                for (int c = threadIdx.x; c < TILE; c += blockDim.x) {
                    float s = part[c];
                    for (int q = 1; q < ksplit; ++q) s += cluster.map_shared_rank(part, q)[c];
                    const int64_t o = tile * TILE + c;
                    if (o < p.rows) out[o * p.out_os] = Elem<T>::from_f(s);
                }
            }
            cluster.sync();  // keep the other CTAs' shared memory alive until read
        } else {
            __syncthreads();
            for (int c = threadIdx.x; c < TILE; c += blockDim.x) {
                const int64_t o = tile * TILE + c;
                if (o < p.rows) out[o * p.out_os] = Elem<T>::from_f(part[c]);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// coldot, staged: the same column-dot GEMV with the matrix streamed by TMA.
// The register-fed kernel above keeps four 16-byte loads in flight per
// thread (~37 KB per SM), far fewer bytes than HBM's latency needs, and its
// long-scoreboard stalls set its pace.  Here a producer warp copies boxes of
// 512 bytes of outputs x 64 k rows (32 KB) into a two-stage shared-memory
// ring (three CTAs per SM, so the decode shape's 43 tiles x 8-way k split run
// in one wave), so the bytes in flight no longer depend on registers; 8 consumer
// warps reduce each stage (a thread owns 16 bytes of outputs, warp w rows
// w, w + 8, ... of the stage), then the warps' partial sums are added in
// shared memory and, with a k split, across the cluster through distributed
// shared memory in rank order.  Every wait is bounded.
// ---------------------------------------------------------------------------

constexpr int kCsWarps = 8;                 // consumer warps
constexpr int kCsThreads = (kCsWarps + 1) * 32;
constexpr int kCsRows = 64;                 // k rows per stage
constexpr uint32_t kCsRowBytes = 512;       // one 16-byte vector per consumer lane
constexpr int kCsStages = 2;
constexpr uint32_t kCsStageBytes = kCsRows * kCsRowBytes;
constexpr uint32_t kCsSmem = kCsStages * kCsStageBytes + 2 * kCsStages * 8 + 16 + 1024;
static_assert(kCsWarps * kCsRowBytes / 2 * 4 <= kCsStages * kCsStageBytes,
              "the warps' partial sums fit in the drained ring");

template <typename T>
__global__ void __launch_bounds__(kCsThreads, 3)
gemv_coldot_stream_kernel(const __grid_constant__ CUtensorMap map, const GemvParams p, int ksplit) {
    constexpr int V = Elem<T>::kVec;
    constexpr int TW = kCsRowBytes / sizeof(T);  // outputs per tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t s0 = raw + pad;
    const uint32_t bar0 = s0 + kCsStages * kCsStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kCsStages + s); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kCsStages * kCsStageBytes + 2 * kCsStages * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t tile = blockIdx.x / ksplit;
    const int rank = static_cast<int>(blockIdx.x % ksplit);  // == rank in the cluster (cluster dims = ksplit)
    const int64_t kbt = (p.k + kCsRows - 1) / kCsRows;
    const int64_t kb0 = kbt * rank / ksplit, kb1 = kbt * (rank + 1) / ksplit;
    const uint64_t lim = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kCsStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kCsWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kCsWarps && lane == 0) tma_prefetch_desc(&map);
    __syncthreads();

    float acc[V];
    for (int64_t bat = blockIdx.y; bat < p.batch; bat += gridDim.y) {
        // every stage of the previous batch item was consumed before this one's fills
        const int64_t it0 = (bat - blockIdx.y) / gridDim.y * (kb1 - kb0);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        if (warp == kCsWarps) {
            if (lane == 0) {
                // ---------------- producer ----------------
                int64_t it = it0;
                bool ok = true;
                for (int64_t kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = static_cast<int>(it % kCsStages);
                    const uint32_t use = static_cast<uint32_t>(it / kCsStages);
                    if (use > 0 && !mbar_wait_bounded(empty_bar(s), (use - 1u) & 1u, lim, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), kCsStageBytes);
                    tma_load_3d(s0 + s * kCsStageBytes, &map, full_bar(s), static_cast<int32_t>(tile * TW),
                                static_cast<int32_t>(kb * kCsRows), static_cast<int32_t>(bat));
                }
                if (!ok) {
                    *abort_flag = 1;
                    report_device_error(p.err, kKidGemvColdotStream);
                    // this thread's copies still in flight: its last kCsStages fills at most
                    for (int64_t j = it - 1; j >= it0 && j >= it - kCsStages; --j)
                        mbar_wait_bounded(full_bar(static_cast<int>(j % kCsStages)),
                                          static_cast<uint32_t>(j / kCsStages) & 1u, lim, nullptr);
                }
            }
        } else {
            // ---------------- consumers ----------------
            const T *vec = static_cast<const T *>(p.vec) + bat * p.vec_bs;
            int64_t it = it0;
            for (int64_t kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = static_cast<int>(it % kCsStages);
                int ready = 0;
                if (lane == 0)
                    ready = mbar_wait_bounded(full_bar(s), static_cast<uint32_t>(it / kCsStages) & 1u, lim, abort_flag);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (!ready) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_device_error(p.err, kKidGemvColdotStream);
                    }
                    break;
                }
                const uint4 *st = reinterpret_cast<const uint4 *>(smem + s * kCsStageBytes);
#pragma unroll
                for (int r = warp; r < kCsRows; r += kCsWarps) {
                    const int64_t x = kb * kCsRows + r;
                    // rows past k were zero-filled by the copy; their vector entry is not read
                    const float v = x < p.k ? Elem<T>::to_f(vec[x * p.vec_ks]) : 0.f;
                    float wf[V];
                    unpack16<T>(st[r * (kCsRowBytes / 16) + lane], wf);
#pragma unroll
                    for (int i = 0; i < V; ++i) acc[i] = fmaf(wf[i], v, acc[i]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
            }
        }
        // every stage of this batch item is consumed (or the CTA aborted): the
        // ring is free for the partial sums of the warps
        __syncthreads();
        float *red = reinterpret_cast<float *>(smem);  // [kCsWarps][TW]
        if (warp < kCsWarps) {
#pragma unroll
            for (int i = 0; i < V; ++i) red[warp * TW + lane * V + i] = acc[i];
        }
        __syncthreads();
        float *part = red + kCsWarps * TW;  // [TW]: this CTA's sums
        for (int c = threadIdx.x; c < TW; c += blockDim.x) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kCsWarps; ++w) sum += red[w * TW + c];
            part[c] = sum;
        }
        T *out = static_cast<T *>(p.out) + bat * p.out_bs;
        if (ksplit > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();  // every CTA's partial sums are visible cluster-wide
            if (rank == 0) {
                for (int c = threadIdx.x; c < TW; c += blockDim.x) {
                    float sum = part[c];
                    for (int q = 1; q < ksplit; ++q) sum += cluster.map_shared_rank(part, q)[c];
                    const int64_t o = tile * TW + c;
                    if (o < p.rows) out[o * p.out_os] = Elem<T>::from_f(sum);
                }
            }
            cluster.sync();  // keep the other CTAs' shared memory alive until read
        } else {
            __syncthreads();
            for (int c = threadIdx.x; c < TW; c += blockDim.x) {
                const int64_t o = tile * TW + c;
                if (o < p.rows) out[o * p.out_os] = Elem<T>::from_f(part[c]);
            }
        }
        __syncthreads();
    }
}

template <typename T>
__global__ void fill_zero_kernel(T *c, int64_t batch, int64_t m, int64_t n, int64_t ldc, int64_t sc) {
    const int64_t total = batch * m * n;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < total;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = q / (m * n);
        const int64_t r = q % (m * n);
        c[b * sc + (r / n) * ldc + (r % n)] = Elem<T>::from_f(0.f);
    }
}

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 1;
    }
    return cached[dev];
}

template <typename T, int NV>
cudaError_t rowdot_nv(const GemvParams &p, cudaStream_t s) {
    const int64_t warps = kRowdotThreads / 32;
    int64_t blocks = (p.rows + warps - 1) / warps;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const unsigned gy = static_cast<unsigned>(p.batch < 65535 ? p.batch : 65535);
    gemv_rowdot_kernel<T, NV><<<dim3(static_cast<unsigned>(blocks), gy), kRowdotThreads, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t rowdot_t(const GemvParams &p, cudaStream_t s) {
    if (p.nvec <= 1) return rowdot_nv<T, 1>(p, s);
    if (p.nvec <= 2) return rowdot_nv<T, 2>(p, s);
    if (p.nvec <= 4) return rowdot_nv<T, 4>(p, s);
    if (p.nvec <= 8) return rowdot_nv<T, 8>(p, s);
    return rowdot_nv<T, 16>(p, s);
}

template <typename T>
cudaError_t coldot_t(const GemvParams &p, cudaStream_t s) {
    constexpr int TILE = 32 * Elem<T>::kVec;
    const int64_t tiles = (p.rows + TILE - 1) / TILE;
    const int64_t bgrid = p.batch < 65535 ? p.batch : 65535;
    // split k over a cluster when the output tiles cannot fill the GPU
    int ksplit = 1;
    while (ksplit < 8 && tiles * bgrid * ksplit < 2LL * num_sms() && p.k >= 512LL * ksplit * 2)
        ksplit *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * ksplit), static_cast<unsigned>(bgrid), 1);
    cfg.blockDim = dim3(kColdotThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ksplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_coldot_kernel<T>, p, ksplit);
}

template <typename T>
cudaError_t coldot_stream_t(const CUtensorMap &map, const GemvParams &p, cudaStream_t s) {
    constexpr int TW = kCsRowBytes / sizeof(T);
    const int64_t tiles = (p.rows + TW - 1) / TW;
    const int64_t bgrid = p.batch < 65535 ? p.batch : 65535;
    const int64_t kbt = (p.k + kCsRows - 1) / kCsRows;
    // split k over a cluster (at most 8) until the grid holds two CTAs per SM,
    // keeping at least four k-blocks per CTA
    int ksplit = 1;
    while (ksplit < 8 && tiles * bgrid * ksplit < 2LL * num_sms() && kbt >= 4LL * ksplit * 2) ksplit *= 2;
    static unsigned long long attr_set = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemv_coldot_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kCsSmem);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * ksplit), static_cast<unsigned>(bgrid), 1);
    cfg.blockDim = dim3(kCsThreads, 1, 1);
    cfg.dynamicSmemBytes = kCsSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ksplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_coldot_stream_kernel<T>, map, p, ksplit);
}

template <typename T>
cudaError_t fill_t(void *c, int64_t batch, int64_t m, int64_t n, int64_t ldc, int64_t sc,
                   cudaStream_t s) {
    const int64_t total = batch * m * n;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fill_zero_kernel<T><<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<T *>(c), batch, m,
                                                                      n, ldc, sc);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_rowdot(int dt, const GemvParams &p, cudaStream_t s) {
    switch (dt) {
    case kF32: return rowdot_t<float>(p, s);
    case kF16: return rowdot_t<__half>(p, s);
    case kBF16: return rowdot_t<__nv_bfloat16>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv_coldot(int dt, const GemvParams &p, cudaStream_t s) {
    switch (dt) {
    case kF32: return coldot_t<float>(p, s);
    case kF16: return coldot_t<__half>(p, s);
    case kBF16: return coldot_t<__nv_bfloat16>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv_coldot_stream(int dt, const CUtensorMap &map, const GemvParams &p, cudaStream_t s) {
    switch (dt) {
    case kF32: return coldot_stream_t<float>(map, p, s);
    case kF16: return coldot_stream_t<__half>(map, p, s);
    case kBF16: return coldot_stream_t<__nv_bfloat16>(map, p, s);
    default: return cudaErrorInvalidValue;
    }
}

int gemv_coldot_stream_box_cols(int dt) { return static_cast<int>(kCsRowBytes) / (dt == kF32 ? 4 : 2); }
int gemv_coldot_stream_box_rows() { return kCsRows; }

cudaError_t launch_fill_zero(int dt, void *c, int64_t batch, int64_t m, int64_t n, int64_t ldc,
                             int64_t sc, cudaStream_t s) {
    switch (dt) {
    case kF32: return fill_t<float>(c, batch, m, n, ldc, sc, s);
    case kF16: return fill_t<__half>(c, batch, m, n, ldc, sc, s);
    case kBF16: return fill_t<__nv_bfloat16>(c, batch, m, n, ldc, sc, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbmm
