// gemv_tc.cu -- the skinny decode GEMV y[m, n] = x[m, k] W[n, k]^T for 2..15
// tokens (f16/bf16, batch 1) on the sm_103a tensor cores, computed as
// y^T = W x^T: the weight rows are the MMA's M side (128 per tile) and the
// tokens its N side (16, the rows past m read as zeros by TMA).
//
// Semantics: tract-metal 0.23.6, src/kernels/matmul/mlx_gemm/mod.rs,
// `dispatch_metal_mlx_gemv_wide` (c[m, n] = a[m, k] @ b[n, k]^T for m in
// 2..=15, gated by `gemv_wide_config`).
//
// Every weight byte is read once, so the kernel is HBM-bound; the MMA work
// (M=128, N=16, K=16 per instruction) is a small fraction of the stream time,
// where a CUDA-core kernel's dot products grow with every token.  One
// thread-block cluster of `ksplit` CTAs per 128-row tile of W: a decode shape
// has too few tiles to occupy every SM (11008 rows = 86 tiles), and one CTA
// streams no faster than ~70 GB/s, so the contraction is split over the
// cluster's CTAs (an even share of the 64-wide k-blocks each) and the partial
// accumulators are added through distributed shared memory -- no scratch
// buffer, no atomics, a fixed summation order.  6 warps per CTA:
//   warp 0      TMA: the 128x64 weight tile and the 16x64 token tile of each
//               k-block (128-byte swizzle) into a ring of kStages stages; the
//               weights with the L2 evict-first policy
//   warp 1      allocates 32 TMEM columns and issues 4 x tcgen05.mma per
//               k-block from one thread
//   warps 2..5  epilogue: tcgen05.ld of the 16 accumulator columns of their
//               TMEM lane quarter (one weight row per lane); with a split,
//               each CTA parks its partial sums in its own (by then idle)
//               ring memory and the cluster's rank 0 adds the others' in rank
//               order; then round to the output dtype and store element
//               (j, n0 + row) for every token j < m -- a warp writes 32
//               contiguous outputs of each row
// The ring is sized so that two CTAs share an SM.  Every mbarrier wait is
// bounded; on a timeout the kernel records it in the device error word, waits
// (bounded) for its own copies and MMAs, still takes part in both cluster
// barriers, releases its TMEM and returns.
#include <cooperative_groups.h>

#include "device_common.cuh"

namespace cg = cooperative_groups;

namespace gbmm {

namespace {

constexpr int kBM = 128;   // weight rows per tile (MMA M)
constexpr int kBN = 16;    // tokens (MMA N)
constexpr int kBK = 64;    // one 128-byte swizzle row of 16-bit elements
constexpr int kStages = 6;   // 110.6 KB: two CTAs per SM
constexpr int kThreads = 192;
constexpr uint32_t kWBytes = kBM * kBK * 2;
constexpr uint32_t kXBytes = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kWBytes + kXBytes;  // 18 KB: every tile base stays 1024-byte aligned
constexpr uint32_t kTmemCols = 32;                   // the allocation minimum; 16 are used
constexpr uint32_t kSmemBytes = kStages * kStageBytes + 256 + 1024;
constexpr int kMaxSplit = 8;                             // the portable cluster size
constexpr uint32_t kPartBytes = kBM * kBN * 4;           // one CTA's f32 partial sums
static_assert(kStageBytes % 1024 == 0 && kWBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kPartBytes <= kStages * kStageBytes, "the partial sums are parked in the ring");
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");

// Each thread of the warp reads its TMEM lane, 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

template <typename TC, uint32_t kFmt>
__global__ void __launch_bounds__(kThreads, 1)
gemv_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
               const GemvTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t s0 = raw_addr + pad;  // stage s: W at s0 + s * kStageBytes, x kWBytes after it
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    // barrier slots: full[kStages], empty[kStages], tfull, drain
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * kStages);
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ksplit = p.ksplit;
    const int rank = static_cast<int>(blockIdx.x) % ksplit;  // == rank in the cluster (cluster dims = ksplit)
    const int n0 = static_cast<int>(blockIdx.x) / ksplit * kBM;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_w);
        tma_prefetch_desc(&map_x);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // this CTA's share of the k-blocks: [kb0, kb0 + kblocks)
    const int kb_total = (p.k + kBK - 1) / kBK;
    const int kb0 = static_cast<int>(static_cast<int64_t>(kb_total) * rank / ksplit);
    const int kblocks = static_cast<int>(static_cast<int64_t>(kb_total) * (rank + 1) / ksplit) - kb0;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t pol = policy_evict_first();
            uint32_t issued = 0;
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb) {
                const int stage = kb % kStages;
                const uint32_t use = static_cast<uint32_t>(kb / kStages);
                if (use > 0 && !mbar_wait_bounded(empty_bar(stage), (use - 1u) & 1u, p.wait_limit_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sw = s0 + stage * kStageBytes;
                mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
                tma_load_3d_hint(sw, &map_w, full_bar(stage), (kb0 + kb) * kBK, n0, 0, pol);
                tma_load_3d(sw + kWBytes, &map_x, full_bar(stage), (kb0 + kb) * kBK, 0, 0);
                ++issued;
            }
            if (!ok) {
                *abort_flag = 1;
                report_device_error(p.err, kKidGemvTc);
                // wait for this CTA's own copies still in flight
                for (int s = 0; s < kStages; ++s) {
                    const uint32_t n_s = issued / kStages + (static_cast<uint32_t>(s) < issued % kStages ? 1u : 0u);
                    if (n_s > 0) mbar_wait_bounded(full_bar(s), (n_s - 1u) & 1u, p.wait_limit_ns, nullptr);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t kIdesc = idesc_f16(kFmt, kBM, kBN);
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb) {
                const int stage = kb % kStages;
                if (!mbar_wait_bounded(full_bar(stage), static_cast<uint32_t>(kb / kStages) & 1u, p.wait_limit_ns,
                                       abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sw = s0 + stage * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    umma_f16_ss(tmem_base, sdesc_kmajor_sw128(sw + kk * 32), sdesc_kmajor_sw128(sw + kWBytes + kk * 32),
                                kIdesc, (kb | kk) != 0 ? 1u : 0u);
                umma_commit(empty_bar(stage));
            }
            if (ok) {
                umma_commit(tfull_bar);
            } else {
                *abort_flag = 1;
                report_device_error(p.err, kKidGemvTc);
            }
            // every MMA this thread issued has completed once this arrives
            umma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, p.wait_limit_ns, nullptr);
        }
    }
    __syncwarp();  // the producer and MMA warps reconverge before the cluster barriers

    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 = weight rows
    const int rrow = quarter * 32 + lane;
    float acc[kBN];
    if (warp >= 2) {
        int ready = 0;
        if (lane == 0) ready = mbar_wait_bounded(tfull_bar, 0, p.wait_limit_ns, abort_flag);
        ready = __shfl_sync(0xffffffffu, ready, 0);
        __syncwarp();
        if (ready && kblocks > 0) {
            tc_fence_after();
            uint32_t r[kBN];
            tmem_ld16(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16), r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < kBN; ++j) acc[j] = __uint_as_float(r[j]);
        } else {
#pragma unroll
            for (int j = 0; j < kBN; ++j) acc[j] = 0.f;
            if (!ready && lane == 0) {
                *abort_flag = 1;
                report_device_error(p.err, kKidGemvTc);
            }
        }
    }

    float *part = reinterpret_cast<float *>(smem);  // [kBM][kBN], over the drained ring
    if (ksplit > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        // every thread of the cluster reaches both barriers, on every path
        if (warp >= 2 && rank != 0) {
#pragma unroll
            for (int j = 0; j < kBN; j += 4)
                *reinterpret_cast<float4 *>(part + rrow * kBN + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        }
        cluster.sync();  // the partial sums of every rank are visible cluster-wide
        if (warp >= 2 && rank == 0) {
            for (int q = 1; q < ksplit; ++q) {
                const float *rp = cluster.map_shared_rank(part, q) + rrow * kBN;
#pragma unroll
                for (int j = 0; j < kBN; j += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(rp + j);
                    acc[j] += v.x;
                    acc[j + 1] += v.y;
                    acc[j + 2] += v.z;
                    acc[j + 3] += v.w;
                }
            }
        }
        cluster.sync();  // keep every rank's shared memory alive until rank 0 has read it
    }
    if (warp >= 2 && rank == 0) {
        const int64_t row = static_cast<int64_t>(n0) + rrow;
        if (row < p.n) {
            TC *c = static_cast<TC *>(p.c);
#pragma unroll
            for (int j = 0; j < kBN; ++j)
                if (j < p.m) c[static_cast<int64_t>(j) * p.ldc + row] = Elem<TC>::from_f(acc[j]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <typename TC, uint32_t kFmt>
cudaError_t gemv_tc_t(const CUtensorMap &mw, const CUtensorMap &mx, const GemvTcParams &p, cudaStream_t s) {
    static unsigned long long attr_set = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel<TC, kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    const unsigned tiles = static_cast<unsigned>((p.n + kBM - 1) / kBM);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * static_cast<unsigned>(p.ksplit), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.ksplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_tc_kernel<TC, kFmt>, mw, mx, p);
}

}  // namespace

int gemv_tc_block_rows() { return kBM; }
int gemv_tc_max_tokens() { return kBN; }
int gemv_tc_block_k() { return kBK; }

int gemv_tc_split(int64_t n, int64_t k, int num_sms) {
    // the largest cluster that keeps the grid within 1.25 CTAs per SM, each CTA
    // still with at least four k-blocks of its own.  Measured (f16, 8 tokens,
    // k 4096, L2 flushed): 11008 rows = 86 tiles take 26.6 / 24.6 / 24.6 /
    // 30.7 us at splits 1 / 2 / 3 / 4, 4096 rows 24.6 / 18.4 / 16.4 / 16.4 /
    // 18.4 us at 1 / 2 / 3 / 4 / 8: past about one CTA per SM every extra
    // CTA adds its own prologue and pipeline fill to an SM's time
    const int64_t tiles = (n + kBM - 1) / kBM;
    const int64_t kb = (k + kBK - 1) / kBK;
    int split = 1;
    while (split < kMaxSplit && 4 * tiles * (split + 1) <= 5LL * num_sms && kb >= 4LL * (split + 1)) ++split;
    return split;
}

cudaError_t launch_gemv_tc(int dt, const CUtensorMap &map_w, const CUtensorMap &map_x, const GemvTcParams &p,
                           cudaStream_t s) {
    if (p.ksplit < 1 || p.ksplit > kMaxSplit) return cudaErrorInvalidValue;
    switch (dt) {
    case kF16: return gemv_tc_t<__half, 0>(map_w, map_x, p, s);
    case kBF16: return gemv_tc_t<__nv_bfloat16, 1>(map_w, map_x, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbmm
