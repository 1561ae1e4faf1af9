// gemm_tc.cu -- batched f16/bf16 GEMM on the sm_103a tensor cores:
// C[b] = op(A[b]) * op(B[b]) for every combination of the transpose flags,
// f32 accumulation in tensor memory, f16/bf16 output.  Each operand is read
// as stored: K-contiguous (A [m, k] untransposed, B [n, k] transposed) or
// M/N-contiguous (A stored [k, m], B stored [k, n]); the MMA takes either
// major-ness from its instruction descriptor.
//
// Semantics: tract-metal 0.23.6, src/kernels/matmul/mlx_gemm/mod.rs,
// `dispatch_metal_mlx_gemm` (B stored [n, k] when transposed; batch strides
// per operand) and rlx-metal 0.2.14, src/mps_blas.rs (transposeRight).
//
// Two kernels: gemm_tc_pair_kernel (256 x 256 tiles on CTA pairs, see its
// section below) for long-k problems with at least two rounds of such tiles,
// and gemm_tc_kernel (128 x 256 tiles) for the rest; the host picks one.
//
// Design of gemm_tc_kernel (one persistent CTA per SM, 6 warps, warp-specialised):
//   warp 0      TMA producer: 128x64 A tiles and 256x64 B tiles, 128-byte
//               swizzled, into a 4-stage shared-memory ring (48 KB/stage);
//               a K-major tile is one box of 64 k x 128 / 256 rows, an
//               M/N-major tile two / four boxes of 64 m-or-n x 64 k, 8 KB apart.
//   warp 1      allocates 512 TMEM columns (two 128x256 f32 accumulators)
//               and issues tcgen05.mma (M=128, N=256, K=16) from one thread;
//               tcgen05.commit releases a stage when its MMAs are done and
//               signals the epilogue when a tile's accumulator is complete.
//   warps 2..5  epilogue: tcgen05.ld of their TMEM lane quarter, round to the
//               output dtype, store; then hand the accumulator back, so the
//               next tile's MMAs overlap this tile's stores.
// Tiles are visited in a grouped raster (8 m-blocks x all n-blocks per group)
// so the CTAs running at the same time share A and B panels in L2.  When the
// last round of tiles would leave at least half of the CTAs idle, each of its
// tiles runs as two 128x128 half units (N = 128 MMAs, the same rate per
// column), so that round takes half a tile's time.
// Every mbarrier wait is bounded; on a timeout the kernel records it in the
// device error word, waits (bounded) for its own copies and MMAs in flight,
// releases its TMEM and returns.
#include "device_common.cuh"

namespace gbmm {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;  // 64 x 2 bytes = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kGroupM = 8;
constexpr uint32_t kABytes = kBM * kBK * 2;
constexpr uint32_t kBBytes = kBN * kBK * 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kMNBox = 64 * kBK * 2;  // one 64 (m or n) x 64 (k) box of an M/N-major tile
constexpr uint32_t kSmemBytes = kStages * (kABytes + kBBytes) + 256 + 1024;

struct TileCoord {
    int bat, mb, nb;
    int h;       // half of the tile's columns a half unit computes
    int halves;  // 2: whole tile, 1: half unit h, 0: nothing (half past n)
};

__device__ __forceinline__ TileCoord decode_tile(int tile, const GemmTcParams &p) {
    const int per_batch = p.tiles_m * p.tiles_n;
    TileCoord t;
    t.bat = tile / per_batch;
    const int r = tile % per_batch;
    const int group = r / (kGroupM * p.tiles_n);
    const int first_m = group * kGroupM;
    const int gm = min(kGroupM, p.tiles_m - first_m);
    const int local = r % (kGroupM * p.tiles_n);
    t.mb = first_m + local % gm;
    t.nb = local / gm;
    t.h = 0;
    t.halves = 2;
    return t;
}

// Tiles that do not split over the grid evenly: with tail = num_tiles mod
// grid at most grid / 2, units [0, split_from) are whole tiles and every
// tile from split_from on becomes two half units (units split_from + 2i and
// split_from + 2i + 1).
__device__ __forceinline__ int gemm_tail_tiles(int num_tiles, int grid) {
    int tail = num_tiles > grid ? num_tiles % grid : (2 * num_tiles <= grid ? num_tiles : 0);
    if (2 * tail > grid) tail = 0;
    return tail;
}

__device__ __forceinline__ TileCoord decode_unit(int u, int split_from, const GemmTcParams &p) {
    if (u < split_from) return decode_tile(u, p);
    TileCoord t = decode_tile(split_from + (u - split_from) / 2, p);
    t.h = (u - split_from) & 1;
    t.halves = static_cast<int64_t>(t.nb) * kBN + t.h * (kBN / 2) < p.n ? 1 : 0;
    return t;
}

template <typename TC>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// kAMN / kBMN: A / B stored M- / N-contiguous (see the file comment)
template <typename TC, uint32_t kFmt, bool kAMN, bool kBMN>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const GemmTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t s_a = raw_addr + pad;
    const uint32_t s_b = s_a + kStages * kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * (kABytes + kBBytes));
    // barrier slots: full[kStages], empty[kStages], tfull[2], tempty[2], drain
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kblocks = (p.k + kBK - 1) / kBK;
    const int tail = gemm_tail_tiles(p.num_tiles, static_cast<int>(gridDim.x));
    const int split_from = p.num_tiles - tail;
    const int num_units = split_from + 2 * tail;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                const TileCoord tc = decode_unit(u, split_from, p);
                if (tc.halves == 0) continue;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.wait_limit_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(stage), kABytes + kBBytes);
                    const int abat = p.a_bcast ? 0 : tc.bat, bbat = p.b_bcast ? 0 : tc.bat;
                    if (kAMN) {
#pragma unroll
                        for (int j = 0; j < kBM / 64; ++j)
                            tma_load_3d(s_a + stage * kABytes + j * kMNBox, &map_a, full_bar(stage),
                                        tc.mb * kBM + j * 64, kb * kBK, abat);
                    } else {
                        tma_load_3d(s_a + stage * kABytes, &map_a, full_bar(stage), kb * kBK, tc.mb * kBM, abat);
                    }
                    if (kBMN) {
#pragma unroll
                        for (int j = 0; j < kBN / 64; ++j)
                            tma_load_3d(s_b + stage * kBBytes + j * kMNBox, &map_b, full_bar(stage),
                                        tc.nb * kBN + j * 64, kb * kBK, bbat);
                    } else {
                        tma_load_3d(s_b + stage * kBBytes, &map_b, full_bar(stage), kb * kBK, tc.nb * kBN, bbat);
                    }
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                report_device_error(p.err, kKidGemmTc);
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
            constexpr uint32_t kIdesc = idesc_f16(kFmt, kBM, kBN, kAMN ? 1u : 0u, kBMN ? 1u : 0u);
            constexpr uint32_t kIdescHalf = idesc_f16(kFmt, kBM, kBN / 2, kAMN ? 1u : 0u, kBMN ? 1u : 0u);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                const TileCoord tc = decode_unit(u, split_from, p);
                if (tc.halves == 0) continue;
                // a half unit multiplies by B rows [h * 128, h * 128 + 128) of the
                // stage: 16 KB further on in both B layouts
                const uint32_t b_off = static_cast<uint32_t>(tc.h) * (kBBytes / 2);
                const uint32_t idesc = tc.halves == 2 ? kIdesc : kIdescHalf;
                if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, p.wait_limit_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, p.wait_limit_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t da = kAMN ? sdesc_mnmajor_sw128(s_a + stage * kABytes + kk * 2048, kMNBox)
                                                 : sdesc_kmajor_sw128(s_a + stage * kABytes + kk * 32);
                        const uint64_t db = kBMN ? sdesc_mnmajor_sw128(s_b + stage * kBBytes + b_off + kk * 2048, kMNBox)
                                                 : sdesc_kmajor_sw128(s_b + stage * kBBytes + b_off + kk * 32);
                        umma_f16_ss(d_tmem, da, db, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit(empty_bar(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(tfull_bar(acc));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                *abort_flag = 1;
                report_device_error(p.err, kKidGemmTc);
            }
            // every MMA this thread issued has completed once this arrives
            umma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, p.wait_limit_ns, nullptr);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            const TileCoord tc = decode_unit(u, split_from, p);
            if (tc.halves == 0) continue;
            // one lane waits and the warp follows its verdict, so the warp stays
            // converged for the .sync.aligned TMEM loads below
            int ready = 0;
            if (lane == 0) ready = mbar_wait_bounded(tfull_bar(acc), acc_phase, p.wait_limit_ns, abort_flag);
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report_device_error(p.err, kKidGemmTc);
                }
                break;
            }
            __syncwarp();
            tc_fence_after();
            const int64_t row = static_cast<int64_t>(tc.mb) * kBM + quarter * 32 + lane;
            TC *crow = static_cast<TC *>(p.c) + static_cast<int64_t>(tc.bat) * p.sc + row * p.ldc;
            const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                    static_cast<uint32_t>(acc * kBN);
#pragma unroll 1
            for (int chunk = 0; chunk < tc.halves * (kBN / 64); ++chunk) {
                uint32_t r[32];
                tmem_ld32(t_addr + chunk * 32, r);
                tmem_ld_wait();
                const int64_t col0 = static_cast<int64_t>(tc.nb) * kBN + tc.h * (kBN / 2) + chunk * 32;
                if (row < p.m && col0 < p.n) {
                    if (p.c_vec_ok && col0 + 32 <= p.n) {
                        uint4 *dst = reinterpret_cast<uint4 *>(crow + col0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 o;
                            o.x = pack2<TC>(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                            o.y = pack2<TC>(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                            o.z = pack2<TC>(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                            o.w = pack2<TC>(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                            dst[v] = o;
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (col0 + c < p.n) crow[col0 + c] = Elem<TC>::from_f(__uint_as_float(r[c]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

constexpr int kWBM = 256;  // rows of a wide (CTA-pair) tile

// ---------------------------------------------------------------------------
// CTA-pair tiles: 256 x 256 outputs per pair of CTAs, computed by
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), for every layout of
// the operands (K-contiguous: one 64 k x 128 row box per CTA and operand;
// M/N-contiguous: two 64 x 64 boxes 8 KB apart, as in gemm_tc_kernel).
// Each CTA of the pair holds 128 rows of the A tile and 128 rows of the B
// tile per k-block (16 KB + 16 KB: half the operand bytes per SM of the
// 256 x 256 single-CTA tile for the same MMA work per SM) and its tensor
// memory holds its 128 rows of the accumulator.  A 128 x 256 accumulator
// per CTA leaves room for a second one, so the epilogue of a tile overlaps
// the MMAs of the next, and the smaller stages allow a six-deep ring.
//   warp 0      TMA (both CTAs): this CTA's A and B rows of each k-block,
//               completion counted on the even CTA's full barrier
//               (cp.async.bulk.tensor .cta_group::2)
//   warp 1      allocates 512 TMEM columns in both CTAs (one warp of each
//               executes the pair allocation); in the even CTA, one thread
//               issues the pair MMAs and commits them to both CTAs' barriers
//   warps 2..5  epilogue (both CTAs): their TMEM lane quarter of the tile's
//               accumulator, rounded and stored; the accumulator is handed
//               back to the even CTA's MMA issuer (8 arrivals per use)
// Tiles are visited by clusters in the grouped raster of the other kernels;
// when the last round of tiles would leave at least half of the pairs idle,
// its tiles run as two 256 x 128 half units each (N = 128 MMAs, each CTA
// using the first 64 of the 128 B rows it loads).  Every wait is bounded; a timeout raises both CTAs' abort flags and the
// device error word; both CTAs meet at a cluster barrier before the tensor
// memory is released.
// ---------------------------------------------------------------------------

constexpr int kPStages = 6;
constexpr uint32_t kPABytes = kBM * kBK * 2;     // this CTA's 128 A rows of a k-block
constexpr uint32_t kPBBytes = kBM * kBK * 2;     // this CTA's 128 B rows of a k-block
constexpr uint32_t kPStageBytes = kPABytes + kPBBytes;
constexpr uint32_t kPSmemBytes = kPStages * kPStageBytes + 256 + 1024;
static_assert(kPStageBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");

template <typename TC, uint32_t kFmt, bool kAMN, bool kBMN>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const GemmTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t s0 = raw_addr + pad;  // stage s: A at s0 + s * kPStageBytes, B kPABytes after it
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPStages * kPStageBytes);
    // barrier slots: full[kPStages] (used in the even CTA: both CTAs' copies),
    // empty[kPStages], tfull[2], tempty[2] (used in the even CTA), drain
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kPStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kPStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kPStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kPStages + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kPStages + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs
    const bool leader = rank == 0;
    const uint64_t lim = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(full_bar(s), 1);   // the even CTA's producer arrive + both CTAs' bytes
            mbar_init(empty_bar(s), 1);  // the pair MMAs' commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 8);  // four epilogue warps in each CTA
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers exist before any copy, commit or arrival can reach them
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kblocks = (p.k + kBK - 1) / kBK;
    const int cl = static_cast<int>(blockIdx.x) >> 1;
    const int ncl = static_cast<int>(gridDim.x) >> 1;
    // the last round of tiles, when it would leave at least half of the pairs
    // idle, runs as 256 x 128 half units (N = 128 pair MMAs)
    const int tail = gemm_tail_tiles(p.num_tiles, ncl);
    const int split_from = p.num_tiles - tail;
    const int num_units = split_from + 2 * tail;
    // a timeout stops both CTAs of the pair
    const uint32_t peer_abort = mapa_shared(smem_addr(const_cast<int *>(abort_flag)), rank ^ 1u);
    auto raise_abort = [&]() {
        *abort_flag = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
        report_device_error(p.err, kKidGemmTc);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = cl; u < num_units && ok; u += ncl) {
                const TileCoord tc = decode_unit(u, split_from, p);
                if (tc.halves == 0) continue;
                const int abat = p.a_bcast ? 0 : tc.bat, bbat = p.b_bcast ? 0 : tc.bat;
                const int arow = tc.mb * 2 * kBM + static_cast<int>(rank) * kBM;
                // a half unit needs 64 B rows per CTA: the first half of the box
                const int brow = tc.halves == 2 ? tc.nb * kBN + static_cast<int>(rank) * kBM
                                                : tc.nb * kBN + tc.h * (kBN / 2) + static_cast<int>(rank) * (kBM / 2);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded_cluster(empty_bar(stage), phase ^ 1u, lim, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * kPStageBytes);
                    const uint32_t sa = s0 + stage * kPStageBytes, sb = sa + kPABytes;
                    const uint32_t fb = mapa_shared(full_bar(stage), 0);
                    if (kAMN) {
                        tma_load_3d_pair(sa, &map_a, fb, arow, kb * kBK, abat);
                        tma_load_3d_pair(sa + kMNBox, &map_a, fb, arow + 64, kb * kBK, abat);
                    } else {
                        tma_load_3d_pair(sa, &map_a, fb, kb * kBK, arow, abat);
                    }
                    if (kBMN) {
                        tma_load_3d_pair(sb, &map_b, fb, brow, kb * kBK, bbat);
                        tma_load_3d_pair(sb + kMNBox, &map_b, fb, brow + 64, kb * kBK, bbat);
                    } else {
                        tma_load_3d_pair(sb, &map_b, fb, kb * kBK, brow, bbat);
                    }
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                raise_abort();
                // copies still in flight land within microseconds; give them 200 us
                const uint64_t t0 = global_ns();
                while (global_ns() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- pair MMA issuer (even CTA) ----------------
            constexpr uint32_t kIdesc = idesc_f16(kFmt, 2 * kBM, kBN, kAMN ? 1u : 0u, kBMN ? 1u : 0u);
            constexpr uint32_t kIdescHalf = idesc_f16(kFmt, 2 * kBM, kBN / 2, kAMN ? 1u : 0u, kBMN ? 1u : 0u);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_phase[2] = {0u, 0u};
            bool ok = true;
            int local = 0;
            for (int u = cl; u < num_units && ok; u += ncl) {
                const TileCoord tc = decode_unit(u, split_from, p);
                if (tc.halves == 0) continue;
                const uint32_t idesc = tc.halves == 2 ? kIdesc : kIdescHalf;
                const int a = local++ & 1;
                // both CTAs' epilogues have read this accumulator's previous tile
                if (!mbar_wait_bounded_cluster(tempty_bar(a), acc_phase[a] ^ 1u, lim, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * kBN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded_cluster(full_bar(stage), phase, lim, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = s0 + stage * kPStageBytes, sb = sa + kPABytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t da = kAMN ? sdesc_mnmajor_sw128(sa + kk * 2048, kMNBox)
                                                 : sdesc_kmajor_sw128(sa + kk * 32);
                        const uint64_t db = kBMN ? sdesc_mnmajor_sw128(sb + kk * 2048, kMNBox)
                                                 : sdesc_kmajor_sw128(sb + kk * 32);
                        umma_f16_ss_pair(d_tmem, da, db, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit_pair_mc(empty_bar(stage), 0x3);  // the stage is free in both CTAs
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(tfull_bar(a), 0x3);
                acc_phase[a] ^= 1u;
            }
            if (!ok) raise_abort();
            umma_commit_pair_mc(drain_bar, 0x1);
            mbar_wait_bounded(drain_bar, 0, lim, nullptr);
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        uint32_t tphase[2] = {0u, 0u};
        int local = 0;
        for (int u = cl; u < num_units; u += ncl) {
            const TileCoord tc = decode_unit(u, split_from, p);
            if (tc.halves == 0) continue;
            const int a = local++ & 1;
            int ready = 0;
            if (lane == 0) ready = mbar_wait_bounded_cluster(tfull_bar(a), tphase[a], lim, abort_flag);
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) {
                if (lane == 0) raise_abort();
                break;
            }
            __syncwarp();
            tc_fence_after();
            const int64_t row = static_cast<int64_t>(tc.mb) * 2 * kBM + static_cast<int64_t>(rank) * kBM +
                                quarter * 32 + lane;
            TC *crow = static_cast<TC *>(p.c) + static_cast<int64_t>(tc.bat) * p.sc + row * p.ldc;
            const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                    static_cast<uint32_t>(a * kBN);
            const int nchunks = tc.halves == 2 ? kBN / 32 : kBN / 64;
            const int64_t cbase = static_cast<int64_t>(tc.nb) * kBN + (tc.halves == 2 ? 0 : tc.h * (kBN / 2));
#pragma unroll 1
            for (int chunk = 0; chunk < nchunks; ++chunk) {
                uint32_t r[32];
                tmem_ld32(t_addr + chunk * 32, r);
                tmem_ld_wait();
                const int64_t col0 = cbase + chunk * 32;
                if (row < p.m && col0 < p.n) {
                    if (p.c_vec_ok == 2 && col0 + 32 <= p.n) {
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint32_t o[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                o[q] = pack2<TC>(__uint_as_float(r[16 * v + 2 * q]),
                                                 __uint_as_float(r[16 * v + 2 * q + 1]));
                            asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(
                                             crow + col0 + 16 * v),
                                         "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]),
                                         "r"(o[7])
                                         : "memory");
                        }
                    } else if (p.c_vec_ok && col0 + 32 <= p.n) {
                        uint4 *dst = reinterpret_cast<uint4 *>(crow + col0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 o;
                            o.x = pack2<TC>(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                            o.y = pack2<TC>(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                            o.z = pack2<TC>(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                            o.w = pack2<TC>(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                            __stcs(dst + v, o);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (col0 + c < p.n) crow[col0 + c] = Elem<TC>::from_f(__uint_as_float(r[c]));
                    }
                }
            }
            // this CTA's rows of the accumulator are read: hand it back to the even CTA's issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(a), 0));
            tphase[a] ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    // every pair MMA has completed (the even CTA waited for its drain) and
    // both CTAs' epilogues are done before either CTA releases the columns
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <typename TC, uint32_t kFmt, bool kAMN, bool kBMN>
cudaError_t tc_pair_t(const CUtensorMap &ma, const CUtensorMap &mb, const GemmTcParams &p, int num_sms,
                      cudaStream_t s) {
    static unsigned long long attr_set = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_pair_kernel<TC, kFmt, kAMN, kBMN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    const int pairs = num_sms / 2;
    const int clusters = 2 * p.num_tiles <= pairs ? 2 * p.num_tiles : (p.num_tiles < pairs ? p.num_tiles : pairs);
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<TC, kFmt, kAMN, kBMN>, ma, mb, p);
}

template <typename TC, uint32_t kFmt>
cudaError_t tc_pair_major(const CUtensorMap &ma, const CUtensorMap &mb, const GemmTcParams &p, int num_sms,
                          cudaStream_t s) {
    if (p.a_mn) return p.b_mn ? tc_pair_t<TC, kFmt, true, true>(ma, mb, p, num_sms, s)
                              : tc_pair_t<TC, kFmt, true, false>(ma, mb, p, num_sms, s);
    return p.b_mn ? tc_pair_t<TC, kFmt, false, true>(ma, mb, p, num_sms, s)
                  : tc_pair_t<TC, kFmt, false, false>(ma, mb, p, num_sms, s);
}

template <typename TC, uint32_t kFmt, bool kAMN, bool kBMN>
cudaError_t tc_t(const CUtensorMap &ma, const CUtensorMap &mb, const GemmTcParams &p, int num_sms,
                 cudaStream_t s) {
    static unsigned long long attr_set = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<TC, kFmt, kAMN, kBMN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    // at most half an SM's worth of tiles: every tile runs as two half units
    const int grid = 2 * p.num_tiles <= num_sms ? 2 * p.num_tiles : (p.num_tiles < num_sms ? p.num_tiles : num_sms);
    gemm_tc_kernel<TC, kFmt, kAMN, kBMN><<<grid, kThreads, kSmemBytes, s>>>(ma, mb, p);
    return cudaGetLastError();
}

template <typename TC, uint32_t kFmt>
cudaError_t tc_major(const CUtensorMap &ma, const CUtensorMap &mb, const GemmTcParams &p, int num_sms,
                     cudaStream_t s) {
    if (p.a_mn) return p.b_mn ? tc_t<TC, kFmt, true, true>(ma, mb, p, num_sms, s)
                              : tc_t<TC, kFmt, true, false>(ma, mb, p, num_sms, s);
    return p.b_mn ? tc_t<TC, kFmt, false, true>(ma, mb, p, num_sms, s)
                  : tc_t<TC, kFmt, false, false>(ma, mb, p, num_sms, s);
}

}  // namespace

int gemm_tc_block_m() { return kBM; }
int gemm_tc_wide_block_m() { return kWBM; }
int gemm_tc_block_n() { return kBN; }
int gemm_tc_block_k() { return kBK; }

cudaError_t launch_gemm_tc(int dt, const CUtensorMap &map_a, const CUtensorMap &map_b,
                           const GemmTcParams &p, int num_sms, cudaStream_t s) {
    switch (dt) {
    case kF16: return tc_major<__half, 0>(map_a, map_b, p, num_sms, s);
    case kBF16: return tc_major<__nv_bfloat16, 1>(map_a, map_b, p, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_tc_pair(int dt, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                const GemmTcParams &p, int num_sms, cudaStream_t s) {
    switch (dt) {
    case kF16: return tc_pair_major<__half, 0>(map_a, map_b, p, num_sms, s);
    case kBF16: return tc_pair_major<__nv_bfloat16, 1>(map_a, map_b, p, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbmm
