// direct_tc.cu -- the Direct route of the expert-ID matmul on the sm_103a
// tensor cores, for bf16 or f16 expert weights and f32 activations.
//
// Semantics: mlx-native 0.13.0, src/ops/dense_matmul_id.rs,
// `dense_matmul_id` (Direct: for routed row r = t*top_k + s with
// e = ids[r] < n_experts, out[r, j] = sum_x W_e[j, x] * xrow(t, s)[x], W_e the
// row-major [n, k] matrix of expert e; a row whose id is out of range is
// all zeros).
//
// A decode call selects a few distinct experts, each by a handful of routed
// rows, so the work is streaming each selected expert's weights from HBM
// once.  Per selected expert the product is a skinny GEMM, computed as
// out^T = W_e x^T: 128 weight rows are the MMA's M side, the expert's routed
// rows its N side.  The f32 activations are split exactly as x = hi + lo
// (hi = bf16(x), lo = bf16(x - hi), relative error <= 2^-16) and the two
// halves are the two 16-row halves of one N = 32 operand, so each K = 16
// step is a single MMA and the epilogue adds accumulator columns c and
// c + 16.  f16 weights need f16 activations (one MMA takes one operand
// type), and f16's 5-bit exponent cannot hold every f32: each routed row is
// first scaled by a power of two that puts its largest magnitude over this
// CTA's k-range in [2^14, 2^15) (one warp per row reads the row once before
// its first k-block), split into f16 hi + lo (relative error <= 2^-22 for
// elements within 2^-10 of that maximum, absolute <= 2^-25 in scaled units
// below), and its accumulator column is scaled back exactly before any
// partial sums are added.
//
// Grid: one CTA per (distinct-expert index d, 128-row weight tile, k-split
// rank).  The host sizes it for min(n_experts, m * top_k) distinct experts,
// d-major, so the CTAs of absent experts are the last ones and return at
// once.  Every CTA finds its expert itself: the ids are staged in shared
// memory, the selected experts marked in a bitmap, the d-th set bit (experts
// in ascending order) is its expert, and one warp compacts the routed rows
// that chose it in ascending order.  Routed rows beyond 16 run as further
// passes over the same weight tile.  When no expert can be chosen by more
// than 16 rows (DistinctPerToken with m <= 16, or m * top_k <= 16) and the
// tiles alone cannot occupy the SMs, the k-blocks are split over a cluster of
// up to 8 CTAs whose partial sums rank 0 adds through distributed shared
// memory.  The d = 0, rank-0 CTA of each tile writes the zero rows of
// out-of-range ids.  6 warps, three CTAs per SM (a decode call's selected
// experts x tiles fill the SMs in one wave):
//   warp 0      TMA: the 128x64 weight box of W_e per k-block (128-byte
//               swizzle, 3-D tensor map over (k, n, expert))
//   warp 1      TMEM allocation (32 columns) and one MMA per K = 16 step
//   warps 2..5  during a pass: gather 16 routed rows x 64 activations per
//               k-block, split into bf16 hi / lo, write the swizzled K-major
//               operand; after it: tcgen05.ld, hi + lo, f32 stores (a warp
//               writes 32 consecutive outputs of a routed row)
// Every mbarrier wait is bounded; a timeout is recorded in the device error
// word, the CTA waits (bounded) for its own copies and MMAs, still takes part
// in the cluster barriers, releases its TMEM and returns.
#include <cooperative_groups.h>

#include "device_common.cuh"

namespace cg = cooperative_groups;

namespace gbmm {

namespace {

constexpr int kBM = 128;      // weight rows per tile (MMA M)
constexpr int kBR = 16;       // routed rows per pass
constexpr int kBN = 2 * kBR;  // MMA N: hi rows 0..15, lo rows 16..31
constexpr int kBK = 64;
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr uint32_t kWBytes = kBM * kBK * 2;
constexpr uint32_t kXBytes = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kWBytes + kXBytes;  // 20 KB: tile bases stay 1024-byte aligned
constexpr int kMaxIds = 1024;
constexpr int kMaxExperts = 4096;
constexpr int kMaxSplit = 8;
constexpr uint32_t kTmemCols = 32;
constexpr int kNumBars = 2 * kStages + 5;  // full, empty, tfull, tempty, drain, scale-ready x 2
constexpr uint32_t kRingBytes = kStages * kStageBytes;
constexpr uint32_t kIdsOff = kRingBytes;
constexpr uint32_t kRowsOff = kIdsOff + kMaxIds * 4;
constexpr uint32_t kMapOff = kRowsOff + kMaxIds * 4;
constexpr uint32_t kBarOff = kMapOff + kMaxExperts / 8;
constexpr uint32_t kCtlOff = kBarOff + kNumBars * 8;
constexpr uint32_t kScaleOff = kCtlOff + 32;  // [2][kBR] f32 row scales + [2][kBR] inverses (f16 weights)
constexpr uint32_t kSmemBytes = kScaleOff + 4 * kBR * 4 + 1024;
static_assert(kStageBytes % 1024 == 0 && kWBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kBM * kBR * 4 <= kRingBytes, "the partial sums are parked in the ring");
static_assert(3 * (kSmemBytes + 1024) <= 228 * 1024, "three CTAs per SM");

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float bf16_lo_half(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi_half(uint32_t packed) { return __uint_as_float(packed & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t packed) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&packed));
}

// hi = round(a), lo = round(a - hi) for a pair, in the 16-bit type of the weights
template <bool kF16>
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
    if (kF16) {
        hi = pack_f16x2(a, b);
        const float2 h = f16x2_to_float2(hi);
        lo = pack_f16x2(a - h.x, b - h.y);
    } else {
        hi = pack_bf16x2(a, b);
        lo = pack_bf16x2(a - bf16_lo_half(hi), b - bf16_hi_half(hi));
    }
}

__device__ __forceinline__ const float *x_row_of(const MatmulIdParams &p, uint32_t r) {
    const int64_t t = r / p.top_k;
    const int64_t s = r % p.top_k;
    return p.x + t * p.x_token_stride + s * p.x_slot_stride;
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 3)
direct_tc_kernel(const __grid_constant__ CUtensorMap map_w, const MatmulIdParams p, int ksplit, int tiles,
                 int x_vec_ok) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t s0 = raw_addr + pad;  // stage s: W at s0 + s * kStageBytes, x kWBytes after it
    uint32_t *ids_s = reinterpret_cast<uint32_t *>(smem + kIdsOff);
    uint32_t *rows_s = reinterpret_cast<uint32_t *>(smem + kRowsOff);
    uint32_t *emap = reinterpret_cast<uint32_t *>(smem + kMapOff);
    const uint32_t bar0 = s0 + kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * kStages);
    const uint32_t tempty_bar = tfull_bar + 8u;
    const uint32_t drain_bar = tfull_bar + 16u;
    auto sready_bar = [&](int b) { return tfull_bar + 24u + 8u * b; };  // row scales of a pass written
    float *scale_s = reinterpret_cast<float *>(smem + kScaleOff);  // [2][kBR] row scales, by pass parity
    float *unscale_s = scale_s + 2 * kBR;                             // [2][kBR] their inverses
    uint32_t *ctl = reinterpret_cast<uint32_t *>(smem + kCtlOff);  // tmem slot, abort, expert, count
    volatile int *abort_flag = reinterpret_cast<volatile int *>(ctl + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = static_cast<int>(blockIdx.x) % ksplit;  // == rank in the cluster (cluster dims = ksplit)
    const int unit = static_cast<int>(blockIdx.x) / ksplit;
    const int tile = unit % tiles;
    const int d = unit / tiles;
    const int n0 = tile * kBM;
    const int n_ids = static_cast<int>(p.total_rows);
    const uint32_t E = static_cast<uint32_t>(p.n_experts);
    const int nwords = static_cast<int>((E + 31) / 32);
    const uint64_t lim = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 5);  // the TMA thread (+ bytes) and the four activation warps
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, 4);
        mbar_init(drain_bar, 1);
        mbar_init(sready_bar(0), 4);
        mbar_init(sready_bar(1), 4);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&map_w);
    if (warp == 1) {
        tmem_alloc(smem_addr(ctl), kTmemCols);
        tmem_relinquish();
    }
    {
        // ---- this CTA's expert: the d-th distinct in-range id, ascending ----
        for (int i = threadIdx.x; i < nwords; i += kThreads) emap[i] = 0u;
        __syncthreads();
        for (int r = threadIdx.x; r < n_ids; r += kThreads) {
            const uint32_t e = p.ids[r];
            ids_s[r] = e;
            if (e < E) atomicOr(&emap[e >> 5], 1u << (e & 31));
        }
        __syncthreads();
        if (warp == 0) {
            int sel = -1;
            uint32_t base = 0;
            for (int w0 = 0; w0 < nwords; w0 += 32) {
                const uint32_t word = w0 + lane < nwords ? emap[w0 + lane] : 0u;
                const uint32_t c = static_cast<uint32_t>(__popc(word));
                uint32_t incl = c;
    #pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint32_t excl = base + incl - c;
                const uint32_t want = static_cast<uint32_t>(d);
                int mine = -1;
                if (sel < 0 && want >= excl && want < excl + c) {
                    uint32_t wbits = word;
                    for (uint32_t j = 0; j < want - excl; ++j) wbits &= wbits - 1u;  // drop the lower set bits
                    mine = (w0 + lane) * 32 + __ffs(static_cast<int>(wbits)) - 1;
                }
                const unsigned who = __ballot_sync(0xffffffffu, mine >= 0);
                if (who != 0u) sel = __shfl_sync(0xffffffffu, mine, __ffs(static_cast<int>(who)) - 1);
                base += __shfl_sync(0xffffffffu, incl, 31);
            }
            // the routed rows that chose it, ascending
            int cnt = 0;
            if (sel >= 0) {
                const unsigned lt = (1u << lane) - 1u;
                for (int b = 0; b < n_ids; b += 32) {
                    const int r = b + lane;
                    const bool hit = r < n_ids && ids_s[r] == static_cast<uint32_t>(sel);
                    const unsigned bal = __ballot_sync(0xffffffffu, hit);
                    if (hit) rows_s[cnt + __popc(bal & lt)] = static_cast<uint32_t>(r);
                    cnt += __popc(bal);
                }
            }
            if (lane == 0) {
                ctl[2] = static_cast<uint32_t>(sel);
                ctl[3] = static_cast<uint32_t>(cnt);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl[0];
    const int e_sel = static_cast<int>(ctl[2]);
    const int cnt = static_cast<int>(ctl[3]);
    // routed row c of this CTA's expert
    auto row_of = [&](int c) -> uint32_t { return rows_s[c]; };
    const int passes = e_sel >= 0 ? (cnt + kBR - 1) / kBR : 0;
    const int kb_total = static_cast<int>((p.k + kBK - 1) / kBK);
    const int kb0 = static_cast<int>(static_cast<int64_t>(kb_total) * rank / ksplit);
    const int kblocks = static_cast<int>(static_cast<int64_t>(kb_total) * (rank + 1) / ksplit) - kb0;
    const int iters = passes * kblocks;

    float acc[kBR];  // epilogue warps: this lane's weight row, one value per routed row of the pass
#pragma unroll
    for (int c = 0; c < kBR; ++c) acc[c] = 0.f;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- weight tiles (TMA) ----------------
            const uint64_t pol = passes > 1 ? policy_evict_normal() : policy_evict_first();
            int it = 0;
            for (; it < iters; ++it) {
                const int stage = it % kStages;
                const uint32_t use = static_cast<uint32_t>(it / kStages);
                if (use > 0 && !mbar_wait_bounded(empty_bar(stage), (use - 1u) & 1u, lim, abort_flag)) break;
                mbar_arrive_expect_tx(full_bar(stage), kWBytes);
                tma_load_3d_hint(s0 + stage * kStageBytes, &map_w, full_bar(stage), (kb0 + it % kblocks) * kBK, n0,
                                 e_sel, pol);
            }
            if (it < iters) {
                *abort_flag = 1;
                report_device_error(p.err, kKidDirectTc);
                // this thread's copies still in flight: its last kStages fills at most
                for (int j = it - 1; j >= 0 && j >= it - kStages; --j)
                    mbar_wait_bounded(full_bar(j % kStages), static_cast<uint32_t>(j / kStages) & 1u, lim, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t kIdesc = idesc_f16(kF16 ? 0u : 1u, kBM, kBN);  // 16-bit x 16-bit -> f32
            bool ok = true;
            int it = 0;
            for (int pass = 0; pass < passes && ok; ++pass) {
                // the epilogue has read the previous pass's accumulator
                if (pass > 0 && !mbar_wait_bounded(tempty_bar, static_cast<uint32_t>(pass - 1) & 1u, lim, abort_flag)) {
                    ok = false;
                    break;
                }
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int stage = it % kStages;
                    if (!mbar_wait_bounded(full_bar(stage), static_cast<uint32_t>(it / kStages) & 1u, lim,
                                           abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sw = s0 + stage * kStageBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        umma_f16_ss(tmem_base, sdesc_kmajor_sw128(sw + kk * 32),
                                    sdesc_kmajor_sw128(sw + kWBytes + kk * 32), kIdesc, (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(empty_bar(stage));
                }
                if (ok) umma_commit(tfull_bar);
            }
            if (!ok) {
                *abort_flag = 1;
                report_device_error(p.err, kKidDirectTc);
            }
            umma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, lim, nullptr);
        }
    } else {
        // ---------------- activations, then epilogue (warps 2..5) ----------------
        // activations: thread t routes row t / 8 of the pass, activations
        // 8 (t % 8) .. +7 of the k-block = 16-byte chunk t % 8 of its hi row
        // and of its lo row (16 rows further)
        const int t = threadIdx.x - 64;
        const int row = t >> 3;
        const uint32_t ch = static_cast<uint32_t>(t & 7);
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 = weight rows
        const int64_t j = static_cast<int64_t>(n0) + quarter * 32 + lane;
        int it = 0;
        for (int pass = 0; pass < passes; ++pass) {
            const int c = pass * kBR + row;
            const float *src = c < cnt ? x_row_of(p, row_of(c)) : nullptr;
            float scale = 1.f;  // power of two applied before the f16 split
            bool sok = true;
            if (kF16) {
                // row scales: activation warp w takes rows w, w + 4, w + 8, w + 12 of the
                // pass, its lanes reading the row's k-range with 16-byte loads
                const int b = pass & 1;
                for (int rr = warp - 2; rr < kBR; rr += 4) {
                    const int cr = pass * kBR + rr;
                    float mx = 0.f;
                    if (cr < cnt) {
                        const float *xs = x_row_of(p, row_of(cr));
                        const int64_t k_lo = static_cast<int64_t>(kb0) * kBK;
                        const int64_t k_hi = min(p.k, static_cast<int64_t>(kb0 + kblocks) * kBK);
                        if (x_vec_ok) {
                            const float4 *x4 = reinterpret_cast<const float4 *>(xs);
#pragma unroll 8
                            for (int64_t q = k_lo / 4 + lane; q < k_hi / 4; q += 32) {
                                const float4 a = x4[q];
                                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
                            }
                        } else {
                            for (int64_t q = k_lo + lane; q < k_hi; q += 32) mx = fmaxf(mx, fabsf(xs[q]));
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    }
                    // mx in [2^(eb-127), 2^(eb-126)): scale by 2^(141 - eb), kept within the normal range
                    int sexp = 0;
                    if (mx > 0.f) {
                        const int eb = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu);
                        sexp = min(126, max(-126, 141 - eb));
                    }
                    if (lane == 0) {
                        scale_s[b * kBR + rr] = __uint_as_float(static_cast<uint32_t>(127 + sexp) << 23);
                        unscale_s[b * kBR + rr] = __uint_as_float(static_cast<uint32_t>(127 - sexp) << 23);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sready_bar(b));
                // every activation warp's rows
                int r_ok = 0;
                if (lane == 0) r_ok = mbar_wait_bounded(sready_bar(b), static_cast<uint32_t>(pass >> 1) & 1u, lim, abort_flag);
                r_ok = __shfl_sync(0xffffffffu, r_ok, 0);
                __syncwarp();
                sok = r_ok != 0;
                if (sok) scale = scale_s[b * kBR + row];
            }
            bool ok = sok;
            for (int kb = 0; kb < kblocks && ok; ++kb, ++it) {
                const int stage = it % kStages;
                const uint32_t use = static_cast<uint32_t>(it / kStages);
                int ready = 1;
                if (use > 0 && lane == 0) ready = mbar_wait_bounded(empty_bar(stage), (use - 1u) & 1u, lim, abort_flag);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                __syncwarp();
                if (!ready) {
                    ok = false;
                    break;
                }
                float f[8];
                const int64_t kx = static_cast<int64_t>(kb0 + kb) * kBK + ch * 8;
                if (src == nullptr) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = 0.f;
                } else if (x_vec_ok && kx + 8 <= p.k) {
                    const float4 a = *reinterpret_cast<const float4 *>(src + kx);
                    const float4 b = *reinterpret_cast<const float4 *>(src + kx + 4);
                    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
                    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = kx + e < p.k ? src[kx + e] : 0.f;
                }
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) split_pair<kF16>(f[2 * h] * scale, f[2 * h + 1] * scale, hi[h], lo[h]);
                // 128-byte swizzle: 16-byte chunk ch of operand row i at chunk ch ^ (i % 8)
                const uint32_t xb = s0 + stage * kStageBytes + kWBytes;
                const uint32_t a_hi = xb + static_cast<uint32_t>(row) * 128u + ((ch ^ (row & 7)) << 4);
                const uint32_t a_lo = xb + static_cast<uint32_t>(row + kBR) * 128u + ((ch ^ ((row + kBR) & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a_hi), "r"(hi[0]), "r"(hi[1]),
                             "r"(hi[2]), "r"(hi[3])
                             : "memory");
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a_lo), "r"(lo[0]), "r"(lo[1]),
                             "r"(lo[2]), "r"(lo[3])
                             : "memory");
                fence_async_smem();  // generic-proxy writes -> visible to the tensor cores
                __syncwarp();
                if (lane == 0) mbar_arrive(full_bar(stage));
            }
            int ready = 0;
            if (ok && lane == 0) ready = mbar_wait_bounded(tfull_bar, static_cast<uint32_t>(pass) & 1u, lim, abort_flag);
            ready = __shfl_sync(0xffffffffu, ready, 0);
            __syncwarp();
            if (!ready) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report_device_error(p.err, kKidDirectTc);
                }
                break;
            }
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16), v);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < kBR; ++cc) acc[cc] = __uint_as_float(v[cc]) + __uint_as_float(v[cc + kBR]);
            if (kF16) {
                // every activation warp has written its rows' scales for this pass
                int sok = 0;
                if (lane == 0)
                    sok = mbar_wait_bounded(sready_bar(pass & 1), static_cast<uint32_t>(pass >> 1) & 1u, lim, abort_flag);
                sok = __shfl_sync(0xffffffffu, sok, 0);
                __syncwarp();
                if (!sok && lane == 0) {
                    *abort_flag = 1;
                    report_device_error(p.err, kKidDirectTc);
                }
#pragma unroll
                for (int cc = 0; cc < kBR; ++cc) acc[cc] *= unscale_s[(pass & 1) * kBR + cc];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar);
            if (ksplit == 1 && j < p.n) {
                for (int cc = 0; cc < kBR && pass * kBR + cc < cnt; ++cc)
                    p.out[static_cast<int64_t>(row_of(pass * kBR + cc)) * p.n + j] = acc[cc];
            }
        }
    }
    __syncwarp();  // the TMA and MMA warps reconverge before the cluster barriers

    if (ksplit > 1 && passes > 0) {
        // at most one pass here: every CTA of the cluster has the same expert and rows
        float *part = reinterpret_cast<float *>(smem);  // [kBM][kBR], over the drained ring
        cg::cluster_group cluster = cg::this_cluster();
        const int rrow = (warp & 3) * 32 + lane;
        const bool epi = warp >= 2;
        if (epi && rank != 0) {
#pragma unroll
            for (int c = 0; c < kBR; c += 4)
                *reinterpret_cast<float4 *>(part + rrow * kBR + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
        }
        cluster.sync();  // the partial sums of every rank are visible cluster-wide
        if (epi && rank == 0) {
            for (int qr = 1; qr < ksplit; ++qr) {
                const float *rp = cluster.map_shared_rank(part, qr) + rrow * kBR;
#pragma unroll
                for (int c = 0; c < kBR; c += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(rp + c);
                    acc[c] += v.x;
                    acc[c + 1] += v.y;
                    acc[c + 2] += v.z;
                    acc[c + 3] += v.w;
                }
            }
            const int64_t j = static_cast<int64_t>(n0) + rrow;
            if (j < p.n)
                for (int c = 0; c < kBR && c < cnt; ++c) p.out[static_cast<int64_t>(row_of(c)) * p.n + j] = acc[c];
        }
        cluster.sync();  // keep every rank's shared memory alive until rank 0 has read it
    }

    // zero rows of out-of-range ids, once per output column
    if (d == 0 && rank == 0 && warp >= 2) {
        const int64_t j = static_cast<int64_t>(n0) + (warp & 3) * 32 + lane;
        if (j < p.n)
            for (int r = 0; r < n_ids; ++r)
                if (ids_s[r] >= E) p.out[static_cast<int64_t>(r) * p.n + j] = 0.f;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

int direct_tc_max_ids() { return kMaxIds; }
int direct_tc_max_experts() { return kMaxExperts; }
int direct_tc_block_rows() { return kBM; }
int direct_tc_block_k() { return kBK; }

int direct_tc_split(int64_t n, int64_t k, int64_t max_distinct, int64_t max_rows_per_expert, int num_sms) {
    // a cluster split only when one pass covers every expert's rows; the
    // largest that keeps the grid within one wave of three CTAs per SM with
    // at least four k-blocks per CTA.  A CTA keeps only three 16 KB weight
    // stages in flight (~30 GB/s alone), so a call with few experts needs
    // the split to fill the SMs: 8 experts x 12 tiles (one token, top-8)
    // took 45.7 us unsplit against 35.5 us on the FFMA kernel
    if (max_rows_per_expert > kBR) return 1;
    const int64_t units = (n + kBM - 1) / kBM * max_distinct;
    const int64_t kb = (k + kBK - 1) / kBK;
    int split = 1;
    while (split < kMaxSplit && units * (split + 1) <= 3LL * num_sms && kb >= 4LL * (split + 1)) ++split;
    return split;
}

namespace {
template <bool kF16>
cudaError_t direct_tc_t(const CUtensorMap &map_w, const MatmulIdParams &p, int max_distinct, int ksplit,
                        int x_vec_ok, cudaStream_t s) {
    static unsigned long long attr_set = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(direct_tc_kernel<kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    const int64_t tiles = (p.n + kBM - 1) / kBM;
    const int64_t grid = tiles * max_distinct * ksplit;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ksplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, direct_tc_kernel<kF16>, map_w, p, ksplit, static_cast<int>(tiles),
                              x_vec_ok);
}
}  // namespace

cudaError_t launch_matmul_id_direct_tc(int wdt, const CUtensorMap &map_w, const MatmulIdParams &p,
                                       int max_distinct, int ksplit, int x_vec_ok, cudaStream_t s) {
    if (ksplit < 1 || ksplit > kMaxSplit || max_distinct < 1 || p.total_rows > kMaxIds ||
        p.n_experts > kMaxExperts)
        return cudaErrorInvalidValue;
    switch (wdt) {
    case kF16: return direct_tc_t<true>(map_w, p, max_distinct, ksplit, x_vec_ok, s);
    case kBF16: return direct_tc_t<false>(map_w, p, max_distinct, ksplit, x_vec_ok, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbmm
