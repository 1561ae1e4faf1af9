// grouped_tc.cu -- the grouped GEMM of the GroupedPrefill route on the sm_103a
// tensor cores, for bf16 or f16 expert weights and f32 activations.
//
// Semantics: mlx-native 0.13.0, src/ops/dense_matmul_id.rs, `dense_matmul_id`
// (GroupedPrefill: per expert, the routed rows listed by the map dispatch
// times that expert's row-major [n, k] matrix, f32 output rows).
//
// For expert e and its routed rows r_0 < r_1 < ... (routed_rows[e*m + i],
// i < expert_counts[e]) the kernel computes the GEMM
//     out[r_i, j] = sum_x W_e[j, x] * xrow(r_i)[x]
// with M = routed rows (gathered), N = n, K = k, in tiles of 128 rows x 512
// outputs.  The activations are f32; tensor cores take bf16 pairs, so every
// activation is split exactly as x = hi + lo with hi = bf16(x) and
// lo = bf16(x - hi) and both halves are multiplied by the same bf16 weight
// tiles into one f32 accumulator.  The split leaves a relative error of at
// most 2^-16 on each activation (against 2^-8 for a single bf16 rounding),
// so the result stays an f32-accurate expert product.
//
// The costly operand is the activation tile: its rows are gathered, and each
// gathered row must be split into hi / lo on the SMs.  A tile 512 outputs
// wide (two 128x256 f32 accumulators, the whole tensor memory) amortises one
// gather + split over twice the weight columns of a 256-wide tile.
//
// One persistent CTA per SM, 14 warps:
//   warp 0     TMA: two 256x64 bf16 weight tiles of W_e per k-block (3-D
//              tensor map over (k, n, expert), 128-byte swizzle, L2
//              evict-normal) into a ring of its own.  No L2 prefetch of the
//              weights: with three stages in flight it only took TMA issue
//              slots (3 % slower with a prefetch 4 k-blocks ahead)
//   warp 1     TMEM allocation (512 columns) and the MMA issuer:
//              16 x tcgen05.mma (M=128, N=256, K=16) per 64-wide k-block
//   warps 2..5 epilogue: TMEM -> registers -> f32 rows of `out`, scattered to
//              their routed rows (each thread writes 128 contiguous bytes per
//              32 columns, L1 bypassed, L2 evict-first); the next 32 TMEM
//              columns are read while the current ones are stored, and each
//              256-column accumulator half has its own full / empty barrier
//              pair, so a half is drained and handed back while the MMAs of
//              the other still run
//   warps 6..13 activation producers: gather the 128 routed x rows (f32, L2
//              evict-last: each token row serves top_k experts) two k-blocks
//              ahead of use, split into bf16 hi / lo, write the 128-byte-
//              swizzled K-major smem layout the MMA descriptors expect.
// Shared memory: an activation ring of 4 stages x (x_hi 16 KB + x_lo 16 KB)
// and a weight ring of 3 stages x one 256x64 tile (32 KB).  The weight ring
// runs a half k-block at a time: a weight stage is refilled as soon as the
// MMAs of its half are done.  The activation ring's depth is what the time
// follows (measured on the MoE prefill workload): 4 + 3 stages run 4 %
// faster than 3 + 3, 3 + 4 are slower than 3 + 3, 5 + 2 13 % slower than
// 4 + 3, and at 192 KB 3 + 3 beat 4 weight + 2 activation stages by 9 %.
// Tile list: every CTA derives it from expert_counts (written by the map
// launch before this one): tiles ordered by expert, then row block, then
// output block, located through a tile prefix kept for every 8th expert (to
// leave the shared memory to the rings).  Every mbarrier wait is bounded;
// see gemm_tc.cu.
//
// Tail units.  An expert's last row block often holds only a few routed rows
// (on the Zipf prefill workload 69 of 128 experts end on a block of at most
// 64), yet an M = 128 MMA costs the same for 38 rows as for 128.  A unit
// whose row block holds r <= 64 routed rows therefore swaps the operands:
// the weights are the MMA's M side (each 256-row weight stage is two
// 128-row A tiles) and the routed rows its N side, hi in operand rows 0..r-1
// and lo in rows 64..63+r of the activation stage, N = 64 + round16(r)
// (round16(r) without the lo half).  MMAs with N below ~112 cost a fixed ~55
// cycles, so the unit's 16 MMAs per k-block cost 16 x ~55-64 cycles instead
// of 16 x 128.  Its four accumulators (one per 128 outputs) sit 128 TMEM
// columns apart; the epilogue adds columns c and 64 + c of a lane (an output
// column) and writes routed row c, a warp covering 32 consecutive outputs.
// The arithmetic is the same bf16 hi + lo products as the other units.
//
// f16 weights.  One MMA takes one operand type, so with f16 weights the
// activations are split into f16 hi + lo, and f16's range (largest finite
// 65504, normal down to 2^-14) cannot hold every f32.  Each routed row of a
// unit is therefore scaled by a power of two that puts its largest magnitude
// over the whole k range in [2^14, 2^15) (the rule of the Direct kernel),
// split, and its accumulator row multiplied back exactly in the epilogue.
// The row maxima (8 lanes per row, 16-byte loads) of a CTA's first unit are
// found by the producer warps before its first k-block, those of every later
// unit by the epilogue warps, which are idle while the tensor cores work on
// the unit before it; the scale exponents pass through shared memory,
// double-buffered by unit.
#include "device_common.cuh"

namespace gbmm {

namespace {

constexpr int kBM = 128;
constexpr int kTailRows = 64;      // row blocks of at most this many routed rows run as tail units
constexpr int kTailLo = 64;        // operand row of the lo half of routed row 0 in a tail unit
constexpr uint32_t kTailCols = 128;  // TMEM columns between the accumulators of a tail unit
constexpr int kBNH = 256;          // one accumulator / one MMA N
constexpr int kBN = 2 * kBNH;      // tile width
constexpr int kBK = 64;
constexpr int kXStages = 4;         // activation stages (x_hi + x_lo of one k-block)
constexpr int kWStages = 3;         // weight stages (one 256-row half of a k-block)
constexpr int kThreads = 448;
constexpr int kRowsPerProducer = 4;  // 8 producer warps x 32 row groups x 4 = 128 rows
constexpr int kProducerWarp0 = 6;
constexpr int kXPrefetch = 4;      // k-blocks of activation L2 prefetch ahead of the loads
constexpr uint32_t kXBytes = kBM * kBK * 2;   // one bf16 half of the activation tile
constexpr uint32_t kWBytes = kBNH * kBK * 2;  // one weight tile
constexpr uint32_t kXStageBytes = 2 * kXBytes;
constexpr uint32_t kWBase = kXStages * kXStageBytes;  // weight ring after the activation ring
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxExperts = 1024;
constexpr uint32_t kRingBytes = kWBase + kWStages * kWBytes;
constexpr int kNumBars = 2 * kXStages + 2 * kWStages + 10;  // + row-scale barriers (f16 weights)
// Tile prefix kept for every kPrefixStep-th expert only (the experts between
// are walked from their counts), so that four activation stages fit.
constexpr int kPrefixStep = 8;
constexpr uint32_t kPrefixBytes = (kMaxExperts / kPrefixStep + 2) * 4;  // coarse prefix + total tiles
constexpr uint32_t kRexpBytes = 2 * kBM;                                 // int8 row-scale exponents (f16)
constexpr uint32_t kSmemBytes = kRingBytes + kPrefixBytes + kRexpBytes + 8 * kNumBars + 16 + 1024;
static_assert((kPrefixBytes + kRexpBytes) % 8 == 0, "mbarriers need 8-byte alignment");
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM: shared memory within the opt-in limit");

static_assert(kTailLo % 8 == 0 && kTailRows <= kTailLo && kTailLo + kTailRows <= kBM,
              "a tail unit's hi and lo rows share the 128-row x_hi operand, in the same swizzle phase");
static_assert(4 * kTailCols <= kTmemCols && kTailLo + kTailRows <= static_cast<int>(kTailCols),
              "four tail accumulators of at most 128 columns fill the tensor memory");

struct GroupedTile {
    int e, mb, nb, rows;
    int n0;      // first output column of the work unit
    int halves;  // 256-column accumulator halves it computes (0: nothing to do)
    bool tail;   // rows <= kTailRows: routed rows on the MMA's N side
};

// MMA N of a tail unit with `rows` routed rows: hi rows at 0.., lo rows at kTailLo..
template <bool kSplit>
__device__ __forceinline__ uint32_t tail_n(int rows) {
    const uint32_t r16 = static_cast<uint32_t>(rows + 15) & ~15u;
    return kSplit ? static_cast<uint32_t>(kTailLo) + r16 : r16;
}

// row blocks x output blocks of expert e (its count read from the map's scratch)
__device__ __forceinline__ int expert_tiles(const uint32_t *counts, int e, int m, int nblk) {
    const int c = min(static_cast<int>(counts[e]), m);
    return (c + kBM - 1) / kBM * nblk;
}

// Tile t: expert e, row block, output block.  coarse[j] = tiles of experts
// below kPrefixStep * j; the largest j with coarse[j] <= t (of ceil(E / step)
// entries) gives the expert group, whose experts are then walked.
__device__ __forceinline__ GroupedTile decode_grouped(int t, const uint32_t *coarse, int E, int nblk,
                                                      const uint32_t *counts, int m) {
    int lo = 0, hi = (E + kPrefixStep - 1) / kPrefixStep;  // coarse[lo] <= t; t < coarse[hi] if hi < count
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (coarse[mid] <= static_cast<uint32_t>(t)) lo = mid; else hi = mid;
    }
    int e = lo * kPrefixStep;
    int base = static_cast<int>(coarse[lo]);
    const int e_end = min(E, e + kPrefixStep);
    for (; e + 1 < e_end; ++e) {
        const int te = expert_tiles(counts, e, m, nblk);
        if (t < base + te) break;
        base += te;
    }
    GroupedTile g;
    g.e = e;
    const int local = t - base;
    g.mb = local / nblk;
    g.nb = local % nblk;
    const int cnt = min(static_cast<int>(counts[e]), m);
    g.rows = min(kBM, cnt - g.mb * kBM);
    g.tail = g.rows <= kTailRows;
    return g;
}

// Work units.  Tiles [0, split_from) run whole; when the tile count does not
// divide evenly over the CTAs, each tile from split_from on is cut into two
// 256-column units, so no CTA runs more than half a tile longer than another.
// A unit whose columns start at or past n computes nothing (halves = 0), and
// a whole tile whose second half lies past n computes one half.
__device__ __forceinline__ GroupedTile decode_unit(int u, int split_from, const uint32_t *prefix, int E, int nblk,
                                                   const uint32_t *counts, int m, int64_t n) {
    const bool cut = u >= split_from;
    const int t = cut ? split_from + (u - split_from) / 2 : u;
    GroupedTile g = decode_grouped(t, prefix, E, nblk, counts, m);
    g.n0 = g.nb * kBN + (cut ? ((u - split_from) & 1) * kBNH : 0);
    const int want = cut ? 1 : 2;
    g.halves = g.n0 >= n ? 0 : (g.n0 + kBNH >= n ? 1 : want);
    return g;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float bf16_half(uint32_t packed, int half) {
    return __uint_as_float(half ? (packed & 0xffff0000u) : (packed << 16));
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// hi = round(a) (and lo = round(a - hi)) for a pair, in the weights' 16-bit type
template <bool kF16, bool kSplit>
__device__ __forceinline__ void split16(float a, float b, uint32_t &hi, uint32_t &lo) {
    if (kF16) {
        hi = pack_f16(a, b);
        if (kSplit) {
            const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
            lo = pack_f16(a - h.x, b - h.y);
        }
    } else {
        hi = pack_bf16(a, b);
        if (kSplit) lo = pack_bf16(a - bf16_half(hi, 0), b - bf16_half(hi, 1));
    }
}

// power-of-two exponent that puts a row maximum mx in [2^14, 2^15), kept
// within f32's normal range (0 for a zero row)
__device__ __forceinline__ int row_scale_exp(float mx) {
    if (!(mx > 0.f)) return 0;
    const int eb = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu);
    return min(126, max(-126, 141 - eb));
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// Parity of the row-scale full barrier of buffer j & 1 for the CTA's j-th
// unit (j >= 1): buffer 1 completes for j = 1, 3, 5, ..., buffer 0 for
// j = 2, 4, ... (the first unit's scales use their own barrier).
__device__ __forceinline__ uint32_t sfull_parity(uint32_t j) {
    return (j & 1u) ? ((j >> 1) & 1u) : (((j >> 1) & 1u) ^ 1u);
}

// one lane waits, the warp follows its verdict (keeps the warp converged)
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit,
                                          volatile int *abort_flag, int lane) {
    int ready = 0;
    if (lane == 0) ready = mbar_wait_bounded(bar, parity, limit, abort_flag);
    ready = __shfl_sync(0xffffffffu, ready, 0);
    __syncwarp();
    return ready != 0;
}

// kSplit: activations as hi + lo (two MMAs per weight tile); without it a
// single rounding (opt-in, half the tensor work).  kF16: f16 weights (row-
// scaled f16 activations), else bf16.
template <bool kSplit, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
grouped_tc_kernel(const __grid_constant__ CUtensorMap map_w, const MatmulIdParams p, int out_vec_ok) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t s_base = raw_addr + pad;
    // activation stage s at s_base + s*kXStageBytes (x_hi, x_lo); weight stage
    // s at s_base + kWBase + s*kWBytes
    uint32_t *prefix = reinterpret_cast<uint32_t *>(smem + kRingBytes);
    // coarse tile prefix, then the total tile count at prefix[kMaxExperts / kPrefixStep + 1]
    int8_t *rexp_s = reinterpret_cast<int8_t *>(smem + kRingBytes + kPrefixBytes);  // [2][kBM] (f16)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kRingBytes + kPrefixBytes + kRexpBytes);
    const uint32_t bar0 = smem_addr(bars);
    auto xfull_bar = [&](int s) { return bar0 + 8u * s; };
    auto xempty_bar = [&](int s) { return bar0 + 8u * (kXStages + s); };
    auto wfull_bar = [&](int s) { return bar0 + 8u * (2 * kXStages + s); };
    auto wempty_bar = [&](int s) { return bar0 + 8u * (2 * kXStages + kWStages + s); };
    // one full / empty pair per 256-column accumulator half
    const uint32_t acc_bar0 = bar0 + 8u * (2 * kXStages + 2 * kWStages);
    auto tfull_bar = [&](int h) { return acc_bar0 + 8u * h; };
    auto tempty_bar = [&](int h) { return acc_bar0 + 8u * (2 + h); };
    const uint32_t drain_bar = acc_bar0 + 32u;
    // f16 weights: row scales of the CTA's j-th unit, in buffer j & 1, written
    // (by the producers for j = 0: s0_bar; by the epilogue after: sfull_bar)
    // and read by the producers (sempty_bar)
    auto sfull_bar = [&](int b) { return acc_bar0 + 40u + 8u * b; };
    auto sempty_bar = [&](int b) { return acc_bar0 + 56u + 8u * b; };
    const uint32_t s0_bar = acc_bar0 + 72u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ uint32_t warp_tot[kThreads / 32];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = static_cast<int>(p.n_experts);
    const int m = static_cast<int>(p.m);
    const int nblk = static_cast<int>((p.n + kBN - 1) / kBN);
    const uint64_t lim = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(xfull_bar(s), 8);   // one arrive per producer warp
            mbar_init(xempty_bar(s), 1);  // MMA commit
        }
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(wfull_bar(s), 1);   // TMA thread's arrive + the copy's bytes
            mbar_init(wempty_bar(s), 1);  // MMA commit
        }
        mbar_init(tfull_bar(0), 1);
        mbar_init(tfull_bar(1), 1);
        mbar_init(tempty_bar(0), 4);
        mbar_init(tempty_bar(1), 4);
        mbar_init(drain_bar, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(sfull_bar(b), 4);   // one arrive per epilogue warp
            mbar_init(sempty_bar(b), 8);  // one arrive per producer warp
        }
        mbar_init(s0_bar, 8);  // one arrive per producer warp
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&map_w);
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }

    // Launched right behind the map kernel with programmatic stream
    // serialisation: the set-up above may overlap the map's tail; nothing
    // global is read or written before the map grid has completed.
    grid_dep_wait();

    // tile prefix over experts, sum_{e' < e} ceil(count/128) * nblk, kept for
    // e a multiple of kPrefixStep, and the total
    {
        constexpr int kPer = 3;  // 448 threads x 3 >= 1024 + 1 entries
        uint32_t v[kPer];
        uint32_t sum = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int e = threadIdx.x * kPer + q;
            uint32_t t = 0;
            if (e < E) {
                const uint32_t c = min(p.counts[e], static_cast<uint32_t>(m));
                t = (c + kBM - 1) / kBM * static_cast<uint32_t>(nblk);
            }
            v[q] = t;
            sum += t;
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        uint32_t base = 0;
        for (int w = 0; w < warp; ++w) base += warp_tot[w];
        uint32_t run = base + incl - sum;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int e = threadIdx.x * kPer + q;
            if (e == E) prefix[kMaxExperts / kPrefixStep + 1] = run;
            else if (e < E && e % kPrefixStep == 0) prefix[e / kPrefixStep] = run;
            run += v[q];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int num_tiles = static_cast<int>(prefix[kMaxExperts / kPrefixStep + 1]);
    const int grid = static_cast<int>(gridDim.x);
    const int tail = num_tiles > grid ? num_tiles % grid : (2 * num_tiles <= grid ? num_tiles : 0);
    const int split_from = num_tiles - tail;
    const int num_units = split_from + 2 * tail;
    const int kblocks = static_cast<int>((p.k + kBK - 1) / kBK);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- weight tiles (TMA) ----------------
            // evict-normal: the row blocks of an expert read its weight slab
            // close together in time (evict-first measured 7 % slower)
            const uint64_t pol = policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0, issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                const GroupedTile g = decode_unit(u, split_from, prefix, E, nblk, p.counts, m, p.n);
                if (g.halves == 0) continue;
                const int n0 = g.n0;
                for (int kb = 0; kb < kblocks && ok; ++kb) {
                    for (int h = 0; h < g.halves; ++h) {
                        if (!mbar_wait_bounded(wempty_bar(stage), phase ^ 1u, lim, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(wfull_bar(stage), kWBytes);
                        tma_load_3d_hint(s_base + kWBase + stage * kWBytes, &map_w, wfull_bar(stage), kb * kBK,
                                         n0 + h * kBNH, g.e, pol);
                        ++issued;
                        if (++stage == kWStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                report_device_error(p.err, kKidGroupedTc);
                // let the copies in flight land before the CTA can exit
                for (int s = 0; s < kWStages; ++s) {
                    const uint32_t n_s = issued / kWStages + (static_cast<uint32_t>(s) < issued % kWStages ? 1u : 0u);
                    if (n_s > 0) mbar_wait_bounded(wfull_bar(s), (n_s - 1u) & 1u, lim, nullptr);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t kFmt = kF16 ? 0u : 1u;                 // f16 or bf16 operands
            constexpr uint32_t kIdesc = idesc_f16(kFmt, kBM, kBNH);  // 16-bit x 16-bit -> f32
            int xs = 0, ws = 0;
            uint32_t xph = 0, wph = 0, acc_phase[2] = {0u, 0u};
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                const GroupedTile g = decode_unit(u, split_from, prefix, E, nblk, p.counts, m, p.n);
                if (g.halves == 0) continue;
                // tail unit: weights as A (M = 128), the routed rows as B (N rows)
                const uint32_t idesc_tail = idesc_f16(kFmt, kBM, tail_n<kSplit>(g.rows));
                for (int kb = 0; kb < kblocks && ok; ++kb) {
                    if (!mbar_wait_bounded(xfull_bar(xs), xph, lim, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t s_hi = s_base + xs * kXStageBytes;
                    const uint32_t s_lo = s_hi + kXBytes;
                    for (int h = 0; h < g.halves && g.tail; ++h) {
                        if (kb == 0 && !mbar_wait_bounded(tempty_bar(h), acc_phase[h] ^ 1u, lim, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait_bounded(wfull_bar(ws), wph, lim, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t s_w = s_base + kWBase + ws * kWBytes;
#pragma unroll
                        for (int m2 = 0; m2 < 2; ++m2) {
                            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(2 * h + m2) * kTailCols;
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk)
                                umma_f16_ss(d_tmem, sdesc_kmajor_sw128(s_w + m2 * (kBM * 128) + kk * 32),
                                            sdesc_kmajor_sw128(s_hi + kk * 32), idesc_tail, (kb | kk) != 0 ? 1u : 0u);
                        }
                        umma_commit(wempty_bar(ws));
                        // this half's accumulator is final: the epilogue may start on it
                        // while the other half's last MMAs run
                        if (kb == kblocks - 1) umma_commit(tfull_bar(h));
                        if (++ws == kWStages) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    }
                    for (int h = 0; h < g.halves && !g.tail; ++h) {
                        // accumulator half h drained by the epilogue of the previous unit
                        if (kb == 0 && !mbar_wait_bounded(tempty_bar(h), acc_phase[h] ^ 1u, lim, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait_bounded(wfull_bar(ws), wph, lim, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t s_w = s_base + kWBase + ws * kWBytes;
                        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(h * kBNH);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            const uint64_t dw = sdesc_kmajor_sw128(s_w + kk * 32);
                            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                            umma_f16_ss(d_tmem, sdesc_kmajor_sw128(s_hi + kk * 32), dw, kIdesc, acc);
                            if (kSplit) umma_f16_ss(d_tmem, sdesc_kmajor_sw128(s_lo + kk * 32), dw, kIdesc, 1u);
                        }
                        umma_commit(wempty_bar(ws));
                        // this half's accumulator is final: the epilogue may start on it
                        // while the other half's last MMAs run
                        if (kb == kblocks - 1) umma_commit(tfull_bar(h));
                        if (++ws == kWStages) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(xempty_bar(xs));
                    if (++xs == kXStages) {
                        xs = 0;
                        xph ^= 1u;
                    }
                }
                if (!ok) break;
                for (int h = 0; h < g.halves; ++h) acc_phase[h] ^= 1u;
            }
            if (!ok) {
                *abort_flag = 1;
                report_device_error(p.err, kKidGroupedTc);
            }
            umma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, lim, nullptr);
        }
    } else if (warp < kProducerWarp0) {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;
        uint32_t acc_phase = 0;  // bit h: phase of accumulator half h
        bool ok = true;
        // wait until accumulator half h of the current unit is final
        auto wait_half = [&](int h) -> bool {
            if (!warp_wait(tfull_bar(h), (acc_phase >> h) & 1u, lim, abort_flag, lane)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report_device_error(p.err, kKidGroupedTc);
                }
                return false;
            }
            tc_fence_after();
            return true;
        };
        // all of half h is in registers or stored: hand it back to the MMA issuer
        auto hand_back = [&](int h) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(h));
        };
        // the CTA's next unit with work after u (num_units: none)
        auto next_unit = [&](int u) -> int {
            for (u += gridDim.x; u < num_units; u += gridDim.x)
                if (decode_unit(u, split_from, prefix, E, nblk, p.counts, m, p.n).halves > 0) return u;
            return num_units;
        };
        // f16 weights: the scale exponents of unit u (the CTA's j-th unit with
        // work) into buffer j & 1, each warp taking rows 16 g + 4 quarter +
        // lane / 8 (g < 8), 8 lanes per row with 16 loads of 16 bytes in flight
        const uint64_t xpol = policy_evict_last();
        auto row_scales = [&](int u, uint32_t j) -> bool {
            const GroupedTile g = decode_unit(u, split_from, prefix, E, nblk, p.counts, m, p.n);
            const int b = static_cast<int>(j & 1u);
            // the producers have read buffer b's scales of unit j - 2
            if (!warp_wait(sempty_bar(b), ((j >> 1) & 1u) ^ 1u, lim, abort_flag, lane)) return false;
            const int sub = lane & 7;
            for (int g4 = 0; g4 < kBM / 16; ++g4) {
                const int i = 16 * g4 + 4 * quarter + (lane >> 3);
                if (16 * g4 >= g.rows) break;  // warp-uniform: no row of this group or later
                const float *src = nullptr;
                if (i < g.rows) {
                    const uint32_t r = p.routed_rows[static_cast<int64_t>(g.e) * m + g.mb * kBM + i];
                    const int64_t tok = r / p.top_k, slot = r % p.top_k;
                    src = p.x + tok * p.x_token_stride + slot * p.x_slot_stride + sub * 4;
                }
                float mx = 0.f;
                for (int64_t c0 = 0; c0 < p.k; c0 += 32 * 16) {
                    float4 a[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const int64_t kk = c0 + 32 * t;
                        a[t] = (src != nullptr && kk + sub * 4 < p.k) ? ld_f4_policy(src + kk, xpol)
                                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(a[t].x), fabsf(a[t].y)), fmaxf(fabsf(a[t].z), fabsf(a[t].w))));
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (sub == 0) rexp_s[b * kBM + i] = static_cast<int8_t>(row_scale_exp(mx));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sfull_bar(b));
            return true;
        };
        uint32_t uc = 0;  // units with work so far (row-scale buffer uc & 1)
        int u = blockIdx.x;
        while (u < num_units && decode_unit(u, split_from, prefix, E, nblk, p.counts, m, p.n).halves == 0)
            u += gridDim.x;
        int u1 = u < num_units ? next_unit(u) : num_units;
        // unit 1's scales while the producers find unit 0's
        if (kF16 && u1 < num_units && !(ok = row_scales(u1, 1)) && lane == 0) {
            *abort_flag = 1;
            report_device_error(p.err, kKidGroupedTc);
        }
        for (; u < num_units && ok;) {
            const GroupedTile g = decode_unit(u, split_from, prefix, E, nblk, p.counts, m, p.n);
            const int sb = static_cast<int>(uc & 1u);
            const int8_t *rexp = rexp_s + sb * kBM;
            if (kF16) {
                // this unit's scales, complete from all their writers
                const bool ready = uc == 0 ? warp_wait(s0_bar, 0u, lim, abort_flag, lane)
                                           : warp_wait(sfull_bar(sb), sfull_parity(uc), lim, abort_flag, lane);
                ok = ready;
                if (!ok) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_device_error(p.err, kKidGroupedTc);
                    }
                    break;
                }
            }
            // after this unit's rows are stored: the scales of the unit after
            // the next one (its buffer is this unit's), while the next runs
            auto advance = [&]() {
                const int u2 = u1 < num_units ? next_unit(u1) : num_units;
                if (kF16 && ok && u2 < num_units && !(ok = row_scales(u2, uc + 2)) && lane == 0) {
                    *abort_flag = 1;
                    report_device_error(p.err, kKidGroupedTc);
                }
                ++uc;
                u = u1;
                u1 = u2;
            };
            if (g.tail) {
                // lane = output column n0 + 128 q + 32 quarter + lane; TMEM column
                // c (hi) + column kTailLo + c (lo) of accumulator q = routed row c
                const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
                const int64_t row_base = static_cast<int64_t>(g.e) * m + g.mb * kBM;
                for (int q = 0; q < 2 * g.halves && ok; ++q) {
                    if (!(q & 1) && !(ok = wait_half(q >> 1))) break;
                    const int64_t j = static_cast<int64_t>(g.n0) + q * kBM + quarter * 32 + lane;
                    for (int c0 = 0; c0 < g.rows; c0 += 32) {
                        uint32_t vh[32], vl[32];
                        tmem_ld32(t_lane + static_cast<uint32_t>(q) * kTailCols + c0, vh);
                        if (kSplit) tmem_ld32(t_lane + static_cast<uint32_t>(q) * kTailCols + kTailLo + c0, vl);
                        tmem_ld_wait();
                        const uint32_t my_r = c0 + lane < g.rows ? p.routed_rows[row_base + c0 + lane] : 0u;
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const uint32_t r = __shfl_sync(0xffffffffu, my_r, c);
                            if (c0 + c < g.rows && j < p.n) {
                                float v = kSplit ? __uint_as_float(vh[c]) + __uint_as_float(vl[c])
                                                 : __uint_as_float(vh[c]);
                                if (kF16) v *= pow2f(-rexp[c0 + c]);
                                __stcs(p.out + static_cast<int64_t>(r) * p.n + j, v);
                            }
                        }
                    }
                    // both accumulators of this 256-column half are read
                    if (q & 1) hand_back(q >> 1);
                }
                acc_phase ^= (1u << g.halves) - 1u;
                advance();
                continue;
            }
            const int i = quarter * 32 + lane;
            const bool valid = i < g.rows;
            const int64_t r = valid ? static_cast<int64_t>(p.routed_rows[static_cast<int64_t>(g.e) * m +
                                                                         g.mb * kBM + i])
                                    : 0;
            float *orow = p.out + r * p.n;
            const float rs = kF16 ? pow2f(-rexp[i]) : 1.f;  // exact power of two
            const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            const uint64_t spol = policy_evict_first();
            constexpr int kChunksPerHalf = kBNH / 32;
            static_assert(kChunksPerHalf % 2 == 0, "chunks are read in pairs");
            const int nch = g.halves * kChunksPerHalf;
            auto store_chunk = [&](uint32_t (&v)[32], int chunk) {
                const int64_t j0 = static_cast<int64_t>(g.n0) + chunk * 32;
                if (!valid || j0 >= p.n) return;
                if (kF16) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * rs);
                }
                if (out_vec_ok == 2 && j0 + 32 <= p.n) {
                    // whole 32-byte sectors per store: no partial-sector writes in L2;
                    // not kept in L1, evict-first in L2 (1 % faster than .cs stores)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        asm volatile(
                            "st.global.L1::no_allocate.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(orow + j0 + 8 * q),
                            "r"(v[8 * q]), "r"(v[8 * q + 1]), "r"(v[8 * q + 2]), "r"(v[8 * q + 3]),
                            "r"(v[8 * q + 4]), "r"(v[8 * q + 5]), "r"(v[8 * q + 6]), "r"(v[8 * q + 7]), "l"(spol)
                            : "memory");
                } else if (out_vec_ok && j0 + 32 <= p.n) {
                    float4 *dst = reinterpret_cast<float4 *>(orow + j0);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        __stcs(dst + q, make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                    __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (j0 + c < p.n) orow[j0 + c] = __uint_as_float(v[c]);
                }
            };
            // Two register buffers: chunk c + 1 is read from tensor memory while
            // chunk c is stored.  A half goes back to the MMA issuer as soon as
            // its last chunk has arrived in registers.
            uint32_t va[32], vb[32];
            if (!(ok = wait_half(0))) break;
            tmem_ld32(t_addr, va);
#pragma unroll 1
            for (int chunk = 0; chunk < nch && ok; chunk += 2) {
                tmem_ld_wait();  // va = chunk
                tmem_ld32(t_addr + (chunk + 1) * 32, vb);
                store_chunk(va, chunk);
                tmem_ld_wait();  // vb = chunk + 1
                if ((chunk + 2) % kChunksPerHalf == 0) hand_back((chunk + 1) / kChunksPerHalf);
                if (chunk + 2 < nch) {
                    if ((chunk + 2) % kChunksPerHalf == 0 && !(ok = wait_half((chunk + 2) / kChunksPerHalf))) break;
                    tmem_ld32(t_addr + (chunk + 2) * 32, va);
                }
                store_chunk(vb, chunk + 1);
            }
            acc_phase ^= (1u << g.halves) - 1u;
            advance();
        }
    } else {
        // ---------------- activation producers (warps 6..13) ----------------
        // Each thread owns one 16-byte chunk (8 elements) of the 64-wide k-block
        // in 4 rows.  Loads run two k-blocks ahead of the conversion, in a
        // ring of registers, so gathered rows stream in while earlier stages
        // are converted and while the tensor cores are busy.
        const int tid = threadIdx.x - kProducerWarp0 * 32;  // 0..255
        const int sub = tid & 7;
        const int rsub = tid >> 3;  // rows rsub + 32 q, q < 4
        const uint64_t pol = policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t uc = 0;  // units with work so far (row-scale buffer uc & 1)
        bool ok = true;
        for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
            const GroupedTile g = decode_unit(u, split_from, prefix, E, nblk, p.counts, m, p.n);
            if (g.halves == 0) continue;
            const float *src[kRowsPerProducer];
#pragma unroll
            for (int q = 0; q < kRowsPerProducer; ++q) {
                const int i = rsub + 32 * q;
                src[q] = nullptr;
                if (i < g.rows) {
                    const uint32_t r = p.routed_rows[static_cast<int64_t>(g.e) * m + g.mb * kBM + i];
                    const int64_t tok = r / p.top_k, slot = r % p.top_k;
                    src[q] = p.x + tok * p.x_token_stride + slot * p.x_slot_stride + sub * 8;
                }
            }
            // f16 weights: each row's scale from its largest magnitude over k
            float scl[kRowsPerProducer];
#pragma unroll
            for (int q = 0; q < kRowsPerProducer; ++q) scl[q] = 1.f;
            if (kF16 && uc == 0) {
                // the CTA's first unit: its row maxima over k, before its first k-block
                float mx[kRowsPerProducer];
#pragma unroll
                for (int q = 0; q < kRowsPerProducer; ++q) mx[q] = 0.f;
                for (int kb = 0; kb < kblocks; kb += 2) {
                    float4 a[2][kRowsPerProducer][2];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const bool in_k = kb + t < kblocks && static_cast<int64_t>(kb + t) * kBK + sub * 8 < p.k;
#pragma unroll
                        for (int q = 0; q < kRowsPerProducer; ++q) {
                            if (in_k && src[q] != nullptr) {
                                a[t][q][0] = ld_f4_policy(src[q] + static_cast<int64_t>(kb + t) * kBK, pol);
                                a[t][q][1] = ld_f4_policy(src[q] + static_cast<int64_t>(kb + t) * kBK + 4, pol);
                            } else {
                                a[t][q][0] = make_float4(0.f, 0.f, 0.f, 0.f);
                                a[t][q][1] = a[t][q][0];
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int q = 0; q < kRowsPerProducer; ++q)
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                mx[q] = fmaxf(mx[q], fmaxf(fmaxf(fabsf(a[t][q][h].x), fabsf(a[t][q][h].y)),
                                                           fmaxf(fabsf(a[t][q][h].z), fabsf(a[t][q][h].w))));
                }
                // the 8 lanes of a row (sub = lane & 7) combine their maxima
#pragma unroll
                for (int q = 0; q < kRowsPerProducer; ++q) {
#pragma unroll
                    for (int o = 1; o < 8; o <<= 1) mx[q] = fmaxf(mx[q], __shfl_xor_sync(0xffffffffu, mx[q], o));
                    const int se = row_scale_exp(mx[q]);
                    scl[q] = pow2f(se);
                    if (sub == 0) rexp_s[rsub + 32 * q] = static_cast<int8_t>(se);  // buffer 0, for the epilogue
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(s0_bar);
                    mbar_arrive(sempty_bar(0));  // scales kept in registers
                }
            } else if (kF16) {
                // the epilogue warps have found this unit's row scales
                const int sb = static_cast<int>(uc & 1u);
                if (!warp_wait(sfull_bar(sb), sfull_parity(uc), lim, abort_flag, lane)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_device_error(p.err, kKidGroupedTc);
                    }
                    ok = false;
                    break;
                }
#pragma unroll
                for (int q = 0; q < kRowsPerProducer; ++q) scl[q] = pow2f(rexp_s[sb * kBM + rsub + 32 * q]);
                __syncwarp();
                if (lane == 0) mbar_arrive(sempty_bar(sb));
            }
            ++uc;
            float4 ring0[kRowsPerProducer][2], ring1[kRowsPerProducer][2], ring2[kRowsPerProducer][2];
            auto issue = [&](float4 (&buf)[kRowsPerProducer][2], int kb) {
                // L2 prefetch of the rows' segment kXPrefetch k-blocks further on:
                // one thread per 128-byte line (chunks 0 and 4 of the 256-byte segment)
                if ((sub & 3) == 0 && kb + kXPrefetch < kblocks &&
                    static_cast<int64_t>(kb + kXPrefetch) * kBK + sub * 8 < p.k) {
#pragma unroll
                    for (int q = 0; q < kRowsPerProducer; ++q)
                        if (src[q] != nullptr)
                            prefetch_l2_evict_last(src[q] + static_cast<int64_t>(kb + kXPrefetch) * kBK);
                }
                const bool in_k = kb < kblocks && static_cast<int64_t>(kb) * kBK + sub * 8 < p.k;
#pragma unroll
                for (int q = 0; q < kRowsPerProducer; ++q) {
                    if (in_k && src[q] != nullptr) {
                        buf[q][0] = ld_f4_policy(src[q] + static_cast<int64_t>(kb) * kBK, pol);
                        buf[q][1] = ld_f4_policy(src[q] + static_cast<int64_t>(kb) * kBK + 4, pol);
                    } else {
                        buf[q][0] = make_float4(0.f, 0.f, 0.f, 0.f);
                        buf[q][1] = buf[q][0];
                    }
                }
            };
            auto consume = [&](float4 (&buf)[kRowsPerProducer][2]) -> bool {
                if (!warp_wait(xempty_bar(stage), phase ^ 1u, lim, abort_flag, lane)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_device_error(p.err, kKidGroupedTc);
                    }
                    return false;
                }
                const uint32_t s_hi = s_base + stage * kXStageBytes;
#pragma unroll
                for (int q = 0; q < kRowsPerProducer; ++q) {
                    const int i = rsub + 32 * q;
                    // a tail unit keeps its lo rows where the hi rows past its count would go
                    if (g.tail && i >= g.rows) continue;
                    const float f[8] = {buf[q][0].x, buf[q][0].y, buf[q][0].z, buf[q][0].w,
                                        buf[q][1].x, buf[q][1].y, buf[q][1].z, buf[q][1].w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (kF16)
                            split16<true, kSplit>(f[2 * h] * scl[q], f[2 * h + 1] * scl[q], hi[h], lo[h]);
                        else
                            split16<false, kSplit>(f[2 * h], f[2 * h + 1], hi[h], lo[h]);
                    }
                    // 128-byte swizzle: 16-byte chunk c of row i sits at chunk c ^ (i % 8)
                    const uint32_t off = static_cast<uint32_t>(i) * 128u +
                                         (static_cast<uint32_t>(sub ^ (i & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(s_hi + off), "r"(hi[0]),
                                 "r"(hi[1]), "r"(hi[2]), "r"(hi[3])
                                 : "memory");
                    // lo: row kTailLo + i of the same operand in a tail unit (same
                    // swizzle phase: kTailLo is a multiple of 8), else row i of x_lo
                    const uint32_t lo_addr = g.tail ? s_hi + off + static_cast<uint32_t>(kTailLo) * 128u
                                                    : s_hi + kXBytes + off;
                    if (kSplit)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(lo_addr),
                                     "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                                     : "memory");
                }
                fence_async_smem();  // generic-proxy writes -> visible to the tensor cores
                __syncwarp();
                if (lane == 0) mbar_arrive(xfull_bar(stage));
                if (++stage == kXStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                return true;
            };
            issue(ring0, 0);
            issue(ring1, 1);
            for (int kb = 0; kb < kblocks && ok; kb += 3) {
                issue(ring2, kb + 2);
                ok = consume(ring0);
                if (!ok || kb + 1 >= kblocks) break;
                issue(ring0, kb + 3);
                ok = consume(ring1);
                if (!ok || kb + 2 >= kblocks) break;
                issue(ring1, kb + 4);
                ok = consume(ring2);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

namespace {
template <bool kSplit, bool kF16>
cudaError_t grouped_tc_t(const CUtensorMap &map_w, const MatmulIdParams &p, int out_vec_ok, int num_sms,
                         cudaStream_t s) {
    static unsigned long long attr_set = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(grouped_tc_kernel<kSplit, kF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    // may start while the map kernel before it finishes (it waits for it
    // before touching global memory)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, grouped_tc_kernel<kSplit, kF16>, map_w, p, out_vec_ok);
}
}  // namespace

cudaError_t launch_matmul_id_grouped_tc(const CUtensorMap &map_w, const MatmulIdParams &p, int out_vec_ok,
                                        int split, int f16, int num_sms, cudaStream_t s) {
    if (f16)
        return split ? grouped_tc_t<true, true>(map_w, p, out_vec_ok, num_sms, s)
                     : grouped_tc_t<false, true>(map_w, p, out_vec_ok, num_sms, s);
    return split ? grouped_tc_t<true, false>(map_w, p, out_vec_ok, num_sms, s)
                 : grouped_tc_t<false, false>(map_w, p, out_vec_ok, num_sms, s);
}

int grouped_tc_max_experts() { return kMaxExperts; }
int grouped_tc_block_k() { return kBK; }

}  // namespace gbmm
