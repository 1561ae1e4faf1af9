// matmul_id.cu -- expert-ID matrix multiplication: the Direct route, the
// routing map of the GroupedPrefill route, and the FFMA grouped GEMM used
// for weight dtypes the tensor-core grouped kernel does not take.
//
// Semantics: mlx-native 0.13.0, src/ops/dense_matmul_id.rs -- module
// contract (a strided stack of row-major [n, k] expert matrices, f32
// activations, f32 output), `dense_matmul_id` (input token/slot strides per
// layout; an id outside n_experts gives a zero output row without forming a
// weight address), `DenseMatmulIdScratch` (expert_counts, routed_rows).
//
// Direct route.  The pages launch one thread group per (8 outputs, routed
// row).  Here a CTA owns (routed row r, a tile of 32 expert rows j).  The
// routed rows are cut into windows of 256; the CTA of the FIRST routed row
// in a window that selects expert e computes every row of that window that
// selects e, and the CTAs of later rows with the same expert exit at once.
// So each distinct expert of a window is streamed from HBM once, whatever
// the number of tokens that picked it.  Rows of W are read as coalesced
// 16-byte vectors (L1 bypassed), activations through L1.
//
// Routing map.  One cluster of 8 CTAs x 32 warps builds expert_counts and
// routed_rows without atomics: each warp owns a contiguous segment of routed
// rows and counts it per expert (lanes holding the same id are found with
// one warp match instruction; one leader lane per distinct id updates the
// warp's private counter row in shared memory), the per
// expert counts are scanned across warps and, through distributed shared
// memory, across the cluster's CTAs in row order, and a second pass
// scatters every row index to its final, ascending position.  Extra CTAs of
// the same launch zero-fill output rows whose id is out of range.
#include <cooperative_groups.h>

#include <type_traits>

#include "device_common.cuh"

namespace cg = cooperative_groups;

namespace gbmm {

namespace {

constexpr int kDirectThreads = 256;
constexpr int kDirectRows = 32;     // expert rows (outputs j) per CTA
constexpr int kDirectWindow = 256;  // routed rows searched for sharers (== threads)
constexpr int kDirectXR = 4;        // routed rows per pass over the W tile
constexpr int kDirectUnroll = 8;    // 16-byte W vectors in flight per lane

__device__ __forceinline__ const float *x_row(const MatmulIdParams &p, uint32_t r) {
    const int64_t t = r / p.top_k;
    const int64_t s = r % p.top_k;
    return p.x + t * p.x_token_stride + s * p.x_slot_stride;
}

// One pass of a warp over its expert rows j (j0 + warp, step 8) for up to NR
// routed rows (nr of them live) that selected the same expert.
template <typename TW, int NR>
__device__ __forceinline__ void direct_pass(const MatmulIdParams &p, const TW *W, const uint32_t *rows,
                                            int nr, int64_t j0, int64_t j1, int warp, int lane,
                                            int vec_ok) {
    constexpr int V = Elem<TW>::kVec;
    const float *xr[NR];
    uint32_t orow[NR];
#pragma unroll
    for (int q = 0; q < NR; ++q) {
        orow[q] = rows[q < nr ? q : 0];
        xr[q] = x_row(p, orow[q]);
    }
    for (int64_t j = j0 + warp; j < j1; j += kDirectThreads / 32) {
        const TW *wrow = W + j * p.k;
        float acc[NR];
#pragma unroll
        for (int q = 0; q < NR; ++q) acc[q] = 0.f;
        int64_t x_done = 0;
        if (vec_ok) {
            const int64_t nch = p.k / V;
            int64_t c0 = 0;
            for (; c0 + 32 * kDirectUnroll <= nch; c0 += 32 * kDirectUnroll) {
                uint4 wv[kDirectUnroll];
#pragma unroll
                for (int u = 0; u < kDirectUnroll; ++u) wv[u] = ld_stream16(wrow + (c0 + u * 32 + lane) * V);
#pragma unroll
                for (int u = 0; u < kDirectUnroll; ++u) {
                    float wf[V];
                    unpack16<TW>(wv[u], wf);
                    const int64_t xo = (c0 + u * 32 + lane) * V;
#pragma unroll
                    for (int q = 0; q < NR; ++q) {
                        if (NR == 1 || q < nr) {
#pragma unroll
                            for (int h = 0; h < V / 4; ++h) {
                                const float4 xv = __ldg(reinterpret_cast<const float4 *>(xr[q] + xo) + h);
                                acc[q] = fmaf(wf[4 * h + 0], xv.x, acc[q]);
                                acc[q] = fmaf(wf[4 * h + 1], xv.y, acc[q]);
                                acc[q] = fmaf(wf[4 * h + 2], xv.z, acc[q]);
                                acc[q] = fmaf(wf[4 * h + 3], xv.w, acc[q]);
                            }
                        }
                    }
                }
            }
            for (int64_t c = c0 + lane; c < nch; c += 32) {
                float wf[V];
                unpack16<TW>(ld_stream16(wrow + c * V), wf);
#pragma unroll
                for (int q = 0; q < NR; ++q) {
                    if (NR == 1 || q < nr) {
#pragma unroll
                        for (int h = 0; h < V / 4; ++h) {
                            const float4 xv = __ldg(reinterpret_cast<const float4 *>(xr[q] + c * V) + h);
                            acc[q] = fmaf(wf[4 * h + 0], xv.x, acc[q]);
                            acc[q] = fmaf(wf[4 * h + 1], xv.y, acc[q]);
                            acc[q] = fmaf(wf[4 * h + 2], xv.z, acc[q]);
                            acc[q] = fmaf(wf[4 * h + 3], xv.w, acc[q]);
                        }
                    }
                }
            }
            x_done = nch * V;
        }
        for (int64_t x = x_done + lane; x < p.k; x += 32) {
            const float wv = Elem<TW>::to_f(wrow[x]);
#pragma unroll
            for (int q = 0; q < NR; ++q)
                if (NR == 1 || q < nr) acc[q] = fmaf(wv, xr[q][x], acc[q]);
        }
#pragma unroll
        for (int q = 0; q < NR; ++q) acc[q] = warp_sum(acc[q]);
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < NR; ++q)
                if (NR == 1 || q < nr) p.out[static_cast<int64_t>(orow[q]) * p.n + j] = acc[q];
        }
    }
}

// The decode case: one routed row per expert.  A warp streams two expert rows
// (j and j + 8) at once, so twice the 16-byte loads are in flight per lane.
template <typename TW>
__device__ __forceinline__ void direct_pass_single(const MatmulIdParams &p, const TW *W, uint32_t orow,
                                                   int64_t j0, int64_t j1, int warp, int lane) {
    constexpr int V = Elem<TW>::kVec;
    const float *xr = x_row(p, orow);
    const int64_t nch = p.k / V;
    constexpr int kStep = kDirectThreads / 32;
    for (int64_t ja = j0 + warp; ja < j1; ja += 2 * kStep) {
        const int64_t jb = ja + kStep;
        const bool has_b = jb < j1;
        const TW *wa = W + ja * p.k;
        const TW *wb = W + (has_b ? jb : ja) * p.k;
        float acc_a = 0.f, acc_b = 0.f;
        for (int64_t c0 = 0; c0 < nch; c0 += 32 * kDirectUnroll) {
            uint4 va[kDirectUnroll], vb[kDirectUnroll];
#pragma unroll
            for (int u = 0; u < kDirectUnroll; ++u) {
                const int64_t c = c0 + u * 32 + lane;
                const bool in = c < nch;
                va[u] = in ? ld_stream16(wa + c * V) : make_uint4(0u, 0u, 0u, 0u);
                vb[u] = in && has_b ? ld_stream16(wb + c * V) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kDirectUnroll; ++u) {
                const int64_t c = c0 + u * 32 + lane;
                if (c < nch) {
                    float fa[V], fb[V];
                    unpack16<TW>(va[u], fa);
                    unpack16<TW>(vb[u], fb);
#pragma unroll
                    for (int h = 0; h < V / 4; ++h) {
                        const float4 xv = __ldg(reinterpret_cast<const float4 *>(xr + c * V) + h);
                        acc_a = fmaf(fa[4 * h + 0], xv.x, acc_a);
                        acc_a = fmaf(fa[4 * h + 1], xv.y, acc_a);
                        acc_a = fmaf(fa[4 * h + 2], xv.z, acc_a);
                        acc_a = fmaf(fa[4 * h + 3], xv.w, acc_a);
                        acc_b = fmaf(fb[4 * h + 0], xv.x, acc_b);
                        acc_b = fmaf(fb[4 * h + 1], xv.y, acc_b);
                        acc_b = fmaf(fb[4 * h + 2], xv.z, acc_b);
                        acc_b = fmaf(fb[4 * h + 3], xv.w, acc_b);
                    }
                }
            }
        }
        for (int64_t x = nch * V + lane; x < p.k; x += 32) {
            acc_a = fmaf(Elem<TW>::to_f(wa[x]), xr[x], acc_a);
            acc_b = fmaf(Elem<TW>::to_f(wb[x]), xr[x], acc_b);
        }
        acc_a = warp_sum(acc_a);
        acc_b = warp_sum(acc_b);
        if (lane == 0) {
            p.out[static_cast<int64_t>(orow) * p.n + ja] = acc_a;
            if (has_b) p.out[static_cast<int64_t>(orow) * p.n + jb] = acc_b;
        }
    }
}

template <typename TW>
__global__ void __launch_bounds__(kDirectThreads)
matmul_id_direct_kernel(MatmulIdParams p, int vec_ok) {
    __shared__ uint32_t s_list[kDirectWindow];
    __shared__ int s_warp_cnt[kDirectThreads / 32];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    for (int64_t r = blockIdx.x; r < p.total_rows; r += gridDim.x) {
        for (int64_t jt = blockIdx.y; jt * kDirectRows < p.n; jt += gridDim.y) {
            const int64_t j0 = jt * kDirectRows;
            const int64_t j1 = j0 + kDirectRows < p.n ? j0 + kDirectRows : p.n;
            const uint32_t e = p.ids[r];
            if (e >= static_cast<uint32_t>(p.n_experts)) {
                for (int64_t j = j0 + tid; j < j1; j += blockDim.x) p.out[r * p.n + j] = 0.f;
                continue;
            }
            const int64_t w0 = (r / kDirectWindow) * kDirectWindow;
            const int64_t w1 = w0 + kDirectWindow < p.total_rows ? w0 + kDirectWindow : p.total_rows;
            const int64_t rr = w0 + tid;
            const uint32_t my_e = rr < w1 ? p.ids[rr] : 0xffffffffu;
            // an earlier row of the window selected the same expert: it owns the work
            if (__syncthreads_or(rr < r && my_e == e)) continue;
            const bool mine = rr >= r && rr < w1 && my_e == e;
            const unsigned bal = __ballot_sync(0xffffffffu, mine);
            if (lane == 0) s_warp_cnt[warp] = __popc(bal);
            __syncthreads();
            int off = 0, total = 0;
            for (int w = 0; w < kDirectThreads / 32; ++w) {
                if (w < warp) off += s_warp_cnt[w];
                total += s_warp_cnt[w];
            }
            if (mine) s_list[off + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint32_t>(rr);
            __syncthreads();

            const TW *W = static_cast<const TW *>(p.w) + static_cast<int64_t>(e) * p.expert_stride_elems;
            for (int l0 = 0; l0 < total; l0 += kDirectXR) {
                const int nr = total - l0 < kDirectXR ? total - l0 : kDirectXR;
                // the common decode case is one routed row per expert: specialise
                if (nr == 1 && vec_ok)
                    direct_pass_single<TW>(p, W, s_list[l0], j0, j1, warp, lane);
                else if (nr == 1)
                    direct_pass<TW, 1>(p, W, s_list + l0, 1, j0, j1, warp, lane, vec_ok);
                else if (nr == 2)
                    direct_pass<TW, 2>(p, W, s_list + l0, 2, j0, j1, warp, lane, vec_ok);
                else
                    direct_pass<TW, kDirectXR>(p, W, s_list + l0, nr, j0, j1, warp, lane, vec_ok);
            }
            __syncthreads();  // s_list / s_warp_cnt are rewritten by the next (r, jt)
        }
    }
}

// ---------------------------------------------------------------------------
// routing map
// ---------------------------------------------------------------------------

constexpr int kMapThreads = 1024;
constexpr int kMapWarps = kMapThreads / 32;
constexpr int kMapBatch = 16;  // ids per lane held in registers per step
constexpr int kMapCluster = 8; // CTAs of the cluster that builds the map

__global__ void __launch_bounds__(kMapThreads) matmul_id_map_kernel(MatmulIdParams p) {
    // the grouped GEMM launched after this kernel may start its prologue now;
    // it waits for this grid's completion before it reads the map
    grid_dep_launch_dependents();
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t E = static_cast<uint32_t>(p.n_experts);
    const int64_t total = p.total_rows;

    if (static_cast<int>(blockIdx.x) >= kMapCluster) {
        // zero-fill output rows whose id is outside [0, n_experts)
        __shared__ uint32_t s_rows[kMapThreads];
        __shared__ int s_wc[kMapWarps];
        const int64_t zb = blockIdx.x - kMapCluster, nz = gridDim.x - kMapCluster;
        for (int64_t base = zb * kMapThreads; base < total; base += nz * kMapThreads) {
            const int64_t r = base + tid;
            const bool bad = r < total && p.ids[r] >= E;
            const unsigned bal = __ballot_sync(0xffffffffu, bad);
            if (lane == 0) s_wc[warp] = __popc(bal);
            __syncthreads();
            int off = 0, cnt = 0;
            for (int w = 0; w < kMapWarps; ++w) {
                if (w < warp) off += s_wc[w];
                cnt += s_wc[w];
            }
            if (bad) s_rows[off + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint32_t>(r);
            __syncthreads();
            for (int q = 0; q < cnt; ++q) {
                float *orow = p.out + static_cast<int64_t>(s_rows[q]) * p.n;
                for (int64_t j = tid; j < p.n; j += kMapThreads) orow[j] = 0.f;
            }
            __syncthreads();
        }
        return;
    }

    // the map proper: one cluster of kMapCluster CTAs, CTA c owns the c-th
    // contiguous segment of routed rows, each of its warps a sub-segment
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = static_cast<int>(blockIdx.x);  // == rank in the first cluster
    extern __shared__ uint32_t cnt[];  // [kMapWarps][E] counts, then tot[E]
    uint32_t *tot = cnt + static_cast<int64_t>(kMapWarps) * E;
    uint32_t *mine = cnt + static_cast<int64_t>(warp) * E;
    int64_t cseg = (total + kMapCluster - 1) / kMapCluster;
    cseg = (cseg + 32 * kMapWarps - 1) / (32 * kMapWarps) * (32 * kMapWarps);
    const int64_t cbeg = crank * cseg;
    const int64_t cend = cbeg + cseg < total ? cbeg + cseg : total;
    const int64_t wseg = cseg / kMapWarps;
    const int64_t beg = cbeg + static_cast<int64_t>(warp) * wseg;
    const int64_t end = beg + wseg < cend ? beg + wseg : cend;
    for (uint32_t e = lane; e < E; e += 32) mine[e] = 0;
    __syncwarp();
    // keys 0..E-1 are experts, E marks an out-of-range id; batches wholly
    // past the segment's end are skipped (the same test for every lane)

    // pass 1: per-warp counts
    for (int64_t base = beg; base < end; base += 32 * kMapBatch) {
        uint32_t v[kMapBatch];
#pragma unroll
        for (int b = 0; b < kMapBatch; ++b) {
            const int64_t r = base + b * 32 + lane;
            v[b] = r < end ? p.ids[r] : 0xffffffffu;
        }
#pragma unroll
        for (int b = 0; b < kMapBatch; ++b) {
            if (base + b * 32 >= end) break;
            const uint32_t key = v[b] < E ? v[b] : E;
            const unsigned grp = __match_any_sync(0xffffffffu, key);
            if (key != E && lane == __ffs(grp) - 1) mine[key] += __popc(grp);
            __syncwarp();
        }
    }
    __syncthreads();

    // exclusive scan across this CTA's warps (row order) per expert
    for (uint32_t e = tid; e < E; e += kMapThreads) {
        uint32_t run = 0;
        for (int w = 0; w < kMapWarps; ++w) {
            const uint32_t c = cnt[static_cast<int64_t>(w) * E + e];
            cnt[static_cast<int64_t>(w) * E + e] = run;
            run += c;
        }
        tot[e] = run;
    }
    cluster.sync();  // every CTA's per-expert totals are visible cluster-wide
    // rows of lower-ranked CTAs come first: read their totals through DSMEM
    for (uint32_t e = tid; e < E; e += kMapThreads) {
        uint32_t below = 0;
        for (int c = 0; c < crank; ++c) below += cluster.map_shared_rank(tot, c)[e];
        for (int w = 0; w < kMapWarps; ++w) cnt[static_cast<int64_t>(w) * E + e] += below;
        if (crank == kMapCluster - 1) p.counts[e] = below + tot[e];
    }
    cluster.sync();  // remote reads done before any CTA moves on (and later exits)

    // pass 2: scatter row indices to their ascending positions
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int64_t base = beg; base < end; base += 32 * kMapBatch) {
        uint32_t v[kMapBatch];
#pragma unroll
        for (int b = 0; b < kMapBatch; ++b) {
            const int64_t r = base + b * 32 + lane;
            v[b] = r < end ? p.ids[r] : 0xffffffffu;
        }
#pragma unroll
        for (int b = 0; b < kMapBatch; ++b) {
            if (base + b * 32 >= end) break;
            const int64_t r = base + b * 32 + lane;
            const uint32_t key = v[b] < E ? v[b] : E;
            const unsigned grp = __match_any_sync(0xffffffffu, key);
            if (key != E) {
                const uint32_t pos = mine[key] + __popc(grp & lt_mask);
                if (pos < static_cast<uint32_t>(p.m))
                    p.routed_rows[static_cast<int64_t>(key) * p.m + pos] = static_cast<uint32_t>(r);
            }
            __syncwarp();
            if (key != E && lane == __ffs(grp) - 1) mine[key] += __popc(grp);
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------------------------
// grouped GEMM on the FFMA pipe (any weight dtype)
// ---------------------------------------------------------------------------
//
// One CTA per (128 routed rows of expert e, 128 outputs): the rows are
// gathered through routed_rows, the weights widened to f32 as they land in
// shared memory.  256 threads, each an 8 x 8 block of outputs (rows
// {4 ty .. 4 ty + 3, 64 + 4 ty ..}, columns likewise with tx), so every
// 16-wide k step reads four 16-byte shared-memory vectors per 64 FMAs.  The
// next k step's tiles are loaded into registers while the current one is
// multiplied (two shared-memory buffers, one barrier per step).
// A row block of at most 64 routed rows runs as a 64 x 256 tile instead
// (threads 8 x 32, rows {4 ty .., 32 + 4 ty ..}, columns {4 tx .., 128 +
// 4 tx ..}): the same 64 FMAs per four 16-byte shared-memory reads per
// thread, where half of a 128 x 128 tile would idle.  The CTA of the even
// 128-column index computes both 128-column tiles; the odd one returns.

constexpr int kGM = 128;
constexpr int kGN = 128;
constexpr int kGK = 16;
constexpr int kGThreads = 256;
constexpr int kGPitch = kGM + 4;  // keeps 16-byte alignment of each k row

constexpr int kG64M = 64;
constexpr int kG64N = 256;
constexpr int kG64PitchA = kG64M + 4;
constexpr int kG64PitchB = kG64N + 4;

// the 64 x 256 tile of a row block of at most 64 routed rows (see above)
template <typename TW>
__device__ __forceinline__ void grouped_simt64(const MatmulIdParams &p, int vec_ok, int out_vec_ok, int64_t e,
                                               int64_t cnt, int64_t i0, int64_t n0, float *smem_f,
                                               const uint32_t *s_rows) {
    constexpr int kV = 16 / static_cast<int>(sizeof(TW));
    float (*As)[kGK][kG64PitchA] = reinterpret_cast<float (*)[kGK][kG64PitchA]>(smem_f);
    float (*Bs)[kGK][kG64PitchB] =
        reinterpret_cast<float (*)[kGK][kG64PitchB]>(smem_f + 2 * kGK * kG64PitchA);
    const int tid = threadIdx.x;
    const int tx = tid & 31;
    const int ty = tid >> 5;
    const TW *W = static_cast<const TW *>(p.w) + e * p.expert_stride_elems;
    // x: row tid / 4, k 4 (tid % 4); weights: kV k of column (tid / (16 / kV)) + 64 h (f32) or 128 h (16-bit)
    const int akc = (tid & 3) * 4;
    const uint32_t rr = s_rows[tid >> 2];
    const float *arow = rr != 0xffffffffu ? x_row(p, rr) : nullptr;
    constexpr int kBPer = kG64N * kGK / kV / kGThreads;  // weight vectors per thread: 4 (f32) or 2
    constexpr int kColStep = kG64N / kBPer;
    const int bcol0 = kV == 4 ? (tid >> 2) : (tid >> 1);
    const int bkc = kV == 4 ? (tid & 3) * 4 : (tid & 1) * 8;

    auto load = [&](int64_t k0, float4 &ra, float (&rb)[kBPer * kV]) {
        const int64_t kx = k0 + akc;
        if (arow == nullptr) {
            ra = make_float4(0.f, 0.f, 0.f, 0.f);
        } else if (vec_ok && kx + 4 <= p.k) {
            ra = *reinterpret_cast<const float4 *>(arow + kx);
        } else {
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = kx + j < p.k ? arow[kx + j] : 0.f;
            ra = make_float4(v[0], v[1], v[2], v[3]);
        }
#pragma unroll
        for (int h = 0; h < kBPer; ++h) {
            const int64_t col = n0 + bcol0 + kColStep * h;
            const int64_t bx = k0 + bkc;
            float *dst = rb + h * kV;
            if (col >= p.n) {
#pragma unroll
                for (int j = 0; j < kV; ++j) dst[j] = 0.f;
            } else if (vec_ok && bx + kV <= p.k) {
                unpack16<TW>(ld_stream16(W + col * p.k + bx), dst);
            } else {
#pragma unroll
                for (int j = 0; j < kV; ++j) dst[j] = bx + j < p.k ? Elem<TW>::to_f(W[col * p.k + bx + j]) : 0.f;
            }
        }
    };
    auto store = [&](int buf, const float4 &ra, const float (&rb)[kBPer * kV]) {
        const int r = tid >> 2;
        As[buf][akc + 0][r] = ra.x;
        As[buf][akc + 1][r] = ra.y;
        As[buf][akc + 2][r] = ra.z;
        As[buf][akc + 3][r] = ra.w;
#pragma unroll
        for (int h = 0; h < kBPer; ++h) {
            const int c = bcol0 + kColStep * h;
#pragma unroll
            for (int j = 0; j < kV; ++j) Bs[buf][bkc + j][c] = rb[h * kV + j];
        }
    };

    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
    float4 ra;
    float rb[kBPer * kV];
    load(0, ra, rb);
    store(0, ra, rb);
    __syncthreads();
    int cur = 0;
    for (int64_t k0 = 0; k0 < p.k; k0 += kGK) {
        const bool more = k0 + kGK < p.k;
        if (more) load(k0 + kGK, ra, rb);
#pragma unroll
        for (int kk = 0; kk < kGK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[cur][kk][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[cur][kk][32 + 4 * ty]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][4 * tx]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][128 + 4 * tx]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
        }
        if (more) store(cur ^ 1, ra, rb);
        __syncthreads();
        cur ^= 1;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const uint32_t orr = s_rows[(r < 4 ? 0 : 32) + 4 * ty + (r & 3)];
        if (orr == 0xffffffffu) continue;
        float *orow = p.out + static_cast<int64_t>(orr) * p.n;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t c0 = n0 + 128 * h + 4 * tx;
            if (out_vec_ok && c0 + 4 <= p.n) {
                *reinterpret_cast<float4 *>(orow + c0) =
                    make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2], acc[r][4 * h + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (c0 + c < p.n) orow[c0 + c] = acc[r][4 * h + c];
            }
        }
    }
}

template <typename TW>
__global__ void __launch_bounds__(kGThreads, 2) matmul_id_grouped_simt_kernel(MatmulIdParams p, int vec_ok,
                                                                               int out_vec_ok) {
    constexpr int kV = 16 / static_cast<int>(sizeof(TW));  // weight elements per 16-byte vector
    // the 128 x 128 tile's two buffers, or the 64 x 256 tile's
    constexpr int kSmemF128 = 2 * 2 * kGK * kGPitch;
    constexpr int kSmemF64 = 2 * kGK * (kG64PitchA + kG64PitchB);
    __shared__ __align__(16) float smem_f[kSmemF128 > kSmemF64 ? kSmemF128 : kSmemF64];
    float (*As)[kGK][kGPitch] = reinterpret_cast<float (*)[kGK][kGPitch]>(smem_f);
    float (*Bs)[kGK][kGPitch] = reinterpret_cast<float (*)[kGK][kGPitch]>(smem_f + 2 * kGK * kGPitch);
    __shared__ uint32_t s_rows[kGM];
    const int tid = threadIdx.x;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int64_t e = blockIdx.z;
    const uint32_t cnt_raw = p.counts[e];
    const int64_t cnt = cnt_raw < static_cast<uint32_t>(p.m) ? cnt_raw : p.m;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kGM;
    if (i0 >= cnt) return;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kGN;
    if (tid < kGM) s_rows[tid] = i0 + tid < cnt ? p.routed_rows[e * p.m + i0 + tid] : 0xffffffffu;
    __syncthreads();
    if (cnt - i0 <= kG64M) {
        // at most 64 routed rows: the 64 x 256 tile, computed by the CTA of the
        // even 128-column index
        if (blockIdx.y & 1) return;
        grouped_simt64<TW>(p, vec_ok, out_vec_ok, e, cnt, i0, n0, smem_f, s_rows);
        return;
    }
    const TW *W = static_cast<const TW *>(p.w) + e * p.expert_stride_elems;

    // this thread's global sources
    const int akc = (tid & 3) * 4;
    const float *arow[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t rr = s_rows[(tid >> 2) + 64 * h];
        arow[h] = rr != 0xffffffffu ? x_row(p, rr) : nullptr;
    }
    const int bcol0 = kV == 4 ? (tid >> 2) : (tid >> 1);
    const int bkc = kV == 4 ? (tid & 3) * 4 : (tid & 1) * 8;

    auto load = [&](int64_t k0, float4 (&ra)[2], float (&rb)[8]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t kx = k0 + akc;
            if (arow[h] == nullptr) {
                ra[h] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (vec_ok && kx + 4 <= p.k) {
                ra[h] = *reinterpret_cast<const float4 *>(arow[h] + kx);
            } else {
                float v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = kx + j < p.k ? arow[h][kx + j] : 0.f;
                ra[h] = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
        // weights: f32 -> 2 columns x 4 k; 16-bit -> 1 column x 8 k
#pragma unroll
        for (int h = 0; h < 8 / kV; ++h) {
            const int64_t col = n0 + bcol0 + 64 * h;
            const int64_t kx = k0 + bkc;
            float *dst = rb + h * kV;
            if (col >= p.n) {
#pragma unroll
                for (int j = 0; j < kV; ++j) dst[j] = 0.f;
            } else if (vec_ok && kx + kV <= p.k) {
                unpack16<TW>(ld_stream16(W + col * p.k + kx), dst);
            } else {
#pragma unroll
                for (int j = 0; j < kV; ++j) dst[j] = kx + j < p.k ? Elem<TW>::to_f(W[col * p.k + kx + j]) : 0.f;
            }
        }
    };
    auto store = [&](int buf, const float4 (&ra)[2], const float (&rb)[8]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = (tid >> 2) + 64 * h;
            As[buf][akc + 0][r] = ra[h].x;
            As[buf][akc + 1][r] = ra[h].y;
            As[buf][akc + 2][r] = ra[h].z;
            As[buf][akc + 3][r] = ra[h].w;
        }
#pragma unroll
        for (int h = 0; h < 8 / kV; ++h) {
            const int c = bcol0 + 64 * h;
#pragma unroll
            for (int j = 0; j < kV; ++j) Bs[buf][bkc + j][c] = rb[h * kV + j];
        }
    };

    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;

    // all 128 rows (blocks of at most 64 took the 64 x 256 tile above)
    auto mainloop = [&](auto rows_c) {
        constexpr int RN = decltype(rows_c)::value;
        float4 ra[2];
        float rb[8];
        load(0, ra, rb);
        store(0, ra, rb);
        __syncthreads();
        int cur = 0;
        for (int64_t k0 = 0; k0 < p.k; k0 += kGK) {
            const bool more = k0 + kGK < p.k;
            if (more) load(k0 + kGK, ra, rb);
#pragma unroll
            for (int kk = 0; kk < kGK; ++kk) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[cur][kk][4 * ty]);
                const float4 a1 = RN == 8 ? *reinterpret_cast<const float4 *>(&As[cur][kk][64 + 4 * ty]) : a0;
                const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][4 * tx]);
                const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][64 + 4 * tx]);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int r = 0; r < RN; ++r)
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
            }
            if (more) store(cur ^ 1, ra, rb);
            __syncthreads();
            cur ^= 1;
        }
    };
    mainloop(std::integral_constant<int, 8>{});

#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const uint32_t rr = s_rows[(r < 4 ? 0 : 64) + 4 * ty + (r & 3)];
        if (rr == 0xffffffffu) continue;
        float *orow = p.out + static_cast<int64_t>(rr) * p.n;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t c0 = n0 + 64 * h + 4 * tx;
            if (out_vec_ok && c0 + 4 <= p.n) {
                *reinterpret_cast<float4 *>(orow + c0) =
                    make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2], acc[r][4 * h + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (c0 + c < p.n) orow[c0 + c] = acc[r][4 * h + c];
            }
        }
    }
}

int sm_count() {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v > 0 ? v : 1;
}

template <typename TW>
cudaError_t direct_t(const MatmulIdParams &p, int vec_ok, cudaStream_t s) {
    const int64_t gx = p.total_rows < 0x7fffffffLL ? p.total_rows : 0x7fffffffLL;
    const int64_t tiles = (p.n + kDirectRows - 1) / kDirectRows;
    const int64_t gy = tiles < 65535 ? tiles : 65535;
    matmul_id_direct_kernel<TW><<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                                   kDirectThreads, 0, s>>>(p, vec_ok);
    return cudaGetLastError();
}

template <typename TW>
cudaError_t grouped_simt_t(const MatmulIdParams &p, int vec_ok, int out_vec_ok, cudaStream_t s) {
    const int64_t gx = (p.m + kGM - 1) / kGM;
    const int64_t gy = (p.n + kGN - 1) / kGN;
    if (gx > 0x7fffffffLL || gy > 65535 || p.n_experts > 65535) return cudaErrorInvalidConfiguration;
    matmul_id_grouped_simt_kernel<TW><<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
                                             static_cast<unsigned>(p.n_experts)),
                                        kGThreads, 0, s>>>(p, vec_ok, out_vec_ok);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_matmul_id_direct(int wdt, const MatmulIdParams &p, cudaStream_t s) {
    // 16-byte vectors need 16-byte aligned expert rows and activation rows
    const int size = dtype_size(wdt);
    const bool vec_ok = (reinterpret_cast<uintptr_t>(p.w) % 16 == 0) &&
                        ((p.expert_stride_elems * size) % 16 == 0) && ((p.k * size) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(p.x) % 16 == 0) &&
                        ((p.x_token_stride * 4) % 16 == 0) && ((p.x_slot_stride * 4) % 16 == 0);
    switch (wdt) {
    case kF32: return direct_t<float>(p, vec_ok, s);
    case kF16: return direct_t<__half>(p, vec_ok, s);
    case kBF16: return direct_t<__nv_bfloat16>(p, vec_ok, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_matmul_id_map(const MatmulIdParams &p, cudaStream_t s) {
    const size_t smem = (static_cast<size_t>(kMapWarps) + 1) * static_cast<size_t>(p.n_experts) * 4;
    static unsigned long long attr_set = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set & bit)) {
        cudaError_t e = cudaFuncSetAttribute(matmul_id_map_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (kMapWarps + 1) * 1024 * 4);
        if (e != cudaSuccess) return e;
        attr_set |= bit;
    }
    // the first cluster builds the map; the other clusters zero-fill the rows of
    // out-of-range ids
    int64_t zero_ctas = (p.total_rows + kMapThreads - 1) / kMapThreads;
    const int64_t cap = 2LL * sm_count();
    if (zero_ctas > cap) zero_ctas = cap;
    zero_ctas = (zero_ctas + kMapCluster - 1) / kMapCluster * kMapCluster;
    if (zero_ctas < kMapCluster) zero_ctas = kMapCluster;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(kMapCluster + zero_ctas), 1, 1);
    cfg.blockDim = dim3(kMapThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kMapCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, matmul_id_map_kernel, p);
}

cudaError_t launch_matmul_id_grouped_simt(int wdt, const MatmulIdParams &p, cudaStream_t s) {
    // 16-byte vectors need 16-byte aligned expert rows and activation rows
    const int size = dtype_size(wdt);
    const int vec_ok = (reinterpret_cast<uintptr_t>(p.w) % 16 == 0) && ((p.expert_stride_elems * size) % 16 == 0) &&
                       ((p.k * size) % 16 == 0) && ((p.k * 4) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(p.x) % 16 == 0) && ((p.x_token_stride * 4) % 16 == 0) &&
                       ((p.x_slot_stride * 4) % 16 == 0);
    const int out_vec_ok = (reinterpret_cast<uintptr_t>(p.out) % 16 == 0) && (p.n % 4 == 0);
    switch (wdt) {
    case kF32: return grouped_simt_t<float>(p, vec_ok, out_vec_ok, s);
    case kF16: return grouped_simt_t<__half>(p, vec_ok, out_vec_ok, s);
    case kBF16: return grouped_simt_t<__nv_bfloat16>(p, vec_ok, out_vec_ok, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbmm
