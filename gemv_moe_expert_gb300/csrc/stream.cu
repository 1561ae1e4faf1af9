// stream.cu -- the HBM-bound row-dot matrix x vector (m == 1, or n == 1
// with A stored row-major) as a staged stream.
//
// Semantics: tract-metal 0.23.6, src/kernels/matmul/mlx_gemm/mod.rs,
// `dispatch_metal_mlx_gemv` (each output is a dot product along a contiguous
// matrix row).  Two to fifteen vectors (the skinny case) go to the tensor
// cores instead (gemv_tc.cu).
//
// Every matrix byte is read exactly once, so the kernel runs at the speed
// HBM delivers bytes to the SMs.  A kernel that keeps loads in
// registers stalls whenever its warps are busy reducing or between short
// blocks; here the bytes in flight do not depend on the consumers:
//   * one persistent CTA per SM owns a contiguous range of matrix rows;
//   * a producer warp streams them into a ring of kSlots shared-memory slots
//     of kSlotBytes with 1-D bulk copies (cp.async.bulk, completion counted
//     on one mbarrier per slot, L2 evict-first), refilling a slot as soon as
//     all its rows are consumed.  A slot holds as many whole rows as fit,
//     moved by one copy when the rows are contiguous: one issuing thread
//     sustains roughly one bulk copy per ~0.3 us, so copies of 16 KB are
//     needed for an SM's share of HBM bandwidth (4 KB copies reach a third
//     of it); padded rows are copied one per producer lane in parallel;
//   * the consumer warps take the staged rows round-robin (row slot t of the
//     CTA goes to warp t mod 8), dot each with the vector (staged once per
//     CTA in shared memory) using four independent partial sums, reduce
//     across the warp with shuffles and write the outputs; a slot is free
//     again once every one of its row slots was released.
// Every wait is bounded: on timeout the kernel raises its abort flag and the
// device error word, lets its copies in flight land and returns.
#include "device_common.cuh"

namespace gbmm {

namespace {

constexpr int kGemvWarps = 8;     // consumer warps
constexpr int kSlots = 8;
constexpr uint32_t kSlotBytes = 16384;
constexpr uint32_t kRingBytes = kSlots * kSlotBytes;
constexpr uint32_t kStageXMax = kSlotBytes;   // vector bytes staged per CTA: one row

// shared-memory layout after the ring (byte offsets from the 1024-aligned base)
constexpr uint32_t kBarOff = kRingBytes;                      // full[kSlots], empty[kSlots]
constexpr uint32_t kCtlOff = kBarOff + 2 * kSlots * 8;        // abort flag, pieces issued
constexpr uint32_t kCtlBytes = 16;
constexpr uint32_t kXOff = kCtlOff + kCtlBytes;
constexpr uint32_t kStreamSmem = 1024 + kXOff + kStageXMax;

__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Copy n16 16-byte chunks from global (chunk c at src(c)) to shared memory
// (chunk c at dst[dst_index(c)]), eight loads in flight per thread before
// their stores.
template <typename SrcFn, typename DstFn>
__device__ __forceinline__ void stage16(uint4 *dst, int64_t n16, SrcFn src, DstFn dst_index, int tid, int nthreads) {
    constexpr int kB = 8;
    for (int64_t c0 = tid; c0 < n16; c0 += static_cast<int64_t>(nthreads) * kB) {
        uint4 v[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int64_t c = c0 + static_cast<int64_t>(b) * nthreads;
            v[b] = c < n16 ? ld_cached16(src(c)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int64_t c = c0 + static_cast<int64_t>(b) * nthreads;
            if (c < n16) dst[dst_index(c)] = v[b];
        }
    }
}

// named barrier over the consumer warps only (the producer keeps streaming)
template <int NW>
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

// CTA b of g gets the balanced share [lo, hi) of `total` units
__device__ __forceinline__ void share_of(int64_t total, int64_t &lo, int64_t &hi) {
    lo = total * blockIdx.x / gridDim.x;
    hi = total * (blockIdx.x + 1) / gridDim.x;
}

struct Ring {
    uint32_t base, bar0;
    volatile int *abort_flag;
    volatile long long *issued;  // pieces the producer has issued so far
    __device__ uint32_t slot(int s) const { return base + static_cast<uint32_t>(s) * kSlotBytes; }
    __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar0 + 8u * (kSlots + s); }
};

__device__ __forceinline__ Ring ring_setup(uint8_t *smem, uint32_t s_base, uint32_t rows_per_slot) {
    Ring r;
    r.base = s_base;
    r.bar0 = s_base + kBarOff;
    r.abort_flag = reinterpret_cast<volatile int *>(smem + kCtlOff);
    r.issued = reinterpret_cast<volatile long long *>(smem + kCtlOff + 8);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(r.full(s), 1);               // producer's arrive + the copies' bytes
            mbar_init(r.empty(s), rows_per_slot);  // one release per row slot
        }
        *r.abort_flag = 0;
        *r.issued = 0;
        fence_mbar_init();
    }
    return r;
}

__device__ __forceinline__ void raise_abort(const Ring &r, uint32_t *err, uint32_t kid) {
    *r.abort_flag = 1;
    report_device_error(err, kid);
}

// Producer warp: before the i-th fill of the ring, wait until the slot's
// previous contents were released (lane 0 waits, the warp follows).
__device__ __forceinline__ bool ring_acquire(const Ring &r, int64_t i, uint64_t lim, int lane) {
    int ok = 1;
    if (lane == 0 && i >= kSlots) {
        const uint32_t use = static_cast<uint32_t>(i / kSlots);  // >= 1
        ok = mbar_wait_bounded(r.empty(static_cast<int>(i % kSlots)), (use - 1u) & 1u, lim, r.abort_flag);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// Producer warp: one fill of slot s with nr rows of row_bytes each, row q at
// src(q).  Contiguous rows go as one copy; otherwise the lanes copy one row
// each.  Lane 0 posts the byte count first (copies landing before it only
// drive the count negative; the phase cannot complete without lane 0's arrive).
template <typename SrcFn>
__device__ __forceinline__ void ring_fill(const Ring &r, int s, int64_t nr, uint32_t row_bytes, bool contiguous,
                                          SrcFn src, uint64_t pol, int lane) {
    if (lane == 0) mbar_arrive_expect_tx(r.full(s), static_cast<uint32_t>(nr) * row_bytes);
    __syncwarp();
    if (contiguous) {
        if (lane == 0) bulk_load_hint(r.slot(s), src(0), static_cast<uint32_t>(nr) * row_bytes, r.full(s), pol);
    } else {
        for (int64_t q = lane; q < nr; q += 32)
            bulk_load_hint(r.slot(s) + static_cast<uint32_t>(q) * row_bytes, src(q), row_bytes, r.full(s), pol);
    }
}

// Producer, abort path: wait (bounded) for every issued copy to land.
__device__ __forceinline__ void ring_drain(const Ring &r, int64_t issued, uint64_t lim) {
    for (int s = 0; s < kSlots; ++s) {
        const int64_t n_s = issued / kSlots + (s < issued % kSlots ? 1 : 0);
        if (n_s > 0) mbar_wait_bounded(r.full(s), static_cast<uint32_t>((n_s - 1) & 1), lim, nullptr);
    }
}

// Consumer side: wait (one lane, the warp follows) for the i-th fill.  A
// parity wait on fill u of a slot is only sound once fill u - 1 has
// completed (until then the previous phase carries the same parity), so
// the wait starts only after the producer has issued piece i: it issues
// piece i after piece i - kSlots, the previous fill of the slot, was
// consumed and released.
__device__ __forceinline__ bool ring_wait(const Ring &r, int64_t i, uint64_t lim, int lane) {
    int ok = 0;
    if (lane == 0) {
        ok = 1;
        if (*r.issued <= i) {
            const uint64_t start = global_ns();
            uint32_t iter = 0;
            while (*r.issued <= i) {
                __nanosleep(128);  // leave the issue slots to the warps that compute
                if ((++iter & 15u) == 0 && (*r.abort_flag || global_ns() - start > lim)) {
                    ok = 0;
                    break;
                }
            }
        }
        if (ok)
            ok = mbar_wait_bounded(r.full(static_cast<int>(i % kSlots)), static_cast<uint32_t>((i / kSlots) & 1), lim,
                                   r.abort_flag);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// Producer warp: publish that piece i has been issued.
__device__ __forceinline__ void ring_published(const Ring &r, int64_t i, int lane) {
    __syncwarp();
    if (lane == 0) *r.issued = i + 1;
}

__device__ __forceinline__ void ring_release(const Ring &r, int64_t i, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(r.empty(static_cast<int>(i % kSlots)));
}

// Row slots of a consumer warp: t = warp, warp + NW, ... of the CTA, as
// (piece i, row q) = (t / rp, t % rp), advanced without dividing.
template <int NW>
struct RowCursor {
    int64_t i;
    int q;
    __device__ RowCursor(int warp, int rp) : i(warp / rp), q(warp % rp) {}
    __device__ void advance(int rp) {
        q += NW;
        while (q >= rp) {
            q -= rp;
            ++i;
        }
    }
};

// ---------------------------------------------------------------------------
// row-dot GEMV
// ---------------------------------------------------------------------------
//
// Pieces: groups of rp = kSlotBytes / row bytes consecutive rows, one per
// slot fill; CTA b streams its balanced share of the pieces.  Each dot
// product keeps kAcc independent partial sums, so the FMA chain latency is
// hidden with only two consumer warps per scheduler.
template <typename T>
__global__ void __launch_bounds__((kGemvWarps + 1) * 32, 1) gemv_stream_kernel(GemvParams p, int rp) {
    constexpr int V = Elem<T>::kVec;
    constexpr int NW = kGemvWarps;
    constexpr int kAcc = 4;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t s_base = raw + pad;
    const Ring ring = ring_setup(smem, s_base, static_cast<uint32_t>(rp));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t k = p.k;
    const uint32_t row_bytes = static_cast<uint32_t>(k * sizeof(T));
    int64_t g_lo, g_hi;
    share_of((p.rows + rp - 1) / rp, g_lo, g_hi);
    const int64_t pieces = g_hi - g_lo;
    const uint64_t lim = p.wait_limit_ns;
    const T *mat = static_cast<const T *>(p.mat);
    __syncthreads();

    if (warp == NW) {
        // ---------------- producer warp ----------------
        const uint64_t pol = policy_evict_first();
        const bool contiguous = p.mat_rs == k;
        int64_t i = 0;
        for (; i < pieces; ++i) {
            if (!ring_acquire(ring, i, lim, lane)) break;
            const int64_t r0 = (g_lo + i) * rp;
            const int64_t nr = p.rows - r0 < rp ? p.rows - r0 : rp;
            ring_fill(ring, static_cast<int>(i % kSlots), nr, row_bytes, contiguous,
                      [&](int64_t q) { return static_cast<const void *>(mat + (r0 + q) * p.mat_rs); }, pol, lane);
            ring_published(ring, i, lane);
        }
        if (i < pieces && lane == 0) {
            raise_abort(ring, p.err, kKidGemvStream);
            ring_drain(ring, i, lim);
        }
    } else {
        // ---------------- consumers ----------------
        // the vector: chunk c at xs[c]
        const T *vec = static_cast<const T *>(p.vec);
        const int64_t nch = row_bytes / 16;
        const uint4 *xs = reinterpret_cast<const uint4 *>(smem + kXOff);
        stage16(reinterpret_cast<uint4 *>(smem + kXOff), nch,
                [&](int64_t c) { return static_cast<const void *>(vec + c * V); }, [](int64_t c) { return c; },
                threadIdx.x, NW * 32);
        consumers_sync<NW>();

        T *out = static_cast<T *>(p.out);
        const int nc = static_cast<int>(nch);
        for (RowCursor<NW> rc(warp, rp); rc.i < pieces; rc.advance(rp)) {
            const int64_t i = rc.i;
            if (!ring_wait(ring, i, lim, lane)) {
                if (lane == 0) raise_abort(ring, p.err, kKidGemvStream);
                break;
            }
            const int64_t row = (g_lo + i) * rp + rc.q;
            if (row < p.rows) {
                const uint4 *wr = reinterpret_cast<const uint4 *>(smem + (i % kSlots) * kSlotBytes +
                                                                  static_cast<uint32_t>(rc.q) * row_bytes);
                float acc[kAcc];
#pragma unroll
                for (int a = 0; a < kAcc; ++a) acc[a] = 0.f;
#pragma unroll 2
                for (int c = lane; c < nc; c += 32) {
                    float wf[V], xf[V];
                    unpack16<T>(wr[c], wf);
                    unpack16<T>(xs[c], xf);
#pragma unroll
                    for (int e = 0; e < V; ++e) acc[e % kAcc] = fmaf(wf[e], xf[e], acc[e % kAcc]);
                }
                float v = acc[0];
#pragma unroll
                for (int a = 1; a < kAcc; ++a) v += acc[a];
                v = warp_sum(v);
                if (lane == 0) out[row * p.out_os] = Elem<T>::from_f(v);
            }
            ring_release(ring, i, lane);
        }
    }
    __syncthreads();
}

// one attribute call per (kernel, device): `done` is the caller's own flag
// set, one per kernel (kernels of the same signature share a K)
template <typename K>
cudaError_t set_smem_once(K kernel, uint32_t bytes, unsigned long long &done) {
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (done & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done |= bit;
    return e;
}

template <typename T>
cudaError_t gemv_stream_t(const GemvParams &p, int num_sms, cudaStream_t s) {
    const uint32_t row_bytes = static_cast<uint32_t>(p.k * sizeof(T));
    const int rp = static_cast<int>(kSlotBytes / row_bytes);
    const int64_t pieces = (p.rows + rp - 1) / rp;
    const int64_t grid = pieces < num_sms ? pieces : num_sms;
    static unsigned long long done = 0;
    cudaError_t e = set_smem_once(gemv_stream_kernel<T>, kStreamSmem, done);
    if (e != cudaSuccess) return e;
    gemv_stream_kernel<T><<<static_cast<unsigned>(grid), (kGemvWarps + 1) * 32, kStreamSmem, s>>>(p, rp);
    return cudaGetLastError();
}

}  // namespace

bool gemv_stream_eligible(int dt, const GemvParams &p) {
    const int64_t size = dtype_size(dt);
    return p.vec_ok && p.batch == 1 && p.mat_ks == 1 && p.vec_ks == 1 && p.nvec == 1 &&
           (p.k * size) % 16 == 0 && p.k * size <= static_cast<int64_t>(kSlotBytes);
}

cudaError_t launch_gemv_stream(int dt, const GemvParams &p, int num_sms, cudaStream_t s) {
    switch (dt) {
    case kF32: return gemv_stream_t<float>(p, num_sms, s);
    case kF16: return gemv_stream_t<__half>(p, num_sms, s);
    case kBF16: return gemv_stream_t<__nv_bfloat16>(p, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbmm
