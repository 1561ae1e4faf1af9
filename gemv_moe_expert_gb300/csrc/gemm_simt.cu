// gemm_simt.cu -- general strided GEMM on the FFMA pipe (f32 accumulation),
// any transposes, leading dims, batch strides and tails.  It serves the f32
// GEMM and every f16/bf16 layout the tensor-core path does not take.
//
// Semantics: tract-metal 0.23.6, src/kernels/matmul/mlx_gemm/mod.rs,
// `dispatch_metal_mlx_gemm` (A stored [k, m] when transposed, B stored
// [n, k] when transposed), and rlx-metal 0.2.14, src/mps_blas.rs,
// `encode_mps_sgemm_t`.
//
// Two tilings, both with operands staged through shared memory as f32 and the
// global loads ordered along the contiguous dimension of each operand
// (coalesced for every transpose flag):
//   128 x 128 x 16 per CTA, 256 threads, 8 x 8 outputs per thread (four
//   16-byte shared-memory reads per 64 FMAs), the next k step's tiles loaded
//   into registers while the current one is multiplied (two buffers, one
//   barrier per step) -- for grids of at least one 128 x 128 tile per SM;
//   64 x 64 x 16, 4 x 4 outputs per thread -- for smaller grids, where the
//   larger tile would leave SMs idle.
// f32 grids of interior tiles only, with 16-byte-loadable operands, take a
// variant of the 128 x 128 tile with 16-byte global loads and no bounds
// checks (f32 4096^3: 55 TFLOP/s against 37 for the general tile).
#include "device_common.cuh"

namespace gbmm {

namespace {

constexpr int kBM = 64;
constexpr int kBN = 64;
constexpr int kBK = 16;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmParams p) {
    __shared__ float As[kBK][kBM + 4];
    __shared__ float Bs[kBK][kBN + 4];
    const int tid = threadIdx.x;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kBM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBN;

    for (int64_t bat = blockIdx.z; bat < p.batch; bat += gridDim.z) {
        const T *A = static_cast<const T *>(p.a) + bat * p.sa;
        const T *B = static_cast<const T *>(p.b) + bat * p.sb;
        T *C = static_cast<T *>(p.c) + bat * p.sc;
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;

        for (int64_t k0 = 0; k0 < p.k; k0 += kBK) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int idx = tid + e * 256;
                int i, x;
                if (p.ta) {  // A stored [k][m]: walk i fastest
                    i = idx % kBM;
                    x = idx / kBM;
                } else {     // A stored [m][k]: walk x fastest
                    x = idx % kBK;
                    i = idx / kBK;
                }
                const int64_t gi = m0 + i, gx = k0 + x;
                float v = 0.f;
                if (gi < p.m && gx < p.k)
                    v = Elem<T>::to_f(A[p.ta ? gx * p.lda + gi : gi * p.lda + gx]);
                As[x][i] = v;

                int j, y;
                if (p.tb) {  // B stored [n][k]: walk x fastest
                    y = idx % kBK;
                    j = idx / kBK;
                } else {     // B stored [k][n]: walk j fastest
                    j = idx % kBN;
                    y = idx / kBN;
                }
                const int64_t gj = n0 + j, gy = k0 + y;
                float w = 0.f;
                if (gj < p.n && gy < p.k)
                    w = Elem<T>::to_f(B[p.tb ? gj * p.ldb + gy : gy * p.ldb + gj]);
                Bs[y][j] = w;
            }
            __syncthreads();
#pragma unroll
            for (int x = 0; x < kBK; ++x) {
                float av[4], bv[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) av[r] = As[x][ty + 16 * r];
#pragma unroll
                for (int c = 0; c < 4; ++c) bv[c] = Bs[x][tx + 16 * c];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int64_t gi = m0 + ty + 16 * r;
            if (gi >= p.m) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int64_t gj = n0 + tx + 16 * c;
                if (gj < p.n) C[gi * p.ldc + gj] = Elem<T>::from_f(acc[r][c]);
            }
        }
    }
}

constexpr int kWM = 128;
constexpr int kWN = 128;
constexpr int kWK = 16;
constexpr int kWPitch = kWM + 4;  // keeps each k row of a tile 16-byte aligned

template <typename T>
__global__ void __launch_bounds__(256, 2) gemm_ffma128_kernel(GemmParams p, int c_vec_ok) {
    __shared__ __align__(16) float As[2][kWK][kWPitch];
    __shared__ __align__(16) float Bs[2][kWK][kWPitch];
    const int tid = threadIdx.x;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kWM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kWN;

    for (int64_t bat = blockIdx.z; bat < p.batch; bat += gridDim.z) {
        const T *A = static_cast<const T *>(p.a) + bat * p.sa;
        const T *B = static_cast<const T *>(p.b) + bat * p.sb;
        T *C = static_cast<T *>(p.c) + bat * p.sc;

        // element e (< 8) of this thread's share of the 128 x 16 tiles: A as
        // (row i, k x), B as (column j, k y), walked along the stored dimension
        auto load = [&](int64_t k0, float (&ra)[8], float (&rb)[8]) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int idx = tid + 256 * e;  // 0 .. 2047
                int i, x;
                if (p.ta) { i = idx % kWM; x = idx / kWM; } else { x = idx % kWK; i = idx / kWK; }
                const int64_t gi = m0 + i, gx = k0 + x;
                ra[e] = (gi < p.m && gx < p.k) ? Elem<T>::to_f(A[p.ta ? gx * p.lda + gi : gi * p.lda + gx]) : 0.f;
                int j, y;
                if (p.tb) { y = idx % kWK; j = idx / kWK; } else { j = idx % kWN; y = idx / kWN; }
                const int64_t gj = n0 + j, gy = k0 + y;
                rb[e] = (gj < p.n && gy < p.k) ? Elem<T>::to_f(B[p.tb ? gj * p.ldb + gy : gy * p.ldb + gj]) : 0.f;
            }
        };
        auto store = [&](int buf, const float (&ra)[8], const float (&rb)[8]) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int idx = tid + 256 * e;
                if (p.ta) As[buf][idx / kWM][idx % kWM] = ra[e]; else As[buf][idx % kWK][idx / kWK] = ra[e];
                if (p.tb) Bs[buf][idx % kWK][idx / kWK] = rb[e]; else Bs[buf][idx / kWN][idx % kWN] = rb[e];
            }
        };

        float acc[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;

        float ra[8], rb[8];
        load(0, ra, rb);
        store(0, ra, rb);
        __syncthreads();
        int cur = 0;
        for (int64_t k0 = 0; k0 < p.k; k0 += kWK) {
            const bool more = k0 + kWK < p.k;
            if (more) load(k0 + kWK, ra, rb);
#pragma unroll
            for (int kk = 0; kk < kWK; ++kk) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[cur][kk][4 * ty]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[cur][kk][64 + 4 * ty]);
                const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][4 * tx]);
                const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][64 + 4 * tx]);
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
            const int64_t gi = m0 + (r < 4 ? 0 : 64) + 4 * ty + (r & 3);
            if (gi >= p.m) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t gj = n0 + 64 * h + 4 * tx;
                if (c_vec_ok && gj + 4 <= p.n) {
                    *reinterpret_cast<float4 *>(reinterpret_cast<float *>(C) + gi * p.ldc + gj) =
                        make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2], acc[r][4 * h + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (gj + c < p.n) C[gi * p.ldc + gj + c] = Elem<T>::from_f(acc[r][4 * h + c]);
                }
            }
        }
    }
}

// f32 problems whose tiles are all interior (m and n multiples of 128, k of
// 16) with operands that allow 16-byte loads (16-byte aligned bases, leading
// dimensions and batch strides multiples of 4 elements): the same 128 x 128 x
// 16 tile and 8 x 8 outputs per thread, with each thread's two 16-byte loads
// per operand and k step read through pointers set up once, and no bounds
// checks.  Piece q (< 512) of an operand tile is (row q / 4, k 4 (q % 4)) of
// a k-contiguous operand (stored into shared memory as four k rows), (k q /
// 32, rows 4 (q % 32)) of an M/N-contiguous one (one 16-byte store).
template <bool kTA, bool kTB>
__global__ void __launch_bounds__(256, 2) gemm_ffma128_fast_kernel(GemmParams p) {
    __shared__ __align__(16) float As[2][kWK][kWPitch];
    __shared__ __align__(16) float Bs[2][kWK][kWPitch];
    const int tid = threadIdx.x;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kWM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kWN;

    // this thread's pieces q = tid and tid + 256: the second lies 64 rows
    // (k-contiguous) or 8 k rows (M/N-contiguous) after the first
    constexpr int kOA2 = kTA ? 8 * kWPitch : 64;
    constexpr int kOB2 = kTB ? 64 : 8 * kWPitch;

    for (int64_t bat = blockIdx.z; bat < p.batch; bat += gridDim.z) {
        float4 va[2], vb[2];
        // addresses recomputed from the parameters at each k step (keeps no
        // pointer registers live across the multiply)
        auto load = [&](int64_t k0) {
            const int t = threadIdx.x;
            const float *pa = static_cast<const float *>(p.a) + bat * p.sa +
                              (kTA ? (k0 + (t >> 5)) * p.lda + m0 + 4 * (t & 31)
                                   : (m0 + (t >> 2)) * p.lda + k0 + 4 * (t & 3));
            const float *pb = static_cast<const float *>(p.b) + bat * p.sb +
                              (kTB ? (n0 + (t >> 2)) * p.ldb + k0 + 4 * (t & 3)
                                   : (k0 + (t >> 5)) * p.ldb + n0 + 4 * (t & 31));
            va[0] = *reinterpret_cast<const float4 *>(pa);
            va[1] = *reinterpret_cast<const float4 *>(pa + (kTA ? 8 : 64) * p.lda);
            vb[0] = *reinterpret_cast<const float4 *>(pb);
            vb[1] = *reinterpret_cast<const float4 *>(pb + (kTB ? 64 : 8) * p.ldb);
        };
        auto store = [&](int buf) {
            const int t = threadIdx.x;
            float *sa = &As[buf][0][0] + (kTA ? (t >> 5) * kWPitch + 4 * (t & 31) : 4 * (t & 3) * kWPitch + (t >> 2));
            float *sb = &Bs[buf][0][0] + (kTB ? 4 * (t & 3) * kWPitch + (t >> 2) : (t >> 5) * kWPitch + 4 * (t & 31));
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (kTA) {
                    *reinterpret_cast<float4 *>(sa + e * kOA2) = va[e];
                } else {
                    sa[e * kOA2] = va[e].x;
                    sa[e * kOA2 + kWPitch] = va[e].y;
                    sa[e * kOA2 + 2 * kWPitch] = va[e].z;
                    sa[e * kOA2 + 3 * kWPitch] = va[e].w;
                }
                if (kTB) {
                    sb[e * kOB2] = vb[e].x;
                    sb[e * kOB2 + kWPitch] = vb[e].y;
                    sb[e * kOB2 + 2 * kWPitch] = vb[e].z;
                    sb[e * kOB2 + 3 * kWPitch] = vb[e].w;
                } else {
                    *reinterpret_cast<float4 *>(sb + e * kOB2) = vb[e];
                }
            }
        };

        float acc[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;

        load(0);
        store(0);
        __syncthreads();
        int cur = 0;
        for (int64_t k0 = 0; k0 < p.k; k0 += kWK) {
            const bool more = k0 + kWK < p.k;
            if (more) load(k0 + kWK);
#pragma unroll
            for (int kk = 0; kk < kWK; ++kk) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[cur][kk][4 * ty]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[cur][kk][64 + 4 * ty]);
                const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][4 * tx]);
                const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][64 + 4 * tx]);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
            }
            if (more) store(cur ^ 1);
            __syncthreads();
            cur ^= 1;
        }

        float *C = static_cast<float *>(p.c) + bat * p.sc;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int64_t gi = m0 + (r < 4 ? 0 : 64) + 4 * ty + (r & 3);
#pragma unroll
            for (int h = 0; h < 2; ++h)
                *reinterpret_cast<float4 *>(C + gi * p.ldc + n0 + 64 * h + 4 * tx) =
                    make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2], acc[r][4 * h + 3]);
        }
    }
}

// Small problems are latency-bound.  A CTA owns 16 x 16 outputs; per chunk of
// 128 along k it first issues every load of its A rows and B columns at once
// (one memory round trip), stages them in shared memory as f32, then each
// thread computes one output.  For k <= 128 the whole problem costs one round
// trip plus the launch.
constexpr int kSmallT = 16;
constexpr int kSmallK = 128;

template <typename T>
__global__ void __launch_bounds__(256) gemm_small_kernel(GemmParams p) {
    __shared__ float As[kSmallT][kSmallK + 1];
    __shared__ float Bs[kSmallK][kSmallT + 1];
    const int tj = threadIdx.x & 15, ti = threadIdx.x >> 4;
    const int64_t i0 = static_cast<int64_t>(blockIdx.y) * kSmallT;
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kSmallT;
    for (int64_t bat = blockIdx.z; bat < p.batch; bat += gridDim.z) {
        const T *A = static_cast<const T *>(p.a) + bat * p.sa;
        const T *B = static_cast<const T *>(p.b) + bat * p.sb;
        float acc = 0.f;
        for (int64_t k0 = 0; k0 < p.k; k0 += kSmallK) {
            // 16 x 128 of op(A) and 128 x 16 of op(B): 8 + 8 independent loads per thread,
            // ordered along each operand's contiguous dimension
            float av[8], bv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = threadIdx.x + 256 * u;  // 0..2047
                int r, x;
                if (p.ta) { r = idx % kSmallT; x = idx / kSmallT; } else { x = idx % kSmallK; r = idx / kSmallK; }
                const int64_t gi = i0 + r, gx = k0 + x;
                av[u] = (gi < p.m && gx < p.k) ? Elem<T>::to_f(A[p.ta ? gx * p.lda + gi : gi * p.lda + gx]) : 0.f;
                int c, y;
                if (p.tb) { y = idx % kSmallK; c = idx / kSmallK; } else { c = idx % kSmallT; y = idx / kSmallT; }
                const int64_t gj = j0 + c, gy = k0 + y;
                bv[u] = (gj < p.n && gy < p.k) ? Elem<T>::to_f(B[p.tb ? gj * p.ldb + gy : gy * p.ldb + gj]) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = threadIdx.x + 256 * u;
                if (p.ta) As[idx % kSmallT][idx / kSmallT] = av[u]; else As[idx / kSmallK][idx % kSmallK] = av[u];
                if (p.tb) Bs[idx % kSmallK][idx / kSmallK] = bv[u]; else Bs[idx / kSmallT][idx % kSmallT] = bv[u];
            }
            __syncthreads();
            const int64_t kn = p.k - k0 < kSmallK ? p.k - k0 : kSmallK;
            float part[4] = {0.f, 0.f, 0.f, 0.f};
            int x = 0;
            for (; x + 4 <= kn; x += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) part[u] = fmaf(As[ti][x + u], Bs[x + u][tj], part[u]);
            }
            for (; x < kn; ++x) part[0] = fmaf(As[ti][x], Bs[x][tj], part[0]);
            acc += (part[0] + part[1]) + (part[2] + part[3]);
            __syncthreads();
        }
        const int64_t gi = i0 + ti, gj = j0 + tj;
        if (gi < p.m && gj < p.n)
            static_cast<T *>(p.c)[bat * p.sc + gi * p.ldc + gj] = Elem<T>::from_f(acc);
    }
}

template <typename T>
cudaError_t small_t(const GemmParams &p, cudaStream_t s) {
    const int64_t gx = (p.n + 15) / 16, gy = (p.m + 15) / 16;
    if (gx > 0x7fffffffLL || gy > 65535) return cudaErrorInvalidConfiguration;
    const unsigned gz = static_cast<unsigned>(p.batch < 65535 ? p.batch : 65535);
    gemm_small_kernel<T><<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), gz), 256, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t simt_t(const GemmParams &p, cudaStream_t s) {
    // the 128 x 128 tile once it gives every SM at least one CTA
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t wx = (p.n + kWN - 1) / kWN, wy = (p.m + kWM - 1) / kWM;
    const int64_t wbatch = p.batch < 65535 ? p.batch : 65535;
    if (wx * wy * wbatch >= sms && wx <= 0x7fffffffLL && wy <= 65535) {
        auto a16 = [](const void *q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
        const bool fast = sizeof(T) == 4 && p.m % kWM == 0 && p.n % kWN == 0 && p.k % kWK == 0 && a16(p.a) &&
                          a16(p.b) && a16(p.c) && p.lda % 4 == 0 && p.ldb % 4 == 0 && p.ldc % 4 == 0 &&
                          (p.batch == 1 || (p.sa % 4 == 0 && p.sb % 4 == 0 && p.sc % 4 == 0));
        if (fast) {
            const dim3 grid(static_cast<unsigned>(wx), static_cast<unsigned>(wy), static_cast<unsigned>(wbatch));
            if (p.ta) {
                if (p.tb) gemm_ffma128_fast_kernel<true, true><<<grid, 256, 0, s>>>(p);
                else gemm_ffma128_fast_kernel<true, false><<<grid, 256, 0, s>>>(p);
            } else {
                if (p.tb) gemm_ffma128_fast_kernel<false, true><<<grid, 256, 0, s>>>(p);
                else gemm_ffma128_fast_kernel<false, false><<<grid, 256, 0, s>>>(p);
            }
            return cudaGetLastError();
        }
        // 16-byte f32 stores: C 16-byte aligned with rows and batches a multiple of 4 elements apart
        const int c_vec_ok = sizeof(T) == 4 && reinterpret_cast<uintptr_t>(p.c) % 16 == 0 && p.ldc % 4 == 0 &&
                             p.sc % 4 == 0;
        gemm_ffma128_kernel<T><<<dim3(static_cast<unsigned>(wx), static_cast<unsigned>(wy),
                                      static_cast<unsigned>(wbatch)),
                                 256, 0, s>>>(p, c_vec_ok);
        return cudaGetLastError();
    }
    const int64_t gx = (p.n + kBN - 1) / kBN;
    const int64_t gy = (p.m + kBM - 1) / kBM;
    if (gx > 0x7fffffffLL || gy > 65535) return cudaErrorInvalidConfiguration;
    const unsigned gz = static_cast<unsigned>(p.batch < 65535 ? p.batch : 65535);
    gemm_simt_kernel<T><<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), gz), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_small(int dt, const GemmParams &p, cudaStream_t s) {
    switch (dt) {
    case kF32: return small_t<float>(p, s);
    case kF16: return small_t<__half>(p, s);
    case kBF16: return small_t<__nv_bfloat16>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_simt(int dt, const GemmParams &p, cudaStream_t s) {
    switch (dt) {
    case kF32: return simt_t<float>(p, s);
    case kF16: return simt_t<__half>(p, s);
    case kBF16: return simt_t<__nv_bfloat16>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbmm
