// api.cu -- the extern "C" entry points declared in include/gbmm.h: argument
// validation (all of it before the first launch), routing, tensor-map
// encoding, the launch log and the host-side fault injection hook.
//
// Sources: tract-metal 0.23.6, src/kernels/matmul/mlx_gemm/mod.rs
// (`MlxGemm::dispatch_eval`: dtype rules, gemv / wide / gemm routing;
// `dispatch_metal_mlx_gemm`: operand layouts), mlx-native 0.13.0,
// src/ops/dense_matmul_id.rs (`dense_matmul_id_capability`,
// `validate_dense_matmul_id_call`, `dense_matmul_id`, `DenseMatmulIdScratch`).
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "../../include/gbmm.h"
#include "kernel_params.h"

using namespace gbmm;

namespace {

thread_local std::string t_last_error;
thread_local const char *t_last_kernel = "";
std::atomic<uint64_t> g_launches{0};
std::mutex g_inject_mu;
std::string g_inject_name;

gbmm_status fail(gbmm_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

// A kernel is "resolved" unless a test injected a failure for it: a one-shot
// failure for one kernel name, or, with the name "*", a failure of every
// kernel until the injection is cleared.
bool resolve(const char *name) {
    std::lock_guard<std::mutex> g(g_inject_mu);
    if (g_inject_name == "*") {
        t_last_error = std::string("kernel unavailable: ") + name + " (every launch blocked)";
        return false;
    }
    if (!g_inject_name.empty() && g_inject_name == name) {
        g_inject_name.clear();
        t_last_error = std::string("kernel unavailable: ") + name;
        return false;
    }
    return true;
}

bool debug_sync() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("GBMM_DEBUG_SYNC");
        v = (e && e[0] == '1') ? 1 : 0;
    }
    return v == 1;
}

gbmm_status after_launch(cudaError_t e, const char *name, cudaStream_t s) {
    if (e != cudaSuccess)
        return fail(GBMM_ERR_LAUNCH, "%s launch failed: %s", name, cudaGetErrorString(e));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    t_last_kernel = name;
    if (debug_sync()) {
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess)
            return fail(GBMM_ERR_CUDA, "%s failed on the device: %s", name, cudaGetErrorString(e));
    }
    return GBMM_OK;
}

bool aligned(const void *p, uint64_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// overflow-checked a * b (non-negative)
bool mul_ok(uint64_t a, uint64_t b, uint64_t *out) {
    if (a != 0 && b > UINT64_MAX / a) return false;
    *out = a * b;
    return true;
}
bool add_ok(uint64_t a, uint64_t b, uint64_t *out) {
    if (b > UINT64_MAX - a) return false;
    *out = a + b;
    return true;
}

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo < a.hi && b.lo < b.hi; }

// bytes spanned by a strided [batch][rows][cols] operand (last element + 1)
bool extent_bytes(int64_t batch, int64_t rows, int64_t cols, int64_t ld, int64_t bs, int size,
                  uint64_t *out) {
    if (batch == 0 || rows == 0 || cols == 0) {
        *out = 0;
        return true;
    }
    uint64_t t1, t2, t3, last;
    if (!mul_ok(static_cast<uint64_t>(batch - 1), static_cast<uint64_t>(bs), &t1)) return false;
    if (!mul_ok(static_cast<uint64_t>(rows - 1), static_cast<uint64_t>(ld), &t2)) return false;
    if (!add_ok(t1, t2, &t3)) return false;
    if (!add_ok(t3, static_cast<uint64_t>(cols), &last)) return false;
    return mul_ok(last, static_cast<uint64_t>(size), out);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Tensor map of a 16-bit operand stored [batch][outer][inner] with row pitch
// ld elements, box [box_outer][64 inner], 128-byte swizzle: with inner = k
// the UMMA K-major SW128 layout (box_outer = the tile's rows), with inner =
// m or n the M/N-major one (box_outer = 64 k-rows).
bool encode_operand(CUtensorMap *map, int dt, const void *base, int64_t inner, int64_t outer, int64_t batch,
                    int64_t ld, int64_t bs, bool bcast, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const int size = 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer),
                          static_cast<cuuint64_t>(bcast ? 1 : batch)};
    cuuint64_t row_bytes = static_cast<cuuint64_t>(ld) * size;
    cuuint64_t batch_bytes = bcast ? row_bytes * static_cast<cuuint64_t>(outer)
                                   : static_cast<cuuint64_t>(bs) * size;
    cuuint64_t strides[2] = {row_bytes, batch_bytes};
    cuuint32_t box[3] = {64u, box_outer, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, dt == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map of a column-dot GEMV's matrix: (outputs, k, batch), outputs
// contiguous, boxes of `box_cols` outputs x `box_rows` k rows, no swizzle.
bool encode_coldot(CUtensorMap *map, int dt, const void *base, int64_t rows, int64_t k, int64_t batch,
                   int64_t ks, int64_t bs, uint32_t box_cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const int64_t size = dtype_size(dt);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ks * size),
                             static_cast<cuuint64_t>(batch > 1 ? bs * size : ks * size * k)};
    cuuint32_t box[3] = {box_cols, box_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapDataType ty = dt == kF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dt == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(map, ty, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

gbmm_status gemm_impl(bool gemv_only, gbmm_dtype dt, int64_t batch, int64_t m, int64_t n,
                      int64_t k, int ta_i, int tb_i, const void *a, int64_t a_off, int64_t lda,
                      int64_t sa, const void *b, int64_t b_off, int64_t ldb, int64_t sb, void *c,
                      int64_t c_off, int64_t ldc, int64_t sc, gbmm_stream stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const char *fn = gemv_only ? "gbmm_gemv" : "gbmm_gemm";
    if (dt != GBMM_F32 && dt != GBMM_F16 && dt != GBMM_BF16)
        return fail(GBMM_ERR_UNSUPPORTED_DTYPE, "%s: dtype %d is not f32, f16 or bf16", fn, (int)dt);
    const bool ta = ta_i != 0, tb = tb_i != 0;
    if (batch < 0 || m < 0 || n < 0 || k < 0)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: negative dimension", fn);
    if (gemv_only && !(m == 1 || n == 1))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: requires m == 1 or n == 1 (m=%lld n=%lld)", fn,
                    (long long)m, (long long)n);
    if (a_off < 0 || b_off < 0 || c_off < 0)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: negative byte offset", fn);
    const int64_t lda_min = ta ? m : k, ldb_min = tb ? k : n;
    if (lda < 1 || lda < lda_min)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: lda %lld < %lld", fn, (long long)lda,
                    (long long)(lda_min > 1 ? lda_min : 1));
    if (ldb < 1 || ldb < ldb_min)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: ldb %lld < %lld", fn, (long long)ldb,
                    (long long)(ldb_min > 1 ? ldb_min : 1));
    if (ldc < 1 || ldc < n)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: ldc %lld < n %lld", fn, (long long)ldc,
                    (long long)n);
    if (sa < 0 || sb < 0 || sc < 0)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: negative batch stride", fn);
    if (batch == 0 || m == 0 || n == 0) return GBMM_OK;  // nothing to compute

    const int size = dtype_size(dt);
    if (c == nullptr || (k > 0 && (a == nullptr || b == nullptr)))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: null matrix pointer", fn);
    const char *pa = static_cast<const char *>(a) + a_off;
    const char *pb = static_cast<const char *>(b) + b_off;
    char *pc = static_cast<char *>(c) + c_off;
    if ((k > 0 && (!aligned(pa, size) || !aligned(pb, size))) || !aligned(pc, size))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: matrix base not aligned to the %d-byte element",
                    fn, size);
    if (batch > 1 && sc < (m - 1) * ldc + n)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: batches of C overlap (batch_stride_c %lld)", fn,
                    (long long)sc);
    uint64_t ext_a = 0, ext_b = 0, ext_c = 0;
    bool ok = extent_bytes(batch, m, n, ldc, sc, size, &ext_c);
    if (k > 0) {
        ok = ok && extent_bytes(batch, ta ? k : m, ta ? m : k, lda, sa, size, &ext_a) &&
             extent_bytes(batch, tb ? n : k, tb ? k : n, ldb, sb, size, &ext_b);
    }
    if (!ok) return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: operand extent overflows", fn);
    const Range rc{reinterpret_cast<uintptr_t>(pc), reinterpret_cast<uintptr_t>(pc) + ext_c};
    if (k > 0) {
        const Range ra{reinterpret_cast<uintptr_t>(pa), reinterpret_cast<uintptr_t>(pa) + ext_a};
        const Range rb{reinterpret_cast<uintptr_t>(pb), reinterpret_cast<uintptr_t>(pb) + ext_b};
        if (overlap(rc, ra)) return fail(GBMM_ERR_OVERLAP, "%s: C overlaps A", fn);
        if (overlap(rc, rb)) return fail(GBMM_ERR_OVERLAP, "%s: C overlaps B", fn);
    }

    if (k == 0) {
        if (!resolve("gbmm_fill_zero")) return GBMM_ERR_KERNEL_UNAVAILABLE;
        return after_launch(launch_fill_zero(dt, pc, batch, m, n, ldc, sc, stream), "gbmm_fill_zero",
                            stream);
    }

    auto a16 = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    auto s16 = [size](int64_t elems) { return (elems * size) % 16 == 0; };

    // ---- skinny / wide: a few rows of A against B stored [n, k] ----
    const bool wide = !gemv_only && dt != GBMM_F32 && !ta && tb && batch == 1 && m >= 2 && m <= 15 &&
                      n > 1;
    // the skinny case on the tensor cores: y^T = W x^T, the weight rows as the
    // MMA's M side and the (up to 15) tokens as its N side
    if (wide && a16(pa) && a16(pb) && s16(lda) && s16(ldb) && k < (1LL << 31) && n < (1LL << 31) &&
        gemv_tc_block_k() == 64) {
        CUtensorMap map_w, map_x;
        if (encode_operand(&map_w, dt, pb, k, n, 1, ldb, sb, true, static_cast<uint32_t>(gemv_tc_block_rows())) &&
            encode_operand(&map_x, dt, pa, k, m, 1, lda, sa, true, static_cast<uint32_t>(gemv_tc_max_tokens()))) {
            if (!resolve("gbmm_gemv_tc")) return GBMM_ERR_KERNEL_UNAVAILABLE;
            uint32_t *err = device_error_word();
            if (err == nullptr) return fail(GBMM_ERR_CUDA, "%s: device error word unavailable", fn);
            GemvTcParams tp{};
            tp.c = pc;
            tp.ldc = ldc;
            tp.m = static_cast<int32_t>(m);
            tp.n = static_cast<int32_t>(n);
            tp.k = static_cast<int32_t>(k);
            tp.ksplit = gemv_tc_split(n, k, device_sm_count());
            tp.err = err;
            tp.wait_limit_ns = kWaitLimitNs;
            return after_launch(launch_gemv_tc(dt, map_w, map_x, tp, stream), "gbmm_gemv_tc", stream);
        }
    }
    if (wide || m == 1 || n == 1) {
        GemvParams g{};
        g.k = k;
        g.batch = batch;
        g.nvec = 1;
        g.vec_rr = 0;
        g.out_rr = 0;
        bool rowdot;
        if (wide || m == 1) {
            // the matrix is B: outputs run over n; the vector(s) are rows of op(A)
            g.mat = pb;
            g.rows = n;
            g.mat_bs = sb;
            g.vec = pa;
            g.vec_ks = ta ? lda : 1;
            g.vec_bs = sa;
            g.out = pc;
            g.out_os = 1;
            g.out_bs = sc;
            if (wide) {
                g.nvec = static_cast<int32_t>(m);
                g.vec_rr = lda;
                g.out_rr = ldc;
            }
            rowdot = tb;
            g.mat_rs = tb ? ldb : 1;
            g.mat_ks = tb ? 1 : ldb;
        } else {
            // n == 1: the matrix is A: outputs run over m; the vector is column 0 of op(B)
            g.mat = pa;
            g.rows = m;
            g.mat_bs = sa;
            g.vec = pb;
            g.vec_ks = tb ? 1 : ldb;
            g.vec_bs = sb;
            g.out = pc;
            g.out_os = ldc;
            g.out_bs = sc;
            rowdot = !ta;
            g.mat_rs = ta ? 1 : lda;
            g.mat_ks = ta ? lda : 1;
        }
        if (rowdot) {
            g.vec_ok = g.mat_ks == 1 && g.vec_ks == 1 && a16(g.mat) && s16(g.mat_rs) &&
                       s16(g.mat_bs) && a16(g.vec) && s16(g.vec_bs) && (g.nvec == 1 || s16(g.vec_rr));
            if (!resolve("gbmm_gemv_rowdot")) return GBMM_ERR_KERNEL_UNAVAILABLE;
            g.err = device_error_word();
            g.wait_limit_ns = kWaitLimitNs;
            if (g.err != nullptr && gemv_stream_eligible(dt, g))
                return after_launch(launch_gemv_stream(dt, g, device_sm_count(), stream), "gbmm_gemv_stream",
                                    stream);
            return after_launch(launch_gemv_rowdot(dt, g, stream), "gbmm_gemv_rowdot", stream);
        }
        g.vec_ok = g.mat_rs == 1 && a16(g.mat) && s16(g.mat_ks) && s16(g.mat_bs);
        if (!resolve("gbmm_gemv_coldot")) return GBMM_ERR_KERNEL_UNAVAILABLE;
        // aligned matrices (and no broadcast matrix across a batch) stream by TMA
        if (g.vec_ok && (g.batch == 1 || g.mat_bs != 0) && g.rows < (1LL << 31) && g.k < (1LL << 31) &&
            g.batch < (1LL << 31)) {
            g.err = device_error_word();
            g.wait_limit_ns = kWaitLimitNs;
            CUtensorMap map_m;
            if (g.err != nullptr &&
                encode_coldot(&map_m, dt, g.mat, g.rows, g.k, g.batch, g.mat_ks, g.mat_bs,
                              static_cast<uint32_t>(gemv_coldot_stream_box_cols(dt)),
                              static_cast<uint32_t>(gemv_coldot_stream_box_rows())))
                return after_launch(launch_gemv_coldot_stream(dt, map_m, g, stream), "gbmm_gemv_coldot", stream);
        }
        return after_launch(launch_gemv_coldot(dt, g, stream), "gbmm_gemv_coldot", stream);
    }

    // ---- tensor-core GEMM (every transpose combination; each operand read as stored) ----
    const bool tc_layout = (dt == GBMM_F16 || dt == GBMM_BF16) && a16(pa) && a16(pb) && s16(lda) && s16(ldb) &&
                           s16(sa) && s16(sb) && m < (1LL << 31) && n < (1LL << 31) && k < (1LL << 31) &&
                           batch < (1LL << 31);
    if (tc_layout) {
        const int bn = gemm_tc_block_n(), bk = gemm_tc_block_k();
        // 256 x 256 tiles on CTA pairs: taken for long k and at least two
        // rounds of tiles over the SMs
        const int wbm = gemm_tc_wide_block_m();
        const int64_t tiles_n = (n + bn - 1) / bn;
        const bool wide = k >= 512 && ((m + wbm - 1) / wbm) * tiles_n * batch >= 2LL * device_sm_count();
        const int bm = wide ? wbm : gemm_tc_block_m();
        const int64_t tiles_m = (m + bm - 1) / bm;
        const int64_t tiles = tiles_m * tiles_n * batch;
        const bool a_bc = sa == 0 || batch == 1, b_bc = sb == 0 || batch == 1;
        // the wide tiles run on CTA pairs, each CTA loading 128 rows (or
        // columns) of A and of B
        const bool pair = wide;
        const uint32_t abox = static_cast<uint32_t>(pair ? gemm_tc_block_m() : bm);
        const uint32_t bbox = static_cast<uint32_t>(pair ? gemm_tc_block_m() : bn);
        // A: [m, k] K-contiguous, or stored [k, m] when transposed; B: [n, k]
        // K-contiguous when transposed, else stored [k, n]
        CUtensorMap map_a, map_b;
        const bool maps_ok =
            (ta ? encode_operand(&map_a, dt, pa, m, k, batch, lda, sa, a_bc, static_cast<uint32_t>(bk))
                : encode_operand(&map_a, dt, pa, k, m, batch, lda, sa, a_bc, abox)) &&
            (tb ? encode_operand(&map_b, dt, pb, k, n, batch, ldb, sb, b_bc, bbox)
                : encode_operand(&map_b, dt, pb, n, k, batch, ldb, sb, b_bc, static_cast<uint32_t>(bk)));
        if (tiles < (1LL << 31) && maps_ok) {
            if (!resolve("gbmm_gemm_tc")) return GBMM_ERR_KERNEL_UNAVAILABLE;
            uint32_t *err = device_error_word();
            if (err == nullptr) return fail(GBMM_ERR_CUDA, "%s: device error word unavailable", fn);
            GemmTcParams p{};
            p.c = pc;
            p.ldc = ldc;
            p.sc = sc;
            p.m = static_cast<int32_t>(m);
            p.n = static_cast<int32_t>(n);
            p.k = static_cast<int32_t>(k);
            p.batch = static_cast<int32_t>(batch);
            p.a_bcast = a_bc ? 1 : 0;
            p.b_bcast = b_bc ? 1 : 0;
            p.a_mn = ta ? 1 : 0;
            p.b_mn = tb ? 0 : 1;
            // 1: rows 16-byte aligned; 2: 32-byte aligned
            const bool c32 = reinterpret_cast<uintptr_t>(pc) % 32 == 0 && (ldc * 2) % 32 == 0 && (sc * 2) % 32 == 0;
            p.c_vec_ok = (a16(pc) && s16(ldc) && s16(sc)) ? (c32 ? 2 : 1) : 0;
            p.tiles_m = static_cast<int32_t>(tiles_m);
            p.tiles_n = static_cast<int32_t>(tiles_n);
            p.num_tiles = static_cast<int32_t>(tiles);
            p.err = err;
            p.wait_limit_ns = kWaitLimitNs;
            return after_launch(pair ? launch_gemm_tc_pair(dt, map_a, map_b, p, device_sm_count(), stream)
                                     : launch_gemm_tc(dt, map_a, map_b, p, device_sm_count(), stream),
                                "gbmm_gemm_tc", stream);
        }
    }

    // ---- FFMA GEMM ----
    if (!resolve("gbmm_gemm_simt")) return GBMM_ERR_KERNEL_UNAVAILABLE;
    GemmParams p{};
    p.a = pa;
    p.b = pb;
    p.c = pc;
    p.batch = batch;
    p.m = m;
    p.n = n;
    p.k = k;
    p.lda = lda;
    p.ldb = ldb;
    p.ldc = ldc;
    p.sa = sa;
    p.sb = sb;
    p.sc = sc;
    p.ta = ta;
    p.tb = tb;
    // a few thousand outputs: latency-bound, one output per thread
    if (batch * m * n <= 16384 && k <= 4096)
        return after_launch(launch_gemm_small(dt, p, stream), "gbmm_gemm_small", stream);
    return after_launch(launch_gemm_simt(dt, p, stream), "gbmm_gemm_simt", stream);
}

int weight_size(gbmm_dtype dt) {
    switch (dt) {
    case GBMM_F32: return 4;
    case GBMM_F16:
    case GBMM_BF16: return 2;
    default: return 0;
    }
}

gbmm_status capability_impl(gbmm_dtype wdt, const gbmm_matmul_id_params *p,
                            gbmm_matmul_id_capability_t *out) {
    const char *fn = "gbmm_matmul_id";
    if (p == nullptr || out == nullptr) return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: null argument", fn);
    if (p->m == 0 || p->n == 0 || p->k == 0 || p->top_k == 0 || p->n_experts == 0)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: m, n, k, top_k and n_experts must be nonzero", fn);
    if (p->input_layout > 1 || p->multiplicity > 1 || p->route > 1)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: unknown layout, multiplicity or route", fn);
    if (p->activation_precision > 1 || p->reserved != 0)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: unknown activation precision or nonzero reserved field",
                    fn);
    if (p->top_k > p->n_experts && p->multiplicity == GBMM_IDS_DISTINCT_PER_TOKEN)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: distinct top_k %u exceeds n_experts %u", fn,
                    p->top_k, p->n_experts);
    const int size = weight_size(wdt);
    if (size == 0)
        return fail(GBMM_ERR_UNSUPPORTED_DTYPE, "%s: weights must be f32, f16 or bf16 (got %d)", fn,
                    (int)wdt);
    uint64_t matrix_bytes, t;
    if (!mul_ok(p->n, p->k, &t) || !mul_ok(t, static_cast<uint64_t>(size), &matrix_bytes))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: expert matrix byte extent overflow", fn);
    if (p->expert_stride_bytes < matrix_bytes)
        return fail(GBMM_ERR_INVALID_ARGUMENT,
                    "%s: expert stride %llu is smaller than one %llu-byte matrix", fn,
                    (unsigned long long)p->expert_stride_bytes, (unsigned long long)matrix_bytes);
    if (p->expert_stride_bytes % static_cast<uint64_t>(size) != 0)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: expert stride %llu is not aligned to the weight dtype",
                    fn, (unsigned long long)p->expert_stride_bytes);
    uint64_t last_off, weight_bytes;
    if (!mul_ok(static_cast<uint64_t>(p->n_experts - 1), p->expert_stride_bytes, &last_off))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: expert weight offset overflow", fn);
    if (!add_ok(last_off, matrix_bytes, &weight_bytes))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: weight extent overflow", fn);
    uint64_t total_rows;
    mul_ok(p->m, p->top_k, &total_rows);  // two u32 factors cannot overflow u64
    if (total_rows > UINT32_MAX)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: flattened routed rows exceed the u32 ABI", fn);
    const uint64_t input_rows = p->input_layout == GBMM_INPUT_SHARED_PER_TOKEN ? p->m : total_rows;
    uint64_t input_bytes, ids_bytes, out_bytes;
    if (!mul_ok(input_rows, p->k, &t) || !mul_ok(t, 4, &input_bytes))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: input byte extent overflow", fn);
    if (!mul_ok(total_rows, 4, &ids_bytes))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: expert IDs byte extent overflow", fn);
    if (!mul_ok(total_rows, p->n, &t) || !mul_ok(t, 4, &out_bytes))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: output byte extent overflow", fn);
    if (p->route == GBMM_ROUTE_GROUPED_PREFILL && p->multiplicity != GBMM_IDS_DISTINCT_PER_TOKEN)
        return fail(GBMM_ERR_INVALID_ARGUMENT,
                    "%s: grouped prefill requires distinct expert IDs per token", fn);
    if (p->route == GBMM_ROUTE_GROUPED_PREFILL && p->n_experts > GBMM_GROUPED_MAX_EXPERTS)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: grouped prefill supports at most %u experts", fn,
                    GBMM_GROUPED_MAX_EXPERTS);
    gbmm_matmul_id_capability_t cap{};
    cap.schema_version = GBMM_MATMUL_ID_SCHEMA_VERSION;
    cap.weight_dtype = static_cast<uint32_t>(wdt);
    cap.route = p->route;
    cap.required_weight_bytes = weight_bytes;
    cap.required_input_bytes = input_bytes;
    cap.required_ids_bytes = ids_bytes;
    cap.required_output_bytes = out_bytes;
    if (p->route == GBMM_ROUTE_GROUPED_PREFILL) {
        cap.has_scratch = 1;
        cap.expert_counts_bytes = static_cast<uint64_t>(p->n_experts) * 4;
        uint64_t rr;
        if (!mul_ok(static_cast<uint64_t>(p->n_experts) * p->m, 4, &rr))
            return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: scratch routed rows byte extent overflow", fn);
        cap.routed_rows_bytes = rr;
    }
    *out = cap;
    return GBMM_OK;
}

Range range_of(const void *p, uint64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

}  // namespace

namespace gbmm {
// Lets other translation units of the library set gbmm_last_error().
int record_error(int status, const char *message) {
    t_last_error = message ? message : "";
    return status;
}
}  // namespace gbmm

extern "C" {

gbmm_status gbmm_gemm(gbmm_dtype dt, int64_t batch, int64_t m, int64_t n, int64_t k,
                      int transpose_a, int transpose_b, const void *a, int64_t a_offset_bytes,
                      int64_t lda, int64_t batch_stride_a, const void *b, int64_t b_offset_bytes,
                      int64_t ldb, int64_t batch_stride_b, void *c, int64_t c_offset_bytes,
                      int64_t ldc, int64_t batch_stride_c, gbmm_stream stream) {
    t_last_error.clear();
    return gemm_impl(false, dt, batch, m, n, k, transpose_a, transpose_b, a, a_offset_bytes, lda,
                     batch_stride_a, b, b_offset_bytes, ldb, batch_stride_b, c, c_offset_bytes, ldc,
                     batch_stride_c, stream);
}

gbmm_status gbmm_gemv(gbmm_dtype dt, int64_t batch, int64_t m, int64_t n, int64_t k,
                      int transpose_a, int transpose_b, const void *a, int64_t a_offset_bytes,
                      int64_t lda, int64_t batch_stride_a, const void *b, int64_t b_offset_bytes,
                      int64_t ldb, int64_t batch_stride_b, void *c, int64_t c_offset_bytes,
                      int64_t ldc, int64_t batch_stride_c, gbmm_stream stream) {
    t_last_error.clear();
    return gemm_impl(true, dt, batch, m, n, k, transpose_a, transpose_b, a, a_offset_bytes, lda,
                     batch_stride_a, b, b_offset_bytes, ldb, batch_stride_b, c, c_offset_bytes, ldc,
                     batch_stride_c, stream);
}

gbmm_status gbmm_matmul_id_scratch_bytes(uint32_t max_experts, uint32_t max_tokens,
                                         uint64_t *expert_counts_bytes, uint64_t *routed_rows_bytes) {
    t_last_error.clear();
    if (max_experts == 0 || max_tokens == 0)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "gbmm_matmul_id_scratch_bytes: capacities must be nonzero");
    if (expert_counts_bytes == nullptr || routed_rows_bytes == nullptr)
        return fail(GBMM_ERR_INVALID_ARGUMENT, "gbmm_matmul_id_scratch_bytes: null output");
    uint64_t rr;
    if (!mul_ok(static_cast<uint64_t>(max_experts) * max_tokens, 4, &rr))
        return fail(GBMM_ERR_INVALID_ARGUMENT, "gbmm_matmul_id_scratch_bytes: overflow");
    *expert_counts_bytes = static_cast<uint64_t>(max_experts) * 4;
    *routed_rows_bytes = rr;
    return GBMM_OK;
}

gbmm_status gbmm_matmul_id_capability(gbmm_dtype weight_dtype, const gbmm_matmul_id_params *p,
                                      gbmm_matmul_id_capability_t *out) {
    t_last_error.clear();
    return capability_impl(weight_dtype, p, out);
}

gbmm_status gbmm_matmul_id(const gbmm_matmul_id_params *p, gbmm_dtype weight_dtype,
                           const void *weights, uint64_t weights_bytes, const float *input,
                           uint64_t input_bytes, const uint32_t *ids, uint64_t ids_bytes, float *out,
                           uint64_t out_bytes, const gbmm_matmul_id_scratch *scratch,
                           gbmm_stream stream_, gbmm_matmul_id_receipt *receipt) {
    t_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const char *fn = "gbmm_matmul_id";
    gbmm_matmul_id_capability_t cap;
    gbmm_status st = capability_impl(weight_dtype, p, &cap);
    if (st != GBMM_OK) return st;
    const int size = weight_size(weight_dtype);
    struct Buf {
        const char *label;
        const void *ptr;
        uint64_t len, need;
        int align;
    } bufs[4] = {{"weights", weights, weights_bytes, cap.required_weight_bytes, size},
                 {"input", input, input_bytes, cap.required_input_bytes, 4},
                 {"expert IDs", ids, ids_bytes, cap.required_ids_bytes, 4},
                 {"output", out, out_bytes, cap.required_output_bytes, 4}};
    for (const Buf &b : bufs) {
        if (b.ptr == nullptr) return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: %s is null", fn, b.label);
        if (b.len < b.need)
            return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: %s requires %llu bytes, got %llu", fn, b.label,
                        (unsigned long long)b.need, (unsigned long long)b.len);
        if (!aligned(b.ptr, b.align))
            return fail(GBMM_ERR_INVALID_ARGUMENT, "%s: %s is not aligned to its element", fn, b.label);
    }
    const Range r_out = range_of(out, cap.required_output_bytes);
    const Range r_w = range_of(weights, cap.required_weight_bytes);
    const Range r_in = range_of(input, cap.required_input_bytes);
    const Range r_ids = range_of(ids, cap.required_ids_bytes);
    if (overlap(r_out, r_w)) return fail(GBMM_ERR_OVERLAP, "%s: output must not overlap weights", fn);
    if (overlap(r_out, r_in)) return fail(GBMM_ERR_OVERLAP, "%s: output must not overlap input", fn);
    if (overlap(r_out, r_ids)) return fail(GBMM_ERR_OVERLAP, "%s: output must not overlap expert IDs", fn);

    const bool grouped = p->route == GBMM_ROUTE_GROUPED_PREFILL;
    if (grouped) {
        if (scratch == nullptr)
            return fail(GBMM_ERR_SCRATCH, "%s: grouped prefill requires caller-owned scratch", fn);
        if (scratch->max_experts < p->n_experts || scratch->max_tokens < p->m)
            return fail(GBMM_ERR_SCRATCH, "%s: scratch capacity experts/tokens=%u/%u is smaller than %u/%u",
                        fn, scratch->max_experts, scratch->max_tokens, p->n_experts, p->m);
        if (scratch->expert_counts == nullptr || scratch->routed_rows == nullptr)
            return fail(GBMM_ERR_SCRATCH, "%s: scratch buffer is null", fn);
        if (!aligned(scratch->expert_counts, 4) || !aligned(scratch->routed_rows, 4))
            return fail(GBMM_ERR_SCRATCH, "%s: scratch buffer not aligned to u32", fn);
        if (scratch->expert_counts_bytes < cap.expert_counts_bytes)
            return fail(GBMM_ERR_SCRATCH, "%s: scratch expert counts requires %llu bytes, got %llu", fn,
                        (unsigned long long)cap.expert_counts_bytes,
                        (unsigned long long)scratch->expert_counts_bytes);
        if (scratch->routed_rows_bytes < cap.routed_rows_bytes)
            return fail(GBMM_ERR_SCRATCH, "%s: scratch routed rows requires %llu bytes, got %llu", fn,
                        (unsigned long long)cap.routed_rows_bytes,
                        (unsigned long long)scratch->routed_rows_bytes);
        const Range r_c = range_of(scratch->expert_counts, cap.expert_counts_bytes);
        const Range r_r = range_of(scratch->routed_rows, cap.routed_rows_bytes);
        const Range others[4] = {r_out, r_w, r_in, r_ids};
        for (const Range &o : others)
            if (overlap(r_c, o) || overlap(r_r, o))
                return fail(GBMM_ERR_OVERLAP, "%s: scratch overlaps an operand", fn);
        if (overlap(r_c, r_r)) return fail(GBMM_ERR_OVERLAP, "%s: scratch buffers overlap", fn);
    }

    MatmulIdParams mp{};
    mp.w = weights;
    mp.x = input;
    mp.ids = ids;
    mp.out = out;
    mp.m = p->m;
    mp.n = p->n;
    mp.k = p->k;
    mp.top_k = p->top_k;
    mp.n_experts = p->n_experts;
    mp.expert_stride_elems = static_cast<int64_t>(p->expert_stride_bytes / size);
    if (p->input_layout == GBMM_INPUT_SHARED_PER_TOKEN) {
        mp.x_token_stride = p->k;
        mp.x_slot_stride = 0;
    } else {
        mp.x_token_stride = static_cast<int64_t>(p->k) * p->top_k;
        mp.x_slot_stride = p->k;
    }
    mp.total_rows = static_cast<int64_t>(p->m) * p->top_k;
    mp.err = nullptr;
    mp.wait_limit_ns = kWaitLimitNs;

    if (!grouped) {
        if (!resolve("gbmm_matmul_id_direct")) return GBMM_ERR_KERNEL_UNAVAILABLE;
        // tensor cores for bf16 / f16 weights read by TMA (16-byte aligned base,
        // expert stride and rows) with at most direct_tc_max_ids() routed rows
        CUtensorMap map_w;
        bool tc = (weight_dtype == GBMM_BF16 || weight_dtype == GBMM_F16) && aligned(weights, 16) && p->expert_stride_bytes % 16 == 0 &&
                  p->expert_stride_bytes < (1ull << 40) && p->k % 8 == 0 &&
                  mp.total_rows <= direct_tc_max_ids() && p->n_experts <= static_cast<uint32_t>(direct_tc_max_experts()) &&
                  p->n < (1u << 31) && p->k < (1u << 31) && direct_tc_block_k() == 64;
        if (tc) {
            PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
            cuuint64_t wdims[3] = {p->k, p->n, p->n_experts};
            cuuint64_t wstrides[2] = {static_cast<cuuint64_t>(p->k) * 2, p->expert_stride_bytes};
            cuuint32_t wbox[3] = {static_cast<cuuint32_t>(direct_tc_block_k()),
                                  static_cast<cuuint32_t>(direct_tc_block_rows()), 1u};
            cuuint32_t estr[3] = {1u, 1u, 1u};
            tc = enc != nullptr &&
                 enc(&map_w,
                     weight_dtype == GBMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void *>(weights), wdims, wstrides, wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
        if (tc) {
            mp.err = device_error_word();
            if (mp.err == nullptr) return fail(GBMM_ERR_CUDA, "%s: device error word unavailable", fn);
            const int64_t max_distinct = std::min<int64_t>(p->n_experts, mp.total_rows);
            // a cluster split of k needs one pass per expert: at most 16 routed
            // rows can choose one expert whatever the ids are
            const int split = direct_tc_split(p->n, p->k, max_distinct, mp.total_rows, device_sm_count());
            const int x_vec_ok = aligned(input, 16) && (mp.x_token_stride % 4 == 0) && (mp.x_slot_stride % 4 == 0);
            st = after_launch(launch_matmul_id_direct_tc(weight_dtype, map_w, mp, static_cast<int>(max_distinct), split,
                                                         x_vec_ok, stream),
                              "gbmm_matmul_id_direct_tc", stream);
            if (st != GBMM_OK) return st;
            if (receipt) *receipt = gbmm_matmul_id_receipt{static_cast<uint32_t>(weight_dtype), p->route, 1};
            return GBMM_OK;
        }
        st = after_launch(launch_matmul_id_direct(weight_dtype, mp, stream), "gbmm_matmul_id_direct",
                          stream);
        if (st != GBMM_OK) return st;
        if (receipt) *receipt = gbmm_matmul_id_receipt{static_cast<uint32_t>(weight_dtype), p->route, 1};
        return GBMM_OK;
    }

    // resolve both kernels before the first launch: a failure leaves nothing enqueued
    if (!resolve("gbmm_matmul_id_map")) return GBMM_ERR_KERNEL_UNAVAILABLE;
    if (!resolve("gbmm_matmul_id_grouped")) return GBMM_ERR_KERNEL_UNAVAILABLE;
    mp.counts = scratch->expert_counts;
    mp.routed_rows = scratch->routed_rows;
    // tensor-core grouped GEMM: bf16 or f16 weights read by TMA (16-byte aligned
    // base, expert stride and rows), 16-byte aligned activation rows
    CUtensorMap map_w;
    const bool w16 = weight_dtype == GBMM_BF16 || weight_dtype == GBMM_F16;
    bool tc = w16 && aligned(weights, 16) && p->expert_stride_bytes % 16 == 0 &&
              p->expert_stride_bytes < (1ull << 40) && p->k % 8 == 0 && aligned(input, 16) &&
              p->n_experts <= static_cast<uint32_t>(grouped_tc_max_experts()) && p->n < (1u << 31) &&
              p->k < (1u << 31);
    if (tc) {
        PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
        // weights: (k, n, expert), 256 x bk boxes; a box row of bk bf16 is one
        // swizzle row (64 bytes -> 64-byte swizzle, 128 bytes -> 128-byte)
        const int bk = grouped_tc_block_k();
        cuuint64_t wdims[3] = {p->k, p->n, p->n_experts};
        cuuint64_t wstrides[2] = {static_cast<cuuint64_t>(p->k) * 2, p->expert_stride_bytes};
        cuuint32_t wbox[3] = {static_cast<cuuint32_t>(bk), 256u, 1u};
        cuuint32_t estr[3] = {1u, 1u, 1u};
        tc = enc != nullptr &&
             enc(&map_w, weight_dtype == GBMM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                 3, const_cast<void *>(weights), wdims, wstrides,
                 wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 bk == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    if (tc) {
        mp.err = device_error_word();
        if (mp.err == nullptr) return fail(GBMM_ERR_CUDA, "%s: device error word unavailable", fn);
    }
    st = after_launch(launch_matmul_id_map(mp, stream), "gbmm_matmul_id_map", stream);
    if (st != GBMM_OK) return st;
    if (tc) {
        // 2: 32-byte stores (rows 32-byte aligned), 1: 16-byte stores, 0: scalar
        const int out_vec_ok = (aligned(out, 32) && p->n % 8 == 0) ? 2 : (aligned(out, 16) && p->n % 4 == 0) ? 1 : 0;
        const int split = p->activation_precision == GBMM_ACT_SPLIT ? 1 : 0;
        st = after_launch(launch_matmul_id_grouped_tc(map_w, mp, out_vec_ok, split, weight_dtype == GBMM_F16 ? 1 : 0,
                                                      device_sm_count(), stream),
                          "gbmm_matmul_id_grouped_tc", stream);
    } else {
        st = after_launch(launch_matmul_id_grouped_simt(weight_dtype, mp, stream),
                          "gbmm_matmul_id_grouped_simt", stream);
    }
    if (st != GBMM_OK) return st;
    if (receipt) *receipt = gbmm_matmul_id_receipt{static_cast<uint32_t>(weight_dtype), p->route, 2};
    return GBMM_OK;
}

const char *gbmm_last_error(void) { return t_last_error.c_str(); }

const char *gbmm_status_string(gbmm_status s) {
    switch (s) {
    case GBMM_OK: return "GBMM_OK";
    case GBMM_ERR_INVALID_ARGUMENT: return "GBMM_ERR_INVALID_ARGUMENT";
    case GBMM_ERR_UNSUPPORTED_DTYPE: return "GBMM_ERR_UNSUPPORTED_DTYPE";
    case GBMM_ERR_OVERLAP: return "GBMM_ERR_OVERLAP";
    case GBMM_ERR_SCRATCH: return "GBMM_ERR_SCRATCH";
    case GBMM_ERR_KERNEL_UNAVAILABLE: return "GBMM_ERR_KERNEL_UNAVAILABLE";
    case GBMM_ERR_LAUNCH: return "GBMM_ERR_LAUNCH";
    case GBMM_ERR_DEVICE_TIMEOUT: return "GBMM_ERR_DEVICE_TIMEOUT";
    case GBMM_ERR_CUDA: return "GBMM_ERR_CUDA";
    default: return "GBMM_ERR_UNKNOWN";
    }
}

uint32_t gbmm_abi_version(void) { return GBMM_ABI_VERSION; }

gbmm_status gbmm_device_error(gbmm_stream stream_, uint32_t *code) {
    t_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(GBMM_ERR_CUDA, "gbmm_device_error: %s", cudaGetErrorString(e));
    uint32_t *word = device_error_word();
    if (word == nullptr) return fail(GBMM_ERR_CUDA, "gbmm_device_error: error word unavailable");
    uint32_t v = 0;
    e = cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(GBMM_ERR_CUDA, "gbmm_device_error: %s", cudaGetErrorString(e));
    if (code) *code = v;
    if (v != 0) {
        const uint32_t zero = 0;
        cudaMemcpy(word, &zero, sizeof zero, cudaMemcpyHostToDevice);
        return fail(GBMM_ERR_DEVICE_TIMEOUT, "a bounded device wait ran out (word 0x%x)", v);
    }
    return GBMM_OK;
}

void gbmm_test_inject_kernel_failure(const char *name) {
    std::lock_guard<std::mutex> g(g_inject_mu);
    g_inject_name = name ? name : "";
}

uint64_t gbmm_test_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void gbmm_test_reset_launch_count(void) { g_launches.store(0, std::memory_order_relaxed); }

const char *gbmm_test_last_kernel(void) { return t_last_kernel; }

gbmm_status gbmm_test_bounded_wait(uint64_t limit_ns, gbmm_stream stream_, uint32_t *code) {
    t_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (limit_ns < 1000) limit_ns = 1000;
    if (limit_ns > 2000000000ull) limit_ns = 2000000000ull;
    uint32_t *word = device_error_word();
    if (word == nullptr) return fail(GBMM_ERR_CUDA, "gbmm_test_bounded_wait: error word unavailable");
    gbmm_status st = after_launch(launch_bounded_wait_test(word, limit_ns, stream),
                                  "gbmm_bounded_wait_test", stream);
    if (st != GBMM_OK) return st;
    return gbmm_device_error(stream_, code);
}

}  // extern "C"
