// kernel_params.h -- parameter blocks passed by value from the host dispatch
// (api.cu) to the kernels, and the internal launcher declarations.  Plain C++
// structs: no torch types anywhere in the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbmm {

enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

inline int dtype_size(int dt) { return dt == kF32 ? 4 : 2; }

// device error word bits
constexpr uint32_t kErrWaitTimeout = 1u;

// kernel ids reported in bits 8..15 of the device error word
enum KernelId : uint32_t {
    kKidNone = 0,
    kKidGemmTc = 1,
    kKidGroupedTc = 2,
    kKidBoundedWaitTest = 3,
    kKidGemvStream = 4,
    kKidGemvTc = 5,
    kKidDirectTc = 6,
    kKidGemvColdotStream = 7,
};

// default limit of a bounded device wait (1 s)
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Matrix-times-vector problem after the host has mapped (batch, m, n, k,
// transposes, strides) onto "rows" outputs, each a dot product of length k.
// All strides in elements.
//   mat(o, x) = mat[bat*mat_bs + o*mat_rs + x*mat_ks]
//   vec_r(x)  = vec[bat*vec_bs + r*vec_rr + x*vec_ks]     (r < nvec)
//   out_r(o)  = out[bat*out_bs + r*out_rr + o*out_os]
struct GemvParams {
    const void *mat;
    const void *vec;
    void *out;
    int64_t rows, k, batch;
    int64_t mat_rs, mat_ks, mat_bs;
    int64_t vec_ks, vec_rr, vec_bs;
    int64_t out_os, out_rr, out_bs;
    int32_t nvec;     // vectors sharing one pass over the matrix (1..16)
    int32_t vec_ok;   // 16-byte vector path legal (host-checked alignment)
    uint32_t *err;            // device error word (streamed kernel's bounded waits)
    uint64_t wait_limit_ns;
};

// General strided GEMM (FFMA pipe).  Same addressing as the public API.
struct GemmParams {
    const void *a;
    const void *b;
    void *c;
    int64_t batch, m, n, k;
    int64_t lda, ldb, ldc;
    int64_t sa, sb, sc;
    int32_t ta, tb;
};

// Tensor-core GEMM: A and B read by TMA through the two tensor maps, each
// K-contiguous (A [batch][m][k], B [batch][n][k]) or, when a_mn / b_mn is
// set, M/N-contiguous (A [batch][k][m], B [batch][k][n]); C written with
// ldc / sc.
struct GemmTcParams {
    void *c;
    int64_t ldc, sc;
    int32_t m, n, k, batch;
    int32_t a_bcast, b_bcast;   // batch stride 0: always batch coordinate 0
    int32_t a_mn, b_mn;         // operand stored M- / N-contiguous
    int32_t c_vec_ok;           // C rows allow 16-byte stores (1) or 32-byte stores (2)
    int32_t tiles_m, tiles_n;
    int32_t num_tiles;
    uint32_t *err;
    uint64_t wait_limit_ns;
};

// Expert-ID matmul (all routes).
struct MatmulIdParams {
    const void *w;
    const float *x;
    const uint32_t *ids;
    float *out;
    uint32_t *counts;        // grouped route scratch
    uint32_t *routed_rows;   // grouped route scratch, row stride m
    int64_t m, n, k, top_k, n_experts;
    int64_t expert_stride_elems;
    int64_t x_token_stride, x_slot_stride;   // elements
    int64_t total_rows;                      // m * top_k
    uint32_t *err;
    uint64_t wait_limit_ns;
};

// Skinny decode GEMV on the tensor cores: y[m, n] (row stride ldc) =
// x[m, k] W[n, k]^T, the operands read through tensor maps.
struct GemvTcParams {
    void *c;
    int64_t ldc;
    int32_t m, n, k;
    int32_t ksplit;  // CTAs per cluster splitting k (1..8), from gemv_tc_split()
    uint32_t *err;
    uint64_t wait_limit_ns;
};

// ---- launchers (each returns the launch's cudaError_t) --------------------

cudaError_t launch_fill_zero(int dt, void *c, int64_t batch, int64_t m, int64_t n, int64_t ldc,
                             int64_t sc, cudaStream_t s);
cudaError_t launch_gemv_rowdot(int dt, const GemvParams &p, cudaStream_t s);
cudaError_t launch_gemv_coldot(int dt, const GemvParams &p, cudaStream_t s);
// staged-stream GEMV (stream.cu) and the shapes it takes
bool gemv_stream_eligible(int dt, const GemvParams &p);
cudaError_t launch_gemv_stream(int dt, const GemvParams &p, int num_sms, cudaStream_t s);
// column-dot GEMV fed by TMA (gemv.cu): `map` is a 3-D tensor map over
// (outputs, k, batch) of the matrix with gemv_coldot_stream_box_cols() x
// gemv_coldot_stream_box_rows() boxes, no swizzle
cudaError_t launch_gemv_coldot_stream(int dt, const CUtensorMap &map, const GemvParams &p, cudaStream_t s);
int gemv_coldot_stream_box_cols(int dt);
int gemv_coldot_stream_box_rows();
// skinny decode GEMV on the tensor cores (gemv_tc.cu): W boxes of
// gemv_tc_block_rows() rows, x boxes of gemv_tc_max_tokens() rows, both
// gemv_tc_block_k() wide
cudaError_t launch_gemv_tc(int dt, const CUtensorMap &map_w, const CUtensorMap &map_x, const GemvTcParams &p,
                           cudaStream_t s);
int gemv_tc_block_rows();
int gemv_tc_max_tokens();
int gemv_tc_block_k();
int gemv_tc_split(int64_t n, int64_t k, int num_sms);
cudaError_t launch_gemm_simt(int dt, const GemmParams &p, cudaStream_t s);
cudaError_t launch_gemm_small(int dt, const GemmParams &p, cudaStream_t s);
cudaError_t launch_gemm_tc(int dt, const CUtensorMap &map_a, const CUtensorMap &map_b,
                           const GemmTcParams &p, int num_sms, cudaStream_t s);
// 256 x 256 tiles (gemm_tc_wide_block_m() rows) over CTA pairs (tcgen05 cta_group::2); a
// K-contiguous operand's tensor map has gemm_tc_block_m()-row boxes, an
// M/N-contiguous one 64 x 64 boxes
cudaError_t launch_gemm_tc_pair(int dt, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                const GemmTcParams &p, int num_sms, cudaStream_t s);
cudaError_t launch_matmul_id_direct(int wdt, const MatmulIdParams &p, cudaStream_t s);
cudaError_t launch_matmul_id_map(const MatmulIdParams &p, cudaStream_t s);
cudaError_t launch_matmul_id_grouped_simt(int wdt, const MatmulIdParams &p, cudaStream_t s);
cudaError_t launch_matmul_id_grouped_tc(const CUtensorMap &map_w, const MatmulIdParams &p, int out_vec_ok,
                                        int split, int f16, int num_sms, cudaStream_t s);
cudaError_t launch_bounded_wait_test(uint32_t *err, uint64_t limit_ns, cudaStream_t s);
int grouped_tc_max_experts();
// Direct route on the tensor cores (direct_tc.cu): bf16 or f16 weights
// (wdt) through a 3-D tensor map over (k, n, expert) with direct_tc_block_k()
// x direct_tc_block_rows() boxes; at most direct_tc_max_ids() routed rows and
// direct_tc_max_experts() experts
cudaError_t launch_matmul_id_direct_tc(int wdt, const CUtensorMap &map_w, const MatmulIdParams &p,
                                       int max_distinct, int ksplit, int x_vec_ok, cudaStream_t s);
int direct_tc_split(int64_t n, int64_t k, int64_t max_distinct, int64_t max_rows_per_expert, int num_sms);
int direct_tc_max_ids();
int direct_tc_max_experts();
int direct_tc_block_rows();
int direct_tc_block_k();
int grouped_tc_block_k();

int gemm_tc_block_m();
int gemm_tc_wide_block_m();
int gemm_tc_block_n();
int gemm_tc_block_k();
int device_sm_count();

// device address of the error word on the current device (nullptr on failure)
uint32_t *device_error_word();

}  // namespace gbmm
