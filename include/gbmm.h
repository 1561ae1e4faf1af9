/*
 * gbmm.h -- C ABI of the GB300 (sm_103a) dense GEMM / GEMV / expert-ID matmul
 * library (libgbmm.so).
 *
 * Conventions shared by every entry point
 *   - Pointers named a, b, c, weights, input, ids, out, expert_counts and
 *     routed_rows are DEVICE pointers (cudaMalloc / torch CUDA memory of the
 *     current device).  The caller owns all device memory; the library never
 *     allocates device memory on a call path and never synchronises the
 *     stream (except gbmm_device_error and the test hooks, which say so).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and runs asynchronously.  Stream order is the only ordering:
 *     reuse of an output or scratch buffer on the same stream is safe, on
 *     another stream the caller must order it.
 *   - Fail-closed: every argument check runs on the host before the first
 *     launch.  A call that returns an error launched nothing and wrote
 *     nothing.  gbmm_last_error() then describes the failure.
 *   - Thread safety: calls may be made from several host threads; the error
 *     string is per thread.
 *   - CUDA graphs: every call can be captured into a graph once the same
 *     call has run on the device outside the capture (the first call on a
 *     device sets kernel attributes, looks up the device error word and loads
 *     modules, which a capture does not allow); replays read whatever
 *     the captured buffers hold.  GroupedPrefill's grouped kernel is launched
 *     with programmatic stream serialisation behind the map kernel and waits
 *     for it before touching global memory, which a capture keeps.  Not with
 *     GBMM_DEBUG_SYNC=1 (it synchronises the stream).
 *   - Debugging: with the environment variable GBMM_DEBUG_SYNC=1 (read once
 *     per process) every launch is followed by a stream synchronisation, so a
 *     kernel that fails on the device is reported by the call that launched
 *     it (GBMM_ERR_CUDA, with the kernel's name in gbmm_last_error()) -- the
 *     counterpart of [P1]'s debug wait_until_completed.
 *
 * Sources (page titles and the items on them)
 *   [P1] tract-metal 0.23.6, src/kernels/matmul/mlx_gemm/mod.rs
 *   [P2] mlx-native 0.13.0, src/ops/dense_matmul_id.rs
 *   [P3] rlx-metal 0.2.14, src/mps_blas.rs
 */
#ifndef GBMM_H
#define GBMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GBMM_ABI_VERSION 1u
/* Schema version of the expert-ID capability record, as in [P2]
 * `DENSE_MATMUL_ID_SCHEMA_VERSION`. */
#define GBMM_MATMUL_ID_SCHEMA_VERSION 3u
/* Most experts the grouped route accepts, as in [P2] `GROUPED_MAX_EXPERTS`. */
#define GBMM_GROUPED_MAX_EXPERTS 1024u

#if defined(__GNUC__)
#define GBMM_API __attribute__((visibility("default")))
#else
#define GBMM_API
#endif

typedef struct CUstream_st *gbmm_stream; /* == cudaStream_t */

typedef enum gbmm_status {
    GBMM_OK = 0,
    GBMM_ERR_INVALID_ARGUMENT = 1,  /* a shape, stride, size, flag or alignment rule failed */
    GBMM_ERR_UNSUPPORTED_DTYPE = 2, /* dtype outside the call's set */
    GBMM_ERR_OVERLAP = 3,           /* an output range overlaps an input or scratch range */
    GBMM_ERR_SCRATCH = 4,           /* grouped route: scratch missing or too small */
    GBMM_ERR_KERNEL_UNAVAILABLE = 5,/* a kernel this call needs could not be resolved */
    GBMM_ERR_LAUNCH = 6,            /* the CUDA launch itself failed */
    GBMM_ERR_DEVICE_TIMEOUT = 7,    /* a bounded device-side wait ran out (gbmm_device_error) */
    GBMM_ERR_CUDA = 8               /* another CUDA runtime error */
} gbmm_status;

typedef enum gbmm_dtype {
    GBMM_F32 = 0,
    GBMM_F16 = 1,
    GBMM_BF16 = 2
} gbmm_dtype;

/* ------------------------------------------------------------------------ */
/* Dense GEMM / GEMV                                                          */
/* ------------------------------------------------------------------------ */

/*
 * gbmm_gemm -- C[b] = op(A[b]) * op(B[b]) for b < batch.
 *
 * Defined by [P1] `MlxGemm::dispatch_eval` / `dispatch_metal_mlx_gemm` and
 * [P3] `encode_mps_sgemm_t` (transposeLeft / transposeRight):
 *   C[b,i,j] = sum_{x<k} Aop[b,i,x] * Bop[b,x,j],   i < m, j < n
 *   Aop[b,i,x] = A[b*batch_stride_a + (transpose_a ? x*lda + i : i*lda + x)]
 *   Bop[b,x,j] = B[b*batch_stride_b + (transpose_b ? j*ldb + x : x*ldb + j)]
 *   C[b*batch_stride_c + i*ldc + j] receives the result.
 * So A is stored [k, m] when transpose_a, else [m, k]; B is stored [n, k]
 * when transpose_b, else [k, n]; all row-major with leading dims lda/ldb/ldc.
 *
 * dt: one dtype for A, B and C ([P1] homogeneous datum types); f32, f16 and
 *   bf16.  Products accumulate in f32; f16/bf16 results are rounded to
 *   nearest-even once, from the f32 accumulator.
 * a/b/c + *_offset_bytes: the matrix base; the sum must be aligned to the
 *   element size (offsets are in bytes, as Metal buffer offsets are in [P1]).
 * lda >= (transpose_a ? m : k), ldb >= (transpose_b ? k : n), ldc >= n, in
 *   elements.  Batch strides are in elements and >= 0; A or B may broadcast
 *   one matrix to every batch with stride 0; batches of C must not overlap.
 * C must not overlap A or B (GBMM_ERR_OVERLAP).
 * Edge cases: batch, m or n == 0 is a no-op; k == 0 writes zeros to C.
 *
 * Route (host-side, fixed rules, [P1] `dispatch_eval`):
 *   - skinny/wide (16-bit dt, !transpose_a, transpose_b, batch == 1,
 *     2 <= m <= 15): one HBM-streaming pass over B with a register tile of m
 *     rows of A ([P1] `gemv_wide_config` gate on m);
 *   - m == 1 or n == 1: the GEMV kernels (as gbmm_gemv);
 *   - otherwise the tensor-core GEMM (tcgen05 + TMEM, TMA-fed) when dt is
 *     f16/bf16 and the TMA layout rules hold (K-contiguous A and B, leading
 *     dims and batch strides multiples of 16 bytes, 16-byte aligned bases),
 *     else the FFMA GEMM.
 */
GBMM_API gbmm_status gbmm_gemm(gbmm_dtype dt, int64_t batch, int64_t m, int64_t n, int64_t k,
                      int transpose_a, int transpose_b,
                      const void *a, int64_t a_offset_bytes, int64_t lda, int64_t batch_stride_a,
                      const void *b, int64_t b_offset_bytes, int64_t ldb, int64_t batch_stride_b,
                      void *c, int64_t c_offset_bytes, int64_t ldc, int64_t batch_stride_c,
                      gbmm_stream stream);

/*
 * gbmm_gemv -- the matrix x vector special case of gbmm_gemm ([P1]
 * `dispatch_metal_mlx_gemv`): same arguments and definition, and requires
 * m == 1 or n == 1 (else GBMM_ERR_INVALID_ARGUMENT).  With n != 1 the
 * matrix is B (the vector is row 0 of op(A)); otherwise the matrix is A (the
 * vector is column 0 of op(B)).  A matrix whose rows run along the
 * contraction dim is read as one coalesced, 128-bit-vectorised stream with
 * warp-shuffle reductions; the other orientation reduces across rows.
 */
GBMM_API gbmm_status gbmm_gemv(gbmm_dtype dt, int64_t batch, int64_t m, int64_t n, int64_t k,
                      int transpose_a, int transpose_b,
                      const void *a, int64_t a_offset_bytes, int64_t lda, int64_t batch_stride_a,
                      const void *b, int64_t b_offset_bytes, int64_t ldb, int64_t batch_stride_b,
                      void *c, int64_t c_offset_bytes, int64_t ldc, int64_t batch_stride_c,
                      gbmm_stream stream);

/* ------------------------------------------------------------------------ */
/* Expert-ID matmul                                                           */
/* ------------------------------------------------------------------------ */

/* [P2] `DenseMatmulIdInputLayout` */
enum { GBMM_INPUT_SHARED_PER_TOKEN = 0, GBMM_INPUT_SLOTTED = 1 };
/* [P2] `DenseMatmulIdMultiplicity` */
enum { GBMM_IDS_DISTINCT_PER_TOKEN = 0, GBMM_IDS_MAY_REPEAT = 1 };
/* [P2] `DenseMatmulIdRoute`: chosen by the caller; the library never picks. */
enum { GBMM_ROUTE_DIRECT = 0, GBMM_ROUTE_GROUPED_PREFILL = 1 };

/* [P2] `DenseMatmulIdParams` */
typedef struct gbmm_matmul_id_params {
    uint32_t m;            /* tokens */
    uint32_t n;            /* output features = rows of each expert matrix */
    uint32_t k;            /* input features = columns of each expert matrix */
    uint32_t top_k;        /* expert slots per token */
    uint32_t n_experts;    /* experts in the weight stack */
    uint32_t input_layout; /* GBMM_INPUT_* */
    uint32_t multiplicity; /* GBMM_IDS_* */
    uint32_t route;        /* GBMM_ROUTE_* */
    uint64_t expert_stride_bytes; /* bytes from expert e to expert e+1 */
    /* GBMM_ACT_* (an extension of this library; zero = the pages' f32
     * activation product).  Only the GroupedPrefill route with bf16 or f16
     * weights on the tensor cores reads it; elsewhere every value computes in
     * f32. */
    uint32_t activation_precision;
    uint32_t reserved;     /* must be 0 */
} gbmm_matmul_id_params;

/*
 * Activation precision of the tensor-core grouped GEMM (bf16 or f16 weights,
 * f32 activations).  Tensor cores multiply pairs of one 16-bit type, so the
 * f32 activations must be rounded to the weights' type (for f16 weights each
 * routed row first scaled by a power of two that puts its largest magnitude
 * in [2^14, 2^15), and the result scaled back exactly):
 *   GBMM_ACT_SPLIT (default): x = hi + lo with hi = round(x), lo = round(x - hi),
 *     both multiplied by the weights -- activation error <= 2^-16 |x| (bf16),
 *     2^-22 |x| (f16), the product is f32-accurate and every element meets
 *     2e-3 * sum|w||x|.
 *   GBMM_ACT_BF16: x rounded once, half the tensor work -- activation error
 *     <= 2^-8 |x| for bf16 weights, so an element can differ from the f32
 *     product by up to ~2^-8 * sum|w||x| (about 3.9e-3, above the 2e-3 bound
 *     when all products share a sign; far below it for zero-mean data); for
 *     f16 weights <= 2^-11 |x|, inside the bound.
 */
enum { GBMM_ACT_SPLIT = 0, GBMM_ACT_BF16 = 1 };

/* [P2] `DenseMatmulIdCapability` + `DenseMatmulIdScratchRequirement` */
typedef struct gbmm_matmul_id_capability_t {
    uint32_t schema_version;     /* GBMM_MATMUL_ID_SCHEMA_VERSION */
    uint32_t weight_dtype;       /* gbmm_dtype */
    uint32_t route;              /* GBMM_ROUTE_* */
    uint32_t has_scratch;        /* 1 for the grouped route */
    uint64_t required_weight_bytes; /* (n_experts-1)*expert_stride_bytes + n*k*size */
    uint64_t required_input_bytes;  /* (shared ? m : m*top_k) * k * 4 */
    uint64_t required_ids_bytes;    /* m*top_k*4 */
    uint64_t required_output_bytes; /* m*top_k*n*4 */
    uint64_t expert_counts_bytes;   /* n_experts*4 (grouped), else 0 */
    uint64_t routed_rows_bytes;     /* n_experts*m*4 (grouped), else 0 */
} gbmm_matmul_id_capability_t;

/* [P2] `DenseMatmulIdDispatchReceipt` */
typedef struct gbmm_matmul_id_receipt {
    uint32_t weight_dtype;  /* gbmm_dtype */
    uint32_t route;         /* GBMM_ROUTE_* */
    uint32_t launch_count;  /* kernels enqueued: 1 (Direct) or 2 (GroupedPrefill) */
} gbmm_matmul_id_receipt;

/*
 * Caller-owned scratch of the grouped route ([P2] `DenseMatmulIdScratch`):
 *   expert_counts  u32[max_experts]
 *   routed_rows    u32[max_experts * max_tokens]
 * After a grouped call, expert_counts[e] is the number of routed rows with
 * id e and routed_rows[e*m + i], i < expert_counts[e], lists them in
 * increasing order of the flattened routed row r = t*top_k + s.  Both
 * buffers must outlive the work enqueued on them and must not overlap the
 * weights, input, ids, output or each other.
 */
typedef struct gbmm_matmul_id_scratch {
    uint32_t *expert_counts;
    uint64_t expert_counts_bytes;
    uint32_t *routed_rows;
    uint64_t routed_rows_bytes;
    uint32_t max_experts;
    uint32_t max_tokens;
} gbmm_matmul_id_scratch;

/*
 * gbmm_matmul_id_scratch_bytes -- byte sizes of the scratch buffers for a
 * capacity of (max_experts, max_tokens), as [P2] `DenseMatmulIdScratch::new`
 * computes them (both capacities must be nonzero; overflow is an error).
 * Allocates nothing.
 */
GBMM_API gbmm_status gbmm_matmul_id_scratch_bytes(uint32_t max_experts, uint32_t max_tokens,
                                         uint64_t *expert_counts_bytes,
                                         uint64_t *routed_rows_bytes);

/*
 * gbmm_matmul_id_capability -- fail-closed validation and exact byte
 * extents, with the rules of [P2] `dense_matmul_id_capability`:
 *   m, n, k, top_k, n_experts nonzero; DistinctPerToken with top_k >
 *   n_experts rejected; weight dtype f32/f16/bf16; expert_stride_bytes >=
 *   n*k*size and a multiple of size; all extents overflow-checked in u64;
 *   m*top_k <= UINT32_MAX; GroupedPrefill requires DistinctPerToken and
 *   n_experts <= GBMM_GROUPED_MAX_EXPERTS.
 * Writes *out on success only.  Host-only: needs no GPU.
 */
GBMM_API gbmm_status gbmm_matmul_id_capability(gbmm_dtype weight_dtype, const gbmm_matmul_id_params *p,
                                      gbmm_matmul_id_capability_t *out);

/*
 * gbmm_matmul_id -- expert-ID matrix multiplication ([P2] `dense_matmul_id`).
 *
 * For routed row r = t*top_k + s (t < m, s < top_k) with e = ids[r]:
 *   e >= n_experts: out[r, :] = 0 (the whole row is overwritten, no weight
 *                   address is formed);
 *   otherwise:      out[r, j] = sum_{x<k} W_e[j, x] * xrow(t, s)[x],  j < n,
 * W_e = the row-major [n, k] matrix at byte offset e*expert_stride_bytes of
 * `weights`; xrow(t, s) = input + t*k (SharedPerToken) or input +
 * (t*top_k + s)*k (Slotted); out is f32 [m, top_k, n].  Weights are widened
 * to f32; accumulation is f32.
 *
 * weights/input/ids/out (+ *_bytes): device buffers and their lengths; each
 *   length must cover the capability extent and each pointer must be aligned
 *   to its element type ([P2] `validate_buffer`).
 * out must not overlap weights, input or ids ([P2]
 *   `validate_dense_matmul_id_call`), else GBMM_ERR_OVERLAP.
 * scratch: required for GroupedPrefill (max_experts >= n_experts, max_tokens
 *   >= m, byte lengths >= the requirement; else GBMM_ERR_SCRATCH); may be
 *   NULL for Direct.
 * Routes:
 *   Direct: one launch; each distinct expert selected by the call is
 *     streamed from HBM once and applied to every row that selected it (bf16
 *     or f16 weights with 16-byte aligned rows and at most 1024 routed rows:
 *     on the tensor cores, activations split into hi + lo of the weights'
 *     type -- for f16 each routed row first scaled by a power of two into
 *     f16's range, and scaled back exactly; otherwise on the FFMA pipe).
 *   GroupedPrefill: two launches in stream order -- the routing map
 *     (expert_counts / routed_rows, atomic-free count / scan / scatter; also
 *     zero-fills rows with out-of-range ids), then the grouped GEMM over
 *     each expert's row list (tensor cores for bf16 weights with hi + lo
 *     activations, and for f16 weights with per-row scaled f16 hi + lo; FFMA
 *     for f32 weights and strides TMA cannot read).  The second launch reads
 *     the first's scratch; a later call may reuse the scratch on the same
 *     stream.
 * Both kernels this call needs are resolved before the first launch; if one
 * is unavailable the call fails with nothing enqueued ([P2] `dense_matmul_id`
 * resolves every pipeline before touching the encoder).
 * receipt (may be NULL): written on success.
 */
GBMM_API gbmm_status gbmm_matmul_id(const gbmm_matmul_id_params *p, gbmm_dtype weight_dtype,
                           const void *weights, uint64_t weights_bytes,
                           const float *input, uint64_t input_bytes,
                           const uint32_t *ids, uint64_t ids_bytes,
                           float *out, uint64_t out_bytes,
                           const gbmm_matmul_id_scratch *scratch,
                           gbmm_stream stream, gbmm_matmul_id_receipt *receipt);

/*
 * gbmm_matmul_id_static_scratch -- the GroupedPrefill route of
 * gbmm_matmul_id for callers that cannot allocate device memory.  (The
 * pages have no counterpart: their grouped route always takes caller-owned
 * scratch.)
 *
 * Who needs it: a caller that is handed only the operands and outputs of
 * each call while someone else owns all other device memory (a plugin slot
 * in another runtime), or a serving loop that may not call cudaMalloc once
 * it runs, since an allocation can wait on a device-wide synchronisation.
 * Such a caller cannot supply the expert_counts / routed_rows buffers.
 *
 * What it does: exactly gbmm_matmul_id with route GroupedPrefill (same
 * arguments minus `scratch`, same results, two launches), with the scratch
 * taken from one fixed array compiled into the library.  The array holds
 * GBMM_GROUPED_MAX_EXPERTS counts and GBMM_STATIC_SCRATCH_ROUTED_ROWS_BYTES
 * of routed rows, i.e. n_experts * m <= 1,048,576; it is reserved on every
 * GPU that loads the library until the process exits.  The call allocates
 * nothing and calls no allocating routine.
 *
 * Errors: GBMM_ERR_INVALID_ARGUMENT for a NULL params or a route other than
 * GroupedPrefill; GBMM_ERR_SCRATCH (nothing launched) when n_experts * m * 4
 * exceeds the array; otherwise every rule and status of gbmm_matmul_id.
 *
 * Sharing: every call on every stream of a device uses the same array, and
 * the array keeps the last call's contents.  Nothing in it needs to start at
 * zero (each call rewrites what it reads).  Calls whose work overlaps on the
 * GPU -- concurrent streams, or host threads without stream ordering between
 * them -- race on the array and corrupt each other's results; order them.
 *
 * Set-up: the first call on each device (that device current) looks up the
 * array's device address with cudaGetSymbolAddress and caches it.  With the
 * CUDA runtime's lazy module loading (the default) that lookup is also what
 * loads the array onto the device: a one-time device allocation made by the
 * CUDA runtime, not by this library.  So make one call per device as a
 * warm-up, before serving starts and before any stream capture on it.  The
 * cached address belongs to the device's current context: after
 * cudaDeviceReset (or any reset of the primary context) the array may live
 * at another address, and this entry point must not be called again in that
 * process.
 */
#define GBMM_STATIC_SCRATCH_ROUTED_ROWS_BYTES (4u << 20)
GBMM_API gbmm_status gbmm_matmul_id_static_scratch(const gbmm_matmul_id_params *p,
                                                   gbmm_dtype weight_dtype,
                                                   const void *weights, uint64_t weights_bytes,
                                                   const float *input, uint64_t input_bytes,
                                                   const uint32_t *ids, uint64_t ids_bytes,
                                                   float *out, uint64_t out_bytes,
                                                   gbmm_stream stream,
                                                   gbmm_matmul_id_receipt *receipt);

/* ------------------------------------------------------------------------ */
/* Errors, diagnostics                                                        */
/* ------------------------------------------------------------------------ */

/* Message of the last failed call on this host thread ("" if none).  The
 * string stays valid until the next call on the thread. */
GBMM_API const char *gbmm_last_error(void);

/* Name of a status code. */
GBMM_API const char *gbmm_status_string(gbmm_status s);

/* GBMM_ABI_VERSION. */
GBMM_API uint32_t gbmm_abi_version(void);

/*
 * gbmm_device_error -- synchronises `stream`, then reads and clears the
 * device error word of the current device.  Kernels set it (instead of
 * trapping) when a bounded wait on an mbarrier runs out; the kernel then
 * drains its own copies in flight, releases its tensor memory and returns.
 * *code receives the word (0 = no error; otherwise bit 0 = a wait ran out,
 * bits 8..15 = which kernel).  Returns GBMM_ERR_DEVICE_TIMEOUT when the word
 * was nonzero, GBMM_OK otherwise.
 */
GBMM_API gbmm_status gbmm_device_error(gbmm_stream stream, uint32_t *code);

/* ------------------------------------------------------------------------ */
/* Test hooks (host-side fault injection and launch accounting)               */
/* ------------------------------------------------------------------------ */

/* Makes the next resolution of kernel `name` fail (one shot), like [P2]'s
 * `KernelRegistry::inject_next_pipeline_lookup_failure`.  NULL clears it.
 * The name "*" makes every resolution fail until cleared: a call that passes
 * validation then returns GBMM_ERR_KERNEL_UNAVAILABLE with nothing launched
 * (tests that hand the library addresses no kernel may touch use it).
 * Kernel names: "gbmm_gemv_rowdot", "gbmm_gemv_coldot", "gbmm_gemv_tc", "gbmm_gemm_simt",
 * "gbmm_gemm_tc", "gbmm_fill_zero", "gbmm_matmul_id_direct",
 * "gbmm_matmul_id_map", "gbmm_matmul_id_grouped". */
GBMM_API void gbmm_test_inject_kernel_failure(const char *name);

/* Kernels launched by this library since load / the last reset. */
GBMM_API uint64_t gbmm_test_launch_count(void);
GBMM_API void gbmm_test_reset_launch_count(void);

/* Name of the kernel of the most recent launch on this host thread:
 * "gbmm_gemm_tc", "gbmm_gemm_simt", "gbmm_gemm_small", "gbmm_gemv_stream",
 * "gbmm_gemv_rowdot", "gbmm_gemv_coldot", "gbmm_gemv_tc", "gbmm_fill_zero",
 * "gbmm_matmul_id_direct", "gbmm_matmul_id_direct_tc", "gbmm_matmul_id_map",
 * "gbmm_matmul_id_grouped_tc", "gbmm_matmul_id_grouped_simt", and "gbmm_bounded_wait_test" for the wait test below. */
GBMM_API const char *gbmm_test_last_kernel(void);

/*
 * gbmm_test_bounded_wait -- launches one tiny kernel that waits on an
 * mbarrier that nothing ever arrives on, with a limit of `limit_ns`
 * nanoseconds (clamped to [1 us, 2 s]).  The wait runs out, the kernel sets
 * the device error word and returns; then this call synchronises and
 * returns what gbmm_device_error returns (GBMM_ERR_DEVICE_TIMEOUT with *code
 * set).  Exercises the timeout path without faulting or hanging the GPU.
 */
GBMM_API gbmm_status gbmm_test_bounded_wait(uint64_t limit_ns, gbmm_stream stream, uint32_t *code);

/*
 * gbmm_test_static_scratch_copy -- enqueues on `stream` a device-to-device
 * copy of the first `bytes` bytes of the fixed scratch array that
 * gbmm_matmul_id_static_scratch uses on the current device, into the
 * caller's device buffer `dst`: the expert counts (u32[GBMM_GROUPED_MAX_EXPERTS])
 * first, then the routed-row lists (u32, expert e's list at entry e * m of
 * that region, m the last call's token count).  Lets a test check the routing
 * map the last call left there.  GBMM_ERR_INVALID_ARGUMENT when `bytes`
 * exceeds the array or `dst` is NULL.
 */
GBMM_API gbmm_status gbmm_test_static_scratch_copy(void *dst, uint64_t bytes, gbmm_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* GBMM_H */
