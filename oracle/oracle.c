/*
 * oracle.c -- plain, slow CPU oracle for the dense GEMM / GEMV / expert-ID
 * matmul path.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers.  The product (the CUDA library) never
 * links, loads or calls this file, and this file shares no code, header or
 * table with it.
 *
 * Every result is the plain definition written out: one output element is
 * one loop over the contraction index in increasing order, accumulated in
 * IEEE binary64.  Alongside each element the oracle returns sum |a||b| over
 * the same terms, which the parity tolerance is scaled by.  Threads only
 * split the list of requested output elements; they never change the
 * arithmetic of an element.
 *
 * Sources (page titles and the Rust items on them):
 *   [P1] tract-metal 0.23.6, src/kernels/matmul/mlx_gemm/mod.rs --
 *        `MlxGemm::dispatch_eval`, `dispatch_metal_mlx_gemv`,
 *        `dispatch_metal_mlx_gemm` (operand layouts under the transpose flags),
 *        `dispatch_metal_mlx_gemv_wide`, and the naive reference loop of
 *        `gemv_wide_tests::check`.
 *   [P2] mlx-native 0.13.0, src/ops/dense_matmul_id.rs -- module contract,
 *        `DenseMatmulIdInputLayout`, `dense_matmul_id` (input strides per
 *        layout; out-of-range ids give a zero row), `DenseMatmulIdScratch`,
 *        `dense_matmul_id_capability` (scratch extents n_experts x m).
 *   [P3] rlx-metal 0.2.14, src/mps_blas.rs -- `encode_mps_sgemm_t`
 *        (transposeLeft: A stored [k,m]; transposeRight: B stored [n,k]).
 *
 * Readings where the pages leave a step open (each one listed in the design
 * notes of the repository):
 *   - per-expert weights are row-major [n, k] (an output row is a contiguous
 *     k vector);
 *   - routed_rows entries are the flattened routed-row index r = t*top_k + s,
 *     ascending within an expert, expert e's list starting at e*m;
 *   - an id >= n_experts yields an all-zero output row and is not counted.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* ---- element decoding ------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double or_f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = (double)frac / 1024.0 / 16384.0; /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        v = frac ? (0.0 / 0.0) : (1.0 / 0.0);
    } else {
        double scale = 1.0;
        int e = expo - 15;
        while (e > 0) { scale *= 2.0; --e; }
        while (e < 0) { scale *= 0.5; ++e; }
        v = (1.0 + (double)frac / 1024.0) * scale;
    }
    return sign ? -v : v;
}

/* bf16 is the upper half of an IEEE 754 binary32. */
static double or_bf16_value(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double or_load(int dt, const void *base, int64_t idx)
{
    switch (dt) {
    case OR_F32: return (double)((const float *)base)[idx];
    case OR_F16: return or_f16_value(((const uint16_t *)base)[idx]);
    case OR_BF16: return or_bf16_value(((const uint16_t *)base)[idx]);
    default: return 0.0;
    }
}

/* Decode `count` stored elements to binary64 (used to pin the decoders). */
void oracle_decode(int dt, const void *src, int64_t count, double *dst)
{
    for (int64_t i = 0; i < count; ++i)
        dst[i] = or_load(dt, src, i);
}

/* ---- a tiny thread pool over an index range ---------------------------- */

typedef void (*or_range_fn)(void *ctx, int64_t lo, int64_t hi);

struct or_job { or_range_fn fn; void *ctx; int64_t lo, hi; };

static void *or_job_main(void *arg)
{
    struct or_job *j = (struct or_job *)arg;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void or_parallel(or_range_fn fn, void *ctx, int64_t count, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > count) nthreads = (int)(count > 0 ? count : 1);
    if (nthreads == 1) { fn(ctx, 0, count); return; }
    pthread_t th[256];
    struct or_job jobs[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].lo = count * t / nthreads;
        jobs[t].hi = count * (t + 1) / nthreads;
        if (pthread_create(&th[t], NULL, or_job_main, &jobs[t]) == 0) {
            ++started;
        } else {
            or_job_main(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    (void)started;
}

/* ---- dense GEMM / GEMV -------------------------------------------------- */

/*
 * C[b,i,j] = sum_{x<k} Aop[b,i,x] * Bop[b,x,j]                        [P1, P3]
 *   Aop[b,i,x] = A[b*sa + (ta ? x*lda + i : i*lda + x)]   (A stored [k,m] when ta)
 *   Bop[b,x,j] = B[b*sb + (tb ? j*ldb + x : x*ldb + j)]   (B stored [n,k] when tb)
 * A GEMV (m == 1 or n == 1) is the same definition at that shape [P1
 * `dispatch_metal_mlx_gemv`], and so is the wide skinny case (m in 2..15,
 * B stored [n,k]) [P1 `dispatch_metal_mlx_gemv_wide`].
 */
struct or_gemm_ctx {
    int dt;
    int64_t batch, m, n, k;
    int ta, tb;
    const void *a; int64_t lda, sa;
    const void *b; int64_t ldb, sb;
    const int64_t *idx;  /* NULL: every element of [batch, m, n] in order */
    double *c, *c_abs;
};

static void or_gemm_range(void *vctx, int64_t lo, int64_t hi)
{
    const struct or_gemm_ctx *g = (const struct or_gemm_ctx *)vctx;
    for (int64_t q = lo; q < hi; ++q) {
        int64_t flat = g->idx ? g->idx[q] : q;
        int64_t bb = flat / (g->m * g->n);
        int64_t rem = flat % (g->m * g->n);
        int64_t i = rem / g->n;
        int64_t j = rem % g->n;
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t x = 0; x < g->k; ++x) {
            int64_t ia = bb * g->sa + (g->ta ? x * g->lda + i : i * g->lda + x);
            int64_t ib = bb * g->sb + (g->tb ? j * g->ldb + x : x * g->ldb + j);
            double av = or_load(g->dt, g->a, ia);
            double bv = or_load(g->dt, g->b, ib);
            acc += av * bv;
            acc_abs += (av < 0 ? -av : av) * (bv < 0 ? -bv : bv);
        }
        g->c[q] = acc;
        if (g->c_abs) g->c_abs[q] = acc_abs;
    }
}

/*
 * Computes `count` output elements.  With idx == NULL, count must be
 * batch*m*n and the results come back in [batch, m, n] order; otherwise
 * idx[q] is the flat index b*m*n + i*n + j of the q-th requested element.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemm(int dt, int64_t batch, int64_t m, int64_t n, int64_t k, int ta, int tb,
                const void *a, int64_t lda, int64_t sa,
                const void *b, int64_t ldb, int64_t sb,
                int64_t count, const int64_t *idx, double *c, double *c_abs, int nthreads)
{
    if (dt < OR_F32 || dt > OR_BF16 || batch < 0 || m < 0 || n < 0 || k < 0 || count < 0)
        return -1;
    if (!idx && count != batch * m * n) return -1;
    struct or_gemm_ctx g = { dt, batch, m, n, k, ta, tb, a, lda, sa, b, ldb, sb, idx, c, c_abs };
    or_parallel(or_gemm_range, &g, count, nthreads);
    return 0;
}

/* ---- expert-ID matmul ----------------------------------------------------- */

/*
 * For routed row r = t*top_k + s (t < m, s < top_k), e = ids[r]:      [P2]
 *   e >= n_experts : out[r, :] = 0
 *   otherwise      : out[r, j] = sum_{x<k} W_e[j, x] * xrow(t, s)[x]
 * W_e starts expert_stride_bytes * e bytes into the weight buffer and is
 * row-major [n, k].  xrow(t, s) is the f32 row at
 *   SharedPerToken (layout 0): x + t*k
 *   Slotted        (layout 1): x + (t*top_k + s)*k
 * (the token/slot strides of `dense_matmul_id`).  Output is [m, top_k, n].
 */
struct or_mid_ctx {
    int wdt;
    int64_t m, n, k, top_k, n_experts;
    int64_t expert_stride_elems;
    int layout;
    const void *w; const float *x; const uint32_t *ids;
    const int64_t *idx;  /* NULL: every element of [m*top_k, n] */
    double *out, *out_abs;
};

static void or_mid_range(void *vctx, int64_t lo, int64_t hi)
{
    const struct or_mid_ctx *g = (const struct or_mid_ctx *)vctx;
    for (int64_t q = lo; q < hi; ++q) {
        int64_t flat = g->idx ? g->idx[q] : q;
        int64_t r = flat / g->n;
        int64_t j = flat % g->n;
        int64_t t = r / g->top_k;
        int64_t s = r % g->top_k;
        uint32_t e = g->ids[r];
        double acc = 0.0, acc_abs = 0.0;
        if ((int64_t)e < g->n_experts) {
            const float *xrow = g->layout == 0 ? g->x + t * g->k
                                               : g->x + (t * g->top_k + s) * g->k;
            int64_t wbase = (int64_t)e * g->expert_stride_elems + j * g->k;
            for (int64_t x = 0; x < g->k; ++x) {
                double wv = or_load(g->wdt, g->w, wbase + x);
                double xv = (double)xrow[x];
                acc += wv * xv;
                acc_abs += (wv < 0 ? -wv : wv) * (xv < 0 ? -xv : xv);
            }
        }
        g->out[q] = acc;
        if (g->out_abs) g->out_abs[q] = acc_abs;
    }
}

int oracle_matmul_id(int wdt, int64_t m, int64_t n, int64_t k, int64_t top_k, int64_t n_experts,
                     int64_t expert_stride_bytes, int input_layout,
                     const void *w, const float *x, const uint32_t *ids,
                     int64_t count, const int64_t *idx, double *out, double *out_abs,
                     int nthreads)
{
    int64_t size = wdt == OR_F32 ? 4 : 2;
    if (wdt < OR_F32 || wdt > OR_BF16 || expert_stride_bytes % size != 0) return -1;
    if (input_layout != 0 && input_layout != 1) return -1;
    if (!idx && count != m * top_k * n) return -1;
    struct or_mid_ctx g = { wdt, m, n, k, top_k, n_experts, expert_stride_bytes / size,
                            input_layout, w, x, ids, idx, out, out_abs };
    or_parallel(or_mid_range, &g, count, nthreads);
    return 0;
}

/*
 * Routing map of the grouped route                                     [P2]
 * One sequential pass over r = 0 .. m*top_k-1: an id e < n_experts appends r
 * to expert e's list, which starts at routed_rows[e*m]; counts[e] is the
 * list's length.  Ids >= n_experts are skipped.  Entries past counts[e] are
 * left untouched.  Under the distinct-per-token promise a list never exceeds
 * m entries; if the promise is broken, entries past the m-th are dropped
 * (counts[e] still reports the full count).
 */
void oracle_map_distinct(int64_t m, int64_t top_k, int64_t n_experts, const uint32_t *ids,
                         uint32_t *counts, uint32_t *routed_rows)
{
    for (int64_t e = 0; e < n_experts; ++e) counts[e] = 0;
    for (int64_t r = 0; r < m * top_k; ++r) {
        uint32_t e = ids[r];
        if ((int64_t)e >= n_experts) continue;
        if ((int64_t)counts[e] < m) /* only a broken distinct promise overflows */
            routed_rows[(int64_t)e * m + counts[e]] = (uint32_t)r;
        counts[e] += 1;
    }
}
