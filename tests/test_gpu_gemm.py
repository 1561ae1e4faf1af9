"""GPU parity of the dense GEMM / GEMV entry points against the CPU oracle,
called through the C ABI (gbmm_gemm / gbmm_gemv).

Covers every route (tensor-core GEMM, FFMA GEMM, row/column GEMV, the
skinny/wide path, the k == 0 fill), all dtypes and transposes, padded
leading dims, batch strides (including broadcast), byte offsets, ragged
tails, guard bands around C, and the three dense workloads at full size
(the 4 x 4096^3 GEMM on sampled outputs).
"""

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemv_moe_expert_gb300 import binding as gb  # noqa: E402
from gemv_moe_expert_gb300 import synth  # noqa: E402
from tests.gpu_util import (GUARD, DevBuf, StridedGemm, NP_DT, assert_close, to_f64)  # noqa: E402

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemv_moe_expert_gb300 import build
    build.build()
    gb.load()
    torch.cuda.init()


def run_case(oracle_mod, g: StridedGemm, fn=gb.gbmm_gemm, expect_kernel=None, idx=None):
    a, b, c = g.device()
    gb.gbmm_test_reset_launch_count()
    st = fn(*g.args(a, b, c))
    assert st == gb.GBMM_OK, gb.gbmm_last_error()
    torch.cuda.synchronize()
    if expect_kernel is not None:
        assert gb.gbmm_test_last_kernel() == expect_kernel
        assert gb.gbmm_test_launch_count() == 1
    assert gb.gbmm_device_error()[0] == gb.GBMM_OK
    assert a.guards_intact() and b.guards_intact() and c.guards_intact()
    assert g.c_gaps_untouched(c)
    got = g.gather_c(c)
    if idx is None:
        ref, ref_abs = g.oracle(oracle_mod)
        return assert_close(got, ref, ref_abs, g.dtype, g.dtype, f"{g.dtype} {g.m}x{g.n}x{g.k}")
    ref, ref_abs = g.oracle(oracle_mod, idx=idx)
    return assert_close(got.reshape(-1)[idx], ref, ref_abs, g.dtype, g.dtype, "sampled")


# ---------------------------------------------------------------------------
# worked examples printed on the tract-metal page
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_worked_examples(oracle_mod, dtype):
    b, m, n, k = 2, 2, 4, 3
    a = synth._store(np.arange(b * m * k, dtype=np.float32), dtype)
    bb = synth._store(np.arange(b * k * n, dtype=np.float32), dtype)
    da, db, dc = DevBuf(a.nbytes, host=a), DevBuf(bb.nbytes, host=bb), DevBuf(b * m * n * a.itemsize)
    st = gb.gbmm_gemm(dtype, b, m, n, k, 0, 0, da.ptr, 0, k, m * k, db.ptr, 0, n, k * n, dc.ptr, 0,
                      n, m * n)
    assert st == gb.GBMM_OK, gb.gbmm_last_error()
    got = to_f64(dc.read(NP_DT[dtype], b * m * n), dtype)
    expect = np.array([20, 23, 26, 29, 56, 68, 80, 92, 344, 365, 386, 407, 488, 518, 548, 578],
                      dtype=np.float64)
    if dtype == "bf16":
        # 8 significant bits: the printed values, rounded to bf16
        expect = to_f64(synth.f32_to_bf16_bits(expect.astype(np.float32)), "bf16")
    assert np.array_equal(got, expect)
    # all ones, b=10 m=n=32 k=16 -> 16 everywhere
    g = StridedGemm(dtype, 10, 32, 32, 16, False, False, dist="ints")
    g.a[:] = synth._store(np.ones(g.a.size, np.float32), dtype)
    g.b[:] = synth._store(np.ones(g.b.size, np.float32), dtype)
    da, db, dc = g.device()
    assert gb.gbmm_gemm(*g.args(da, db, dc)) == gb.GBMM_OK
    assert np.all(g.gather_c(dc) == 16.0)


# ---------------------------------------------------------------------------
# tensor-core GEMM (f16/bf16, every transpose combination)
# ---------------------------------------------------------------------------

TC_SHAPES = [
    (1, 128, 256, 64),        # exactly one tile, one k-block
    (2, 200, 300, 152),       # ragged m, n and k tails, several tiles
    (1, 257, 513, 1000),      # one past the tile edges
    (3, 384, 256, 4096),      # long k
    (1, 1000, 40, 72),        # narrow n
    (1, 16, 1000, 520),       # m = 16 (just above the skinny path)
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", TC_SHAPES, ids=[str(s) for s in TC_SHAPES])
def test_tc_gemm_parity(oracle_mod, dtype, shape):
    batch, m, n, k = shape
    g = StridedGemm(dtype, batch, m, n, k, False, True, std=1.0 / np.sqrt(k), seed=batch + m)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc")


def _up8(v):
    return (v + 7) // 8 * 8


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("shape", TC_SHAPES, ids=[str(s) for s in TC_SHAPES])
def test_tc_gemm_transposes(oracle_mod, dtype, ta, tb, shape):
    # operands read as stored: A [k, m] when ta (M-contiguous), B [k, n] when
    # not tb (N-contiguous); leading dims rounded up to 8 elements for TMA,
    # plus padding on one of them
    batch, m, n, k = shape
    lda = _up8(m if ta else k) + (8 if ta else 0)
    ldb = _up8(k if tb else n) + (0 if tb else 16)
    g = StridedGemm(dtype, batch, m, n, k, ta, tb, lda=lda, ldb=ldb, std=1.0 / np.sqrt(k),
                    seed=batch + m + 7 * ta + 3 * tb)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (True, True)])
def test_tc_gemm_transposes_exact_and_broadcast(oracle_mod, dtype, ta, tb):
    # small integers: every partial sum exact, so every layout must agree with
    # the oracle to the output rounding; and a broadcast operand (stride 0)
    g = StridedGemm(dtype, 1, 256, 512, 1024, ta, tb, dist="ints", seed=5)
    a, b, c = g.device()
    assert gb.gbmm_gemm(*g.args(a, b, c)) == gb.GBMM_OK
    assert gb.gbmm_test_last_kernel() == "gbmm_gemm_tc"
    got = g.gather_c(c)
    ref, _ = g.oracle(oracle_mod)
    rounded = to_f64(synth._store(ref.astype(np.float32).reshape(-1), dtype), dtype).reshape(ref.shape)
    assert np.array_equal(got, rounded)
    rows_a, cols_a = (1000, 136) if ta else (136, 1000)
    g = StridedGemm(dtype, 3, 136, 200, 1000, ta, tb, lda=_up8(cols_a), ldb=_up8(1000 if tb else 200),
                    sa=0 if ta else None, sb=None if ta else 0, seed=9)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tc_gemm_strides_offsets_broadcast(oracle_mod, dtype):
    # padded leading dims (multiples of 8 elements), batch strides with gaps,
    # 16-byte aligned byte offsets, and a broadcast A (stride 0)
    g = StridedGemm(dtype, 3, 130, 270, 200, False, True, lda=208, ldb=264, ldc=300,
                    sa=0, sb=270 * 264 + 64, sc=130 * 300 + 8, a_off=32, b_off=64, c_off=16)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc")
    # unaligned C (ldc odd) takes the scalar store path of the same kernel
    g = StridedGemm(dtype, 2, 129, 257, 64, False, True, ldc=259, c_off=2)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc")


# 160 tiles of 128 x 256: one full round on 152 SMs plus 8 tiles, which run as
# 128-column half units; n = 1948 leaves 28 columns for the second half of
# the last column block, n = 1892 none (that half unit computes nothing)
LAST_ROUND_CASES = [
    ("f16", False, True, 1948), ("bf16", False, True, 1892),
    ("f16", False, False, 1948), ("bf16", True, True, 1892), ("f16", True, False, 1948),
]


@pytest.mark.parametrize("dtype,ta,tb,n", LAST_ROUND_CASES, ids=[str(c) for c in LAST_ROUND_CASES])
def test_tc_gemm_last_round_half_units(oracle_mod, dtype, ta, tb, n):
    m, k = 2560, 256
    lda = _up8(m if ta else k)
    ldb = _up8(k if tb else n)
    g = StridedGemm(dtype, 1, m, n, k, ta, tb, lda=lda, ldb=ldb, std=1.0 / np.sqrt(k), seed=n + 3 * ta)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc")


# 256 x 256 tiles (k >= 512 and at least two rounds of them over the SMs):
# 4 x 10 x 9 = 360 tiles with ragged m, n and k; the last round (56 tiles on
# 152 SMs) runs as 128-row half units, and with m = 2404 the second half of
# the last row block holds no rows.  Checked on sampled outputs: the corners
# and edges of the sub-tiles, half units and ragged blocks, plus random ones.
# ldc 2148 (rows 8-byte aligned: scalar stores), 2152 (16-byte), 2176 (32-byte)
WIDE_CASES = [
    ("f16", False, True, 2523, 2176), ("bf16", False, True, 2404, 2148), ("f16", False, False, 2404, 2152),
    ("bf16", True, True, 2523, 2176), ("f16", True, False, 2523, 2148), ("bf16", True, False, 2404, 2176),
]


@pytest.mark.parametrize("dtype,ta,tb,m,ldc", WIDE_CASES, ids=[str(c) for c in WIDE_CASES])
def test_tc_gemm_wide_tiles_sampled(oracle_mod, dtype, ta, tb, m, ldc):
    batch, n, k = 4, 2148, 520
    lda = _up8(m if ta else k)
    ldb = _up8(k if tb else n)
    g = StridedGemm(dtype, batch, m, n, k, ta, tb, lda=lda, ldb=ldb, ldc=ldc, std=1.0 / np.sqrt(k),
                    seed=m + 5 * ta + tb)
    rows = sorted({0, 127, 128, 255, 256, 2303, 2304, 2431, 2432, m - 1} - {r for r in range(m, 4096)})
    cols = [0, 31, 255, 256, 2047, 2048, n - 1]
    rng = np.random.default_rng(m + ta + 2 * tb)
    idx = [bi * m * n + i * n + j for bi in range(batch) for i in rows for j in cols]
    idx += list(rng.integers(0, batch * m * n, 6000))
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc", idx=np.array(idx, dtype=np.int64))


@pytest.mark.parametrize("dtype,ta,tb,bcast", [("f16", False, True, "a"), ("bf16", True, False, "b")])
def test_tc_gemm_wide_tiles_broadcast_sampled(oracle_mod, dtype, ta, tb, bcast):
    """256 x 256 tiles (4 x 10 x 8 = 320 of them) with one operand shared by
    every batch (batch stride 0).  Sampled outputs of every batch."""
    batch, m, n, k = 4, 2560, 2048, 520
    lda = _up8(m if ta else k)
    ldb = _up8(k if tb else n)
    g = StridedGemm(dtype, batch, m, n, k, ta, tb, lda=lda, ldb=ldb, sa=0 if bcast == "a" else None,
                    sb=0 if bcast == "b" else None, std=1.0 / np.sqrt(k), seed=7 + ta)
    rng = np.random.default_rng(17)
    idx = [bi * m * n + i * n + j for bi in range(batch) for i in (0, 255, 256, m - 1) for j in (0, 255, 256, n - 1)]
    idx += list(rng.integers(0, batch * m * n, 4000))
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc", idx=np.array(idx, dtype=np.int64))


@pytest.mark.parametrize("dtype,ta,tb,k", [("f16", False, True, 512), ("bf16", True, False, 520)])
def test_tc_gemm_wide_tiles_every_output(oracle_mod, dtype, ta, tb, k):
    """The 256 x 256-tile kernel compared on EVERY output.  m = 4000, n = 5000:
    16 x 20 = 320 tiles with ragged last row and column tiles; on the 152 SMs
    of a GB300 that is two full rounds of tiles (k >= 512 and at least two
    rounds take the wide kernel) and a last round of 16 tiles, run as 128-row
    half units.  k = 512 is eight whole k-blocks; k = 520 ends on a ragged
    ninth one (the three-stage operand ring wraps three times)."""
    batch, m, n = 1, 4000, 5000
    lda = _up8(m if ta else k)
    ldb = _up8(k if tb else n)
    g = StridedGemm(dtype, batch, m, n, k, ta, tb, lda=lda, ldb=ldb, std=1.0 / np.sqrt(k), seed=k + ta)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("reading", ["b_m_k_n", "b_m_n_k"])
def test_tc_gemm_page_shape_25_1280_32000(oracle_mod, dtype, reading):
    """The tract-metal tests' (1, 25, 1280, 32000) matmul on the tensor cores
    (both readings of the tuple order), B stored [n, k]: every output."""
    b, m, x, y = 1, 25, 1280, 32000
    n, k = (y, x) if reading == "b_m_k_n" else (x, y)
    g = StridedGemm(dtype, b, m, n, k, False, True, std=1.0 / np.sqrt(k), seed=25 + k)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_tc")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tc_gemm_exact_small_integers(oracle_mod, dtype):
    # |v| <= 8 integers, k = 1024: every product and partial sum is an exact
    # integer in f32 and every |C| <= 65536; check exact agreement where the
    # output dtype represents the value exactly
    g = StridedGemm(dtype, 1, 256, 512, 1024, False, True, dist="ints")
    a, b, c = g.device()
    assert gb.gbmm_gemm(*g.args(a, b, c)) == gb.GBMM_OK
    got = g.gather_c(c)
    ref, _ = g.oracle(oracle_mod)
    rounded = to_f64(synth._store(ref.astype(np.float32).reshape(-1), dtype), dtype).reshape(ref.shape)
    assert np.array_equal(got, rounded)


# ---------------------------------------------------------------------------
# FFMA GEMM: f32, and the f16/bf16 layouts the tensor-core path does not take
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("ta,tb", [(False, False), (False, True), (True, False), (True, True)])
@pytest.mark.parametrize("size,kernel", [((2, 70, 90, 45), "gbmm_gemm_small"),
                                         ((2, 150, 170, 83), "gbmm_gemm_simt")])
def test_general_gemm_parity(oracle_mod, dtype, ta, tb, size, kernel):
    batch, m, n, k = size
    g = StridedGemm(dtype, batch, m, n, k, ta, tb, lda=(m if ta else k) + 3,
                    ldb=(k if tb else n) + 5, ldc=n + 5, a_off=synth.ITEMSIZE[dtype] * 3)
    # the odd offsets and leading dims rule out the TMA path for every dtype;
    # a few thousand outputs take the latency-bound kernel, more the tiled one
    run_case(oracle_mod, g, expect_kernel=kernel)


def test_f32_gemm_workload_c1(oracle_mod):
    """Single f32 GEMM 64x64x128, NN, U[-1,1], seed 0: every output."""
    w = synth.workload("c1_f32_gemm")
    g = StridedGemm("f32", 1, 64, 64, 128, False, False)
    g.a[:] = w.a.reshape(-1)
    g.b[:] = w.b.reshape(-1)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_small")


def test_f32_gemm_page_shapes(oracle_mod):
    # the pages' f32 matmul shapes, both readings of the tuple order
    for (bb, m, x, y), tb in [((1, 3, 5, 4), False), ((1, 2, 5, 10), True), ((1, 4, 4, 4), True),
                              ((1, 4, 4, 200), True), ((1, 25, 1280, 32000), True)]:
        for (n, k) in ((x, y), (y, x)):
            g = StridedGemm("f32", bb, m, n, k, False, tb, std=1.0, seed=m)
            run_case(oracle_mod, g)


# ---------------------------------------------------------------------------
# GEMV (m == 1 or n == 1) and the skinny/wide path
# ---------------------------------------------------------------------------

GEMV_CASES = [
    # (batch, m, n, k, ta, tb)
    (1, 1, 11, 300, False, True),     # row-dot over B, ragged k
    (1, 1, 700, 1031, False, False),  # column-dot over B
    (3, 1, 129, 64, True, True),      # strided vector (ta)
    (2, 333, 1, 520, False, False),   # row-dot over A, strided vector (B column)
    (2, 77, 1, 999, True, True),      # column-dot over A
    (1, 1, 1, 4097, False, True),     # a dot product
    (10, 1, 4, 4, False, False),      # the pages' mat-vec shapes
    (1, 4, 1, 4, False, False),
    (5, 1, 7, 15, False, True),
    (5, 1, 15, 7, False, True),
    (1, 1, 64, 65536, False, False),  # few outputs, long k: split-k over a cluster
]


@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("case", GEMV_CASES, ids=[str(c) for c in GEMV_CASES])
@pytest.mark.parametrize("entry", ["gemv", "gemm"])
def test_gemv_parity(oracle_mod, dtype, case, entry):
    batch, m, n, k, ta, tb = case
    g = StridedGemm(dtype, batch, m, n, k, ta, tb, std=1.0, seed=k)
    fn = gb.gbmm_gemv if entry == "gemv" else gb.gbmm_gemm
    ratio = run_case(oracle_mod, g, fn=fn)
    assert gb.gbmm_test_last_kernel() in ("gbmm_gemv_rowdot", "gbmm_gemv_coldot", "gbmm_gemv_stream")
    assert ratio <= 1.0


# the column-dot orientation with an aligned matrix: staged through shared
# memory by TMA (boxes of 512 bytes of outputs x 64 k rows)
COLDOT_STREAM_CASES = [
    # (batch, m, n, k, ta, tb)
    (1, 1, 704, 1031, False, False),    # x times B stored [k, n]: ragged output tile and k-block
    (3, 1, 520, 777, False, False),     # batched, batch strides, ragged
    (2, 776, 1, 999, True, True),       # n == 1 with A stored [k, m]
    (1, 1, 64, 65536, False, False),    # few outputs, long k: k split over a cluster
    (1, 1, 11008, 4096, False, False),  # the decode shape, every output
]


@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("case", COLDOT_STREAM_CASES, ids=[str(c) for c in COLDOT_STREAM_CASES])
def test_gemv_coldot_stream_parity(oracle_mod, dtype, case):
    batch, m, n, k, ta, tb = case
    g = StridedGemm(dtype, batch, m, n, k, ta, tb, std=1.0, seed=k + n)
    run_case(oracle_mod, g, fn=gb.gbmm_gemv, expect_kernel="gbmm_gemv_coldot")


def test_gemv_decode_workload_c2(oracle_mod):
    """Decode GEMV f16: x [1,4096] ~N(0,1), W [11008,4096] ~N(0,0.02) (tb): all outputs."""
    w = synth.workload("c2_f16_gemv")
    g = StridedGemm("f16", 1, 1, 11008, 4096, False, True)
    g.a[:] = w.a.reshape(-1)
    g.b[:] = w.b.reshape(-1)
    run_case(oracle_mod, g, fn=gb.gbmm_gemv, expect_kernel="gbmm_gemv_stream")


# (dtype, n, k, ldb, m, kernel): whole rows per 16 KB staging slot (one copy
# when contiguous, one per row when padded), several vectors; rows longer than
# a slot go to the load-in-registers kernel
STREAM_CASES = [
    ("f16", 1000, 4096, None, 1, "gbmm_gemv_stream"),     # two 8 KB rows per slot
    ("f32", 301, 4096, None, 1, "gbmm_gemv_stream"),      # one 16 KB row per slot
    ("bf16", 777, 1000, None, 1, "gbmm_gemv_stream"),     # eight 2000-byte rows per slot, ragged tail
    ("f32", 515, 1024, 1032, 1, "gbmm_gemv_stream"),      # padded rows (ldb > k): one copy per row
    ("f16", 129, 6000, 6008, 1, "gbmm_gemv_stream"),      # padded, one 12000-byte row per slot
    ("f32", 64, 16, None, 1, "gbmm_gemv_stream"),         # 64-byte rows, 256 per slot
    ("f16", 5, 8, None, 1, "gbmm_gemv_stream"),           # fewer rows than CTAs
    ("f32", 301, 5000, None, 1, "gbmm_gemv_rowdot"),      # 20000-byte rows
    ("f16", 129, 12000, None, 1, "gbmm_gemv_rowdot"),     # 24000-byte rows
    # several tokens (2..15, 16-bit, B stored [n, k]): the tensor-core skinny kernel
    ("bf16", 515, 1024, 1032, 3, "gbmm_gemv_tc"),         # padded weight rows
    ("f16", 129, 6000, 6008, 2, "gbmm_gemv_tc"),          # ragged k-block, padded rows
    ("f16", 5, 8, None, 7, "gbmm_gemv_tc"),               # k = 8: one partial k-block
]


@pytest.mark.parametrize("case", STREAM_CASES, ids=[str(c[:5]) for c in STREAM_CASES])
def test_gemv_stream_parity(oracle_mod, case):
    dtype, n, k, ldb, m, kernel = case
    g = StridedGemm(dtype, 1, m, n, k, False, True, ldb=ldb, seed=n)
    run_case(oracle_mod, g, fn=gb.gbmm_gemv if m == 1 else gb.gbmm_gemm, expect_kernel=kernel)


def test_gemv_stream_not_taken_for_batches(oracle_mod):
    # batched GEMV (a different vector per batch): the load-in-registers kernel
    g = StridedGemm("f16", 3, 1, 200, 512, False, True, seed=2)
    run_case(oracle_mod, g, fn=gb.gbmm_gemv, expect_kernel="gbmm_gemv_rowdot")


def _wide_shapes():
    out = []
    with open(os.path.join(GOLDEN, "gemv_wide_gate_shapes.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                dt, m, n, k = line.split()
                out.append((dt, int(m), int(n), int(k)))
    return out


@pytest.mark.parametrize("dtype,m,n,k", _wide_shapes())
def test_wide_skinny_ramp(oracle_mod, dtype, m, n, k):
    """x [m,k] against w [n,k] with the pages' ramp inputs (exact in f32)."""
    g = StridedGemm(dtype, 1, m, n, k, False, True)
    g.a[:] = synth.ramp((m * k,), 1, dtype)
    g.b[:] = synth.ramp((n * k,), 2, dtype)
    run_case(oracle_mod, g)
    if dtype != "f32":
        assert gb.gbmm_test_last_kernel() in ("gbmm_gemv_rowdot", "gbmm_gemv_stream", "gbmm_gemv_tc")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("m", list(range(2, 16)))
def test_wide_skinny_random(oracle_mod, dtype, m):
    # 16-byte multiples for every row stride: the tensor-core skinny kernel (ragged n
    # and k: the last weight tile and k-block are partly outside the operands)
    g = StridedGemm(dtype, 1, m, 256 + 3, 4096 + 8, False, True, lda=4096 + 16, ldc=300, seed=m)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemv_tc")
    # a row stride that is not a multiple of 16 bytes: the CUDA-core kernels
    g = StridedGemm(dtype, 1, m, 256 + 3, 4096 + 8, False, True, lda=4096 + 13, ldc=300, seed=m + 1)
    run_case(oracle_mod, g)
    assert gb.gbmm_test_last_kernel() in ("gbmm_gemv_stream", "gbmm_gemv_rowdot")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("m,n", [(2, 11008), (7, 11008), (15, 11008), (15, 1037)])
def test_skinny_tensor_core_decode_shape(oracle_mod, dtype, m, n):
    """y = x W^T for 2..15 tokens on the decode GEMV's weight shape (k 4096),
    and a ragged n; every output against the oracle."""
    k = 4096
    g = StridedGemm(dtype, 1, m, n, k, False, True, std=1.0 / np.sqrt(k), seed=m + n)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemv_tc")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_skinny_tensor_core_exact_small_integers(oracle_mod, dtype):
    """|v| <= 8 integers, k = 1024: every partial sum is exact in f32, so the
    output equals the oracle's value rounded once to the output dtype."""
    g = StridedGemm(dtype, 1, 11, 700, 1024, False, True, dist="ints", seed=3)
    a, b, c = g.device()
    assert gb.gbmm_gemm(*g.args(a, b, c)) == gb.GBMM_OK
    assert gb.gbmm_test_last_kernel() == "gbmm_gemv_tc"
    got = g.gather_c(c)
    ref, _ = g.oracle(oracle_mod)
    rounded = to_f64(synth._store(ref.astype(np.float32).reshape(-1), dtype), dtype).reshape(ref.shape)
    assert np.array_equal(got, rounded)


FFMA_WIDE_CASES = [
    # dtype, batch, m, n, k, ta, tb, lda, ldc: grids of >= 152 tiles of 128 x 128 take the wide FFMA tile
    ("f32", 4, 1030, 650, 200, False, False, None, None),   # ragged m and n tails, nn
    ("f32", 4, 1030, 650, 200, False, True, None, 656),     # nt, C rows padded (16-byte stores)
    ("f32", 4, 1030, 650, 200, True, False, None, 651),     # tn, C rows padded to an odd pitch (scalar stores)
    ("f32", 4, 1030, 650, 200, True, True, None, None),     # tt
    ("f16", 2, 1664, 1536, 72, False, True, 75, None),      # f16 rows TMA cannot read (odd lda)
    # interior-only grids with 16-byte-loadable f32 operands: the vector-load FFMA kernel
    ("f32", 2, 1280, 1024, 208, False, False, 212, None),  # nn, A rows padded to a multiple of 4
    ("f32", 2, 1280, 1024, 208, False, True, None, 1028),  # nt, C rows padded
    ("f32", 2, 1280, 1024, 208, True, False, 1284, None),  # tn, A stored [k, m] with padded rows
    ("f32", 2, 1280, 1024, 208, True, True, None, None),   # tt
]


@pytest.mark.parametrize("case", FFMA_WIDE_CASES, ids=lambda c: "{}_b{}_{}x{}x{}_ta{}_tb{}".format(*c[:7]))
def test_ffma_wide_tile_parity(oracle_mod, case):
    """The 128 x 128 FFMA tile (8 x 8 outputs per thread, double-buffered
    shared memory) for every transpose pair, ragged tails and padded rows;
    every output against the oracle."""
    dtype, batch, m, n, k, ta, tb, lda, ldc = case
    g = StridedGemm(dtype, batch, m, n, k, ta, tb, lda=lda, ldc=ldc, std=1.0 / np.sqrt(k), seed=m + n + k)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_simt")


@pytest.mark.parametrize("ta,tb,bcast", [(False, True, "a"), (True, False, "b"), (False, False, "a")])
def test_ffma_vector_tile_broadcast_and_offsets(oracle_mod, ta, tb, bcast):
    """The vector-load FFMA tile (f32 grid of interior tiles) with a broadcast
    operand (batch stride 0), padded leading dimensions and 16-byte aligned
    byte offsets; every output against the oracle."""
    batch, m, n, k = 3, 1024, 1024, 48
    lda = (m if ta else k) + 4
    ldb = (k if tb else n) + 8
    g = StridedGemm("f32", batch, m, n, k, ta, tb, lda=lda, ldb=ldb, ldc=n + 4,
                    sa=0 if bcast == "a" else None, sb=0 if bcast == "b" else None,
                    a_off=16, b_off=48, c_off=32, std=1.0 / np.sqrt(k), seed=5 + ta + 2 * tb)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemm_simt")


def test_gemm_and_gemv_replay_from_a_cuda_graph(oracle_mod):
    """A tensor-core GEMM, the m == 1 stream GEMV and the skinny tensor-core
    GEMV captured into one CUDA graph and replayed: every output of each
    against the oracle (stream order inside the graph is the library's only
    synchronisation)."""
    cases = [(StridedGemm("bf16", 2, 512, 640, 520, False, True, std=1.0 / np.sqrt(520), seed=3), "gbmm_gemm_tc"),
             (StridedGemm("f16", 1, 1, 2048, 1024, False, True, std=1.0 / 32, seed=4), "gbmm_gemv_stream"),
             (StridedGemm("f16", 1, 6, 1300, 1024, False, True, std=1.0 / 32, seed=5), "gbmm_gemv_tc")]
    bufs = [g.device() for g, _ in cases]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def launch_all():
        for (g, name), (a, b, c) in zip(cases, bufs):
            st = gb.gbmm_gemm(*g.args(a, b, c))
            assert st == gb.GBMM_OK, gb.gbmm_last_error()
            assert gb.gbmm_test_last_kernel() == name

    with torch.cuda.stream(s):
        launch_all()  # outside the capture: kernel attributes set, modules loaded
    torch.cuda.synchronize()
    for g, (a, b, c) in zip((g for g, _ in cases), bufs):
        c.t[GUARD:GUARD + c.nbytes].fill_(0x7F)  # garbage the graph must overwrite
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch_all()
    graph.replay()
    torch.cuda.synchronize()
    assert gb.gbmm_device_error()[0] == gb.GBMM_OK
    for (g, _), (a, b, c) in zip(cases, bufs):
        ref, ref_abs = g.oracle(oracle_mod)
        assert_close(g.gather_c(c), ref, ref_abs, g.dtype, g.dtype, "graph replay")


SKINNY_SPLIT_CASES = [
    # dtype, m, n, k, lda, ldc: what the case covers (cluster split chosen by the library)
    ("f16", 5, 300, 1000, None, None),    # ragged k (15 blocks + 40), 3 tiles, a 3-way split of 16 k-blocks
    ("bf16", 2, 129, 8, None, None),      # one partial k-block, no split, a one-row last tile
    ("f16", 15, 128, 4096, None, 136),    # one tile, 8-way split, C rows padded (gaps must stay untouched)
    ("bf16", 9, 2000, 520, 528, None),    # padded x rows, 9 k-blocks split 2 ways (4 and 5)
    ("f16", 3, 11008, 64, None, None),    # one whole k-block per tile, 86 tiles
]


@pytest.mark.parametrize("case", SKINNY_SPLIT_CASES, ids=lambda c: f"{c[0]}_m{c[1]}_n{c[2]}_k{c[3]}")
def test_skinny_tensor_core_splits_and_tails(oracle_mod, case):
    """The skinny tensor-core GEMV across its k splits (1 to 8 CTAs per tile
    adding partial sums through distributed shared memory) and its ragged
    edges; every output against the oracle."""
    dtype, m, n, k, lda, ldc = case
    g = StridedGemm(dtype, 1, m, n, k, False, True, lda=lda, ldc=ldc, std=1.0 / np.sqrt(k), seed=n + k)
    run_case(oracle_mod, g, expect_kernel="gbmm_gemv_tc")


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_k_zero_writes_zeros(oracle_mod, dtype):
    g = StridedGemm(dtype, 2, 5, 7, 0, False, False, ldc=9, sc=60)
    a, b, c = g.device()
    assert gb.gbmm_gemm(*g.args(a, b, c)) == gb.GBMM_OK
    assert gb.gbmm_test_last_kernel() == "gbmm_fill_zero"
    assert np.all(g.gather_c(c) == 0.0)
    assert g.c_gaps_untouched(c) and c.guards_intact()


def test_empty_problems_launch_nothing():
    g = StridedGemm("f16", 1, 0, 7, 9, False, True)
    a, b, c = g.device()
    gb.gbmm_test_reset_launch_count()
    assert gb.gbmm_gemm(*g.args(a, b, c)) == gb.GBMM_OK
    assert gb.gbmm_test_launch_count() == 0
    assert c.guards_intact()


def test_batched_gemm_workload_c3_sampled(oracle_mod):
    """Batched f16 GEMM 4 x 4096^3, B stored [b,N,K], ~N(0,1/64): 4096 sampled
    outputs (all corners, tile edges and random) against the oracle."""
    w = synth.workload("c3_f16_gemm")
    b, m, n, k = 4, 4096, 4096, 4096
    da, db = DevBuf(w.a.nbytes, host=w.a), DevBuf(w.b.nbytes, host=w.b)
    dc = DevBuf(b * m * n * 2)
    st = gb.gbmm_gemm("f16", b, m, n, k, 0, 1, da.ptr, 0, k, m * k, db.ptr, 0, k, n * k, dc.ptr, 0,
                      n, m * n)
    assert st == gb.GBMM_OK, gb.gbmm_last_error()
    assert gb.gbmm_test_last_kernel() == "gbmm_gemm_tc"
    torch.cuda.synchronize()
    assert gb.gbmm_device_error()[0] == gb.GBMM_OK
    assert dc.guards_intact()
    rng = np.random.default_rng(1)
    pts = [(bi, i, j) for bi in range(b) for i in (0, 127, 128, m - 1) for j in (0, 255, 256, n - 1)]
    idx = [bi * m * n + i * n + j for bi, i, j in pts]
    idx += list(rng.integers(0, b * m * n, 4096 - len(idx)))
    idx = np.array(idx, dtype=np.int64)
    ref, ref_abs = synth_oracle_gemm(oracle_mod, w, idx)
    got = to_f64(dc.read(np.float16, b * m * n)[idx], "f16")
    assert_close(got, ref, ref_abs, "f16", "f16", "c3 sampled")
    # the full output is finite and not trivially zero
    full = dc.read(np.float16, b * m * n)
    assert np.isfinite(full).all() and np.count_nonzero(full) > 0.99 * full.size


def synth_oracle_gemm(oracle_mod, w, idx):
    return oracle_mod.gemm(w.dtype, w.batch, w.m, w.n, w.k, w.ta, w.tb, w.a.reshape(-1), w.lda,
                           w.stride_a, w.b.reshape(-1), w.ldb, w.stride_b, idx=idx)
