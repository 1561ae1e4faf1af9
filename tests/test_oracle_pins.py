"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- values printed on the pages, closed forms, exact integer
arithmetic, library routines (numpy binary64 matmul / einsum), and brute
force over every id tensor of tiny routing problems.

Sources: tract-metal 0.23.6 ``mlx_gemm/mod.rs`` (tests::test_mlx_gemm,
gemv_wide_tests), mlx-native 0.13.0 ``dense_matmul_id.rs`` (dense_matmul_id,
DenseMatmulIdScratch, dense_matmul_id_capability), rlx-metal 0.2.14
``mps_blas.rs`` (encode_mps_sgemm_t transpose flags).
"""

import itertools
import os

import numpy as np
import pytest

from gemv_moe_expert_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np_value(arr, dtype):
    """binary64 values through numpy (the library decode, independent of the oracle)."""
    if dtype == "bf16":
        with np.errstate(invalid="ignore"):
            return (np.asarray(arr, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(arr).astype(np.float64)


def _op(arr, ld_rows, transposed):
    """Materialise op(X) for a dense [batch, rows, cols] buffer."""
    return np.swapaxes(arr, -1, -2) if transposed else arr


# --------------------------------------------------------------------------
# element decoders
# --------------------------------------------------------------------------

def test_decode_f16_every_pattern(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle_mod.decode(bits.view(np.float16), "f16")
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_decode_bf16_known_values(oracle_mod):
    # bf16 bit patterns of well-known values
    table = {0x3F80: 1.0, 0xBF80: -1.0, 0x4000: 2.0, 0x4049: 3.140625, 0x3E00: 0.125,
             0x0000: 0.0, 0x7F7F: 3.3895313892515355e38, 0x0080: 1.1754943508222875e-38,
             0x0001: 9.183549615799121e-41, 0xC2F7: -123.5}
    bits = np.array(list(table), dtype=np.uint16)
    got = oracle_mod.decode(bits, "bf16")
    assert list(got) == [table[int(b)] for b in bits]


def test_decode_bf16_every_pattern(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = _np_value(bits, "bf16")
    got = oracle_mod.decode(bits, "bf16")
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])


def test_synth_bf16_rounding_is_nearest_even():
    v = np.array([1.0, 1.00390625, 1.01171875, 1.0 + 2 ** -9, 1.0 + 3 * 2 ** -9, -2.5e-3],
                 dtype=np.float32)
    bits = synth.f32_to_bf16_bits(v)
    back = synth.bf16_bits_to_f32(bits).astype(np.float64)
    # ties go to the even neighbour; everything else to the nearest
    assert back[0] == 1.0
    assert back[1] == 1.0           # 1 + 2^-8 is a tie between 1 and 1+2^-7 -> even (1)
    assert back[2] == 1.015625      # 1 + 3*2^-8 ties -> 1 + 2^-6 (even)
    assert back[3] == 1.0
    assert back[4] == 1.0078125
    assert abs(back[5] - (-2.5e-3)) <= 2.5e-3 * 2 ** -8


# --------------------------------------------------------------------------
# dense GEMM / GEMV
# --------------------------------------------------------------------------

def _read_worked_examples():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "mlx_gemm_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            elif key == "dims":
                cur["dims"] = tuple(int(v) for v in vals)
            elif key == "fill":
                cur["fill"] = float(vals[0])
            elif key == "expected":
                cur["expected"] = [float(v) for v in vals]
    return cases


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_gemm_worked_examples_from_page(oracle_mod, dtype):
    for case in _read_worked_examples():
        b, m, n, k = case["dims"]
        if case["name"] == "ones":
            a = np.ones(b * m * k, np.float32)
            bb = np.ones(b * k * n, np.float32)
        else:
            a = np.arange(b * m * k, dtype=np.float32)
            bb = np.arange(b * k * n, dtype=np.float32)
        a = synth._store(a, dtype)
        bb = synth._store(bb, dtype)
        c, c_abs = oracle_mod.gemm(dtype, b, m, n, k, False, False, a, k, m * k, bb, n, k * n)
        if "fill" in case:
            assert np.all(c == case["fill"])
        else:
            assert list(c.reshape(-1)) == case["expected"]
            assert np.array_equal(c, c_abs)   # non-negative inputs


@pytest.mark.parametrize("dtype", synth.DTYPES)
@pytest.mark.parametrize("ta,tb", [(False, False), (False, True), (True, False), (True, True)])
def test_gemm_matches_numpy_matmul(oracle_mod, dtype, ta, tb):
    batch, m, n, k = 3, 7, 5, 11
    pad = 3
    lda = (m if ta else k) + pad
    ldb = (k if tb else n) + pad
    rows_a, rows_b = (k if ta else m), (n if tb else k)
    sa = rows_a * lda + 5
    sb = rows_b * ldb + 2
    rng = np.random.default_rng(7)
    a = synth._store(rng.standard_normal(batch * sa).astype(np.float32), dtype)
    b = synth._store(rng.standard_normal(batch * sb).astype(np.float32), dtype)
    c, c_abs = oracle_mod.gemm(dtype, batch, m, n, k, ta, tb, a, lda, sa, b, ldb, sb)
    av, bv = _np_value(a, dtype), _np_value(b, dtype)
    for i in range(batch):
        A = av[i * sa:i * sa + rows_a * lda].reshape(rows_a, lda)[:, :(m if ta else k)]
        B = bv[i * sb:i * sb + rows_b * ldb].reshape(rows_b, ldb)[:, :(k if tb else n)]
        Aop = A.T if ta else A
        Bop = B.T if tb else B
        np.testing.assert_allclose(c[i], Aop @ Bop, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(c_abs[i], np.abs(Aop) @ np.abs(Bop), rtol=1e-13, atol=1e-13)


def test_gemm_batch_broadcast_stride_zero(oracle_mod):
    batch, m, n, k = 4, 3, 6, 9
    rng = np.random.default_rng(3)
    a = rng.standard_normal(m * k).astype(np.float32)            # shared by every batch
    b = rng.standard_normal(batch * k * n).astype(np.float32)
    c, _ = oracle_mod.gemm("f32", batch, m, n, k, False, False, a, k, 0, b, n, k * n)
    A = a.astype(np.float64).reshape(m, k)
    for i in range(batch):
        np.testing.assert_allclose(c[i], A @ b[i * k * n:(i + 1) * k * n].astype(np.float64)
                                   .reshape(k, n), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("dtype", synth.DTYPES)
def test_gemm_identity_and_permutation(oracle_mod, dtype):
    m = k = 24
    n = 10
    rng = np.random.default_rng(11)
    b_vals = rng.integers(-100, 100, size=(k, n)).astype(np.float32)
    b = synth._store(b_vals.reshape(-1), dtype)
    eye = synth._store(np.eye(m, dtype=np.float32).reshape(-1), dtype)
    c, _ = oracle_mod.gemm(dtype, 1, m, n, k, False, False, eye, k, 0, b, n, 0)
    assert np.array_equal(c[0], b_vals.astype(np.float64))
    perm = rng.permutation(m)
    P = np.zeros((m, k), np.float32)
    P[np.arange(m), perm] = 1.0
    c, _ = oracle_mod.gemm(dtype, 1, m, n, k, False, False, synth._store(P.reshape(-1), dtype),
                           k, 0, b, n, 0)
    assert np.array_equal(c[0], b_vals[perm].astype(np.float64))
    # transposed A: P stored [k, m] with ta -> op(A) = P^T
    c, _ = oracle_mod.gemm(dtype, 1, m, n, k, True, False, synth._store(P.reshape(-1), dtype),
                           m, 0, b, n, 0)
    assert np.array_equal(c[0], (P.T @ b_vals).astype(np.float64))


def test_gemm_rank_one_closed_form(oracle_mod):
    m, n, k = 9, 13, 37
    u = np.arange(1, m + 1, dtype=np.float32) - 5
    v = np.arange(1, n + 1, dtype=np.float32) * 0.5 - 3
    a = np.repeat(u[:, None], k, axis=1).reshape(-1)        # A[i, x] = u_i
    b = np.repeat(v[None, :], k, axis=0).reshape(-1)        # B[x, j] = v_j
    c, c_abs = oracle_mod.gemm("f32", 1, m, n, k, False, False, a, k, 0, b, n, 0)
    for i in range(m):
        for j in range(n):
            assert c[0, i, j] == k * float(u[i]) * float(v[j])
            assert c_abs[0, i, j] == k * abs(float(u[i])) * abs(float(v[j]))


def test_gemm_triangular_number_closed_form(oracle_mod):
    # A = 1, B[x, j] = x  ->  C[i, j] = k (k - 1) / 2, with B stored [n, k] (tb)
    m, n, k = 4, 6, 1000
    a = np.ones(m * k, np.float32)
    b = np.tile(np.arange(k, dtype=np.float32), n)
    c, _ = oracle_mod.gemm("f32", 1, m, n, k, False, True, a, k, 0, b, k, 0)
    assert np.all(c == k * (k - 1) / 2)


def _read_wide_shapes():
    out = []
    with open(os.path.join(GOLDEN, "gemv_wide_gate_shapes.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                dt, m, n, k = line.split()
                out.append((dt, int(m), int(n), int(k)))
    return out


@pytest.mark.parametrize("dtype,m,n,k", _read_wide_shapes())
def test_gemv_wide_ramp_exact(oracle_mod, dtype, m, n, k):
    """Ramp inputs are multiples of 1/64, so 4096 * C is an integer: compare the
    oracle with exact integer arithmetic (brute force in Python ints)."""
    x = synth.ramp((m, k), 1, dtype)
    w = synth.ramp((n, k), 2, dtype)
    c, _ = oracle_mod.gemm(dtype, 1, m, n, k, False, True, x, k, 0, w, k, 0)
    xi = [int(((i * 7 + 13) % 29) - 14) for i in range(m * k)]
    wi = [int(((i * 7 + 26) % 29) - 14) for i in range(n * k)]
    for i in range(m):
        for j in range(n):
            exact = sum(xi[i * k + t] * wi[j * k + t] for t in range(k))
            assert c[0, i, j] * 4096.0 == exact


@pytest.mark.parametrize("shape", [(1, 4, 4, 1), (10, 1, 4, 4), (5, 1, 15, 7), (1, 3, 5, 4),
                                   (1, 2, 5, 10), (1, 4, 4, 200)])
@pytest.mark.parametrize("order", ["bmkn", "bmnk"])
@pytest.mark.parametrize("tb", [False, True])
def test_gemv_and_small_gemm_shapes_match_numpy(oracle_mod, shape, order, tb):
    # the pages' `run_mmm_test_case` tuples; their order (b,m,k,n or b,m,n,k) is
    # not on the page, so both readings are checked
    if order == "bmkn":
        batch, m, k, n = shape
    else:
        batch, m, n, k = shape
    g = synth.gemm_case("t", "f32", batch, m, n, k, False, tb, dist="ints")
    c, _ = oracle_mod.gemm("f32", batch, m, n, k, False, tb, g.a, g.lda, g.stride_a,
                           g.b, g.ldb, g.stride_b)
    A = g.a.astype(np.float64)
    B = g.b.astype(np.float64)
    ref = A @ (np.swapaxes(B, -1, -2) if tb else B)
    assert np.array_equal(c, ref)


def test_gemm_sampled_matches_full(oracle_mod):
    g = synth.gemm_case("t", "f16", 2, 17, 19, 33, True, True)
    full, full_abs = oracle_mod.gemm("f16", 2, 17, 19, 33, True, True, g.a, g.lda, g.stride_a,
                                     g.b, g.ldb, g.stride_b)
    idx = np.array([0, 5, 17 * 19 - 1, 17 * 19, 2 * 17 * 19 - 1, 100], dtype=np.int64)
    s, s_abs = oracle_mod.gemm("f16", 2, 17, 19, 33, True, True, g.a, g.lda, g.stride_a,
                               g.b, g.ldb, g.stride_b, idx=idx)
    assert np.array_equal(s, full.reshape(-1)[idx])
    assert np.array_equal(s_abs, full_abs.reshape(-1)[idx])


# --------------------------------------------------------------------------
# expert-ID matmul
# --------------------------------------------------------------------------

def _np_matmul_id(case):
    """numpy einsum formulation over the gathered expert matrices."""
    W = _np_value(case.w, case.wdtype)
    E, n, k = case.n_experts, case.n, case.k
    stride = case.expert_stride_elems
    mats = np.stack([W[e * stride:e * stride + n * k].reshape(n, k) for e in range(E)])
    ids = case.ids.astype(np.int64)
    valid = ids < E
    safe = np.where(valid, ids, 0)
    x = case.x.astype(np.float64)
    if case.input_layout == 0:
        xr = np.repeat(x[:, None, :], case.top_k, axis=1)
    else:
        xr = x.reshape(case.m, case.top_k, k)
    out = np.einsum("tsjx,tsx->tsj", mats[safe], xr)
    out_abs = np.einsum("tsjx,tsx->tsj", np.abs(mats[safe]), np.abs(xr))
    out[~valid] = 0.0
    out_abs[~valid] = 0.0
    return out, out_abs


@pytest.mark.parametrize("wdtype", synth.DTYPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_matmul_id_matches_numpy_einsum(oracle_mod, wdtype, layout):
    case = synth.matmul_id_case("t", wdtype, 5, 9, 21, 3, 6, input_layout=layout,
                                stride_pad_elems=8, seed=4)
    out, out_abs = oracle_mod.matmul_id(wdtype, case.m, case.n, case.k, case.top_k,
                                        case.n_experts, case.expert_stride_bytes, layout,
                                        case.w, case.x, case.ids)
    ref, ref_abs = _np_matmul_id(case)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out_abs, ref_abs, rtol=1e-12, atol=1e-12)


def test_matmul_id_single_expert_is_plain_gemm(oracle_mod):
    m, n, k, top_k = 6, 8, 40, 1
    case = synth.matmul_id_case("t", "f32", m, n, k, top_k, 1, seed=2)
    out, _ = oracle_mod.matmul_id("f32", m, n, k, top_k, 1, case.expert_stride_bytes, 0,
                                  case.w, case.x, case.ids)
    ref, _ = oracle_mod.gemm("f32", 1, m, n, k, False, True, case.x, k, 0, case.w, k, 0)
    assert np.array_equal(out[:, 0, :], ref[0])
    np.testing.assert_allclose(out[:, 0, :], case.x.astype(np.float64) @
                               case.w.reshape(n, k).astype(np.float64).T, rtol=1e-13, atol=1e-13)


def test_matmul_id_out_of_range_ids_give_zero_rows(oracle_mod):
    m, n, k, top_k, E = 3, 5, 12, 2, 4
    ids = np.array([[0, 4], [3, 1000], [0xFFFFFFFF, 2]], dtype=np.uint32)
    case = synth.matmul_id_case("t", "bf16", m, n, k, top_k, E, ids=ids, multiplicity=1)
    out, out_abs = oracle_mod.matmul_id("bf16", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                        case.w, case.x, ids)
    for t, s in [(0, 1), (1, 1), (2, 0)]:
        assert np.all(out[t, s] == 0.0) and np.all(out_abs[t, s] == 0.0)
    for t, s in [(0, 0), (1, 0), (2, 1)]:
        assert np.any(out[t, s] != 0.0)


def test_matmul_id_stride_padding_is_never_read(oracle_mod):
    m, n, k, top_k, E = 4, 6, 16, 2, 5
    case = synth.matmul_id_case("t", "f32", m, n, k, top_k, E, stride_pad_elems=7, seed=9)
    w = case.w.copy()
    stride = case.expert_stride_elems
    for e in range(E):
        w[e * stride + n * k:(e + 1) * stride] = np.nan
    out, _ = oracle_mod.matmul_id("f32", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                  w, case.x, case.ids)
    assert np.all(np.isfinite(out))
    ref, _ = _np_matmul_id(case)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_matmul_id_slotted_equals_shared_when_rows_replicate(oracle_mod):
    m, n, k, top_k, E = 5, 7, 19, 3, 6
    case = synth.matmul_id_case("t", "f16", m, n, k, top_k, E, seed=5)
    shared, _ = oracle_mod.matmul_id("f16", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                     case.w, case.x, case.ids)
    slotted_x = np.repeat(case.x, top_k, axis=0)
    slotted, _ = oracle_mod.matmul_id("f16", m, n, k, top_k, E, case.expert_stride_bytes, 1,
                                      case.w, slotted_x, case.ids)
    assert np.array_equal(shared, slotted)


def test_matmul_id_repeat_ids_give_identical_rows(oracle_mod):
    m, n, k, top_k, E = 2, 5, 9, 4, 3
    ids = np.array([[1, 1, 2, 1], [0, 0, 0, 0]], dtype=np.uint32)
    case = synth.matmul_id_case("t", "f32", m, n, k, top_k, E, ids=ids, multiplicity=1)
    out, _ = oracle_mod.matmul_id("f32", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                  case.w, case.x, ids)
    assert np.array_equal(out[0, 0], out[0, 1]) and np.array_equal(out[0, 0], out[0, 3])
    assert np.all(out[1] == out[1, 0])


def test_matmul_id_sampled_matches_full(oracle_mod):
    case = synth.matmul_id_case("t", "bf16", 6, 10, 24, 2, 5, seed=1)
    full, full_abs = oracle_mod.matmul_id("bf16", 6, 10, 24, 2, 5, case.expert_stride_bytes, 0,
                                          case.w, case.x, case.ids)
    idx = np.array([0, 9, 10, 57, 6 * 2 * 10 - 1], dtype=np.int64)
    s, s_abs = oracle_mod.matmul_id("bf16", 6, 10, 24, 2, 5, case.expert_stride_bytes, 0,
                                    case.w, case.x, case.ids, idx=idx)
    assert np.array_equal(s, full.reshape(-1)[idx])
    assert np.array_equal(s_abs, full_abs.reshape(-1)[idx])


# --------------------------------------------------------------------------
# routing map (map_distinct)
# --------------------------------------------------------------------------

def _brute_map(m, top_k, E, ids):
    """Independent definition: sort the (expert, row) pairs lexicographically."""
    pairs = sorted((int(e), r) for r, e in enumerate(ids.reshape(-1)) if int(e) < E)
    counts = [0] * E
    lists = [[] for _ in range(E)]
    for e, r in pairs:
        counts[e] += 1
        lists[e].append(r)
    return counts, lists


def test_map_distinct_brute_force_all_id_tensors(oracle_mod):
    checked = 0
    for E in (1, 2, 3, 4):
        for m in (1, 2, 3):
            for top_k in (1, 2):
                if top_k > E:
                    continue
                # each token row: an ordered pair of distinct valid ids, or with an
                # out-of-range value (E or 0xFFFFFFFF) in some slots
                values = list(range(E)) + [E, 0xFFFFFFFF]
                rows = [r for r in itertools.product(values, repeat=top_k)
                        if len({v for v in r if v < E}) == sum(1 for v in r if v < E)]
                for combo in itertools.product(rows, repeat=m):
                    ids = np.array(combo, dtype=np.uint32).reshape(m, top_k)
                    counts, rows_map = oracle_mod.map_distinct(m, top_k, E, ids)
                    bc, bl = _brute_map(m, top_k, E, ids)
                    assert list(counts) == bc
                    for e in range(E):
                        assert list(rows_map[e, :counts[e]]) == bl[e]
                    checked += 1
    assert checked > 10000


def test_map_distinct_invariants_on_zipf_workload(oracle_mod):
    m, top_k, E = 4096, 8, 128
    ids = synth.distinct_ids(m, top_k, E, 0, zipf_s=1.1)
    counts, rows = oracle_mod.map_distinct(m, top_k, E, ids)
    flat = ids.reshape(-1)
    assert counts.sum() == flat.size
    assert counts.max() <= m
    seen = np.zeros(flat.size, dtype=np.int64)
    for e in range(E):
        lst = rows[e, :counts[e]].astype(np.int64)
        assert np.all(np.diff(lst) > 0)
        assert np.all(flat[lst] == e)
        seen[lst] += 1
    assert np.all(seen == 1)


def test_zipf_workload_statistics_reproduce():
    """Seed-0 statistics of the GroupedPrefill workload's Zipf(1.1) ids."""
    ids = synth.distinct_ids(4096, 8, 128, 0, zipf_s=1.1)
    counts = np.bincount(ids.reshape(-1), minlength=128)
    top = sorted(counts.tolist(), reverse=True)
    assert counts[0] == 3647 and top[:3] == [3647, 2711, 2148]
    assert counts.min() == 38 and np.all(counts > 0) and counts.sum() == 32768
