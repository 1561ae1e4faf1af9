"""GPU parity of gbmm_matmul_id (both routes) against the CPU oracle, called
through the C ABI.  Routing maps (expert_counts, and each expert's routed
rows) must be bit-exact; f32 outputs must meet the tolerance of the weight
dtype (1e-5 * sum|a||b| for f32 weights, 2e-3 * sum|a||b| for f16/bf16).

Semantics: mlx-native 0.13.0, src/ops/dense_matmul_id.rs.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemv_moe_expert_gb300 import binding as gb  # noqa: E402
from gemv_moe_expert_gb300 import synth  # noqa: E402
from tests.gpu_util import GUARD, DevBuf, assert_close  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemv_moe_expert_gb300 import build
    build.build()
    gb.load()
    torch.cuda.init()


class Run:
    """Uploads a MatmulIdCase, calls gbmm_matmul_id, reads results back."""

    def __init__(self, case: synth.MatmulIdCase, out_fill=0x7F, precision=0):
        self.case = case
        c = case
        self.params = gb.make_params(c.m, c.n, c.k, c.top_k, c.n_experts, c.expert_stride_bytes,
                                     c.input_layout, c.multiplicity, c.route, precision)
        st, cap = gb.gbmm_matmul_id_capability(c.wdtype, self.params)
        assert st == gb.GBMM_OK, gb.gbmm_last_error()
        self.cap = cap
        self.w = DevBuf(c.w.nbytes, host=c.w)
        self.x = DevBuf(c.x.nbytes, host=c.x)
        self.ids = DevBuf(c.ids.nbytes, host=c.ids)
        # garbage in the output: every row must be fully overwritten
        self.out = DevBuf(cap.required_output_bytes, fill=out_fill)
        self.scratch = None
        if c.route == gb.ROUTE_GROUPED_PREFILL:
            self.counts = DevBuf(cap.expert_counts_bytes, fill=0xEE)
            self.rows = DevBuf(cap.routed_rows_bytes, fill=0xEE)
            self.scratch = gb.make_scratch(self.counts.ptr, cap.expert_counts_bytes, self.rows.ptr,
                                           cap.routed_rows_bytes, c.n_experts, c.m)

    def call(self):
        c = self.case
        gb.gbmm_test_reset_launch_count()
        st, rec = gb.gbmm_matmul_id(self.params, c.wdtype, self.w.ptr, c.w.nbytes, self.x.ptr,
                                    c.x.nbytes, self.ids.ptr, c.ids.nbytes, self.out.ptr,
                                    self.cap.required_output_bytes, self.scratch)
        assert st == gb.GBMM_OK, gb.gbmm_last_error()
        torch.cuda.synchronize()
        assert gb.gbmm_device_error()[0] == gb.GBMM_OK
        expect_launches = 2 if c.route == gb.ROUTE_GROUPED_PREFILL else 1
        assert rec.launch_count == expect_launches and rec.route == c.route
        assert rec.weight_dtype == gb.DTYPE_CODES[c.wdtype]
        assert gb.gbmm_test_launch_count() == expect_launches
        for buf in (self.w, self.x, self.ids, self.out):
            assert buf.guards_intact()
        if self.scratch is not None:
            assert self.counts.guards_intact() and self.rows.guards_intact()
        return self

    def output(self):
        c = self.case
        return self.out.read(np.float32, c.m * c.top_k * c.n).astype(np.float64)

    def check(self, oracle_mod, idx=None):
        c = self.case
        got = self.output()
        ref, ref_abs = oracle_mod.matmul_id(c.wdtype, c.m, c.n, c.k, c.top_k, c.n_experts,
                                            c.expert_stride_bytes, c.input_layout, c.w, c.x,
                                            c.ids, idx=idx)
        if idx is not None:
            got = got[idx]
        ratio = assert_close(got, ref, ref_abs, c.wdtype, "f32", c.name)
        if self.scratch is not None:
            self.check_map(oracle_mod)
        return ratio

    def check_map(self, oracle_mod):
        c = self.case
        counts_ref, rows_ref = oracle_mod.map_distinct(c.m, c.top_k, c.n_experts, c.ids)
        counts = self.counts.read(np.uint32, c.n_experts)
        assert np.array_equal(counts, counts_ref)
        rows = self.rows.read(np.uint32, c.n_experts * c.m).reshape(c.n_experts, c.m)
        for e in range(c.n_experts):
            n_e = min(int(counts_ref[e]), c.m)
            assert np.array_equal(rows[e, :n_e], rows_ref[e, :n_e]), e


def test_direct_decode_workload_c4(oracle_mod):
    """m=4, E=64, top_k=8 distinct uniform ids, k=2048, n=1408, bf16 W: every output."""
    r = Run(synth.workload("c4_moe_direct")).call()
    r.check(oracle_mod)
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_direct_tc"


DIRECT_TC_CASES = [
    # m, top_k, E, n, k, layout: what the case covers
    (1, 2, 8, 1408, 2048, 0),    # 2 routed rows: k split over clusters of 8 CTAs
    (2, 8, 64, 1408, 2048, 1),   # 16 rows, Slotted: 176 units, clusters of 2
    (1, 4, 4, 300, 1000, 0),     # ragged n and k (15 k-blocks + 40), clusters of 4
    (40, 8, 16, 256, 512, 0),    # 320 rows over 16 experts: several 16-row passes per expert, no split
    (9, 1, 1024, 136, 64, 1),    # one k-block, 9 of 1024 experts
]


@pytest.mark.parametrize("wdtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", DIRECT_TC_CASES, ids=lambda c: "m{}_top{}_E{}_n{}_k{}_l{}".format(*c))
def test_direct_tensor_core_splits_and_passes(oracle_mod, case, wdtype):
    """The Direct route's tensor-core kernel across its k splits, its 16-row
    passes and ragged edges, with out-of-range ids mixed in; every output."""
    m, top_k, E, n, k, layout = case
    ids = synth.distinct_ids(m, top_k, E, seed=n + k, zipf_s=None)
    ids[0, top_k - 1] = E          # an out-of-range id: the row must be zero
    c = synth.matmul_id_case(f"dtc-{m}-{E}", wdtype, m, n, k, top_k, E, route=0, input_layout=layout,
                             ids=ids, seed=n + k)
    r = Run(c).call()
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_direct_tc"
    r.check(oracle_mod)
    assert np.all(r.output().reshape(m, top_k, n)[0, top_k - 1] == 0.0)


@pytest.mark.parametrize("split", [False, True])
def test_direct_tensor_core_f16_activation_range(oracle_mod, split):
    """f16 weights take f16 activations on the tensor cores, each routed row
    scaled by a power of two first: rows of magnitude 1e30, 1e-30 and 7e4
    (above f16's largest finite value), a zero row and a row whose elements
    span 2^24 still meet 2e-3 * sum|w||x|.  With two routed rows the k-blocks
    are split over a cluster (each CTA scales over its own k-range)."""
    m, top_k, E, n, k = (1, 2, 8, 1408, 2048) if split else (6, 2, 8, 264, 512)
    c = synth.matmul_id_case("f16range", "f16", m, n, k, top_k, E, route=0, input_layout=1, seed=21)
    rows = c.x.reshape(m * top_k, k)
    factors = [1e30, 1e-30, 7e4, 0.0, 1.0, 3.0e-3][: m * top_k]
    for r, f in enumerate(factors):
        rows[r] *= np.float32(f)
    rows[-1] *= np.exp2(np.linspace(-12, 12, k)).astype(np.float32)
    r = Run(c).call()
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_direct_tc"
    r.check(oracle_mod)


@pytest.mark.parametrize("wdtype", synth.DTYPES)
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("k", [256, 1024])
def test_direct_parity_row_sizes(oracle_mod, wdtype, layout, k):
    # 512 B to 4 KB weight rows, SharedPerToken with 128 routed rows (~11 per
    # expert) or Slotted with 16, ragged n, padded expert stride
    m = 16 if layout == 0 else 2
    case = synth.matmul_id_case(f"dr-{wdtype}-{layout}-{k}", wdtype, m, 300, k, 8, 12, route=0,
                                input_layout=layout, stride_pad_elems=8, seed=k + layout)
    Run(case).call().check(oracle_mod)


def test_direct_repeats_and_out_of_range_short_rows(oracle_mod):
    m, top_k, E = 12, 6, 5
    rng = np.random.default_rng(14)
    ids = rng.integers(0, E, size=(m, top_k)).astype(np.uint32)   # repeats within a token
    ids[1, 2] = E
    ids[11, 5] = 0xFFFFFFFF
    case = synth.matmul_id_case("dr-rep", "bf16", m, 136, 512, top_k, E, route=0, multiplicity=1, ids=ids)
    r = Run(case).call()
    r.check(oracle_mod)
    out = r.output().reshape(m, top_k, -1)
    assert np.all(out[1, 2] == 0.0) and np.all(out[11, 5] == 0.0)


@pytest.mark.parametrize("wdtype", synth.DTYPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_direct_parity_many_rows_per_expert(oracle_mod, wdtype, layout):
    # SharedPerToken: 128 routed rows over 12 experts, ~11 rows per expert
    # (several passes of 4 rows over a weight tile); Slotted: 24 rows.  Ragged
    # 32-row weight tiles (n = 300), padded expert stride.
    m = 16 if layout == 0 else 3
    case = synth.matmul_id_case(f"ds-{wdtype}-{layout}", wdtype, m, 300, 520, 8, 12, route=0,
                                input_layout=layout, stride_pad_elems=8, seed=21)
    Run(case).call().check(oracle_mod)


def test_direct_may_repeat_and_out_of_range(oracle_mod):
    m, top_k, E = 12, 6, 5
    rng = np.random.default_rng(4)
    ids = rng.integers(0, E, size=(m, top_k)).astype(np.uint32)   # repeats within a token
    ids[2, 3] = E
    ids[9, 0] = 0xFFFFFFFF
    case = synth.matmul_id_case("ds-rep", "bf16", m, 136, 256, top_k, E, route=0, multiplicity=1,
                                ids=ids)
    r = Run(case).call()
    r.check(oracle_mod)
    out = r.output().reshape(m, top_k, -1)
    assert np.all(out[2, 3] == 0.0) and np.all(out[9, 0] == 0.0)


def test_grouped_prefill_workload_c5_sampled(oracle_mod):
    """m=4096, E=128, top_k=8 Zipf(1.1) ids, k=4096, n=1536, bf16 W: the routing map
    bit-exact, and 8192 sampled outputs (first/last rows of every expert's list
    and random) against the oracle."""
    case = synth.workload("c5_moe_grouped")
    r = Run(case).call()
    c = case
    counts_ref, rows_ref = oracle_mod.map_distinct(c.m, c.top_k, c.n_experts, c.ids)
    r.check_map(oracle_mod)
    rng = np.random.default_rng(5)
    picks = []
    for e in range(c.n_experts):
        lst = rows_ref[e, :counts_ref[e]]
        for rr in (lst[0], lst[-1], lst[len(lst) // 2]):
            for j in (0, c.n - 1, int(rng.integers(0, c.n))):
                picks.append(int(rr) * c.n + j)
    total = c.m * c.top_k * c.n
    picks += list(rng.integers(0, total, 8192 - len(picks)))
    idx = np.array(picks, dtype=np.int64)
    got = r.output()
    ref, ref_abs = oracle_mod.matmul_id(c.wdtype, c.m, c.n, c.k, c.top_k, c.n_experts,
                                        c.expert_stride_bytes, c.input_layout, c.w, c.x, c.ids,
                                        idx=idx)
    assert_close(got[idx], ref, ref_abs, "bf16", "f32", "c5 sampled")
    assert np.isfinite(got).all()


@pytest.mark.parametrize("wdtype", synth.DTYPES)
@pytest.mark.parametrize("route", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
def test_matmul_id_parity_small(oracle_mod, wdtype, route, layout):
    # several tiles in every dimension, ragged tails, padded expert stride
    case = synth.matmul_id_case(f"{wdtype}-r{route}-l{layout}", wdtype, 150, 300, 520, 4, 12,
                                route=route, input_layout=layout, stride_pad_elems=8, seed=3)
    Run(case).call().check(oracle_mod)
    if route == 1:
        want = {"bf16": "gbmm_matmul_id_grouped_tc", "f16": "gbmm_matmul_id_grouped_tc",
                "f32": "gbmm_matmul_id_grouped_simt"}[wdtype]
        assert gb.gbmm_test_last_kernel() == want


def test_grouped_tc_odd_shapes(oracle_mod):
    # k not a multiple of 64, n not a multiple of 256 nor 4 (scalar epilogue stores),
    # several row blocks for the largest experts, one expert with no rows
    m, top_k, E = 700, 3, 7
    ids = synth.distinct_ids(m, top_k, E - 1, seed=4)  # expert E-1 never selected
    case = synth.matmul_id_case("odd", "bf16", m, 261, 200, top_k, E, route=1, ids=ids)
    Run(case).call().check(oracle_mod)
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"


def test_grouped_tc_tail_units(oracle_mod):
    """More 128 x 512 tiles than CTAs, not a multiple of them: the last tiles run
    as 256-column halves, and with n = 1100 the second half of every last
    column block lies past n and is skipped.  Every output and the map."""
    m, top_k, E = 2048, 4, 8
    case = synth.matmul_id_case("tail", "bf16", m, 1100, 264, top_k, E, route=1, seed=11)
    r = Run(case).call()
    r.check(oracle_mod)
    r.check_map(oracle_mod)
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"


def test_grouped_tc_deep_k_every_output(oracle_mod):
    """k = 4096 (64 k-blocks: the three-stage weight and activation rings wrap
    about 21 times per tile), 1664 tokens x top-2 over 4 experts (about 832
    routed rows each: 7 row blocks of 128), n = 1088 (two 512-column blocks
    and a 64-column one): 84 whole tiles.  Every output and the map."""
    m, top_k, E = 1664, 2, 4
    case = synth.matmul_id_case("deepk", "bf16", m, 1088, 4096, top_k, E, route=1, seed=21)
    r = Run(case).call()
    r.check(oracle_mod)
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"


# routed rows per expert: last row blocks of every size around the tail-unit
# limit (64 rows: such blocks run with the routed rows on the MMA's N side,
# hi rows 0.., lo rows 64..) and the N = 16 steps, plus experts of several
# blocks and one with none
TAIL_COUNTS = [1, 15, 16, 17, 31, 32, 33, 47, 48, 63, 64, 65, 96, 133, 192, 257, 0, 128 + 64]


@pytest.mark.parametrize("n,k,precision", [(1536, 264, 0), (2560, 200, 0), (1100, 104, 0), (1536, 264, 1)],
                         ids=["halves", "whole", "cut-past-n", "single-rounding"])
def test_grouped_tc_tail_units_every_size(oracle_mod, n, k, precision):
    """Last row blocks of 1..65 routed rows (top_k 1, one id per token, the
    tokens shuffled over the experts).  n = 1536: 22 row blocks x 3 column
    blocks = 66 tiles, at most half the CTAs, so every tile runs as two
    256-column halves; n = 2560: 110 whole tiles; n = 1100: the second half
    of each last column block lies past n.  Every output and the map; the
    single-rounding mode within its own bound."""
    counts = np.array(TAIL_COUNTS)
    m, top_k, E = int(counts.sum()), 1, len(counts)
    rng = np.random.default_rng(5)
    ids = rng.permutation(np.repeat(np.arange(E), counts)).astype(np.uint32).reshape(m, 1)
    case = synth.matmul_id_case("tails", "bf16", m, n, k, top_k, E, route=1, ids=ids, seed=k)
    r = Run(case, precision=precision).call()
    if precision == 0:
        r.check(oracle_mod)
    else:
        got = r.output()
        ref, ref_abs = oracle_mod.matmul_id("bf16", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                            case.w, case.x, case.ids)
        assert np.all(np.abs(got - ref.reshape(-1)) <= (2.0 ** -8 + 1e-5) * ref_abs.reshape(-1))
        r.check_map(oracle_mod)
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"


@pytest.mark.parametrize("k", [40, 104, 136, 200, 264, 328, 448])
def test_grouped_tc_k_block_orders(oracle_mod, k):
    """1 to 7 k-blocks of 64 (ragged or whole), the short-k end of the
    activation and weight rings.  9216 routed rows over 6 experts (about 12 row blocks each) x 3 column
    blocks of n = 1300 (the last one cut past n): about 216 tiles, more than
    CTAs, so the last round also runs as half units.  Every output."""
    m, top_k, E = 3072, 3, 6
    case = synth.matmul_id_case(f"korder-{k}", "bf16", m, 1300, k, top_k, E, route=1, seed=k)
    Run(case).call().check(oracle_mod)
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"


@pytest.mark.parametrize("route", [0, 1])
def test_out_of_range_ids_give_zero_rows(oracle_mod, route):
    m, top_k, E = 40, 4, 9
    ids = synth.distinct_ids(m, top_k, E, seed=8)
    ids[3, 1] = E
    ids[7, 0] = 0xFFFFFFFF
    ids[7, 3] = 1000
    ids[39, 2] = E + 1
    case = synth.matmul_id_case("oob", "bf16", m, 72, 136, top_k, E, route=route, ids=ids)
    r = Run(case).call()
    r.check(oracle_mod)
    out = r.output().reshape(m, top_k, -1)
    for t, s in [(3, 1), (7, 0), (7, 3), (39, 2)]:
        assert np.all(out[t, s] == 0.0)


def test_direct_may_repeat(oracle_mod):
    case = synth.matmul_id_case("repeat", "bf16", 6, 200, 264, 5, 3, route=0, multiplicity=1,
                                seed=2)
    Run(case).call().check(oracle_mod)


def test_direct_many_windows(oracle_mod):
    # 800 routed rows: several 256-row sharing windows, experts shared across tokens
    case = synth.matmul_id_case("windows", "f16", 100, 96, 512, 8, 16, route=0, seed=6)
    Run(case).call().check(oracle_mod)


def test_grouped_scratch_reuse_two_calls(oracle_mod):
    """Two grouped calls in a row on the same scratch with different ids: the
    second map overwrites the first in stream order."""
    case = synth.matmul_id_case("reuse", "bf16", 64, 128, 256, 4, 10, route=1, seed=1)
    r = Run(case).call()
    r.check(oracle_mod)
    ids2 = synth.distinct_ids(64, 4, 10, seed=99)
    r.case.ids = ids2
    r.ids.t[4096:4096 + ids2.nbytes].copy_(torch.from_numpy(ids2.view(np.uint8).reshape(-1).copy()))
    r.call().check(oracle_mod)


def test_grouped_all_rows_one_expert(oracle_mod):
    # every token selects expert 0 in slot 0: one expert's list holds all m rows
    m, top_k, E = 300, 2, 4
    ids = np.zeros((m, top_k), dtype=np.uint32)
    ids[:, 1] = 1 + (np.arange(m) % 3)
    case = synth.matmul_id_case("one-expert", "bf16", m, 160, 192, top_k, E, route=1, ids=ids)
    Run(case).call().check(oracle_mod)


def test_split_activations_meet_tolerance_where_single_rounding_cannot(oracle_mod):
    """Activations at a bf16 rounding tie (1 + 2^-8, all positive) against positive
    weights: a single bf16 rounding of x errs by ~3.9e-3 * sum|w||x|, above the
    2e-3 bound, while the default hi/lo split (x = hi + lo exactly) meets it.
    This is why the split is the default of the tensor-core grouped route."""
    m, n, k, top_k, E = 64, 256, 512, 2, 4
    case = synth.matmul_id_case("tie", "bf16", m, n, k, top_k, E, route=1, seed=2)
    case.x[:] = np.float32(1.0 + 2.0 ** -8)
    w = synth.bf16_bits_to_f32(case.w)
    case.w[:] = synth.f32_to_bf16_bits(np.abs(w))
    Run(case).call().check(oracle_mod)  # default: split, stated tolerance
    fast = Run(case, precision=gb.ACT_BF16).call()
    got = fast.output()
    ref, ref_abs = oracle_mod.matmul_id("bf16", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                        case.w, case.x, case.ids)
    err = np.abs(got - ref.reshape(-1)) / ref_abs.reshape(-1)
    assert err.max() > 2e-3          # a single rounding breaks the stated bound here
    assert err.max() <= 2.0 ** -8 + 1e-5


@pytest.mark.parametrize("layout", [0, 1])
def test_grouped_single_rounding_mode(oracle_mod, layout):
    """Opt-in single bf16 rounding of the activations: within its own bound
    (2^-8 + 1e-5) * sum|w||x| everywhere, and on zero-mean data within the
    stated 2e-3 bound too."""
    case = synth.matmul_id_case("fast", "bf16", 300, 520, 1000, 4, 12, route=1,
                                input_layout=layout, seed=7)
    r = Run(case, precision=gb.ACT_BF16).call()
    got = r.output()
    ref, ref_abs = oracle_mod.matmul_id("bf16", case.m, case.n, case.k, case.top_k, case.n_experts,
                                        case.expert_stride_bytes, layout, case.w, case.x, case.ids)
    ref, ref_abs = ref.reshape(-1), ref_abs.reshape(-1)
    assert np.all(np.abs(got - ref) <= (2.0 ** -8 + 1e-5) * ref_abs)
    assert_close(got, ref, ref_abs, "bf16", "f32", "single-rounding mode, zero-mean data")
    r.check_map(oracle_mod)


# ---------------------------------------------------------------------------
# degenerate and maximum cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("route", [0, 1])
def test_single_expert_is_a_plain_gemm(oracle_mod, route):
    """n_experts = 1, top_k = 1, every id 0: out[t, 0, :] = W_0 x_t, the dense
    GEMM x [m, k] times W_0 stored [n, k] -- checked against the oracle's
    expert-ID loop and against its separate dense GEMM loop."""
    m, n, k = 70, 300, 264
    ids = np.zeros((m, 1), dtype=np.uint32)
    case = synth.matmul_id_case("one", "bf16", m, n, k, 1, 1, route=route, ids=ids)
    r = Run(case).call()
    r.check(oracle_mod)
    w32 = synth.bf16_bits_to_f32(case.w)[: n * k]
    ref, ref_abs = oracle_mod.gemm("f32", 1, m, n, k, False, True, case.x.reshape(-1), k, m * k, w32, k, n * k)
    assert_close(r.output().reshape(m, n), ref.reshape(m, n), ref_abs.reshape(m, n), "bf16", "f32", "E=1 as GEMM")


@pytest.mark.parametrize("route", [0, 1])
def test_no_id_in_range(oracle_mod, route):
    """No id selects an expert (all equal to n_experts or above): every output
    row is zero and, on the grouped route, every expert count is zero."""
    m, top_k, E = 33, 3, 5
    ids = np.full((m, top_k), E, dtype=np.uint32)
    ids[::2, 1] = 0xFFFFFFFF
    ids[1::3, 2] = E + 7
    case = synth.matmul_id_case("none", "bf16", m, 136, 64, top_k, E, route=route, ids=ids)
    r = Run(case).call()
    r.check(oracle_mod)
    assert np.all(r.output() == 0.0)
    if route == 1:
        assert np.all(r.counts.read(np.uint32, E) == 0)


@pytest.mark.parametrize("wdtype", ["f32", "f16"])
def test_grouped_ffma_row_block_sizes(oracle_mod, wdtype):
    """The FFMA grouped kernel's row blocks of 128 routed rows, and its
    half-block path for blocks of at most 64: expert lists of 64, 65, 1, 129
    and 0 rows (top-1 routing, so each token's id is its expert), ragged n and
    k; every output and the map."""
    sizes = [64, 65, 1, 129, 0]
    ids = np.concatenate([np.full(c, e, dtype=np.uint32) for e, c in enumerate(sizes)])
    ids = np.random.default_rng(11).permutation(ids).reshape(-1, 1)
    m, E = ids.shape[0], len(sizes)
    case = synth.matmul_id_case("ffma_blocks", wdtype, m, 200, 52, 1, E, route=1, ids=ids)
    r = Run(case).call()
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_simt"
    r.check(oracle_mod)
    r.check_map(oracle_mod)


@pytest.mark.parametrize("wdtype", ["f32"])
@pytest.mark.parametrize("layout", [0, 1])
def test_grouped_ffma_small_blocks_odd_column_tiles(oracle_mod, wdtype, layout):
    """The FFMA grouped kernel's 64 x 256 tile for row blocks of at most 64
    routed rows with an odd number of 128-column tiles (n = 300: the CTAs of
    column tiles 0 and 2 compute 256 columns each, the last one ragged) next to
    128 x 128 tiles of larger blocks; ragged k; every output and the map."""
    sizes = [40, 64, 65, 130, 1, 0, 200]
    ids = np.concatenate([np.full(c_, e, dtype=np.uint32) for e, c_ in enumerate(sizes)])
    ids = np.random.default_rng(7).permutation(ids).reshape(-1, 1)
    m, E = ids.shape[0], len(sizes)
    c = synth.matmul_id_case(f"ffma-small-{layout}", wdtype, m, 300, 70, 1, E, route=1, input_layout=layout,
                             ids=ids, seed=17)
    r = Run(c).call()
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_simt"
    r.check(oracle_mod)
    r.check_map(oracle_mod)


@pytest.mark.parametrize("precision", [0, 1])
def test_grouped_f16_tensor_core_row_scales(oracle_mod, precision):
    """GroupedPrefill with f16 weights on the grouped tensor-core kernel: each
    routed row of a unit is scaled by a power of two from its largest magnitude
    over the whole k range before the f16 split.  1200 Slotted routed rows over
    6 experts (row blocks of 128 and a last block per expert, ragged n and k)
    with rows of magnitude 1e30, 1e-30, 7e4 (above f16's largest finite
    value), zero rows and rows spanning 2^24 mixed in; every output and the
    map.  precision 1 is the opt-in single rounding, which for f16 (11
    significant bits) still meets 2e-3 * sum|w||x|."""
    m, top_k, E, n, k = 300, 4, 6, 264, 1000
    c = synth.matmul_id_case("f16grouped", "f16", m, n, k, top_k, E, route=1, input_layout=1, seed=23)
    rows = c.x.reshape(m * top_k, k)
    rows[::7] *= np.float32(1e30)
    rows[3::11] *= np.float32(1e-30)
    rows[5::13] *= np.float32(7e4)
    rows[9::17] = 0.0
    rows[2::19] *= np.exp2(np.linspace(-12, 12, k)).astype(np.float32)
    r = Run(c, precision=precision).call()
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"
    r.check(oracle_mod)
    r.check_map(oracle_mod)


@pytest.mark.parametrize("wdtype", ["bf16", "f16"])
def test_grouped_tc_expert_groups_with_gaps(oracle_mod, wdtype):
    """21 experts (not a multiple of the tile prefix's 8-expert step) with
    lists of 0 to 500 routed rows, empty experts inside and at the ends of the
    8-expert groups: the tile order walks each group's experts from their
    counts.  Top-1 routing; every output and the map."""
    sizes = [0, 300, 0, 129, 64, 65, 0, 1, 200, 0, 128, 256, 0, 0, 77, 500, 3, 0, 130, 1, 0]
    ids = np.concatenate([np.full(c_, e, dtype=np.uint32) for e, c_ in enumerate(sizes)])
    ids = np.random.default_rng(21).permutation(ids).reshape(-1, 1)
    m, E = ids.shape[0], len(sizes)
    c = synth.matmul_id_case(f"groups-{wdtype}", wdtype, m, 600, 136, 1, E, route=1, ids=ids, seed=21)
    r = Run(c).call()
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"
    r.check(oracle_mod)
    r.check_map(oracle_mod)


def test_grouped_f16_several_units_per_cta(oracle_mod):
    """f16 weights with more work units than SMs (4096 routed rows over 8
    experts x 8 output blocks of 512, the last round cut into 256-column
    halves), so every CTA runs two or three units: the first unit's row scales
    come from the producer warps, the later ones from the epilogue warps
    through both shared-memory buffers.  Rows of mixed magnitude; every
    output."""
    m, top_k, E, n, k = 1024, 4, 8, 4000, 136
    c = synth.matmul_id_case("f16units", "f16", m, n, k, top_k, E, route=1, seed=31)
    rows = c.x.reshape(m, k)
    rows[::3] *= np.float32(5e6)
    rows[1::5] *= np.float32(3e-7)
    r = Run(c).call()
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"
    r.check(oracle_mod)


@pytest.mark.parametrize("count", [1, 17, 64, 65, 128, 200])
def test_grouped_f16_tail_and_full_blocks(oracle_mod, count):
    """f16 weights: an expert list of `count` routed rows (tail units for at
    most 64 rows in the last block, full blocks above) next to a second
    expert of 100 rows, rows of mixed magnitude; every output."""
    sizes = [count, 100]
    ids = np.concatenate([np.full(c_, e, dtype=np.uint32) for e, c_ in enumerate(sizes)])
    ids = np.random.default_rng(count).permutation(ids).reshape(-1, 1)
    m, E = ids.shape[0], len(sizes)
    c = synth.matmul_id_case(f"f16tail{count}", "f16", m, 600, 264, 1, E, route=1, ids=ids, seed=count)
    rows = c.x.reshape(m, 264)
    rows[::5] *= np.float32(3e5)
    rows[1::6] *= np.float32(2e-9)
    r = Run(c).call()
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"
    r.check(oracle_mod)


@pytest.mark.parametrize("wdtype", ["bf16", "f16"])
def test_grouped_call_replays_from_a_cuda_graph(oracle_mod, wdtype):
    """GroupedPrefill captured into a CUDA graph (its map launch, then the
    grouped tensor-core kernel launched with programmatic stream serialisation
    behind it) and replayed twice, with new activations and new expert ids
    copied into the same buffers before the second replay: both replays match
    the oracle, map included."""
    c = synth.matmul_id_case(f"graph-{wdtype}", wdtype, 300, 520, 264, 4, 12, route=1, seed=41)
    r = Run(c)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def launch():
        st, _ = gb.gbmm_matmul_id(r.params, c.wdtype, r.w.ptr, c.w.nbytes, r.x.ptr, c.x.nbytes, r.ids.ptr,
                                  c.ids.nbytes, r.out.ptr, r.cap.required_output_bytes, r.scratch)
        assert st == gb.GBMM_OK, gb.gbmm_last_error()

    with torch.cuda.stream(s):
        launch()  # outside the capture: kernel attributes set, modules loaded
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch()
    graph.replay()
    torch.cuda.synchronize()
    assert gb.gbmm_device_error()[0] == gb.GBMM_OK
    r.check(oracle_mod)
    # new inputs in the same buffers, second replay
    c2 = synth.matmul_id_case(f"graph2-{wdtype}", wdtype, 300, 520, 264, 4, 12, route=1, seed=42)
    c2.w = c.w  # same weights, new activations and ids
    for buf, host in ((r.x, c2.x), (r.ids, c2.ids)):
        raw = np.ascontiguousarray(host).reshape(-1).view(np.uint8)
        buf.t[GUARD:GUARD + raw.size].copy_(torch.from_numpy(raw.copy()))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert gb.gbmm_device_error()[0] == gb.GBMM_OK
    r.case = c2
    r.check(oracle_mod)


def test_grouped_max_experts(oracle_mod):
    """n_experts = 1024, the grouped route's limit: 1200 routed rows over 1024
    experts (most lists hold 0 to 3 rows).  Every output and the map."""
    m, top_k, E = 300, 4, 1024
    case = synth.matmul_id_case("e1024", "bf16", m, 264, 136, top_k, E, route=1, seed=5)
    Run(case).call().check(oracle_mod)
    assert gb.gbmm_test_last_kernel() == "gbmm_matmul_id_grouped_tc"


@pytest.mark.parametrize("route", [0, 1])
def test_single_token_and_every_expert(oracle_mod, route):
    """One token (m = 1), and top_k = n_experts (every token picks every
    expert, in a per-token permuted order)."""
    Run(synth.matmul_id_case("m1", "bf16", 1, 300, 200, 8, 16, route=route, seed=4)).call().check(oracle_mod)
    Run(synth.matmul_id_case("all", "bf16", 40, 136, 264, 6, 6, route=route, seed=6)).call().check(oracle_mod)
