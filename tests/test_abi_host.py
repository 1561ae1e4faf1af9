"""Host-only checks of the C ABI (no GPU): the library builds for sm_103a,
loads, exports every symbol include/gbmm.h declares, and every validation
rule fails closed before any launch.

Rules restated from mlx-native 0.13.0 ``dense_matmul_id.rs``
(``dense_matmul_id_capability``, ``validate_dense_matmul_id_call``,
``DenseMatmulIdScratch::new``, the grouped-pipeline failure test) and
tract-metal 0.23.6 ``mlx_gemm/mod.rs`` (``MlxGemm::dispatch_eval``,
``dispatch_metal_mlx_gemv``, ``dispatch_metal_mlx_gemm``).  The pointers
below are fake but aligned addresses: every call that reaches a launch
would need a GPU, so each case here must be rejected (or be an empty
problem) before touching CUDA.
"""

import os
import re
import subprocess

import pytest

from gemv_moe_expert_gb300 import binding as gb
from gemv_moe_expert_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gb.load()


@pytest.fixture(autouse=True)
def _no_kernel_may_launch():
    """Every kernel launch is blocked while a case here runs: on a machine
    with a GPU, a validation rule that regressed then shows up as
    GBMM_ERR_KERNEL_UNAVAILABLE instead of a kernel reading the fake
    addresses below."""
    gbuild.build()
    gb.load()
    gb.gbmm_test_inject_kernel_failure("*")
    yield
    gb.gbmm_test_inject_kernel_failure(None)


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "gbmm.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"GBMM_API\s+[\w\s\*]*?\b(gbmm_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_symbols() == sorted(gb.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", gb.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing but the API leaks out (the CUDA runtime is linked privately)
    assert all(s.startswith("gbmm_") for s in exported), sorted(exported)


def test_library_is_built_for_sm_103a(lib):
    out = subprocess.run(["cuobjdump", "--list-elf", gb.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_status_strings_and_version(lib):
    assert gb.gbmm_abi_version() == 1
    assert gb.gbmm_status_string(gb.GBMM_ERR_OVERLAP) == "GBMM_ERR_OVERLAP"
    assert gb.gbmm_status_string(99) == "GBMM_ERR_UNKNOWN"


# ---------------------------------------------------------------------------
# expert-ID capability
# ---------------------------------------------------------------------------

def _p2_fixture():
    vals = {}
    with open(os.path.join(GOLDEN, "matmul_id_capability_p2_test.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *rest = line.split()
                vals[key] = [int(v) for v in rest]
    return vals


def test_capability_extents_of_page_test_shape(lib):
    v = _p2_fixture()
    m, n, k, top_k, E, stride = v["params"]
    p = gb.make_params(m, n, k, top_k, E, stride, route=gb.ROUTE_GROUPED_PREFILL)
    st, cap = gb.gbmm_matmul_id_capability("f32", p)
    assert st == gb.GBMM_OK, gb.gbmm_last_error()
    assert cap.schema_version == gb.MATMUL_ID_SCHEMA_VERSION
    assert cap.required_weight_bytes == v["weights"][0]
    assert cap.required_input_bytes == v["input"][0]
    assert cap.required_ids_bytes == v["ids"][0]
    assert cap.required_output_bytes == v["output"][0]
    assert cap.has_scratch == 1
    assert cap.expert_counts_bytes == v["counts"][0]
    assert cap.routed_rows_bytes == v["routed_rows"][0]


@pytest.mark.parametrize("wdt,size", [("f32", 4), ("f16", 2), ("bf16", 2)])
@pytest.mark.parametrize("layout", [0, 1])
def test_capability_closed_forms(lib, wdt, size, layout):
    m, n, k, top_k, E = 37, 19, 130, 3, 11
    stride = n * k * size + 64
    p = gb.make_params(m, n, k, top_k, E, stride, input_layout=layout)
    st, cap = gb.gbmm_matmul_id_capability(wdt, p)
    assert st == gb.GBMM_OK
    assert cap.required_weight_bytes == (E - 1) * stride + n * k * size
    assert cap.required_input_bytes == (m if layout == 0 else m * top_k) * k * 4
    assert cap.required_ids_bytes == m * top_k * 4
    assert cap.required_output_bytes == m * top_k * n * 4
    assert cap.has_scratch == 0 and cap.expert_counts_bytes == 0 and cap.routed_rows_bytes == 0
    assert cap.route == gb.ROUTE_DIRECT and cap.weight_dtype == gb.DTYPE_CODES[wdt]


BAD_PARAMS = [
    # (description, overrides, expected status)
    ("zero m", dict(m=0), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("zero n", dict(n=0), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("zero k", dict(k=0), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("zero top_k", dict(top_k=0), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("zero experts", dict(n_experts=0), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("distinct top_k > experts", dict(top_k=9, n_experts=8), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("stride below one matrix", dict(expert_stride_bytes=8 * 16 * 2 - 2), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("stride not a multiple of the dtype", dict(expert_stride_bytes=8 * 16 * 2 + 1),
     gb.GBMM_ERR_INVALID_ARGUMENT),
    ("weight offset overflow", dict(n_experts=1 << 31, expert_stride_bytes=1 << 40, top_k=1),
     gb.GBMM_ERR_INVALID_ARGUMENT),
    ("routed rows above u32", dict(m=1 << 30, top_k=8, n_experts=8), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("grouped needs distinct", dict(route=1, multiplicity=1), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("grouped at most 1024 experts", dict(route=1, n_experts=1025), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("unknown layout", dict(input_layout=2), gb.GBMM_ERR_INVALID_ARGUMENT),
    ("unknown route", dict(route=5), gb.GBMM_ERR_INVALID_ARGUMENT),
]


@pytest.mark.parametrize("desc,over,expect", BAD_PARAMS, ids=[b[0] for b in BAD_PARAMS])
def test_capability_rejects(lib, desc, over, expect):
    base = dict(m=4, n=8, k=16, top_k=2, n_experts=8, expert_stride_bytes=8 * 16 * 2,
                input_layout=0, multiplicity=0, route=0)
    base.update(over)
    p = gb.make_params(base["m"], base["n"], base["k"], base["top_k"], base["n_experts"],
                       base["expert_stride_bytes"], base["input_layout"], base["multiplicity"],
                       base["route"])
    st, _ = gb.gbmm_matmul_id_capability("bf16", p)
    assert st == expect, (desc, gb.gbmm_last_error())
    assert gb.gbmm_last_error() != ""


def test_capability_accepts_grouped_boundary_and_repeat_direct(lib):
    p = gb.make_params(4, 8, 16, 2, 1024, 8 * 16 * 2, route=1)
    assert gb.gbmm_matmul_id_capability("bf16", p)[0] == gb.GBMM_OK
    p = gb.make_params(4, 8, 16, 9, 8, 8 * 16 * 2, multiplicity=1, route=0)
    assert gb.gbmm_matmul_id_capability("bf16", p)[0] == gb.GBMM_OK


def test_capability_activation_precision_field(lib):
    p = gb.make_params(4, 8, 16, 2, 8, 8 * 16 * 2, route=1, activation_precision=gb.ACT_BF16)
    assert gb.gbmm_matmul_id_capability("bf16", p)[0] == gb.GBMM_OK
    p = gb.make_params(4, 8, 16, 2, 8, 8 * 16 * 2, activation_precision=2)
    assert gb.gbmm_matmul_id_capability("bf16", p)[0] == gb.GBMM_ERR_INVALID_ARGUMENT
    p = gb.make_params(4, 8, 16, 2, 8, 8 * 16 * 2)
    p.reserved = 1
    assert gb.gbmm_matmul_id_capability("bf16", p)[0] == gb.GBMM_ERR_INVALID_ARGUMENT


def test_capability_rejects_unsupported_dtype(lib):
    p = gb.make_params(4, 8, 16, 2, 8, 8 * 16 * 2)
    st, _ = gb.gbmm_matmul_id_capability(7, p)
    assert st == gb.GBMM_ERR_UNSUPPORTED_DTYPE


def test_scratch_bytes(lib):
    assert gb.gbmm_matmul_id_scratch_bytes(128, 4096) == (gb.GBMM_OK, 512, 128 * 4096 * 4)
    assert gb.gbmm_matmul_id_scratch_bytes(0, 10)[0] == gb.GBMM_ERR_INVALID_ARGUMENT
    assert gb.gbmm_matmul_id_scratch_bytes(10, 0)[0] == gb.GBMM_ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------------------
# expert-ID call validation (fake, aligned, disjoint device addresses)
# ---------------------------------------------------------------------------

BASE = 1 << 40


class Call:
    """A grouped call on m=9 n=7 k=35 top_k=2 E=4 (f32 weights) with fake buffers."""

    def __init__(self, route=1):
        self.m, self.n, self.k, self.top_k, self.E = 9, 7, 35, 2, 4
        self.stride = self.n * self.k * 4
        self.p = gb.make_params(self.m, self.n, self.k, self.top_k, self.E, self.stride, route=route)
        st, cap = gb.gbmm_matmul_id_capability("f32", self.p)
        assert st == gb.GBMM_OK
        self.cap = cap
        self.w = BASE
        self.x = BASE + (1 << 20)
        self.ids = BASE + (2 << 20)
        self.out = BASE + (3 << 20)
        self.wb, self.xb = cap.required_weight_bytes, cap.required_input_bytes
        self.ib, self.ob = cap.required_ids_bytes, cap.required_output_bytes
        self.scratch = gb.make_scratch(BASE + (4 << 20), cap.expert_counts_bytes, BASE + (5 << 20),
                                       cap.routed_rows_bytes, self.E, self.m)

    def run(self, scratch="default", **kw):
        args = dict(w=self.w, wb=self.wb, x=self.x, xb=self.xb, ids=self.ids, ib=self.ib,
                    out=self.out, ob=self.ob)
        args.update(kw)
        s = self.scratch if scratch == "default" else scratch
        return gb.gbmm_matmul_id(self.p, "f32", args["w"], args["wb"], args["x"], args["xb"],
                                 args["ids"], args["ib"], args["out"], args["ob"], s, stream=0)


@pytest.mark.parametrize("kw,expect", [
    (dict(wb=3919), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(xb=1259), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(ib=71), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(ob=503), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(w=BASE + 2), gb.GBMM_ERR_INVALID_ARGUMENT),        # not f32-aligned
    (dict(ids=BASE + (2 << 20) + 1), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(out=BASE + 100), gb.GBMM_ERR_OVERLAP),             # output inside the weights
    (dict(out=BASE + (1 << 20) + 8), gb.GBMM_ERR_OVERLAP),   # output inside the input
    (dict(out=BASE + (2 << 20) - 500), gb.GBMM_ERR_OVERLAP),  # output runs into the ids
    (dict(x=0), gb.GBMM_ERR_INVALID_ARGUMENT),
])
def test_matmul_id_call_validation(lib, kw, expect):
    c = Call()
    gb.gbmm_test_reset_launch_count()
    st, _ = c.run(**kw)
    assert st == expect, gb.gbmm_last_error()
    assert gb.gbmm_test_launch_count() == 0


def test_grouped_scratch_rules(lib):
    c = Call()
    gb.gbmm_test_reset_launch_count()
    assert c.run(scratch=None)[0] == gb.GBMM_ERR_SCRATCH
    small = gb.make_scratch(BASE + (4 << 20), 16, BASE + (5 << 20), 144, 3, 9)   # 3 < E
    assert c.run(scratch=small)[0] == gb.GBMM_ERR_SCRATCH
    small = gb.make_scratch(BASE + (4 << 20), 16, BASE + (5 << 20), 144, 4, 8)   # 8 < m
    assert c.run(scratch=small)[0] == gb.GBMM_ERR_SCRATCH
    short = gb.make_scratch(BASE + (4 << 20), 12, BASE + (5 << 20), 144, 4, 9)
    assert c.run(scratch=short)[0] == gb.GBMM_ERR_SCRATCH
    short = gb.make_scratch(BASE + (4 << 20), 16, BASE + (5 << 20), 140, 4, 9)
    assert c.run(scratch=short)[0] == gb.GBMM_ERR_SCRATCH
    clash = gb.make_scratch(c.out, 16, BASE + (5 << 20), 144, 4, 9)             # counts on the output
    assert c.run(scratch=clash)[0] == gb.GBMM_ERR_OVERLAP
    assert gb.gbmm_test_launch_count() == 0


@pytest.mark.parametrize("victim", ["gbmm_matmul_id_grouped", "gbmm_matmul_id_map"])
def test_grouped_kernel_resolution_failure_launches_nothing(lib, victim):
    """A kernel of the grouped route that cannot be resolved fails the call with
    nothing enqueued, and names the kernel (the pages' grouped-pipeline
    failure test, restated for the C ABI)."""
    c = Call()
    gb.gbmm_test_reset_launch_count()
    gb.gbmm_test_inject_kernel_failure(victim)
    st, _ = c.run()
    assert st == gb.GBMM_ERR_KERNEL_UNAVAILABLE
    assert victim in gb.gbmm_last_error()
    assert gb.gbmm_test_launch_count() == 0
    gb.gbmm_test_inject_kernel_failure(None)


def test_direct_resolution_failure_launches_nothing(lib):
    c = Call(route=0)
    gb.gbmm_test_reset_launch_count()
    gb.gbmm_test_inject_kernel_failure("gbmm_matmul_id_direct")
    st, _ = c.run(scratch=None)
    assert st == gb.GBMM_ERR_KERNEL_UNAVAILABLE
    assert gb.gbmm_test_launch_count() == 0


# ---------------------------------------------------------------------------
# dense GEMM / GEMV validation
# ---------------------------------------------------------------------------

def _gemm(fn=gb.gbmm_gemm, dt="f16", batch=1, m=8, n=8, k=8, ta=0, tb=0, a=BASE, ao=0, lda=None,
          sa=64, b=BASE + (1 << 20), bo=0, ldb=None, sb=64, c=BASE + (2 << 20), co=0, ldc=None,
          sc=64):
    # leading dims follow the BLAS rule ld >= max(1, tight)
    lda = lda if lda is not None else max(1, m if ta else k)
    ldb = ldb if ldb is not None else max(1, k if tb else n)
    ldc = ldc if ldc is not None else max(1, n)
    return fn(dt, batch, m, n, k, ta, tb, a, ao, lda, sa, b, bo, ldb, sb, c, co, ldc, sc, stream=0)


@pytest.mark.parametrize("kw,expect", [
    (dict(dt=3), gb.GBMM_ERR_UNSUPPORTED_DTYPE),
    (dict(m=-1), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(k=-1), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(lda=7), gb.GBMM_ERR_INVALID_ARGUMENT),           # < k
    (dict(ta=1, lda=7), gb.GBMM_ERR_INVALID_ARGUMENT),     # < m
    (dict(ldb=7), gb.GBMM_ERR_INVALID_ARGUMENT),           # < n
    (dict(tb=1, ldb=7), gb.GBMM_ERR_INVALID_ARGUMENT),     # < k
    (dict(ldc=7), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(sa=-1), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(ao=-2), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(ao=1), gb.GBMM_ERR_INVALID_ARGUMENT),            # misaligned f16 base
    (dict(dt="f32", co=2), gb.GBMM_ERR_INVALID_ARGUMENT),
    (dict(batch=2, sc=63), gb.GBMM_ERR_INVALID_ARGUMENT),  # batches of C overlap
    (dict(c=BASE + 16), gb.GBMM_ERR_OVERLAP),              # C on top of A
    (dict(c=BASE + (1 << 20) - 64), gb.GBMM_ERR_OVERLAP),  # C runs into B
    (dict(a=0), gb.GBMM_ERR_INVALID_ARGUMENT),
])
def test_gemm_validation(lib, kw, expect):
    gb.gbmm_test_reset_launch_count()
    assert _gemm(**kw) == expect, gb.gbmm_last_error()
    assert gb.gbmm_test_launch_count() == 0


def test_gemv_requires_a_vector_operand(lib):
    assert _gemm(fn=gb.gbmm_gemv, m=2, n=2) == gb.GBMM_ERR_INVALID_ARGUMENT
    assert "m == 1 or n == 1" in gb.gbmm_last_error()


@pytest.mark.parametrize("kw", [dict(m=0), dict(n=0), dict(batch=0), dict(m=0, a=0, b=0)])
def test_empty_problems_launch_nothing(lib, kw):
    gb.gbmm_test_reset_launch_count()
    assert _gemm(**kw) == gb.GBMM_OK
    assert gb.gbmm_test_launch_count() == 0


def test_gemm_kernel_resolution_failure(lib):
    gb.gbmm_test_reset_launch_count()
    gb.gbmm_test_inject_kernel_failure("gbmm_fill_zero")
    assert _gemm(k=0) == gb.GBMM_ERR_KERNEL_UNAVAILABLE
    assert gb.gbmm_test_launch_count() == 0
