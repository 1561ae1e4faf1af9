"""gbmm_matmul_id_static_scratch: the grouped expert-ID matmul for callers
that cannot allocate device memory (their host runtime hands them only the
operands and outputs, or they may not call cudaMalloc while serving).

Through the C ABI, on two calls in a row with different routings, the entry
point must
  * match the CPU oracle within the parity tolerance of bf16 weights
    (2e-3 * sum|a||b| per output element),
  * return exactly the bits gbmm_matmul_id returns for the same inputs with
    caller-owned scratch (same kernels, same routing), and
  * leave in its fixed array the routing map of that call: expert counts and
    each expert's routed rows, bit-exact against the oracle's map.
Sizes beyond the fixed scratch and other routes are refused with nothing
launched.  This file is collected last and also runs on its own in a fresh
process.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemv_moe_expert_gb300 import binding as gb  # noqa: E402
from gemv_moe_expert_gb300 import synth  # noqa: E402
from tests.gpu_util import assert_close  # noqa: E402

pytestmark = pytest.mark.gpu

# the array's layout: GBMM_GROUPED_MAX_EXPERTS u32 counts, then the routed-row lists
COUNTS_CAPACITY = 1024


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemv_moe_expert_gb300 import build
    build.build()
    gb.load()
    torch.cuda.init()


def _up(arr):
    return torch.from_numpy(np.ascontiguousarray(arr).reshape(-1).view(np.uint8).copy()).cuda()


def test_static_scratch_matches_oracle_and_caller_scratch_on_two_calls(oracle_mod):
    m, n, k, top_k, E = 300, 264, 512, 4, 16
    case = synth.matmul_id_case("noalloc", "bf16", m, n, k, top_k, E, route=1, seed=11)
    p = gb.make_params(m, n, k, top_k, E, case.expert_stride_bytes, route=gb.ROUTE_GROUPED_PREFILL)
    st, cap = gb.gbmm_matmul_id_capability("bf16", p)
    assert st == gb.GBMM_OK
    w, x = _up(case.w), _up(case.x)
    counts = torch.empty(cap.expert_counts_bytes, dtype=torch.uint8, device="cuda")
    rows = torch.empty(cap.routed_rows_bytes, dtype=torch.uint8, device="cuda")
    scratch = gb.make_scratch(counts, cap.expert_counts_bytes, rows, cap.routed_rows_bytes, E, m)
    out_ref = torch.empty(cap.required_output_bytes, dtype=torch.uint8, device="cuda")
    out_new = torch.empty(cap.required_output_bytes, dtype=torch.uint8, device="cuda")
    map_copy = torch.empty(4 * COUNTS_CAPACITY + cap.routed_rows_bytes, dtype=torch.uint8, device="cuda")

    for call, seed in enumerate((11, 12)):
        ids_np = synth.distinct_ids(m, top_k, E, seed=seed)
        ids = _up(ids_np)
        out_new.fill_(0xAB)
        out_ref.fill_(0xCD)
        st, rec = gb.gbmm_matmul_id(p, "bf16", w, case.w.nbytes, x, case.x.nbytes, ids,
                                    ids_np.nbytes, out_ref, cap.required_output_bytes, scratch)
        assert st == gb.GBMM_OK, gb.gbmm_last_error()
        gb.gbmm_test_reset_launch_count()
        st, rec = gb.gbmm_matmul_id_static_scratch(p, "bf16", w, case.w.nbytes, x, case.x.nbytes,
                                                   ids, ids_np.nbytes, out_new,
                                                   cap.required_output_bytes)
        assert st == gb.GBMM_OK, gb.gbmm_last_error()
        assert rec.launch_count == 2 and rec.route == gb.ROUTE_GROUPED_PREFILL
        assert gb.gbmm_test_launch_count() == 2
        assert gb.gbmm_test_static_scratch_copy(map_copy, map_copy.numel()) == gb.GBMM_OK
        torch.cuda.synchronize()
        assert gb.gbmm_device_error()[0] == gb.GBMM_OK

        got = out_new.cpu().numpy().view(np.float32)
        want = out_ref.cpu().numpy().view(np.float32)
        # same kernels, same routing: the same bits as the caller-scratch call
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), f"call {call}"
        ref, ref_abs = oracle_mod.matmul_id("bf16", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                            case.w, case.x, ids_np)
        assert_close(got.astype(np.float64), ref.reshape(-1), ref_abs.reshape(-1), "bf16", "f32",
                     f"static scratch, call {call}")

        # the routing map this call left in the fixed array
        counts_ref, rows_ref = oracle_mod.map_distinct(m, top_k, E, ids_np)
        raw = map_copy.cpu().numpy().view(np.uint32)
        assert np.array_equal(raw[:E], counts_ref), f"call {call}"
        lists = raw[COUNTS_CAPACITY:COUNTS_CAPACITY + E * m].reshape(E, m)
        for e in range(E):
            c = int(counts_ref[e])
            assert np.array_equal(lists[e, :c], rows_ref[e, :c]), f"call {call}, expert {e}"


def test_static_scratch_refuses_what_it_cannot_hold():
    # Real buffers of the sizes each call asks for, and every kernel launch
    # blocked meanwhile: a regression in the refusals then fails the test
    # (GBMM_ERR_KERNEL_UNAVAILABLE) without any kernel touching memory.
    def buffers(m, n, k, top_k, E):
        w = torch.empty(E * n * k * 2, dtype=torch.uint8, device="cuda")
        x = torch.empty(m * k * 4, dtype=torch.uint8, device="cuda")
        ids = torch.zeros(m * top_k * 4, dtype=torch.uint8, device="cuda")
        out = torch.empty(m * top_k * n * 4, dtype=torch.uint8, device="cuda")
        return w, x, ids, out

    gb.gbmm_test_inject_kernel_failure("*")
    try:
        gb.gbmm_test_reset_launch_count()
        # n_experts * m * 4 bytes beyond the fixed array
        m, n, k, top_k, E = gb.STATIC_SCRATCH_ROUTED_ROWS_BYTES // (4 * 8) + 1, 64, 64, 2, 8
        w, x, ids, out = buffers(m, n, k, top_k, E)
        p = gb.make_params(m, n, k, top_k, E, n * k * 2, route=gb.ROUTE_GROUPED_PREFILL)
        st, _ = gb.gbmm_matmul_id_static_scratch(p, "bf16", w, w.numel(), x, x.numel(), ids, ids.numel(),
                                                 out, out.numel())
        assert st == gb.GBMM_ERR_SCRATCH
        assert "static scratch holds" in gb.gbmm_last_error()
        # the Direct route needs no scratch: use gbmm_matmul_id
        m = 4
        w, x, ids, out = buffers(m, n, k, top_k, E)
        p = gb.make_params(m, n, k, top_k, E, n * k * 2, route=gb.ROUTE_DIRECT)
        st, _ = gb.gbmm_matmul_id_static_scratch(p, "bf16", w, w.numel(), x, x.numel(), ids, ids.numel(),
                                                 out, out.numel())
        assert st == gb.GBMM_ERR_INVALID_ARGUMENT
        assert gb.gbmm_test_launch_count() == 0
    finally:
        gb.gbmm_test_inject_kernel_failure(None)
    torch.cuda.synchronize()


def test_static_scratch_call_replays_from_a_cuda_graph(oracle_mod):
    """The use the entry point exists for: after one call on the device (which
    loads the array), the call is captured into a CUDA graph and replayed with
    new ids copied into the same buffer; each replay matches the oracle."""
    m, n, k, top_k, E = 200, 264, 256, 4, 12
    case = synth.matmul_id_case("noalloc-graph", "bf16", m, n, k, top_k, E, route=1, seed=31)
    p = gb.make_params(m, n, k, top_k, E, case.expert_stride_bytes, route=gb.ROUTE_GROUPED_PREFILL)
    st, cap = gb.gbmm_matmul_id_capability("bf16", p)
    assert st == gb.GBMM_OK
    w, x = _up(case.w), _up(case.x)
    ids = _up(case.ids)
    out = torch.empty(cap.required_output_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def launch():
        st, _ = gb.gbmm_matmul_id_static_scratch(p, "bf16", w, case.w.nbytes, x, case.x.nbytes, ids,
                                                 case.ids.nbytes, out, cap.required_output_bytes)
        assert st == gb.GBMM_OK, gb.gbmm_last_error()

    with torch.cuda.stream(s):
        launch()  # before any capture: loads the array and sets kernel attributes
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch()
    for seed in (31, 32):
        ids_np = synth.distinct_ids(m, top_k, E, seed=seed)
        ids.copy_(_up(ids_np))
        out.fill_(0xAB)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert gb.gbmm_device_error()[0] == gb.GBMM_OK
        got = out.cpu().numpy().view(np.float32).astype(np.float64)
        ref, ref_abs = oracle_mod.matmul_id("bf16", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                            case.w, case.x, ids_np)
        assert_close(got, ref.reshape(-1), ref_abs.reshape(-1), "bf16", "f32", f"graph replay, ids seed {seed}")
