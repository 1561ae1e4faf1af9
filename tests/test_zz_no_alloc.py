"""gbmm_matmul_id_static_scratch: the grouped expert-ID matmul for callers
that cannot allocate device memory (their host runtime hands them only the
operands and outputs, or they may not call cudaMalloc while serving).

Through the C ABI, two calls in a row with different routings must match
what gbmm_matmul_id returns for the same inputs with caller-owned scratch,
within the parity tolerance (2e-3 * sum|a||b| for bf16 weights); sizes beyond
the fixed scratch and other routes are refused with nothing launched.  This
file is collected last and also runs on its own in a fresh process.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemv_moe_expert_gb300 import binding as gb  # noqa: E402
from gemv_moe_expert_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


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


def _within_tolerance(got, want, ref_abs):
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    return bool(np.all(err <= 2e-3 * ref_abs))


def test_static_scratch_matches_caller_scratch_on_two_calls(oracle_mod):
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

    for call, seed in enumerate((11, 12)):
        ids_np = synth.distinct_ids(m, top_k, E, seed=seed)
        ids = _up(ids_np)
        out_new.fill_(0xAB)
        st, rec = gb.gbmm_matmul_id(p, "bf16", w, case.w.nbytes, x, case.x.nbytes, ids,
                                    ids_np.nbytes, out_ref, cap.required_output_bytes, scratch)
        assert st == gb.GBMM_OK, gb.gbmm_last_error()
        st, rec = gb.gbmm_matmul_id_static_scratch(p, "bf16", w, case.w.nbytes, x, case.x.nbytes,
                                                   ids, ids_np.nbytes, out_new,
                                                   cap.required_output_bytes)
        assert st == gb.GBMM_OK, gb.gbmm_last_error()
        assert rec.launch_count == 2 and rec.route == gb.ROUTE_GROUPED_PREFILL
        torch.cuda.synchronize()
        got = out_new.cpu().numpy().view(np.float32)
        want = out_ref.cpu().numpy().view(np.float32)
        _, ref_abs = oracle_mod.matmul_id("bf16", m, n, k, top_k, E, case.expert_stride_bytes, 0,
                                          case.w, case.x, ids_np)
        assert _within_tolerance(got, want, ref_abs.reshape(-1)), f"call {call}"


def test_static_scratch_refuses_what_it_cannot_hold():
    # n_experts * m * 4 bytes beyond the fixed array
    too_many_tokens = gb.STATIC_SCRATCH_ROUTED_ROWS_BYTES // (4 * 8) + 1
    p = gb.make_params(too_many_tokens, 64, 64, 2, 8, 64 * 64 * 2, route=gb.ROUTE_GROUPED_PREFILL)
    gb.gbmm_test_reset_launch_count()
    base = 1 << 40
    st, _ = gb.gbmm_matmul_id_static_scratch(p, "bf16", base, 1 << 30, base + (1 << 31), 1 << 30,
                                             base + (1 << 32), 1 << 30, base + (1 << 33), 1 << 33)
    assert st == gb.GBMM_ERR_SCRATCH
    assert "static scratch holds" in gb.gbmm_last_error()
    # the Direct route needs no scratch: use gbmm_matmul_id
    p = gb.make_params(4, 64, 64, 2, 8, 64 * 64 * 2, route=gb.ROUTE_DIRECT)
    st, _ = gb.gbmm_matmul_id_static_scratch(p, "bf16", base, 1 << 20, base + (1 << 21), 1 << 20,
                                             base + (1 << 22), 1 << 20, base + (1 << 23), 1 << 20)
    assert st == gb.GBMM_ERR_INVALID_ARGUMENT
    assert gb.gbmm_test_launch_count() == 0
