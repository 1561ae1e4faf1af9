"""GPU checks of the failure-detection path: a bounded device wait that runs
out reports GBMM_ERR_DEVICE_TIMEOUT through the device error word instead
of trapping, and the context stays usable afterwards."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemv_moe_expert_gb300 import binding as gb  # noqa: E402
from tests.gpu_util import StridedGemm, assert_close  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemv_moe_expert_gb300 import build
    build.build()
    gb.load()
    torch.cuda.init()


def test_bounded_wait_reports_timeout_and_context_survives(oracle_mod):
    assert gb.gbmm_device_error()[0] == gb.GBMM_OK
    st, code = gb.gbmm_test_bounded_wait(2_000_000)  # 2 ms; nothing ever arrives
    assert st == gb.GBMM_ERR_DEVICE_TIMEOUT
    assert code & 1 and (code >> 8) & 0xFF == 3
    # the word was cleared and the GPU still computes
    assert gb.gbmm_device_error() == (gb.GBMM_OK, 0)
    g = StridedGemm("bf16", 1, 128, 256, 128, False, True)
    a, b, c = g.device()
    assert gb.gbmm_gemm(*g.args(a, b, c)) == gb.GBMM_OK
    torch.cuda.synchronize()
    ref, ref_abs = g.oracle(oracle_mod)
    assert_close(g.gather_c(c), ref, ref_abs, "bf16", "bf16", "after timeout")


def test_launch_accounting():
    g = StridedGemm("f16", 1, 64, 64, 64, False, False)
    a, b, c = g.device()
    gb.gbmm_test_reset_launch_count()
    for _ in range(3):
        assert gb.gbmm_gemm(*g.args(a, b, c)) == gb.GBMM_OK
    torch.cuda.synchronize()
    assert gb.gbmm_test_launch_count() == 3
    assert np.isfinite(g.gather_c(c)).all()


def test_debug_sync_mode_gemm_routes():
    """GBMM_DEBUG_SYNC=1 (read once per process, so in a child process):
    every launch is followed by a stream synchronisation; the tensor-core,
    small FFMA and GEMV routes still
    return GBMM_OK and correct results."""
    import os
    import subprocess
    import sys
    code = r"""
import numpy as np, torch
from gemv_moe_expert_gb300 import binding as gb
from tests.gpu_util import StridedGemm, assert_close
import oracle
oracle.build()
gb.load()
for dt, m, n, k, ta, tb in (("f16", 256, 512, 256, False, True), ("f32", 64, 64, 128, False, False),
                            ("f16", 1, 1024, 512, False, True)):
    g = StridedGemm(dt, 1, m, n, k, ta, tb, seed=m)
    a, b, c = g.device()
    assert gb.gbmm_gemm(*g.args(a, b, c)) == gb.GBMM_OK, gb.gbmm_last_error()
    ref, ref_abs = g.oracle(oracle)
    assert_close(g.gather_c(c), ref, ref_abs, dt, dt, "debug sync")
print("ok", gb.gbmm_test_launch_count())
"""
    env = dict(os.environ, GBMM_DEBUG_SYNC="1")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env["PYTHONPATH"] = root + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok 3" in r.stdout, r.stdout
