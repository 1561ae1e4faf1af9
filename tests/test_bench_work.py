"""The bench's algorithmic work per call (the numerators of every roofline
fraction it reports) against closed forms for the five workloads: bytes moved
and flops of each call written out from its shapes and dtypes.  Stand-in
objects carry the shapes, so no weights are materialised; the expert-ID calls
use the seeded ids of the real workloads (C4: 26 distinct experts of 64)."""

import types

import numpy as np
import pytest

import bench
from gemv_moe_expert_gb300 import synth


def gemm_standin(dtype, batch, m, n, k):
    return types.SimpleNamespace(dtype=dtype, batch=batch, m=m, n=n, k=k,
                                 a=np.empty(batch * m * k, dtype=np.uint8),
                                 b=np.empty(batch * n * k, dtype=np.uint8))


def matmul_id_standin(wdtype, m, n, k, top_k, n_experts, zipf_s=None):
    ids = synth.distinct_ids(m, top_k, n_experts, 0, zipf_s)
    return types.SimpleNamespace(wdtype=wdtype, m=m, n=n, k=k, top_k=top_k, n_experts=n_experts,
                                 ids=np.ascontiguousarray(ids, dtype=np.uint32),
                                 x=types.SimpleNamespace(nbytes=m * k * 4))


def test_c1_small_f32_gemm():
    wk = bench.work_of("c1", gemm_standin("f32", 1, 64, 64, 128))
    assert wk["flops"] == 2 * 64 * 64 * 128 == 1_048_576
    assert wk["bytes"] == (64 * 128 + 128 * 64 + 64 * 64) * 4 == 81_920


def test_c2_decode_gemv():
    wk = bench.work_of("c2", gemm_standin("f16", 1, 1, 11008, 4096))
    assert wk["bytes"] == 90_177_536 + 8_192 + 22_016 == 90_207_744   # W + x + y
    assert wk["flops"] == 90_177_536
    assert wk["bound"] == "hbm"


def test_c3_batched_f16_gemm():
    wk = bench.work_of("c3", gemm_standin("f16", 4, 4096, 4096, 4096))
    assert wk["flops"] == 549_755_813_888
    assert wk["bytes"] == 3 * 4 * 4096 * 4096 * 2 == 402_653_184
    assert wk["bound"] == "tensor"


def test_c4_direct_reads_each_distinct_expert_once():
    c = matmul_id_standin("bf16", 4, 1408, 2048, 8, 64)
    wk = bench.work_of("c4", c)
    assert wk["distinct_experts"] == 26
    expert = 1408 * 2048 * 2
    assert expert == 5_767_168
    assert wk["bytes"] == 26 * expert + 4 * 2048 * 4 + 4 * 8 * 4 + 4 * 8 * 1408 * 4 == 150_159_488
    assert wk["flops"] == 2 * 4 * 8 * 1408 * 2048 == 184_549_376


def test_c5_grouped_reads_the_whole_stack():
    c = matmul_id_standin("bf16", 4096, 1536, 4096, 8, 128, zipf_s=1.1)
    wk = bench.work_of("c5", c)
    assert wk["distinct_experts"] == 128
    assert wk["bytes"] == 1_610_612_736 + 67_108_864 + 131_072 + 201_326_592 == 1_879_179_264
    assert wk["flops"] == 412_316_860_416


@pytest.mark.parametrize("hbm,tensor", [(6790.3, 1701.9), (8000.0, 2250.0)])
def test_roofline_time_is_the_larger_bound(hbm, tensor):
    peaks = {"hbm_gbs": hbm}
    c3 = bench.work_of("c3", gemm_standin("f16", 4, 4096, 4096, 4096))
    c2 = bench.work_of("c2", gemm_standin("f16", 1, 1, 11008, 4096))
    assert bench.roofline_seconds(c3, peaks, tensor) == pytest.approx(549_755_813_888 / (tensor * 1e12))
    assert bench.roofline_seconds(c2, peaks, tensor) == pytest.approx(90_207_744 / (hbm * 1e9))
