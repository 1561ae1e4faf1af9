"""Seeded synthetic inputs for the dense GEMM / GEMV / expert-ID matmul path.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path's tests and benchmark.  It draws random tensors and expert ids and
nothing else: it holds none of the method's arithmetic (no products, sums,
routing or output rounding).  Every value it returns is already rounded to
the storage dtype, so both sides read identical bits.

Storage conventions
  * ``"f32"``  -> ``numpy.float32``
  * ``"f16"``  -> ``numpy.float16``
  * ``"bf16"`` -> ``numpy.uint16`` holding the bf16 bit pattern (the upper
    half of a binary32, rounded to nearest-even).

Large normal tensors are drawn in fixed chunks of ``CHUNK`` elements, each
from its own ``numpy.random.SeedSequence([seed, stream, chunk])``, so the
values do not depend on how many threads draw them.

The five named workloads are the ones the benchmark and the parity tests use
(shapes and distributions from the expert-ID matmul and MLX GEMM pages:
mlx-native 0.13.0 ``dense_matmul_id.rs`` and tract-metal 0.23.6
``mlx_gemm/mod.rs``).  Expert ids are the first draw of a fresh
``numpy.random.default_rng(seed)``; the activation/weight tensors use the
chunked streams above.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22

DTYPES = ("f32", "f16", "bf16")
ITEMSIZE = {"f32": 4, "f16": 2, "bf16": 2}

# stream ids keep the chunked draws of different tensors independent
STREAM_A = 1
STREAM_B = 2


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (nearest, ties to even); returns the bits."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_in = v.reshape(-1).view(np.uint32)
    flat_out = out.reshape(-1)

    def work(lo_hi):
        lo, hi = lo_hi
        b = flat_in[lo:hi].astype(np.uint64)
        r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
        flat_out[lo:hi] = r.astype(np.uint16)

    _parallel_ranges(flat_in.size, work)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f32(values: np.ndarray, dtype: str) -> np.ndarray:
    """The exact float32 value of every stored element."""
    if dtype == "bf16":
        return bf16_bits_to_f32(values)
    return np.asarray(values).astype(np.float32)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _parallel_ranges(total: int, fn) -> None:
    ranges = [(lo, min(total, lo + CHUNK)) for lo in range(0, total, CHUNK)]
    if len(ranges) <= 1:
        for r in ranges:
            fn(r)
        return
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fn, ranges))


def _store(v32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return v32
    if dtype == "f16":
        return v32.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(v32)
    raise ValueError(dtype)


def _chunked(shape, dtype: str, seed: int, stream: int, draw) -> np.ndarray:
    total = int(np.prod(shape, dtype=np.int64)) if len(shape) else 1
    np_dt = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]
    out = np.empty(total, dtype=np_dt)

    def work(lo_hi):
        lo, hi = lo_hi
        rng = np.random.default_rng(np.random.SeedSequence([seed, stream, lo // CHUNK]))
        out[lo:hi] = _store(draw(rng, hi - lo), dtype)

    _parallel_ranges(total, work)
    return out.reshape(shape)


def normal(shape, std: float, dtype: str, seed: int = 0, stream: int = STREAM_A) -> np.ndarray:
    """N(0, std) (std is the standard deviation), rounded to ``dtype``."""
    std = np.float32(std)
    return _chunked(shape, dtype, seed, stream,
                    lambda rng, n: rng.standard_normal(n, dtype=np.float32) * std)


def uniform(shape, lo: float, hi: float, dtype: str, seed: int = 0,
            stream: int = STREAM_A) -> np.ndarray:
    """U[lo, hi), rounded to ``dtype``."""
    return _chunked(shape, dtype, seed, stream,
                    lambda rng, n: rng.uniform(lo, hi, n).astype(np.float32))


def small_ints(shape, bound: int, dtype: str, seed: int = 0, stream: int = STREAM_A) -> np.ndarray:
    """Integers in [-bound, bound]: exact in every storage dtype for bound <= 256."""
    return _chunked(shape, dtype, seed, stream,
                    lambda rng, n: rng.integers(-bound, bound + 1, n).astype(np.float32))


def ramp(shape, seed: int, dtype: str = "f32") -> np.ndarray:
    """The periodic test ramp of the gemv_wide tests on the tract-metal 0.23.6
    MLX GEMM page (``gemv_wide_tests::ramp``): element i is
    ((7 i + 13 seed) mod 29 - 14) / 64, rounded to ``dtype`` (exact in all three)."""
    total = int(np.prod(shape))
    i = np.arange(total, dtype=np.int64)
    v = (((i * 7 + seed * 13) % 29) - 14).astype(np.float32) / np.float32(64.0)
    return _store(v, dtype).reshape(shape)


def distinct_ids(m: int, top_k: int, n_experts: int, seed: int = 0,
                 zipf_s: float | None = None, rng: np.random.Generator | None = None) -> np.ndarray:
    """Per token, ``top_k`` distinct expert ids drawn without replacement.

    Uniform by default; with ``zipf_s`` the draw weights are
    p(e) proportional to (e + 1) ** -zipf_s (rank = id).  Returns uint32 [m, top_k].
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    p = None
    if zipf_s is not None:
        p = (np.arange(n_experts, dtype=np.float64) + 1.0) ** (-zipf_s)
        p /= p.sum()
    out = np.empty((m, top_k), dtype=np.uint32)
    for t in range(m):
        out[t] = rng.choice(n_experts, top_k, replace=False, p=p)
    return out


def repeat_ids(m: int, top_k: int, n_experts: int, seed: int = 0) -> np.ndarray:
    """Ids with repeats allowed within a token row (uniform, with replacement)."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, n_experts, size=(m, top_k)).astype(np.uint32)


# ---------------------------------------------------------------------------
# Named workloads
# ---------------------------------------------------------------------------

@dataclass
class GemmCase:
    """C[b] = op(A[b]) op(B[b]) with dense, tight storage.

    A is stored [batch, k, m] when ``ta`` else [batch, m, k]; B is stored
    [batch, n, k] when ``tb`` else [batch, k, n].  C is [batch, m, n].
    """
    name: str
    dtype: str
    batch: int
    m: int
    n: int
    k: int
    ta: bool
    tb: bool
    a: np.ndarray
    b: np.ndarray

    @property
    def lda(self) -> int:
        return self.m if self.ta else self.k

    @property
    def ldb(self) -> int:
        return self.k if self.tb else self.n

    @property
    def ldc(self) -> int:
        return self.n

    @property
    def stride_a(self) -> int:
        return self.m * self.k

    @property
    def stride_b(self) -> int:
        return self.n * self.k

    @property
    def stride_c(self) -> int:
        return self.m * self.n

    @property
    def flops(self) -> int:
        return 2 * self.batch * self.m * self.n * self.k


@dataclass
class MatmulIdCase:
    """Expert-ID matmul inputs: W [n_experts, n, k] (row-major per expert,
    ``expert_stride_bytes`` apart), x f32, ids u32 [m, top_k]."""
    name: str
    wdtype: str
    m: int
    n: int
    k: int
    top_k: int
    n_experts: int
    input_layout: int          # 0 = SharedPerToken, 1 = Slotted
    multiplicity: int          # 0 = DistinctPerToken, 1 = MayRepeat
    route: int                 # 0 = Direct, 1 = GroupedPrefill
    w: np.ndarray              # flat storage, expert e at element e*expert_stride_elems
    x: np.ndarray
    ids: np.ndarray
    expert_stride_bytes: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def expert_stride_elems(self) -> int:
        return self.expert_stride_bytes // ITEMSIZE[self.wdtype]


def gemm_case(name, dtype, batch, m, n, k, ta=False, tb=False, dist="normal", std=1.0,
              seed=0) -> GemmCase:
    shape_a = (batch, k, m) if ta else (batch, m, k)
    shape_b = (batch, n, k) if tb else (batch, k, n)
    if dist == "normal":
        a = normal(shape_a, std, dtype, seed, STREAM_A)
        b = normal(shape_b, std, dtype, seed, STREAM_B)
    elif dist == "uniform":
        a = uniform(shape_a, -1.0, 1.0, dtype, seed, STREAM_A)
        b = uniform(shape_b, -1.0, 1.0, dtype, seed, STREAM_B)
    elif dist == "ints":
        a = small_ints(shape_a, 8, dtype, seed, STREAM_A)
        b = small_ints(shape_b, 8, dtype, seed, STREAM_B)
    elif dist == "ramp":
        a = ramp(shape_a, 1, dtype)
        b = ramp(shape_b, 2, dtype)
    else:
        raise ValueError(dist)
    return GemmCase(name, dtype, batch, m, n, k, ta, tb, a, b)


def matmul_id_case(name, wdtype, m, n, k, top_k, n_experts, *, route=0, input_layout=0,
                   multiplicity=0, zipf_s=None, w_std=0.02, seed=0, stride_pad_elems=0,
                   ids=None) -> MatmulIdCase:
    if ids is None:
        if multiplicity == 0:
            ids = distinct_ids(m, top_k, n_experts, seed, zipf_s)
        else:
            ids = repeat_ids(m, top_k, n_experts, seed)
    stride_elems = n * k + stride_pad_elems
    w = normal((n_experts * stride_elems,), w_std, wdtype, seed, STREAM_A)
    rows = m if input_layout == 0 else m * top_k
    x = normal((rows, k), 1.0, "f32", seed, STREAM_B)
    return MatmulIdCase(name, wdtype, m, n, k, top_k, n_experts, input_layout, multiplicity,
                        route, w, x, np.ascontiguousarray(ids, dtype=np.uint32),
                        expert_stride_bytes=stride_elems * ITEMSIZE[wdtype])


WORKLOADS = ("c1_f32_gemm", "c2_f16_gemv", "c3_f16_gemm", "c4_moe_direct", "c5_moe_grouped")


def workload(name: str):
    """The five named workloads (all seed 0)."""
    if name == "c1_f32_gemm":
        # single f32 GEMM 64x64x128, NN, U[-1,1]
        return gemm_case(name, "f32", 1, 64, 64, 128, False, False, dist="uniform")
    if name == "c2_f16_gemv":
        # decode GEMV: x [1,4096] ~N(0,1), W [11008,4096] ~N(0,0.02) stored [n,k] (transpose_b)
        a = normal((1, 1, 4096), 1.0, "f16", 0, STREAM_A)
        b = normal((1, 11008, 4096), 0.02, "f16", 0, STREAM_B)
        return GemmCase(name, "f16", 1, 1, 11008, 4096, False, True, a, b)
    if name == "c3_f16_gemm":
        # batched strided GEMM 4 x 4096^3, B stored [b,N,K], entries ~N(0, 1/sqrt(K))
        return gemm_case(name, "f16", 4, 4096, 4096, 4096, False, True, std=1.0 / 64.0)
    if name == "c4_moe_direct":
        return matmul_id_case(name, "bf16", 4, 1408, 2048, 8, 64, route=0)
    if name == "c5_moe_grouped":
        return matmul_id_case(name, "bf16", 4096, 1536, 4096, 8, 128, route=1, zipf_s=1.1)
    raise KeyError(name)
