"""Helpers shared by the GPU parity tests: raw device buffers with guard bands,
strided operand construction, and the tolerance check.

Tolerance (per output element, against the binary64 oracle value ``ref`` and
its sum |a||b| ``ref_abs``):
    |gpu - ref| <= tau * ref_abs            tau = 1e-5 for f32 inputs,
                                            tau = 2e-3 for f16/bf16 inputs
plus, for bf16 OUTPUTS only, the rounding of the stored result,
2^-8 * |ref| (bf16 keeps 8 significant bits; rounding to nearest can move a
value by up to half an ulp, 2^-8 relative at worst).  f16 outputs need no
such term: their rounding, at most 2^-11 |ref| <= 2^-11 ref_abs, is already
inside 2e-3 ref_abs.  Where ref_abs == 0 the GPU value must be exactly 0.
"""

from __future__ import annotations

import numpy as np
import torch

from gemv_moe_expert_gb300 import synth

GUARD = 4096
SENTINEL = 0xA5

NP_DT = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}
NAN_BITS = {"f32": np.float32(np.nan), "f16": np.float16(np.nan), "bf16": np.uint16(0x7FC0)}


def tau_for(input_dtype: str) -> float:
    return 1e-5 if input_dtype == "f32" else 2e-3


class DevBuf:
    """A device byte buffer with 4 KiB guard bands on both sides."""

    def __init__(self, nbytes: int, fill: int | None = SENTINEL, host: np.ndarray | None = None):
        self.nbytes = int(nbytes)
        total = self.nbytes + 2 * GUARD
        self.t = torch.full((total,), SENTINEL, dtype=torch.uint8, device="cuda")
        if host is not None:
            raw = np.ascontiguousarray(host).reshape(-1).view(np.uint8)
            assert raw.size <= self.nbytes
            self.t[GUARD:GUARD + raw.size].copy_(torch.from_numpy(raw.copy()))
        elif fill is not None and fill != SENTINEL:
            self.t[GUARD:GUARD + self.nbytes].fill_(fill)

    @property
    def ptr(self) -> int:
        return self.t.data_ptr() + GUARD

    def read(self, np_dtype, count: int | None = None, offset_bytes: int = 0) -> np.ndarray:
        raw = self.t[GUARD + offset_bytes:GUARD + self.nbytes].cpu().numpy()
        out = raw.view(np_dtype)
        return out if count is None else out[:count]

    def guards_intact(self) -> bool:
        head = self.t[:GUARD]
        tail = self.t[GUARD + self.nbytes:]
        return bool((head == SENTINEL).all().item()) and bool((tail == SENTINEL).all().item())


def to_f64(values: np.ndarray, dtype: str) -> np.ndarray:
    return synth.as_f32(values, dtype).astype(np.float64)


def assert_close(got, ref, ref_abs, in_dtype: str, out_dtype: str, what: str = "") -> float:
    """Check the tolerance element by element; returns the worst err / tol."""
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    ref_abs = np.asarray(ref_abs, dtype=np.float64).reshape(-1)
    assert got.shape == ref.shape
    tol = tau_for(in_dtype) * ref_abs
    if out_dtype == "bf16":
        tol = tol + 2.0 ** -8 * np.abs(ref)
    err = np.abs(got - ref)
    ok = err <= tol
    if not ok.all():
        bad = np.flatnonzero(~ok)
        i = bad[0]
        raise AssertionError(
            f"{what}: {bad.size}/{got.size} elements outside tolerance; first at flat {i}: "
            f"gpu={got[i]!r} ref={ref[i]!r} ref_abs={ref_abs[i]!r} tol={tol[i]!r}")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / tol, 0.0)
    return float(ratio.max()) if ratio.size else 0.0


class StridedGemm:
    """A GEMM problem with explicit leading dims, batch strides and byte
    offsets; padding elements are NaN, so a kernel that reads one shows it."""

    def __init__(self, dtype, batch, m, n, k, ta, tb, *, lda=None, ldb=None, ldc=None, sa=None,
                 sb=None, sc=None, a_off=0, b_off=0, c_off=0, dist="normal", std=1.0, seed=0):
        self.dtype, self.batch, self.m, self.n, self.k = dtype, batch, m, n, k
        self.ta, self.tb = bool(ta), bool(tb)
        ra, ca = (k, m) if ta else (m, k)
        rb, cb = (n, k) if tb else (k, n)
        self.lda = lda if lda is not None else max(1, ca)
        self.ldb = ldb if ldb is not None else max(1, cb)
        self.ldc = ldc if ldc is not None else max(1, n)
        self.sa = sa if sa is not None else ra * self.lda
        self.sb = sb if sb is not None else rb * self.ldb
        self.sc = sc if sc is not None else m * self.ldc
        self.size = synth.ITEMSIZE[dtype]
        self.a_off, self.b_off, self.c_off = a_off, b_off, c_off
        na = (batch - 1) * self.sa + ra * self.lda if batch > 0 else 0
        nb = (batch - 1) * self.sb + rb * self.ldb if batch > 0 else 0
        self.nc = (batch - 1) * self.sc + m * self.ldc if batch > 0 else 0
        rng = np.random.default_rng(seed)
        self.a = np.full(max(na, 1), NAN_BITS[dtype], dtype=NP_DT[dtype])
        self.b = np.full(max(nb, 1), NAN_BITS[dtype], dtype=NP_DT[dtype])
        for bi in range(batch if self.sa else min(batch, 1)):
            for r in range(ra):
                base = bi * self.sa + r * self.lda
                self.a[base:base + ca] = self._draw(rng, ca, dist, std)
        for bi in range(batch if self.sb else min(batch, 1)):
            for r in range(rb):
                base = bi * self.sb + r * self.ldb
                self.b[base:base + cb] = self._draw(rng, cb, dist, std)

    def _draw(self, rng, count, dist, std):
        if dist == "normal":
            v = rng.standard_normal(count).astype(np.float32) * np.float32(std)
        elif dist == "uniform":
            v = rng.uniform(-1, 1, count).astype(np.float32)
        elif dist == "ints":
            v = rng.integers(-8, 9, count).astype(np.float32)
        else:
            raise ValueError(dist)
        return synth._store(v, self.dtype)

    def device(self):
        a = DevBuf(self.a.nbytes + self.a_off, host=np.concatenate(
            [np.zeros(self.a_off, np.uint8), self.a.view(np.uint8)]))
        b = DevBuf(self.b.nbytes + self.b_off, host=np.concatenate(
            [np.zeros(self.b_off, np.uint8), self.b.view(np.uint8)]))
        c = DevBuf(max(self.nc, 1) * self.size + self.c_off)
        return a, b, c

    def args(self, a, b, c):
        return (self.dtype, self.batch, self.m, self.n, self.k, self.ta, self.tb,
                a.ptr, self.a_off, self.lda, self.sa, b.ptr, self.b_off, self.ldb, self.sb,
                c.ptr, self.c_off, self.ldc, self.sc)

    def gather_c(self, c: DevBuf) -> np.ndarray:
        """Read C back as binary64 [batch, m, n] (elements outside C untouched)."""
        flat = c.read(NP_DT[self.dtype], self.nc, self.c_off)
        vals = to_f64(flat, self.dtype)
        out = np.empty((self.batch, self.m, self.n))
        for bi in range(self.batch):
            for i in range(self.m):
                base = bi * self.sc + i * self.ldc
                out[bi, i] = vals[base:base + self.n]
        return out

    def c_gaps_untouched(self, c: DevBuf) -> bool:
        """Bytes of the C buffer outside the m x n matrices keep the sentinel."""
        raw = c.read(np.uint8, None, 0)
        mask = np.ones(raw.size, dtype=bool)
        for bi in range(self.batch):
            for i in range(self.m):
                lo = self.c_off + (bi * self.sc + i * self.ldc) * self.size
                mask[lo:lo + self.n * self.size] = False
        return bool((raw[mask] == SENTINEL).all())

    def oracle(self, oracle_mod, idx=None):
        return oracle_mod.gemm(self.dtype, self.batch, self.m, self.n, self.k, self.ta, self.tb,
                               self.a, self.lda, self.sa, self.b, self.ldb, self.sb, idx=idx)
