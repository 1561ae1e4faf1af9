"""ctypes binding of libgbmm.so (include/gbmm.h).

Argument marshalling only: every function here forwards to the C entry point
of the same name and returns its status code.  Device pointers may be given
as integers or as objects with ``data_ptr()`` (torch tensors); ``stream``
defaults to torch's current CUDA stream when torch is importable with CUDA,
else to the legacy default stream.  There is no fallback: if the shared
library is missing, loading raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgbmm.so")

GBMM_OK = 0
GBMM_ERR_INVALID_ARGUMENT = 1
GBMM_ERR_UNSUPPORTED_DTYPE = 2
GBMM_ERR_OVERLAP = 3
GBMM_ERR_SCRATCH = 4
GBMM_ERR_KERNEL_UNAVAILABLE = 5
GBMM_ERR_LAUNCH = 6
GBMM_ERR_DEVICE_TIMEOUT = 7
GBMM_ERR_CUDA = 8

GBMM_F32, GBMM_F16, GBMM_BF16 = 0, 1, 2
DTYPE_CODES = {"f32": GBMM_F32, "f16": GBMM_F16, "bf16": GBMM_BF16}

INPUT_SHARED_PER_TOKEN, INPUT_SLOTTED = 0, 1
ACT_SPLIT, ACT_BF16 = 0, 1
IDS_DISTINCT_PER_TOKEN, IDS_MAY_REPEAT = 0, 1
ROUTE_DIRECT, ROUTE_GROUPED_PREFILL = 0, 1
MATMUL_ID_SCHEMA_VERSION = 3
GROUPED_MAX_EXPERTS = 1024

# every symbol include/gbmm.h declares
EXPORTS = (
    "gbmm_gemm", "gbmm_gemv", "gbmm_matmul_id_scratch_bytes", "gbmm_matmul_id_capability",
    "gbmm_matmul_id", "gbmm_last_error", "gbmm_status_string", "gbmm_abi_version",
    "gbmm_device_error", "gbmm_test_inject_kernel_failure", "gbmm_test_launch_count",
    "gbmm_test_reset_launch_count", "gbmm_test_last_kernel", "gbmm_test_bounded_wait",
    "gbmm_matmul_id_static_scratch", "gbmm_test_static_scratch_copy",
)

# n_experts * m * 4 bytes of routed rows fit the fixed scratch of
# gbmm_matmul_id_static_scratch
STATIC_SCRATCH_ROUTED_ROWS_BYTES = 4 << 20


class MatmulIdParams(ctypes.Structure):
    _fields_ = [("m", ctypes.c_uint32), ("n", ctypes.c_uint32), ("k", ctypes.c_uint32),
                ("top_k", ctypes.c_uint32), ("n_experts", ctypes.c_uint32),
                ("input_layout", ctypes.c_uint32), ("multiplicity", ctypes.c_uint32),
                ("route", ctypes.c_uint32), ("expert_stride_bytes", ctypes.c_uint64),
                ("activation_precision", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class MatmulIdCapability(ctypes.Structure):
    _fields_ = [("schema_version", ctypes.c_uint32), ("weight_dtype", ctypes.c_uint32),
                ("route", ctypes.c_uint32), ("has_scratch", ctypes.c_uint32),
                ("required_weight_bytes", ctypes.c_uint64),
                ("required_input_bytes", ctypes.c_uint64),
                ("required_ids_bytes", ctypes.c_uint64),
                ("required_output_bytes", ctypes.c_uint64),
                ("expert_counts_bytes", ctypes.c_uint64),
                ("routed_rows_bytes", ctypes.c_uint64)]


class MatmulIdReceipt(ctypes.Structure):
    _fields_ = [("weight_dtype", ctypes.c_uint32), ("route", ctypes.c_uint32),
                ("launch_count", ctypes.c_uint32)]


class MatmulIdScratch(ctypes.Structure):
    _fields_ = [("expert_counts", ctypes.c_void_p), ("expert_counts_bytes", ctypes.c_uint64),
                ("routed_rows", ctypes.c_void_p), ("routed_rows_bytes", ctypes.c_uint64),
                ("max_experts", ctypes.c_uint32), ("max_tokens", ctypes.c_uint32)]


_lib = None
_lock = threading.Lock()


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libgbmm.so (once).  Raises OSError if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise OSError(f"libgbmm.so not built at {path}; run gemv_moe_expert_gb300.build.build()")
        lib = ctypes.CDLL(path)
        i64, i32, u32, u64, vp = (ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64,
                                  ctypes.c_void_p)
        gemm_args = [i32, i64, i64, i64, i64, i32, i32, vp, i64, i64, i64, vp, i64, i64, i64,
                     vp, i64, i64, i64, vp]
        for name in ("gbmm_gemm", "gbmm_gemv"):
            getattr(lib, name).argtypes = gemm_args
            getattr(lib, name).restype = i32
        lib.gbmm_matmul_id_scratch_bytes.argtypes = [u32, u32, ctypes.POINTER(u64),
                                                     ctypes.POINTER(u64)]
        lib.gbmm_matmul_id_scratch_bytes.restype = i32
        lib.gbmm_matmul_id_capability.argtypes = [i32, ctypes.POINTER(MatmulIdParams),
                                                  ctypes.POINTER(MatmulIdCapability)]
        lib.gbmm_matmul_id_capability.restype = i32
        lib.gbmm_matmul_id.argtypes = [ctypes.POINTER(MatmulIdParams), i32, vp, u64, vp, u64, vp,
                                       u64, vp, u64, ctypes.POINTER(MatmulIdScratch), vp,
                                       ctypes.POINTER(MatmulIdReceipt)]
        lib.gbmm_matmul_id.restype = i32
        lib.gbmm_last_error.argtypes = []
        lib.gbmm_last_error.restype = ctypes.c_char_p
        lib.gbmm_status_string.argtypes = [i32]
        lib.gbmm_status_string.restype = ctypes.c_char_p
        lib.gbmm_abi_version.argtypes = []
        lib.gbmm_abi_version.restype = u32
        lib.gbmm_device_error.argtypes = [vp, ctypes.POINTER(u32)]
        lib.gbmm_device_error.restype = i32
        lib.gbmm_test_inject_kernel_failure.argtypes = [ctypes.c_char_p]
        lib.gbmm_test_inject_kernel_failure.restype = None
        lib.gbmm_test_launch_count.argtypes = []
        lib.gbmm_test_launch_count.restype = u64
        lib.gbmm_test_reset_launch_count.argtypes = []
        lib.gbmm_test_reset_launch_count.restype = None
        lib.gbmm_test_last_kernel.argtypes = []
        lib.gbmm_test_last_kernel.restype = ctypes.c_char_p
        lib.gbmm_test_bounded_wait.argtypes = [u64, vp, ctypes.POINTER(u32)]
        lib.gbmm_test_bounded_wait.restype = i32
        lib.gbmm_matmul_id_static_scratch.argtypes = [ctypes.POINTER(MatmulIdParams), i32, vp, u64,
                                                      vp, u64, vp, u64, vp, u64, vp,
                                                      ctypes.POINTER(MatmulIdReceipt)]
        lib.gbmm_matmul_id_static_scratch.restype = i32
        lib.gbmm_test_static_scratch_copy.argtypes = [vp, u64, vp]
        lib.gbmm_test_static_scratch_copy.restype = i32
        _lib = lib
        return lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    raise TypeError(f"expected a device pointer, got {type(x)!r}")


def _stream(stream) -> int:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return int(torch.cuda.current_stream().cuda_stream)
        except Exception:  # noqa: BLE001 - torch is optional plumbing
            pass
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _dt(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    if isinstance(dtype, str):
        return DTYPE_CODES[dtype]
    import torch
    return {torch.float32: GBMM_F32, torch.float16: GBMM_F16, torch.bfloat16: GBMM_BF16}[dtype]


def gbmm_gemm(dtype, batch, m, n, k, transpose_a, transpose_b, a, a_offset_bytes, lda,
              batch_stride_a, b, b_offset_bytes, ldb, batch_stride_b, c, c_offset_bytes, ldc,
              batch_stride_c, stream=None) -> int:
    return load().gbmm_gemm(_dt(dtype), batch, m, n, k, int(bool(transpose_a)),
                            int(bool(transpose_b)), _ptr(a), a_offset_bytes, lda, batch_stride_a,
                            _ptr(b), b_offset_bytes, ldb, batch_stride_b, _ptr(c), c_offset_bytes,
                            ldc, batch_stride_c, _stream(stream))


def gbmm_gemv(dtype, batch, m, n, k, transpose_a, transpose_b, a, a_offset_bytes, lda,
              batch_stride_a, b, b_offset_bytes, ldb, batch_stride_b, c, c_offset_bytes, ldc,
              batch_stride_c, stream=None) -> int:
    return load().gbmm_gemv(_dt(dtype), batch, m, n, k, int(bool(transpose_a)),
                            int(bool(transpose_b)), _ptr(a), a_offset_bytes, lda, batch_stride_a,
                            _ptr(b), b_offset_bytes, ldb, batch_stride_b, _ptr(c), c_offset_bytes,
                            ldc, batch_stride_c, _stream(stream))


def gbmm_matmul_id_scratch_bytes(max_experts: int, max_tokens: int):
    """Returns (status, expert_counts_bytes, routed_rows_bytes)."""
    a, b = ctypes.c_uint64(0), ctypes.c_uint64(0)
    st = load().gbmm_matmul_id_scratch_bytes(max_experts, max_tokens, ctypes.byref(a),
                                             ctypes.byref(b))
    return st, a.value, b.value


def make_params(m, n, k, top_k, n_experts, expert_stride_bytes, input_layout=0, multiplicity=0,
                route=0, activation_precision=0) -> MatmulIdParams:
    return MatmulIdParams(m, n, k, top_k, n_experts, input_layout, multiplicity, route,
                          expert_stride_bytes, activation_precision, 0)


def gbmm_matmul_id_capability(weight_dtype, params: MatmulIdParams):
    """Returns (status, MatmulIdCapability)."""
    cap = MatmulIdCapability()
    st = load().gbmm_matmul_id_capability(_dt(weight_dtype), ctypes.byref(params),
                                          ctypes.byref(cap))
    return st, cap


def make_scratch(expert_counts, expert_counts_bytes, routed_rows, routed_rows_bytes, max_experts,
                 max_tokens) -> MatmulIdScratch:
    return MatmulIdScratch(_ptr(expert_counts), expert_counts_bytes, _ptr(routed_rows),
                           routed_rows_bytes, max_experts, max_tokens)


def gbmm_matmul_id(params: MatmulIdParams, weight_dtype, weights, weights_bytes, input,
                   input_bytes, ids, ids_bytes, out, out_bytes, scratch: MatmulIdScratch | None,
                   stream=None):
    """Returns (status, MatmulIdReceipt)."""
    rec = MatmulIdReceipt()
    st = load().gbmm_matmul_id(ctypes.byref(params), _dt(weight_dtype), _ptr(weights),
                               weights_bytes, _ptr(input), input_bytes, _ptr(ids), ids_bytes,
                               _ptr(out), out_bytes,
                               ctypes.byref(scratch) if scratch is not None else None,
                               _stream(stream), ctypes.byref(rec))
    return st, rec


def gbmm_matmul_id_static_scratch(params: MatmulIdParams, weight_dtype, weights, weights_bytes,
                                  input, input_bytes, ids, ids_bytes, out, out_bytes, stream=None):
    """GroupedPrefill without caller scratch, for callers that cannot allocate
    device memory (see include/gbmm.h).  Returns (status, MatmulIdReceipt)."""
    rec = MatmulIdReceipt()
    st = load().gbmm_matmul_id_static_scratch(ctypes.byref(params), _dt(weight_dtype),
                                              _ptr(weights), weights_bytes, _ptr(input),
                                              input_bytes, _ptr(ids), ids_bytes, _ptr(out),
                                              out_bytes, _stream(stream), ctypes.byref(rec))
    return st, rec


def gbmm_last_error() -> str:
    return load().gbmm_last_error().decode()


def gbmm_status_string(status: int) -> str:
    return load().gbmm_status_string(status).decode()


def gbmm_abi_version() -> int:
    return load().gbmm_abi_version()


def gbmm_device_error(stream=None):
    """Returns (status, code)."""
    code = ctypes.c_uint32(0)
    st = load().gbmm_device_error(_stream(stream), ctypes.byref(code))
    return st, code.value


def gbmm_test_inject_kernel_failure(name: str | None) -> None:
    load().gbmm_test_inject_kernel_failure(name.encode() if name else None)


def gbmm_test_launch_count() -> int:
    return load().gbmm_test_launch_count()


def gbmm_test_reset_launch_count() -> None:
    load().gbmm_test_reset_launch_count()


def gbmm_test_last_kernel() -> str:
    return load().gbmm_test_last_kernel().decode()


def gbmm_test_bounded_wait(limit_ns: int, stream=None):
    """Returns (status, code)."""
    code = ctypes.c_uint32(0)
    st = load().gbmm_test_bounded_wait(limit_ns, _stream(stream), ctypes.byref(code))
    return st, code.value


def gbmm_test_static_scratch_copy(dst, nbytes: int, stream=None) -> int:
    """Copy the first `nbytes` of the static scratch array into device buffer `dst`."""
    return load().gbmm_test_static_scratch_copy(_ptr(dst), nbytes, _stream(stream))


class GbmmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{gbmm_status_string(status)}: {message}")
        self.status = status


def check(status: int) -> None:
    """Raise GbmmError for a non-OK status (with gbmm_last_error())."""
    if status != GBMM_OK:
        raise GbmmError(status, gbmm_last_error())
