"""ctypes binding of libmma42 (include/mma42.h).

Argument marshalling only: torch supplies device memory and the current
stream, every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or a call fails, this raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmma42.so")

# element-type codes of mma42.h
MMA_F16, MMA_BF16, MMA_E4M3, MMA_E5M2, MMA_I8, MMA_F32, MMA_I32, MMA_U8 = 1, 2, 3, 4, 5, 6, 7, 8
CODE = {torch.float16: MMA_F16, torch.bfloat16: MMA_BF16, torch.float8_e4m3fn: MMA_E4M3,
        torch.float8_e5m2: MMA_E5M2, torch.int8: MMA_I8, torch.uint8: MMA_U8, torch.float32: MMA_F32,
        torch.int32: MMA_I32}
ACC_DTYPE = {torch.float16: torch.float32, torch.bfloat16: torch.float32,
             torch.float8_e4m3fn: torch.float32, torch.float8_e5m2: torch.float32,
             torch.int8: torch.int32, torch.uint8: torch.int32}

STATUS = {0: "MMA_OK", 1: "MMA_ERR_INVALID_ARG", 2: "MMA_ERR_UNSUPPORTED", 3: "MMA_ERR_SHAPE",
          4: "MMA_ERR_ALIGN", 5: "MMA_ERR_NOT_SPARSE", 6: "MMA_ERR_TIMEOUT", 7: "MMA_ERR_CUDA"}
EXPORTS = ("mma_gemm", "mma_gemm_ex", "sparse42_compress", "sparse42_prune", "sparse42_gemm", "mma_quantize",
           "sparse42_quantize_prune", "mma_sync_status",
           "mma_status_string", "mma_abi_version", "mma_set_wait_limit_ns", "mma_debug_inject",
           "mma_launch_count", "mma_gemm_splitk_noalloc", "mma_legacy_mma_peak", "mma_tcgen05_peak",
           "mma_tma_feed_probe")


class MmaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        self.status = STATUS.get(code, str(code))
        super().__init__(f"{what}: {self.status}")


class mma_dtypes_t(ctypes.Structure):
    _fields_ = [("a", ctypes.c_int32), ("b", ctypes.c_int32), ("acc", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load libmma42.so (built by ``tensor_core_matrix_02_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is missing: build it with `python -m tensor_core_matrix_02_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.mma_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, mma_dtypes_t, vp]
        lib.mma_gemm.restype = i32
        lib.mma_gemm_ex.argtypes = [vp, vp, vp, vp, i64, i64, i64, mma_dtypes_t, ctypes.c_uint32, vp]
        lib.mma_gemm_ex.restype = i32
        lib.sparse42_compress.argtypes = [vp, vp, vp, i64, i64, i32, vp, vp]
        lib.sparse42_compress.restype = i32
        lib.sparse42_prune.argtypes = [vp, vp, vp, i64, i64, i32, vp, vp]
        lib.sparse42_prune.restype = i32
        lib.mma_quantize.argtypes = [vp, vp, i64, i32, vp]
        lib.mma_quantize.restype = i32
        lib.sparse42_quantize_prune.argtypes = [vp, vp, vp, i64, i64, i32, vp, vp]
        lib.sparse42_quantize_prune.restype = i32
        lib.sparse42_gemm.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, mma_dtypes_t, vp]
        lib.sparse42_gemm.restype = i32
        lib.mma_sync_status.argtypes = [vp]
        lib.mma_sync_status.restype = i32
        lib.mma_status_string.argtypes = [i32]
        lib.mma_status_string.restype = ctypes.c_char_p
        lib.mma_abi_version.argtypes = []
        lib.mma_abi_version.restype = i32
        lib.mma_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.mma_set_wait_limit_ns.restype = None
        lib.mma_debug_inject.argtypes = [i32]
        lib.mma_debug_inject.restype = None
        lib.mma_gemm_splitk_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, mma_dtypes_t, i32, vp]
        lib.mma_gemm_splitk_noalloc.restype = i32
        lib.mma_launch_count.argtypes = []
        lib.mma_launch_count.restype = ctypes.c_uint64
        lib.mma_legacy_mma_peak.argtypes = [i32, ctypes.POINTER(ctypes.c_double), vp]
        lib.mma_legacy_mma_peak.restype = i32
        lib.mma_tcgen05_peak.argtypes = [i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), vp]
        lib.mma_tcgen05_peak.restype = i32
        pi32, pd = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double)
        lib.mma_tma_feed_probe.argtypes = [i32, pi32, pi32, i32, i32, i64, pd, pd, vp]
        lib.mma_tma_feed_probe.restype = i32
        if path is None:
            _lib = lib
        return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(code: int, what: str):
    if code != 0:
        raise MmaError(code, what)


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensors must live on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous (row-major, no padding)")


def mma_status_string(code: int) -> str:
    return load_library().mma_status_string(code).decode()


def mma_sync_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load_library().mma_sync_status(_stream(stream)))


def mma_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load_library().mma_launch_count())


LEGACY_KINDS = {"s8": 0, "s8_sparse": 1, "bf16": 2, "e4m3": 3}


def mma_legacy_mma_peak(kind: str, stream=None) -> float:
    """Throughput ceiling in ops/s of the warp-level (mma.sync / mma.sp) tensor
    instructions for ``kind`` in LEGACY_KINDS, measured now on the current device
    (about 25 ms; waits for the stream)."""
    out = ctypes.c_double(0.0)
    _check(load_library().mma_legacy_mma_peak(LEGACY_KINDS[kind], ctypes.byref(out), _stream(stream)),
           "mma_legacy_mma_peak")
    return out.value


TCGEN05_KINDS = {"bf16": 0, "e4m3": 1, "bf16_sparse": 2, "e4m3_sparse": 3}


def mma_tcgen05_peak(kind: str, stream=None) -> tuple[float, float]:
    """Throughput ceiling of tcgen05.mma for ``kind`` in TCGEN05_KINDS (dense or
    4:2-sparse kind::f16 / kind::f8f6f4, the CTA-pair GEMMs' instruction shapes),
    measured now on the current device with operands resident in shared memory
    (about 25 ms; waits for the stream).  Returns (ops per second, ops per SM clock
    cycle per SM)."""
    ops = ctypes.c_double(0.0)
    per_clk = ctypes.c_double(0.0)
    _check(load_library().mma_tcgen05_peak(TCGEN05_KINDS[kind], ctypes.byref(ops), ctypes.byref(per_clk),
                                           _stream(stream)), "mma_tcgen05_peak")
    return ops.value, per_clk.value


def mma_tma_feed_probe(boxes, stages: int, clusters: int = 0, src_bytes: int = 64 << 20,
                       stream=None) -> tuple[float, float]:
    """TMA fill rate of the CTA-pair kernels' pipeline ring with nothing consuming
    it, measured now on the current device.  ``boxes``: up to four (rows, row
    bytes) boxes per stage; ``stages`` in the ring; ``clusters`` SM pairs (0: all
    that fit); ``src_bytes`` of source (64 MB stays in L2).  Returns (bytes, box
    rows) per SM clock cycle per SM."""
    n = len(boxes)
    rows = (ctypes.c_int32 * 4)(*[int(r) for r, _ in boxes], *([0] * (4 - n)))
    rb = (ctypes.c_int32 * 4)(*[int(b) for _, b in boxes], *([0] * (4 - n)))
    byts, rws = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _check(load_library().mma_tma_feed_probe(n, rows, rb, stages, clusters, src_bytes, ctypes.byref(byts),
                                             ctypes.byref(rws), _stream(stream)), "mma_tma_feed_probe")
    return byts.value, rws.value


MMA_FLAG_CLAMP = 1


def mma_gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, D: torch.Tensor | None = None,
             stream=None, clamp: bool = False) -> torch.Tensor:
    """D = A @ B + C on the tensor cores (A M x K, B K x N, C M x N).

    ``clamp=True`` (8-bit integer inputs): saturate D to the i32 range instead of
    wrapping."""
    _need_cuda(A, B, C, D)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shapes A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)} do not chain")
    if D is None:
        D = torch.empty((M, N), dtype=C.dtype, device=C.device)
    t = mma_dtypes_t(CODE.get(A.dtype, 0), CODE.get(B.dtype, 0), CODE.get(C.dtype, 0))
    with torch.cuda.device(A.device):
        if clamp:
            _check(load_library().mma_gemm_ex(_ptr(A), _ptr(B), _ptr(C), _ptr(D), M, N, K, t, MMA_FLAG_CLAMP,
                                              _stream(stream)), "mma_gemm_ex")
        else:
            _check(load_library().mma_gemm(_ptr(A), _ptr(B), _ptr(C), _ptr(D), M, N, K, t, _stream(stream)),
                   "mma_gemm")
    return D


def sparse42_compress(A: torch.Tensor, violations: torch.Tensor | None = None, stream=None,
                      check: bool = False):
    """4:2 compression of A (M x K) -> (vals M x K/2, idx M x K/8 uint8).

    ``violations`` (optional, int32 device tensor of one element) receives the
    number of groups of four that held more than two non-zeros.  With
    ``check=True`` the call waits for the count and raises MmaError with
    MMA_ERR_NOT_SPARSE if any group broke the 4:2 contract.
    """
    _need_cuda(A, violations)
    M, K = A.shape
    if check and violations is None:
        violations = torch.zeros(1, dtype=torch.int32, device=A.device)
    vals = torch.empty((M, K // 2), dtype=A.dtype, device=A.device)
    idx = torch.empty((M, K // 8), dtype=torch.uint8, device=A.device)
    with torch.cuda.device(A.device):
        _check(load_library().sparse42_compress(_ptr(A), _ptr(vals), _ptr(idx), M, K, CODE.get(A.dtype, 0),
                                                _ptr(violations), _stream(stream)), "sparse42_compress")
    if check:
        n = int(violations.item())
        if n:
            raise MmaError(5, f"sparse42_compress: {n} groups of four hold more than two non-zeros")
    return vals, idx


def sparse42_prune(A: torch.Tensor, dropped: torch.Tensor | None = None, stream=None):
    """Prune a dense A (M x K) to 4:2 by magnitude and compress it -> (vals, idx).

    In every group of four along K the two elements of largest magnitude stay
    (the lower position on equal magnitude); ``dropped`` (optional, int32 device
    tensor of one element) receives the number of groups that lost a non-zero.
    """
    _need_cuda(A, dropped)
    M, K = A.shape
    vals = torch.empty((M, K // 2), dtype=A.dtype, device=A.device)
    idx = torch.empty((M, K // 8), dtype=torch.uint8, device=A.device)
    with torch.cuda.device(A.device):
        _check(load_library().sparse42_prune(_ptr(A), _ptr(vals), _ptr(idx), M, K, CODE.get(A.dtype, 0),
                                             _ptr(dropped), _stream(stream)), "sparse42_prune")
    return vals, idx


def mma_quantize(x: torch.Tensor, dtype: torch.dtype, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """f32 -> dtype (float16, bfloat16, float8_e4m3fn, float8_e5m2): saturate to the
    largest finite magnitude, round to nearest even; NaN stays NaN."""
    _need_cuda(x, out)
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 tensor")
    if out is None:
        out = torch.empty(x.shape, dtype=dtype, device=x.device)
    with torch.cuda.device(x.device):
        _check(load_library().mma_quantize(_ptr(x), _ptr(out), x.numel(), CODE.get(dtype, 0), _stream(stream)),
               "mma_quantize")
    return out


def sparse42_quantize_prune(A: torch.Tensor, dtype: torch.dtype, dropped: torch.Tensor | None = None,
                            stream=None):
    """f32 A (M x K) -> quantised to dtype, pruned to 4:2 by magnitude and
    compressed in one pass -> (vals M x K/2 of dtype, idx M x K/8 uint8)."""
    _need_cuda(A, dropped)
    if A.dtype != torch.float32 or not A.is_contiguous():
        raise ValueError("A must be a contiguous float32 tensor")
    M, K = A.shape
    vals = torch.empty((M, K // 2), dtype=dtype, device=A.device)
    idx = torch.empty((M, K // 8), dtype=torch.uint8, device=A.device)
    with torch.cuda.device(A.device):
        _check(load_library().sparse42_quantize_prune(_ptr(A), _ptr(vals), _ptr(idx), M, K, CODE.get(dtype, 0),
                                                      _ptr(dropped), _stream(stream)), "sparse42_quantize_prune")
    return vals, idx


def sparse42_gemm(vals: torch.Tensor, idx: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                  D: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """D = A @ B + C with A given compressed as (vals, idx); K = B.shape[0]."""
    _need_cuda(vals, idx, B, C, D)
    M = vals.shape[0]
    K, N = B.shape
    if tuple(vals.shape) != (M, K // 2) or tuple(idx.shape) != (M, K // 8) or tuple(C.shape) != (M, N):
        raise ValueError("shapes of vals, idx, B and C do not chain")
    if D is None:
        D = torch.empty((M, N), dtype=C.dtype, device=C.device)
    t = mma_dtypes_t(CODE.get(vals.dtype, 0), CODE.get(B.dtype, 0), CODE.get(C.dtype, 0))
    with torch.cuda.device(vals.device):
        _check(load_library().sparse42_gemm(_ptr(vals), _ptr(idx), _ptr(B), _ptr(C), _ptr(D), M, N, K, t,
                                            _stream(stream)), "sparse42_gemm")
    return D


def mma_gemm_splitk_noalloc(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, D: torch.Tensor, ksplit: int,
                            stream=None) -> torch.Tensor:
    """D = A @ B + C in ``ksplit`` K slices whose partials live in the library's
    fixed device array (no allocation inside the call; D is the caller's)."""
    _need_cuda(A, B, C, D)
    M, K = A.shape
    N = B.shape[1]
    t = mma_dtypes_t(CODE.get(A.dtype, 0), CODE.get(B.dtype, 0), CODE.get(C.dtype, 0))
    with torch.cuda.device(A.device):
        _check(load_library().mma_gemm_splitk_noalloc(_ptr(A), _ptr(B), _ptr(C), _ptr(D), M, N, K, t,
                                                      int(ksplit), _stream(stream)), "mma_gemm_splitk_noalloc")
    return D
