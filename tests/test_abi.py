"""The C-ABI library builds, loads, exports what include/mma42.h declares, and
rejects bad arguments on the host before touching the GPU (runs without one).

The argument-check calls below pass made-up, never-dereferenced addresses: a
rejected call returns its status before any CUDA call.
"""
import ctypes
import os
import re

import pytest

from tensor_core_matrix_02_gb300 import build, mma42

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mma42.h")

OK, INVALID, UNSUPPORTED, SHAPE, ALIGN = 0, 1, 2, 3, 4
F16, BF16, E4M3, E5M2, I8, F32, I32 = 1, 2, 3, 4, 5, 6, 7


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mma42.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("mma_gemm", "sparse42_compress", "sparse42_gemm", "mma_sync_status", "mma_status_string"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in mma42.h but not exported"
    assert set(declared_functions()) == set(mma42.EXPORTS)


def test_library_has_no_runtime_dependency_beyond_libc(lib):
    # the CUDA runtime is linked statically; the driver is reached by entry point
    import subprocess
    out = subprocess.run(["ldd", mma42.library_path()], capture_output=True, text=True).stdout
    assert "libcudart" not in out and "liboracle" not in out


def test_abi_version_and_status_strings(lib):
    assert lib.mma_abi_version() == 5
    for code, name in mma42.STATUS.items():
        assert lib.mma_status_string(code).decode().startswith(name)
    assert b"unknown" in lib.mma_status_string(99)


def T(a, b, acc):
    return mma42.mma_dtypes_t(a, b, acc)


# made-up device addresses, 16-byte aligned and far apart
A, B, C, D, X = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def gemm(lib, a, b, c, d, M, N, K, t):
    return lib.mma_gemm(a, b, c, d, M, N, K, t, None)


@pytest.mark.parametrize("t", [T(F16, BF16, F32), T(F16, F16, I32), T(I8, I8, F32), T(F32, F32, F32),
                               T(BF16, BF16, I32), T(E4M3, F16, F32), T(0, 0, 0), T(I8, E4M3, I32),
                               T(F16, F16, BF16), T(BF16, BF16, F16), T(E4M3, E4M3, F16)])
def test_gemm_rejects_type_combinations(lib, t):
    assert gemm(lib, A, B, C, D, 128, 128, 128, t) == UNSUPPORTED


def test_gemm_rejects_bad_sizes_and_pointers(lib):
    t = T(F16, F16, F32)
    assert gemm(lib, A, B, C, D, -1, 128, 128, t) == INVALID
    assert gemm(lib, A, B, C, D, 128, 128, -5, t) == INVALID
    assert gemm(lib, A, B, C, D, 1 << 31, 128, 128, t) == SHAPE
    assert gemm(lib, None, B, C, D, 128, 128, 128, t) == INVALID
    assert gemm(lib, A, B, None, D, 128, 128, 128, t) == INVALID
    assert gemm(lib, A, B, C, None, 128, 128, 128, t) == INVALID


def test_gemm_empty_output_is_a_no_op(lib):
    # nothing to compute, nothing launched (works without a GPU)
    t = T(F16, F16, F32)
    assert gemm(lib, None, None, None, None, 0, 128, 128, t) == OK
    assert gemm(lib, None, None, None, None, 128, 0, 128, t) == OK


def test_gemm_rejects_misalignment(lib):
    t = T(F16, F16, F32)
    assert gemm(lib, A + 8, B, C, D, 128, 128, 128, t) == ALIGN
    assert gemm(lib, A, B, C + 4, D, 128, 128, 128, t) == ALIGN
    assert gemm(lib, A, B, C, D, 128, 128, 12, t) == ALIGN          # K*2 = 24 bytes per A row
    assert gemm(lib, A, B, C, D, 128, 12, 128, t) == ALIGN          # N*2 = 24 bytes per B row
    assert gemm(lib, A, B, C, D, 128, 16, 8, T(E4M3, E4M3, F32)) == ALIGN   # K = 8 fp8 bytes
    assert gemm(lib, A, B, C, D, 128, 8, 16, T(I8, I8, I32)) == ALIGN       # N = 8 i8 bytes


def test_gemm_rejects_overlap(lib):
    t = T(F16, F16, F32)
    M = N = K = 128
    assert gemm(lib, A, B, C, C + 16 * 4, M, N, K, t) == INVALID     # D partly over C
    assert gemm(lib, A, B, C, A, M, N, K, t) == INVALID              # D over A
    assert gemm(lib, A, B, C, B + 64, M, N, K, t) == INVALID         # D over B


def test_sparse_rejects_bad_arguments(lib):
    t = T(F16, F16, F32)
    s = lib.sparse42_gemm
    assert s(A, X, B, C, D, 128, 128, 64, t, None) == SHAPE           # K not a multiple of 128
    assert s(A, X, B, C, D, 128, 128, 128, T(F16, BF16, F32), None) == UNSUPPORTED
    assert s(A, X, B, C, D, 128, 128, 128, T(I8, I8, F32), None) == UNSUPPORTED
    assert s(A, None, B, C, D, 128, 128, 128, t, None) == INVALID
    assert s(A, X + 4, B, C, D, 128, 128, 128, t, None) == ALIGN
    assert s(A, X, B, C, X, 128, 128, 128, t, None) == INVALID        # D over idx
    assert s(None, None, None, None, None, 0, 128, 128, t, None) == OK


@pytest.mark.parametrize("entry", ["sparse42_compress", "sparse42_prune"])
def test_compress_rejects_bad_arguments(lib, entry):
    c = getattr(lib, entry)
    assert c(A, B, X, 128, 128, F32, None, None) == UNSUPPORTED
    assert c(A, B, X, 128, 48, F16, None, None) == SHAPE               # K not a multiple of 32
    assert c(A, B, X, -1, 128, F16, None, None) == INVALID
    assert c(None, B, X, 128, 128, F16, None, None) == INVALID
    assert c(A + 2, B, X, 128, 128, F16, None, None) == ALIGN
    assert c(A, A + 64, X, 128, 128, F16, None, None) == INVALID       # vals over A
    assert c(A, B, X, 128, 128, F16, X + 2, None) == ALIGN             # violation counter


def test_gemm_ex_flags(lib):
    g = lib.mma_gemm_ex
    t8 = T(I8, I8, I32)
    assert g(A, B, C, D, 128, 128, 128, t8, 2, None) == INVALID          # unknown flag
    assert g(A, B, C, D, 128, 128, 128, T(F16, F16, F32), 1, None) == UNSUPPORTED   # clamp is integer-only
    assert g(A, B, C, D, 0, 128, 128, t8, 1, None) == OK


def test_quantize_rejects_bad_arguments(lib):
    q = lib.mma_quantize
    assert q(A, B, 64, I8, None) == UNSUPPORTED
    assert q(A, B, 64, F32, None) == UNSUPPORTED
    assert q(A, B, -1, F16, None) == INVALID
    assert q(None, B, 64, F16, None) == INVALID
    assert q(A + 4, B, 64, F16, None) == ALIGN
    assert q(A, A + 64, 64, F16, None) == INVALID          # y over x
    assert q(None, None, 0, E4M3, None) == OK


def test_quantize_prune_rejects_bad_arguments(lib):
    q = lib.sparse42_quantize_prune
    assert q(A, B, X, 128, 128, I8, None, None) == UNSUPPORTED
    assert q(A, B, X, 128, 48, F16, None, None) == SHAPE
    assert q(A, B, X, -1, 128, F16, None, None) == INVALID
    assert q(A + 4, B, X, 128, 128, F16, None, None) == ALIGN
    assert q(A, A + 64, X, 128, 128, F16, None, None) == INVALID       # vals over A
    assert q(None, None, None, 0, 0, E4M3, None, None) == OK


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    a = torch.zeros(128, 128, dtype=torch.float16)
    with pytest.raises(ValueError):
        mma42.mma_gemm(a, a, a.float())


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        mma42.load_library(str(tmp_path / "libmma42.so"))


def test_legacy_peak_rejects_bad_arguments(lib):
    """Checked before any device work, so this runs without a GPU."""
    out = ctypes.c_double(0.0)
    assert lib.mma_legacy_mma_peak(4, ctypes.byref(out), None) == 1
    assert lib.mma_legacy_mma_peak(-1, ctypes.byref(out), None) == 1
    assert lib.mma_legacy_mma_peak(0, None, None) == 1


def test_tcgen05_peak_rejects_bad_arguments(lib):
    """Argument checks come before any device work: they run without a GPU."""
    out = ctypes.c_double(0.0)
    assert lib.mma_tcgen05_peak(4, ctypes.byref(out), None, None) == 1
    assert lib.mma_tcgen05_peak(-1, ctypes.byref(out), None, None) == 1
    assert lib.mma_tcgen05_peak(0, None, None, None) == 1


def test_feed_probe_rejects_bad_arguments(lib):
    """Checked on the host before any CUDA call."""
    out = ctypes.c_double(0.0)
    I4 = ctypes.c_int32 * 4
    ok_rows, ok_bytes = I4(128, 64, 0, 0), I4(64, 128, 0, 0)
    assert lib.mma_tma_feed_probe(0, ok_rows, ok_bytes, 4, 0, 64 << 20, ctypes.byref(out), None, None) == 1
    assert lib.mma_tma_feed_probe(5, ok_rows, ok_bytes, 4, 0, 64 << 20, ctypes.byref(out), None, None) == 1
    assert lib.mma_tma_feed_probe(2, I4(100, 64, 0, 0), ok_bytes, 4, 0, 64 << 20, ctypes.byref(out), None, None) == 1
    assert lib.mma_tma_feed_probe(2, I4(8, 64, 0, 0), ok_bytes, 4, 0, 64 << 20, ctypes.byref(out), None, None) == 1
    assert lib.mma_tma_feed_probe(2, ok_rows, I4(32, 128, 0, 0), 4, 0, 64 << 20, ctypes.byref(out), None, None) == 1
    assert lib.mma_tma_feed_probe(2, ok_rows, ok_bytes, 1, 0, 64 << 20, ctypes.byref(out), None, None) == 1
    assert lib.mma_tma_feed_probe(2, ok_rows, ok_bytes, 4, 0, 64 << 20, None, None, None) == 1
    assert lib.mma_tma_feed_probe(2, ok_rows, ok_bytes, 4, 0, 1 << 20, ctypes.byref(out), None, None) == 3
    assert lib.mma_tma_feed_probe(2, ok_rows, ok_bytes, 16, 0, 64 << 20, ctypes.byref(out), None, None) == 3
