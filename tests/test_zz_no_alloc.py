"""mma_gemm_splitk_noalloc: the split-K GEMM whose partial sums live in a fixed
device array inside the library, for callers that may not allocate device
memory where they call it (memory owned by another framework's caching
allocator, latency-critical loops where cudaMalloc/cudaFree could wait on the
whole device, runtimes that forbid allocation after start-up).

The GPU test first fills the array with the partials of another, larger
problem (other inputs and shape), then calls the entry point through the C ABI
twice in a row and checks each result against the f64 oracle on the same
rounded inputs, within the tolerance of the other parity tests (and against
mma_gemm as a second check).  This file is collected last so that a run stopping at
its first failure has already run every other test; it also passes on its own
in a fresh process (the entry point's first call does the per-device set-up).
"""
import ctypes

import numpy as np
import pytest
import torch

from tensor_core_matrix_02_gb300 import build, mma42
from tensor_core_matrix_02_gb300 import workloads as W

from gpu_helpers import TOL, assert_matches, oracle_dense, rel_frobenius

MMA_OK, MMA_ERR_UNSUPPORTED, MMA_ERR_SHAPE = 0, 2, 3
F16, BF16, E4M3, I8, F32, I32 = 1, 2, 3, 5, 6, 7


def _call(lib, A, B, C, D, M, N, K, t, ksplit, stream=None):
    p = lambda x: ctypes.c_void_p(x) if isinstance(x, int) else ctypes.c_void_p(x.data_ptr())
    return lib.mma_gemm_splitk_noalloc(p(A), p(B), p(C), p(D), M, N, K, mma42.mma_dtypes_t(*t), ksplit, stream)


def test_noalloc_rejects_requests_beyond_its_limits():
    """Checked on the host before any CUDA call (made-up, never-touched addresses)."""
    build.build()
    lib = mma42.load_library()
    A, B, C, D = 0x10000000, 0x20000000, 0x30000000, 0x40000000
    t = (BF16, BF16, F32)
    assert _call(lib, A, B, C, D, 1024, 1024, 65536, t, 9) == MMA_ERR_SHAPE       # 9 * 4 MiB > 32 MiB
    assert _call(lib, A, B, C, D, 1024, 1024, 65536, t, 1) == MMA_ERR_SHAPE       # not a split
    assert _call(lib, A, B, C, D, 1024, 1024, 65536, t, 17) == MMA_ERR_SHAPE
    assert _call(lib, A, B, C, D, 256, 256, 128, t, 4) == MMA_ERR_SHAPE           # 2 K blocks < 4 slices
    assert _call(lib, A, B, C, D, 256, 256, 4096, (I8, I8, I32), 4) == MMA_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("name,ta,tb,shape,ksplit", [
    ("dense_bf16_skinny", None, None, (1024, 1024, 65536), 8),   # the skinny workload: 8 slices = 32 MiB
    ("dense_bf16_skinny", "f16", "f16", (300, 520, 5000), 5),     # ragged in M, N and K
    ("dense_bf16_skinny", None, None, (200, 96, 3000), 3),        # at most 128 wide: 128-column blocks
    ("dense_e4m3_16384", None, "e5m2", (512, 768, 8192), 16),
])
def test_noalloc_matches_oracle_on_two_calls(oracle, name, ta, tb, shape, ksplit):
    build.build()
    lib = mma42.load_library()
    M, N, K = shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # leave other partials in the whole array first: a different problem whose
    # slices fill all 32 MiB, so stale values sit wherever this call's partials go
    q = W.make("dense_bf16_skinny", device="cuda", M=512, N=2048, K=4096, seed_offset=17)
    Dq = torch.empty((512, 2048), device="cuda")
    assert _call(lib, q.A, q.B, q.C, Dq, 512, 2048, 4096, (BF16, BF16, F32), 8, stream) == MMA_OK
    assert mma42.mma_sync_status() == MMA_OK
    p = W.make(name, device="cuda", M=M, N=N, K=K, ta=ta, tb=tb)
    ref = oracle_dense(oracle, p)
    via_gemm = mma42.mma_gemm(p.A, p.B, p.C)
    assert mma42.mma_sync_status() == MMA_OK
    via_gemm = via_gemm.cpu().numpy().astype(np.float64)
    t = (mma42.CODE[p.A.dtype], mma42.CODE[p.B.dtype], F32)
    for call in range(2):
        D = torch.full((M, N), float("nan"), device="cuda")
        assert _call(lib, p.A, p.B, p.C, D, M, N, K, t, ksplit, stream) == MMA_OK
        assert mma42.mma_sync_status() == MMA_OK
        assert_matches(D, ref, p.ta, f"call {call} against the oracle")
        err = rel_frobenius(D.cpu().numpy(), via_gemm)
        assert err <= TOL[p.ta], f"call {call}: relative Frobenius error {err:.3e} against mma_gemm"
