"""A pipeline wait that runs out is reported, and the context stays usable.

The test hook mma_debug_inject(1) makes the next one-SM dense launch arm its
first pipeline stage without issuing that stage's loads; mma_debug_inject(2)
makes the next CTA-pair launch (dense or 4:2-sparse) arm its first cluster's
first stage for 16 bytes more than its loads bring, every load still issued and
landing; mma_debug_inject(3) does the same to the short-K kernel's first k-block.
Either way the MMA thread's bounded wait on that stage runs out.
Nothing faults or hangs: the kernel records MMA_ERR_TIMEOUT in the device error
word, the roles of the CTA (and, in a pair, the peer CTA's own bounded waits)
stop, issued copies are drained, TMEM is freed and the kernel returns.  The
next call on the same context must be correct.
"""
import numpy as np
import pytest

from tensor_core_matrix_02_gb300 import mma42
from tensor_core_matrix_02_gb300 import workloads as W

from gpu_helpers import assert_matches, gpu_dense, oracle_dense, ref_sparse

pytestmark = pytest.mark.gpu

MMA_ERR_TIMEOUT = 6


def test_wait_timeout_reported_then_next_call_correct(oracle):
    lib = mma42.load_library()
    p = W.make("dense_bf16_8192", M=256, N=512, K=512)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    assert mma42.mma_sync_status() == 0
    lib.mma_set_wait_limit_ns(50_000_000)          # 50 ms
    try:
        lib.mma_debug_inject(1)
        mma42.mma_gemm(A, B, C)
        status = mma42.mma_sync_status()
    finally:
        lib.mma_set_wait_limit_ns(2_000_000_000)
        lib.mma_debug_inject(0)
    assert status == MMA_ERR_TIMEOUT
    assert mma42.mma_sync_status() == 0           # the status was cleared
    D = gpu_dense(p)
    assert_matches(D, oracle_dense(oracle, p), "bf16", "after timeout")


def _timeout_then(lib, call, mode=2):
    assert mma42.mma_sync_status() == 0
    lib.mma_set_wait_limit_ns(50_000_000)          # 50 ms
    try:
        lib.mma_debug_inject(mode)
        call()
        status = mma42.mma_sync_status()
    finally:
        lib.mma_set_wait_limit_ns(2_000_000_000)
        lib.mma_debug_inject(0)
    assert status == MMA_ERR_TIMEOUT
    assert mma42.mma_sync_status() == 0


@pytest.mark.parametrize("name", ["dense_bf16_8192", "dense_e4m3_16384", "dense_i8_4096"])
def test_pair_kernel_wait_timeout_then_next_call_correct(oracle, monkeypatch, name):
    monkeypatch.setenv("MMA42_DENSE_KERNEL", "pair")
    lib = mma42.load_library()
    p = W.make(name, M=1024, N=768, K=1024)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    _timeout_then(lib, lambda: mma42.mma_gemm(A, B, C))
    assert_matches(gpu_dense(p), oracle_dense(oracle, p), p.ta, f"{name} pair kernel after timeout")


@pytest.mark.parametrize("name", ["sparse_f16_random", "sparse_e4m3_e5m2", "sparse_i8_8192"])
def test_sparse_kernel_wait_timeout_then_next_call_correct(oracle, name):
    lib = mma42.load_library()
    p = W.make(name, M=512, N=768, K=1024)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    vals, idx = mma42.sparse42_compress(A)
    _timeout_then(lib, lambda: mma42.sparse42_gemm(vals, idx, B, C))
    D = mma42.sparse42_gemm(vals, idx, B, C)
    assert mma42.mma_sync_status() == 0
    ov, oi, _ = oracle.compress(W.bits(p.A), p.ta)
    ref = ref_sparse(oracle, ov, oi, p.ta, W.bits(p.B), p.tb, p.C.numpy(), p.K)
    assert_matches(D, ref, p.ta, f"{name} after timeout")


@pytest.mark.parametrize("name,bn", [("dense_f16_128", "64"), ("dense_f16_128", "128"), ("dense_e4m3_16384", "128")])
def test_small_kernel_wait_timeout_then_next_call_correct(oracle, monkeypatch, name, bn):
    """The short-K kernel's first block gives up on its first k-block; the block's
    issued loads land before it exits, and the next call is correct."""
    monkeypatch.setenv("MMA42_DENSE_KERNEL", "small")
    monkeypatch.setenv("MMA42_SMALL_BN", bn)
    lib = mma42.load_library()
    p = W.make(name, M=256, N=384, K=256)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    _timeout_then(lib, lambda: mma42.mma_gemm(A, B, C), mode=3)
    assert_matches(gpu_dense(p), oracle_dense(oracle, p), p.ta, f"{name} short-K kernel after timeout")
