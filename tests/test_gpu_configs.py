"""GPU parity at the workloads' full sizes, through the same calls the
benchmark times: sampled output rows (first, last and seeded random ones) are
recomputed by the oracle, and the sampled rows of the 4:2 compression must be
bit-identical to the oracle's.  Floating-point rows are checked as a whole, per
32-column run and per element (the f32 accumulation bound).
"""
import numpy as np
import pytest
import torch

from tensor_core_matrix_02_gb300 import mma42
from tensor_core_matrix_02_gb300 import workloads as W

from gpu_helpers import assert_matches, poisoned_like, ref_dense, ref_sparse

pytestmark = pytest.mark.gpu

SUITE = ["dense_f16_128", "dense_i8_4096", "dense_bf16_8192", "dense_bf16_skinny", "sparse_f16_keep02", "sparse_bf16_8192", "sparse_i8_8192", "prune_f16_8192",
         "sparse_f16_random", "sparse_e4m3_e5m2", "dense_e4m3_16384"]


def sample_rows(M, n=6, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, M - 1} | set(rng.integers(0, M, size=n).tolist())
    return sorted(rows)


@pytest.mark.parametrize("name", SUITE)
def test_full_size_workload_sampled_rows(oracle, name):
    torch.cuda.empty_cache()
    p = W.make(name, device="cuda")
    D = poisoned_like(p.C)
    if p.sparse:
        prune = p.sparse == "prune"
        vals, idx = mma42.sparse42_prune(p.A) if prune else mma42.sparse42_compress(p.A)
        mma42.sparse42_gemm(vals, idx, p.B, p.C, D)
    else:
        mma42.mma_gemm(p.A, p.B, p.C, D)
    assert mma42.mma_sync_status() == 0
    rows = sample_rows(p.M)
    A_rows = p.A[rows].cpu()
    B = W.bits(p.B.cpu())
    C_rows = p.C[rows].cpu().numpy()
    if p.sparse:
        ov, oi, viol = (oracle.prune if p.sparse == "prune" else oracle.compress)(W.bits(A_rows), p.ta)
        assert np.array_equal(W.bits(vals[rows].cpu()), ov)
        assert np.array_equal(idx[rows].cpu().numpy(), oi)
        ref = ref_sparse(oracle, ov, oi, p.ta, B, p.tb, C_rows, p.K)
    else:
        ref = ref_dense(oracle, W.bits(A_rows), p.ta, B, p.tb, C_rows)
    # the sampled rows are not neighbours: tiles are 32-column runs of one row
    assert_matches(D[rows], ref, p.ta, f"{name} rows {rows}", tile=(1, 32))
    if p.sparse:
        del vals, idx
    del p, D
    torch.cuda.empty_cache()
