"""The measurement helpers for the tensor-core ceilings: the warp-level (mma.sync /
mma.sp) path and tcgen05.mma.  Each kind runs and reports a plausible, positive
rate, and a GEMM timed beside the tcgen05 ceiling stays below it."""
import math

import pytest
import torch

from tensor_core_matrix_02_gb300 import mma42
from tensor_core_matrix_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", list(mma42.LEGACY_KINDS))
def test_legacy_peak_measures(kind):
    ops = mma42.mma_legacy_mma_peak(kind)
    assert mma42.mma_sync_status() == 0
    assert math.isfinite(ops) and 1e12 < ops < 1e17, ops


@pytest.mark.parametrize("kind", list(mma42.TCGEN05_KINDS))
def test_tcgen05_peak_measures(kind):
    ops, per_clk = mma42.mma_tcgen05_peak(kind)
    assert mma42.mma_sync_status() == 0
    assert math.isfinite(ops) and 1e13 < ops < 1e17, ops
    # ops per SM clock: thousands for every kind (bf16 dense is the smallest)
    assert math.isfinite(per_clk) and 1e3 < per_clk < 1e6, per_clk


def test_sparse_ceiling_is_above_dense():
    """Per SM clock the 4:2 form does more logical work than the dense one."""
    _, dense = mma42.mma_tcgen05_peak("bf16")
    _, sparse = mma42.mma_tcgen05_peak("bf16_sparse")
    assert mma42.mma_sync_status() == 0
    assert sparse > 1.2 * dense, (dense, sparse)


def test_gemm_stays_below_the_tcgen05_ceiling():
    """A full bf16 GEMM cannot beat its tensor cores' ceiling: a rate far above it
    would mean the timed kernel is not doing the work."""
    p = W.make("dense_bf16_8192", device="cuda", M=4096, N=4096, K=4096)
    D = torch.empty_like(p.C)
    for _ in range(3):
        mma42.mma_gemm(p.A, p.B, p.C, D)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(5):
        mma42.mma_gemm(p.A, p.B, p.C, D)
    b.record()
    torch.cuda.synchronize()
    gemm = 5 * p.flops / (a.elapsed_time(b) * 1e-3)
    peak, _ = mma42.mma_tcgen05_peak("bf16")
    assert mma42.mma_sync_status() == 0
    assert 0 < gemm < 1.15 * peak, (gemm, peak)


@pytest.mark.parametrize("boxes,stages", [
    ([(128, 64), (8, 256), (64, 128), (64, 128)], 7),     # the 4:2 f16 kernel's stage
    ([(128, 128), (64, 128), (64, 128)], 6),              # the dense bf16 kernel's stage
    ([(128, 128)], 4),
])
def test_tma_feed_probe_measures(boxes, stages):
    """The TMA fill rate of a pipeline ring: positive, and below what one SM's
    shared memory could take in a clock (a rate far above it would mean the loads
    were not waited for)."""
    byts, rows = mma42.mma_tma_feed_probe(boxes, stages)
    assert mma42.mma_sync_status() == 0
    assert math.isfinite(byts) and 1.0 < byts < 1024.0, byts
    per_row = sum(r * b for r, b in boxes) / sum(r for r, _ in boxes)
    assert abs(rows * per_row - byts) <= 1e-6 * byts
