"""GPU parity of the CTA-pair kernel's tail split: when the output blocks take
more than one round of the SM pairs and the last round would leave most pairs
idle, the blocks of that round are cut into K slices whose partials a separate
reduction sums (in slice order, then C).

Forced splits (every block a tail block) run every pair-kernel variant at ragged
shapes against the oracle; a 4096 x 4096 output (256 blocks over the SM pairs,
a short last round) checks the planner's own choice on sampled rows that cover
the tail blocks.
"""
import numpy as np
import pytest
import torch

from tensor_core_matrix_02_gb300 import mma42
from tensor_core_matrix_02_gb300 import workloads as W

from gpu_helpers import assert_half_close, assert_matches, gpu_dense, half_reference, oracle_dense, rel_frobenius

pytestmark = pytest.mark.gpu

KINDS = {
    "f16": ("dense_f16_128", None, None),
    "bf16": ("dense_bf16_8192", None, None),
    "e4m3xe5m2": ("dense_e4m3_16384", None, "e5m2"),
    "i8": ("dense_i8_4096", None, None),
    "u8": ("dense_i8_4096", "u8", "u8"),
    "u8xi8": ("dense_i8_4096", "u8", None),
}


@pytest.fixture
def pair(monkeypatch):
    monkeypatch.setenv("MMA42_DENSE_KERNEL", "pair")
    return monkeypatch


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("s", ["2", "3"])
@pytest.mark.parametrize("M,N,K", [(300, 528, 1040), (256, 256, 4096)])
def test_forced_tail_split_matches_oracle(oracle, pair, kind, s, M, N, K):
    pair.setenv("MMA42_TAIL_SPLIT", s)
    name, ta, tb = KINDS[kind]
    p = W.make(name, M=M, N=N, K=K, ta=ta, tb=tb)
    n0 = mma42.mma_launch_count()
    D = gpu_dense(p)
    launches = mma42.mma_launch_count() - n0
    assert_matches(D, oracle_dense(oracle, p), p.ta, f"{kind} tail split {s} {M}x{N}x{K}")
    pair.setenv("MMA42_TAIL_SPLIT", "0")
    pair.setenv("MMA42_KSPLIT", "1")
    n0 = mma42.mma_launch_count()
    gpu_dense(p)
    assert launches == mma42.mma_launch_count() - n0 + 1, "the tail reduction must have run"


@pytest.mark.parametrize("kind", ["f16", "bf16"])
def test_forced_tail_split_half_outputs(oracle, pair, kind):
    """f16 / bf16 C and D: f32 partials summed in slice order, plus C, rounded once."""
    pair.setenv("MMA42_TAIL_SPLIT", "2")
    p = W.make(KINDS[kind][0], M=300, N=272, K=1040)
    C = p.C.to(W.TORCH_DTYPE[kind])
    D = mma42.mma_gemm(p.A.cuda(), p.B.cuda(), C.cuda(), torch.full_like(C.cuda(), float("nan")))
    assert mma42.mma_sync_status() == 0
    assert_half_close(D, half_reference(oracle, p, C, kind), f"{kind} out, tail split")


def test_tail_split_is_deterministic(pair):
    """The reduction's order is fixed: two runs give the same bits."""
    pair.setenv("MMA42_TAIL_SPLIT", "3")
    p = W.make("dense_bf16_8192", M=300, N=528, K=2080)
    assert torch.equal(gpu_dense(p), gpu_dense(p))


def test_forced_tail_split_clamp_is_unaffected(pair):
    """Clamping keeps its own K slices (each slice's sum must fit i32): the tail
    split stays off and saturation stays exact."""
    pair.setenv("MMA42_TAIL_SPLIT", "2")
    M, N, K = 64, 128, 4096 + 16
    A = torch.full((M, K), -128, dtype=torch.int8, device="cuda")
    B = torch.full((K, N), -128, dtype=torch.int8, device="cuda")
    C = torch.full((M, N), (1 << 31) - 1000, dtype=torch.int32, device="cuda")
    D = mma42.mma_gemm(A, B, C, clamp=True)
    assert mma42.mma_sync_status() == 0
    assert (D.cpu() == (1 << 31) - 1).all()


# rows 2048.. hold the raster's last blocks; every 16th row of the lower half, and a
# few of the upper half for the whole blocks
SAMPLE_ROWS = np.concatenate([np.arange(0, 2048, 256), np.arange(2048, 4096, 16)])


@pytest.mark.parametrize("kind", ["bf16", "i8"])
def test_planned_tail_split_at_4096(oracle, monkeypatch, kind):
    """256 blocks of 256 x 256 over the SM pairs: the planner splits the short last
    round (one more launch, the reduction); the sampled rows match the oracle, and
    the result without the split matches too (bit for bit for i8)."""
    name, ta, tb = KINDS[kind]
    p = W.make(name, M=4096, N=4096, K=1024, ta=ta, tb=tb)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    n0 = mma42.mma_launch_count()
    D = mma42.mma_gemm(A, B, C)
    with_split = mma42.mma_launch_count() - n0
    assert mma42.mma_sync_status() == 0
    ref = oracle_dense(oracle, p, rows=SAMPLE_ROWS)
    assert_matches(D[torch.from_numpy(SAMPLE_ROWS).cuda()], ref, p.ta, f"{kind} 4096 planned")
    monkeypatch.setenv("MMA42_TAIL_SPLIT", "0")
    n0 = mma42.mma_launch_count()
    D0 = mma42.mma_gemm(A, B, C)
    without = mma42.mma_launch_count() - n0
    assert with_split == without + 1, "the planner should split the last round of 256 blocks"
    if kind == "i8":
        assert torch.equal(D.cpu(), D0.cpu())
    else:
        assert_matches(D0[torch.from_numpy(SAMPLE_ROWS).cuda()], ref, p.ta, f"{kind} 4096 unsplit")
