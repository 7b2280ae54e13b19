"""GPU parity at sizes where element offsets pass 2^31 (and byte offsets 2^32):
every kernel on the path must index its operands in 64 bits.

- Dense: C and D of 65576 x 33040 (2.17e9 elements; 8.7 GB each as f32 / i32),
  both the CTA-pair and the one-SM kernels, f32, i32 and f16 results.
- 4:2 sparse: A of 65552 x 32896 (2.16e9 elements) through compression, the index
  layout pass and the sparse GEMM, for f16, E4M3 x E5M2 and i8.
- Quantisation and the fused quantise-prune pass over 2.16e9 f32 values.

Inputs are drawn on the device by the seeded workload generators.  Sampled rows,
the first and last and those on either side of the 2^31-element and 2^31- and
2^32-byte boundaries, are recomputed by the oracle.
"""
import numpy as np
import pytest
import torch

from tensor_core_matrix_02_gb300 import mma42
from tensor_core_matrix_02_gb300 import workloads as W

from gpu_helpers import assert_half_close, assert_matches, half_reference, poisoned_like, ref_dense, ref_sparse

pytestmark = pytest.mark.gpu

DM, DN, DK = 65536 + 40, 32768 + 272, 80          # dense: M x N > 2^31
SM, SN, SK = 65536 + 16, 256 + 16, 32768 + 128     # sparse: M x K > 2^31


def boundary_rows(M, row_elems, elem_bytes, seed):
    """Rows on either side of element offset 2^31 and byte offsets 2^31 and 2^32 of
    an M x row_elems row-major array, the first and last rows and a few random ones."""
    rows = {0, M - 1, M - 2}
    for limit, unit in ((1 << 31, 1), (1 << 31, elem_bytes), (1 << 32, elem_bytes)):
        r = limit // (row_elems * unit)
        rows |= {r - 1, r, r + 1}
    rng = np.random.default_rng(seed)
    rows |= set(rng.integers(0, M, size=4).tolist())
    return sorted(r for r in rows if 0 <= r < M)


@pytest.fixture(autouse=True)
def _release_device_memory():
    """Each test holds up to ~20 GB; give it back to the device before the next one."""
    import gc
    torch.cuda.empty_cache()
    yield
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("kind", ["bf16", "i8"])
def test_dense_output_past_2_31_elements(oracle, monkeypatch, kind, kernel):
    monkeypatch.setenv("MMA42_DENSE_KERNEL", kernel)
    name = {"bf16": "dense_bf16_8192", "i8": "dense_i8_4096"}[kind]
    p = W.make(name, device="cuda", M=DM, N=DN, K=DK)
    assert p.M * p.N > (1 << 31)
    D = poisoned_like(p.C)
    mma42.mma_gemm(p.A, p.B, p.C, D)
    assert mma42.mma_sync_status() == 0
    rows = boundary_rows(DM, DN, 4, seed=DM)
    sel = torch.tensor(rows, device="cuda")
    ref = ref_dense(oracle, W.bits(p.A[sel].cpu()), p.ta, W.bits(p.B.cpu()), p.tb, p.C[sel].cpu().numpy())
    assert_matches(D[sel], ref, p.ta, f"{kind} {kernel} {DM}x{DN}x{DK} rows {rows}", tile=(1, 32))


def test_dense_half_output_past_2_31_elements(oracle):
    """f16 C and D of 2.17e9 elements (4.3 GB each): byte offsets pass 2^32."""
    p = W.make("dense_f16_128", device="cuda", M=DM, N=DN, K=DK)
    C = p.C.to(torch.float16)
    p.C = None
    torch.cuda.empty_cache()
    D = torch.full_like(C, float("nan"))
    mma42.mma_gemm(p.A, p.B, C, D)
    assert mma42.mma_sync_status() == 0
    rows = boundary_rows(DM, DN, 2, seed=DN)
    sel = torch.tensor(rows, device="cuda")
    rp = W.Problem(p.name, len(rows), p.N, p.K, p.ta, p.tb, "f16", p.A[sel], p.B, None, None, None)
    assert_half_close(D[sel], half_reference(oracle, rp, C[sel], "f16"), f"f16 out rows {rows}", tile=(1, 32))


SPARSE = {"f16": ("sparse_f16_random", None, None), "e4m3xe5m2": ("sparse_e4m3_e5m2", None, None),
          "i8": ("sparse_i8_8192", None, None)}


@pytest.mark.parametrize("kind", list(SPARSE))
def test_sparse_operand_past_2_31_elements(oracle, kind):
    name, ta, tb = SPARSE[kind]
    p = W.make(name, device="cuda", M=SM, N=SN, K=SK, ta=ta, tb=tb)
    assert p.M * p.K > (1 << 31)
    p.pairs = None
    torch.cuda.empty_cache()
    vals, idx = mma42.sparse42_compress(p.A)
    D = poisoned_like(p.C)
    mma42.sparse42_gemm(vals, idx, p.B, p.C, D)
    assert mma42.mma_sync_status() == 0
    rows = boundary_rows(SM, SK, p.A.element_size(), seed=SK)
    sel = torch.tensor(rows, device="cuda")
    ov, oi, viol = oracle.compress(W.bits(p.A[sel].cpu()), p.ta)
    assert viol == 0
    assert np.array_equal(W.bits(vals[sel].cpu()), ov), f"{kind}: compressed values differ on rows {rows}"
    assert np.array_equal(idx[sel].cpu().numpy(), oi), f"{kind}: index differs on rows {rows}"
    ref = ref_sparse(oracle, ov, oi, p.ta, W.bits(p.B.cpu()), p.tb, p.C[sel].cpu().numpy(), SK)
    assert_matches(D[sel], ref, p.ta, f"{kind} sparse {SM}x{SN}x{SK} rows {rows}", tile=(1, 32))
    # pruning a 4:2 matrix keeps exactly its non-zeros: the same compressed form
    pv, pi = mma42.sparse42_prune(p.A)
    assert mma42.mma_sync_status() == 0
    assert np.array_equal(W.bits(pv[sel].cpu()), ov)
    assert np.array_equal(pi[sel].cpu().numpy(), oi)


@pytest.mark.parametrize("t", ["f16", "e4m3"])
def test_quantize_and_quantize_prune_past_2_31_elements(oracle, t):
    """f32 -> t over 2.16e9 values (8.6 GB in), and the fused quantise-prune pass,
    on values spread so that E4M3 saturates."""
    g = torch.Generator(device="cuda")
    g.manual_seed(SM + SK)
    x = torch.randn((SM, SK), generator=g, device="cuda", dtype=torch.float32) * 300.0
    y = mma42.mma_quantize(x, W.TORCH_DTYPE[t])
    vals, idx = mma42.sparse42_quantize_prune(x, W.TORCH_DTYPE[t])
    assert mma42.mma_sync_status() == 0
    rows = boundary_rows(SM, SK, 4, seed=SM)
    sel = torch.tensor(rows, device="cuda")
    xr = x[sel].cpu().numpy()
    q = oracle.quantize(xr, t)
    assert np.array_equal(W.bits(y[sel].cpu()), q), f"{t}: quantised rows {rows} differ"
    ov, oi, _ = oracle.prune(q, t)
    assert np.array_equal(W.bits(vals[sel].cpu()), ov), f"{t}: pruned values differ on rows {rows}"
    assert np.array_equal(idx[sel].cpu().numpy(), oi), f"{t}: pruned index differs on rows {rows}"
