"""The float parity checks themselves (tests/gpu_helpers.py), on the CPU.

A plain f32 product (numpy, products exact, sums rounded in f32) must pass every
check against the oracle; results with a planted mistake that the whole-matrix
relative Frobenius bound lets through must fail the per-tile or the per-element
check: one 32 x 32 tile that skipped one of its 64 K stages (within the FP8
tolerance over the whole matrix), and one element with a product counted twice.
"""
import numpy as np
import pytest

from tensor_core_matrix_02_gb300 import workloads as W

from gpu_helpers import TOL, assert_matches, oracle_dense, rel_frobenius


def f32_product(p: W.Problem, k0=0, k1=None) -> np.ndarray:
    """C + A[:, k0:k1] B[k0:k1] with f32 sums (the inputs are exact in f32)."""
    A = p.A.float().numpy()[:, k0:k1]
    B = p.B.float().numpy()[k0:k1]
    return (A @ B + (p.C.numpy() if k0 == 0 else 0)).astype(np.float32)


def torch_of(x: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x))


@pytest.mark.parametrize("name,ta,tb", [("dense_bf16_8192", None, None), ("dense_e4m3_16384", None, "e5m2")])
def test_f32_product_passes_every_check(oracle, name, ta, tb):
    p = W.make(name, M=96, N=160, K=2048, ta=ta, tb=tb)
    assert_matches(torch_of(f32_product(p)), oracle_dense(oracle, p), p.ta, "f32 product")


def test_one_tile_missing_one_k_stage_fails_the_tile_check(oracle):
    """FP8, K = 64 stages of 128: the whole-matrix error stays under 2e-2."""
    p = W.make("dense_e4m3_16384", M=640, N=512, K=64 * 128, tb="e5m2")
    ref = oracle_dense(oracle, p)
    got = f32_product(p)
    stage = f32_product(p, 5 * 128, 6 * 128)
    got[64:96, 32:64] -= stage[64:96, 32:64]          # tile (2, 1) without stage 5
    assert rel_frobenius(got.astype(np.float64), np.asarray(ref)) <= TOL["e4m3"]
    with pytest.raises(AssertionError, match="tile"):
        assert_matches(torch_of(got), ref, p.ta, "planted")


def test_one_element_off_fails_the_element_check(oracle):
    """One product counted twice in one element (its first term above 1/4)."""
    p = W.make("dense_bf16_8192", M=128, N=128, K=512)
    ref = oracle_dense(oracle, p)
    got = f32_product(p)
    terms = p.A[77].double().numpy() * p.B[:, 13].double().numpy()
    got[77, 13] += terms[np.argmax(np.abs(terms) > 0.25)]
    assert rel_frobenius(got.astype(np.float64), np.asarray(ref)) <= TOL["bf16"]
    with pytest.raises(AssertionError, match="element"):
        assert_matches(torch_of(got), ref, p.ta, "planted")
