"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
(via the thin binding) and the oracle on the same inputs, and compare."""
import numpy as np
import torch

from tensor_core_matrix_02_gb300 import mma42
from tensor_core_matrix_02_gb300 import workloads as W

# tolerance on the relative Frobenius error against the f64 oracle
TOL = {"f16": 1e-3, "bf16": 1e-3, "e4m3": 2e-2, "e5m2": 2e-2}


def rel_frobenius(got: np.ndarray, ref: np.ndarray) -> float:
    got = got.astype(np.float64)
    num = np.linalg.norm(got - ref)
    den = np.linalg.norm(ref)
    return float(num / den) if den > 0 else float(num)


def wrap_i32(x: np.ndarray) -> np.ndarray:
    return ((x.astype(np.int64) + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int64)


# Per-element bound of a float result accumulated in f32.  The products of two
# 16-bit or two 8-bit floating inputs are exact in f32, so every difference from
# the exact sum comes from f32 additions.  Each tensor-core instruction adds a group
# of g products to the accumulator; modelled as g + 1 additions that each truncate
# to 24 bits (relative error 2^-23 of the running magnitude), K products in
# instructions of g >= 1 cost at most 2K additions, and the split-K partial sums,
# their reduction and the final + C at most K more.  That gives
#     |D - D_exact| <= 3 K 2^-23 (|C| + sum_k |a_ik b_kj|)  <  ELEM_C K 2^-24 (...)
# with ELEM_C = 8 (the standard forward bound of a recursive sum, Higham,
# "Accuracy and Stability of Numerical Algorithms", section 3.1, with the unit
# roundoff of truncation).  The magnitude |C| + sum |a||b| is the oracle run on
# |A|, |B| and |C|.
ELEM_C = 8
U_F32 = 2.0 ** -24


class Ref(np.ndarray):
    """An oracle result; ``mag`` (optional) is |C| + sum_k |a_ik b_kj| for each
    element and ``k`` the logical K, which give the per-element bound."""
    mag = None
    k = None


def with_mag(ref: np.ndarray, mag: np.ndarray, k: int) -> Ref:
    r = np.asarray(ref).view(Ref)
    r.mag = np.asarray(mag, dtype=np.float64)
    r.k = int(k)
    return r


def abs_bits(bits: np.ndarray, t: str) -> np.ndarray:
    """|x| of floating-point bit patterns: the sign bit cleared."""
    return bits & (0x7FFF if bits.dtype == np.uint16 else 0x7F)


def ref_dense(oracle, a_bits, ta: str, b_bits, tb: str, C: np.ndarray, rows=None):
    """The oracle's D = A*B + C, with its magnitude for floating-point types."""
    ref = oracle.gemm(a_bits, ta, b_bits, tb, C, rows=rows)
    if ta in ("i8", "u8"):
        return ref
    mag = oracle.gemm(abs_bits(a_bits, ta), ta, abs_bits(b_bits, tb), tb, np.abs(C), rows=rows)
    return with_mag(ref, mag, a_bits.shape[1])


def ref_sparse(oracle, v_bits, idx, ta: str, b_bits, tb: str, C: np.ndarray, K: int):
    """The oracle's sparse product from (vals, idx), with its magnitude."""
    ref = oracle.sparse_gemm(v_bits, idx, ta, b_bits, tb, C, K)
    if ta in ("i8", "u8"):
        return ref
    mag = oracle.sparse_gemm(abs_bits(v_bits, ta), idx, ta, abs_bits(b_bits, tb), tb, np.abs(C), K)
    return with_mag(ref, mag, K)


def tile_errors(got: np.ndarray, ref: np.ndarray, tile=(32, 32)) -> np.ndarray:
    """Relative Frobenius error of every tile (th x tw, the last ones ragged).  A
    tile whose reference norm is below 1e-3 of the root-mean-square tile norm is
    measured against that floor instead."""
    th, tw = tile
    M, N = ref.shape
    num, den = [], []
    for i in range(0, M, th):
        for j in range(0, N, tw):
            r = ref[i:i + th, j:j + tw]
            num.append(np.linalg.norm(got[i:i + th, j:j + tw] - r))
            den.append(np.linalg.norm(r))
    num, den = np.array(num), np.array(den)
    floor = 1e-3 * np.sqrt(np.mean(den ** 2)) if den.size else 0.0
    return num / np.maximum(den, max(floor, np.finfo(np.float64).tiny))


def assert_matches(got: torch.Tensor, ref: np.ndarray, ta: str, what: str = "", tile=(32, 32)):
    """Integers: bit-exact (wrapping i32).  Floating point: the relative Frobenius
    error of the whole result and of every tile within the tolerance, and, when the
    reference carries its magnitude, every element within the f32 accumulation
    bound above.  Returns the whole-result error."""
    g = got.cpu()
    if ta in ("i8", "u8"):
        assert np.array_equal(g.numpy().astype(np.int64), wrap_i32(ref)), f"{what}: integer result not bit-exact"
        return
    gn = g.numpy().astype(np.float64)
    refv = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(gn).all(), f"{what}: non-finite output"
    err = rel_frobenius(gn, refv)
    assert err <= TOL[ta], f"{what}: relative Frobenius error {err:.3e} > {TOL[ta]:.0e}"
    te = tile_errors(gn, refv, tile)
    if te.size:
        worst = int(np.argmax(te))
        assert te[worst] <= TOL[ta], (f"{what}: tile {worst} ({tile[0]}x{tile[1]} tiles, row-major) relative "
                                      f"Frobenius error {te[worst]:.3e} > {TOL[ta]:.0e}")
    mag = getattr(ref, "mag", None)
    if mag is not None:
        bound = ELEM_C * ref.k * U_F32 * mag + np.finfo(np.float32).tiny
        ratio = np.abs(gn - refv) / bound
        worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
        assert ratio[worst] <= 1.0, (f"{what}: element {tuple(int(x) for x in worst)} differs by "
                                     f"{abs(gn[worst] - refv[worst]):.3e}, above the accumulation bound "
                                     f"{bound[worst]:.3e} (K = {ref.k})")
    return err


def poisoned_like(C: torch.Tensor) -> torch.Tensor:
    D = torch.empty_like(C)
    if D.dtype == torch.float32:
        D.fill_(float("nan"))
    else:
        D.fill_(-0x21524111)          # 0xDEADBEEF as i32
    return D


def gpu_dense(p: W.Problem) -> torch.Tensor:
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    D = poisoned_like(C)
    mma42.mma_gemm(A, B, C, D)
    assert mma42.mma_sync_status() == 0
    return D


def oracle_dense(oracle, p: W.Problem, rows=None) -> np.ndarray:
    return ref_dense(oracle, W.bits(p.A.cpu()), p.ta, W.bits(p.B.cpu()), p.tb, p.C.cpu().numpy(), rows=rows)


# Half-precision C and D: the f64 oracle's result rounded to the output type by the
# oracle's quantisation.  Both sides round once, so an element may differ by the
# two roundings (unit roundoff 2^-11 for f16, 2^-8 for bf16, relative to the
# value) on top of the f32 accumulation bound; 2^-24 covers f16's subnormal step.
U_HALF = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def half_reference(oracle, p: W.Problem, C: torch.Tensor, kind: str, rows=None) -> Ref:
    """The oracle's D = A*B + C (C of the half type) rounded to ``kind``, with the
    magnitude |C| + sum |a||b| of every element."""
    a_bits, b_bits = W.bits(p.A.cpu()), W.bits(p.B.cpu())
    Cf = C.cpu().to(torch.float32).numpy()
    exact = ref_dense(oracle, a_bits, p.ta, b_bits, p.tb, Cf, rows=rows)
    q = oracle.quantize(np.asarray(exact).astype(np.float32), kind)
    want = torch.from_numpy(q.view(np.int16)).view(W.TORCH_DTYPE[kind]).to(torch.float64).numpy()
    r = with_mag(want, exact.mag, exact.k)
    r.kind = kind
    return r


def assert_half_close(D: torch.Tensor, want: Ref, what: str, tile=(32, 32)):
    """Relative Frobenius error of the whole result and of every tile <= 1e-3, and
    every element within the two roundings plus the accumulation bound."""
    got = D.cpu().to(torch.float64).numpy()
    wv = np.asarray(want, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = rel_frobenius(got, wv)
    assert err <= 1e-3, f"{what}: relative Frobenius error {err:.3e}"
    te = tile_errors(got, wv, tile)
    if te.size:
        assert te.max() <= 1e-3, f"{what}: tile {int(np.argmax(te))} relative Frobenius error {te.max():.3e}"
    acc = ELEM_C * want.k * U_F32 * want.mag
    bound = 2 * U_HALF[want.kind] * (np.abs(wv) + acc) + acc + 2.0 ** -24
    ratio = np.abs(got - wv) / bound
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    assert ratio[worst] <= 1.0, (f"{what}: element {tuple(int(x) for x in worst)} differs by "
                                 f"{abs(got[worst] - wv[worst]):.3e}, above {bound[worst]:.3e}")
