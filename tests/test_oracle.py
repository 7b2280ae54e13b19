"""Pins for the CPU oracle: each check comes from something other than the oracle.

* decoders        -- every bit pattern against torch's own conversions
* dense GEMM      -- brute force in exact rational arithmetic on tiny shapes,
                     and closed forms (A = 0, A = I, all-ones)
* 4:2 index       -- the keep-{0,2} constants printed on the pages
                     (tests/golden/keep02_index.txt)
* compress        -- round trip, recovery of the generator's own pattern,
                     the padding / violation readings on hand-made groups
* sparse GEMM     -- brute force on the decompressed A in exact arithmetic,
                     and equality with the dense oracle on the decompressed A
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from tensor_core_matrix_02_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_values(t: torch.Tensor):
    """Exact values of a CPU tensor as Python floats/ints (torch's decoding)."""
    if t.dtype in (torch.int8, torch.int32):
        return t.to(torch.int64).tolist()
    return t.to(torch.float64).tolist()


def _exact_gemm(A, B, C):
    """Plain definition D = C + sum_k A[i][k] B[k][j] in exact rationals."""
    a, b, c = _torch_values(A), _torch_values(B), _torch_values(C)
    M, K, N = len(a), len(b), len(c[0]) if c else 0
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = Fraction(c[i][j])
            for k in range(K):
                s += Fraction(a[i][k]) * Fraction(b[k][j])
            row.append(s)
        out.append(row)
    return out


def _abs_sum(A, B, C):
    a = np.abs(np.array(_torch_values(A), dtype=np.float64)).reshape(A.shape)
    b = np.abs(np.array(_torch_values(B), dtype=np.float64)).reshape(B.shape)
    c = np.abs(np.array(_torch_values(C), dtype=np.float64)).reshape(C.shape)
    return c + a @ b


# ----------------------------------------------------------------- decoders

@pytest.mark.parametrize("t,bits_dtype,n", [("f16", torch.int16, 1 << 16), ("bf16", torch.int16, 1 << 16),
                                            ("e4m3", torch.uint8, 256), ("e5m2", torch.uint8, 256)])
def test_decoder_every_bit_pattern(oracle, t, bits_dtype, n):
    raw = torch.arange(n, dtype=torch.int64)
    if bits_dtype == torch.int16:
        raw = raw.to(torch.int32).to(torch.int16)        # wraps 0x8000.. to negative int16
    else:
        raw = raw.to(torch.uint8)
    ref = raw.view(W.TORCH_DTYPE[t]).to(torch.float64).numpy()
    got = oracle.decode(W.bits(raw.view(W.TORCH_DTYPE[t])), t)
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    assert (nan_ref == nan_got).all()
    assert np.array_equal(got[~nan_got], ref[~nan_ref])
    # signed zeros decode to signed zeros
    assert np.array_equal(np.signbit(got[~nan_got]), np.signbit(ref[~nan_ref]))


def test_decoder_format_landmarks(oracle):
    # largest finite values and NaN encodings of the OCP FP8 formats
    assert oracle.decode(np.array([0x7E], np.uint8), "e4m3")[0] == 448.0
    assert math.isnan(oracle.decode(np.array([0x7F], np.uint8), "e4m3")[0])
    assert oracle.decode(np.array([0x7B], np.uint8), "e5m2")[0] == 57344.0
    assert math.isinf(oracle.decode(np.array([0x7C], np.uint8), "e5m2")[0])
    assert oracle.decode(np.array([0x01], np.uint8), "e4m3")[0] == 2.0 ** -9
    assert oracle.decode(np.array([0x01], np.uint8), "e5m2")[0] == 2.0 ** -16
    assert oracle.decode(np.array([0x0001], np.uint16), "f16")[0] == 2.0 ** -24
    assert oracle.decode(np.array([0x3F80], np.uint16), "bf16")[0] == 1.0


# --------------------------------------------------------------- dense GEMM

TYPE_PAIRS = [("f16", "f16"), ("bf16", "bf16"), ("e4m3", "e4m3"), ("e4m3", "e5m2"),
              ("e5m2", "e4m3"), ("e5m2", "e5m2"), ("i8", "i8"), ("u8", "u8"), ("u8", "i8"), ("i8", "u8")]
INTS = ("i8", "u8")
SHAPES = [(1, 1, 1), (2, 3, 5), (3, 5, 2), (5, 2, 8), (8, 8, 16), (16, 5, 3)]


def _tiny(ta, tb, M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    tacc = "i32" if ta in INTS else "f32"
    dist = {"f16": "normal1", "bf16": "normal1", "e4m3": "normal05", "e5m2": "normal05", "i8": "int8", "u8": "int8"}
    A = W._draw(dist[ta], (M, K), ta, g, "cpu")
    B = W._draw(dist[tb], (K, N), tb, g, "cpu")
    C = W._draw("int20" if tacc == "i32" else "normal1", (M, N), tacc, g, "cpu")
    return A, B, C, tacc


@pytest.mark.parametrize("ta,tb", TYPE_PAIRS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_dense_against_exact_rationals(oracle, ta, tb, M, N, K):
    A, B, C, tacc = _tiny(ta, tb, M, N, K, seed=M * 100 + N * 10 + K)
    D = oracle.gemm(W.bits(A), ta, W.bits(B), tb, C.numpy())
    exact = _exact_gemm(A, B, C)
    if ta in INTS:
        assert D.dtype == np.int64
        assert D.tolist() == [[int(x) for x in row] for row in exact]
        return
    # f64 accumulation of K+1 terms: |error| <= (K+1) u sum|terms|, u = 2^-53
    bound = 2 * (K + 1) * 2.0 ** -53 * _abs_sum(A, B, C)
    err = np.array([[abs(Fraction(D[i][j]) - exact[i][j]) for j in range(N)] for i in range(M)],
                   dtype=np.float64)
    assert (err <= bound).all()


@pytest.mark.parametrize("ta,tb", TYPE_PAIRS)
def test_dense_zero_A_gives_C(oracle, ta, tb):
    M, N, K = 7, 9, 12
    _, B, C, tacc = _tiny(ta, tb, M, N, K, seed=7)
    A = torch.zeros((M, K), dtype=W.TORCH_DTYPE[ta])
    D = oracle.gemm(W.bits(A), ta, W.bits(B), tb, C.numpy())
    assert np.array_equal(D, C.numpy().astype(D.dtype))


@pytest.mark.parametrize("ta,tb", TYPE_PAIRS)
def test_dense_identity_A_gives_B_plus_C(oracle, ta, tb):
    M = K = 8
    N = 6
    _, B, C, tacc = _tiny(ta, tb, M, N, K, seed=11)
    A = torch.eye(K, dtype=torch.float32).to(W.TORCH_DTYPE[ta])
    D = oracle.gemm(W.bits(A), ta, W.bits(B), tb, C.numpy())
    want = np.array(_torch_values(B)) + np.array(_torch_values(C))   # exact here: few bits
    assert np.array_equal(D, want.astype(D.dtype))


@pytest.mark.parametrize("ta,tb", TYPE_PAIRS)
def test_dense_all_ones_gives_K_plus_C(oracle, ta, tb):
    M, N, K = 4, 5, 37
    _, _, C, tacc = _tiny(ta, tb, M, N, K, seed=3)
    A = torch.ones((M, K), dtype=torch.float32).to(W.TORCH_DTYPE[ta])
    B = torch.ones((K, N), dtype=torch.float32).to(W.TORCH_DTYPE[tb])
    D = oracle.gemm(W.bits(A), ta, W.bits(B), tb, C.numpy())
    want = np.array(_torch_values(C)) + K
    assert np.array_equal(D, want.astype(D.dtype))


def test_dense_row_selection_matches_full(oracle):
    p = W.make("dense_bf16_8192", M=33, N=24, K=40)
    full = oracle.gemm(W.bits(p.A), p.ta, W.bits(p.B), p.tb, p.C.numpy())
    rows = [32, 0, 17, 17]
    part = oracle.gemm(W.bits(p.A), p.ta, W.bits(p.B), p.tb, p.C.numpy(), rows=rows)
    assert np.array_equal(part, full[rows])


def test_dense_i8_extreme_values_exact(oracle):
    # (-128)(-128) summed: the largest magnitudes the i8 path can meet
    M, N, K = 3, 4, 1024
    A = torch.full((M, K), -128, dtype=torch.int8)
    B = torch.full((K, N), -128, dtype=torch.int8)
    C = torch.full((M, N), -(1 << 20), dtype=torch.int32)
    D = oracle.gemm(A.numpy(), "i8", B.numpy(), "i8", C.numpy())
    assert (D == K * 16384 - (1 << 20)).all()


@pytest.mark.parametrize("ta,va,tb,vb", [("u8", 255, "u8", 255), ("u8", 255, "i8", -128), ("i8", -128, "u8", 255),
                                         ("i8", -1, "u8", 1)])
def test_dense_8bit_signedness_closed_forms(oracle, ta, va, tb, vb):
    """Constant matrices: D = C + K * a * b, with each operand read as its own
    type ("RDNA3 dense WMMA builtins", section "Common parameters", a_neg/b_neg)."""
    M, N, K = 3, 4, 640
    A = torch.full((M, K), va, dtype=W.TORCH_DTYPE[ta])
    B = torch.full((K, N), vb, dtype=W.TORCH_DTYPE[tb])
    C = torch.full((M, N), 5, dtype=torch.int32)
    D = oracle.gemm(W.bits(A), ta, W.bits(B), tb, C.numpy())
    assert (D == 5 + K * va * vb).all()


# ------------------------------------------------------------------- 4:2 index

def _golden_index():
    rows = []
    with open(os.path.join(GOLDEN, "keep02_index.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                t, groups, value = line.split()
                rows.append((t, int(groups), int(value, 16)))
    return rows


@pytest.mark.parametrize("t,groups,value", _golden_index())
def test_keep02_index_matches_page_constants(oracle, t, groups, value):
    M, K = 3, 64
    p = W.make({"f16": "sparse_f16_keep02", "e4m3": "sparse_e4m3_e5m2",
                "e5m2": "sparse_e4m3_e5m2"}[t], M=M, N=8, K=K, sparse="keep02")
    A = p.A if p.ta == t else p.A.to(torch.float32).to(W.TORCH_DTYPE[t])
    A_bits = W.bits(A).copy()
    # make every kept element non-zero so the pattern is exactly keep {0,2}
    kept = np.zeros((M, K), bool)
    kept[:, 0::4] = kept[:, 2::4] = True
    one = W.bits(torch.ones(1).to(W.TORCH_DTYPE[t]))[0]
    A_bits[kept & (W.bits(A.to(torch.float32).abs().to(W.TORCH_DTYPE[t])) == 0)] = one
    vals, idx, viol = oracle.compress(A_bits, t)
    assert viol == 0
    # an index value covering `groups` groups is `groups` nibbles, lowest group first
    nbytes = groups // 2
    for r in range(M):
        for start in range(0, K // 8, nbytes):
            word = int.from_bytes(bytes(idx[r, start:start + nbytes]), "little")
            assert word == value
    # compressed A keeps positions 0 and 2 of every group, in order, half as long as K
    assert vals.shape == (M, K // 2)
    assert np.array_equal(vals[:, 0::2], A_bits[:, 0::4])
    assert np.array_equal(vals[:, 1::2], A_bits[:, 2::4])


# -------------------------------------------------------------- compress

@pytest.mark.parametrize("name", ["sparse_f16_keep02", "sparse_f16_random", "sparse_e4m3_e5m2"])
@pytest.mark.parametrize("M,K", [(1, 8), (5, 64), (33, 136)])
def test_compress_round_trip(oracle, name, M, K):
    p = W.make(name, M=M, N=8, K=K)
    A = W.bits(p.A)
    vals, idx, viol = oracle.compress(A, p.ta)
    assert viol == 0
    back = oracle.decompress(vals, idx, p.ta, K)
    assert np.array_equal(oracle.decode(back, p.ta), oracle.decode(A, p.ta))
    # the two kept positions of each group carry the generator's pattern
    # wherever the generator's kept values are both non-zero
    pos = np.array(W.PAIRS)[p.pairs.numpy()]                 # M x G x 2
    nib = np.stack([(idx >> 0) & 0xF, (idx >> 4) & 0xF], axis=-1).reshape(M, K // 4)
    got = np.stack([nib & 3, (nib >> 2) & 3], axis=-1)
    zero = oracle.decode(A, p.ta).reshape(M, K // 4, 4) == 0
    both_nonzero = ~np.take_along_axis(zero, pos, axis=2).any(axis=2)
    assert np.array_equal(got[both_nonzero], pos[both_nonzero])
    assert both_nonzero.mean() > 0.9


def _group_case(oracle, group, t="f16"):
    A = torch.tensor([group + [1.0, 0.0, 2.0, 0.0]], dtype=torch.float32).to(W.TORCH_DTYPE[t])
    vals, idx, viol = oracle.compress(W.bits(A), t)
    nib = int(idx[0, 0]) & 0xF
    return (nib & 3, nib >> 2), oracle.decode(vals, t)[0, :2].tolist(), viol, vals


def test_compress_padding_and_violation_readings(oracle):
    # two non-zeros: kept as they are
    assert _group_case(oracle, [0.0, 3.0, 0.0, 5.0])[:3] == ((1, 3), [3.0, 5.0], 0)
    # one non-zero at position 3: padded with the lowest unused position, +0
    pos, v, viol, vals = _group_case(oracle, [0.0, 0.0, 0.0, 7.0])
    assert (pos, v, viol) == ((0, 3), [0.0, 7.0], 0)
    assert W.bits(torch.zeros(1, dtype=torch.float16))[0] == vals[0, 0]   # +0 bits
    # one non-zero at position 0: the padded slot is position 1
    assert _group_case(oracle, [4.0, 0.0, 0.0, 0.0])[:3] == ((0, 1), [4.0, 0.0], 0)
    # no non-zero: positions 0 and 1, both +0
    assert _group_case(oracle, [0.0, 0.0, 0.0, 0.0])[:3] == ((0, 1), [0.0, 0.0], 0)
    # -0 counts as zero and becomes +0
    pos, v, viol, vals = _group_case(oracle, [-0.0, 2.0, 0.0, 0.0])
    assert pos == (0, 1) and vals[0, 0] == 0 and viol == 0
    # three non-zeros violate the contract: the two lowest kept, one violation
    assert _group_case(oracle, [1.0, 0.0, 2.0, 3.0])[:3] == ((0, 2), [1.0, 2.0], 1)
    # NaN and infinity are non-zero
    pos, v, viol, _ = _group_case(oracle, [0.0, float("inf"), 0.0, float("nan")])
    assert pos == (1, 3) and v[0] == math.inf and math.isnan(v[1]) and viol == 0


def test_compress_violations_are_counted(oracle):
    p = W.make("dense_bf16_8192", M=4, N=8, K=32)          # dense: most groups have 4 non-zeros
    _, _, viol = oracle.compress(W.bits(p.A), p.ta)
    nz = (oracle.decode(W.bits(p.A), p.ta).reshape(4, 8, 4) != 0).sum(axis=2)
    assert viol == int((nz > 2).sum()) and viol > 0


# ------------------------------------------------------------------ sparse GEMM

SPARSE_CASES = [("sparse_f16_random", None), ("sparse_f16_keep02", None),
                ("sparse_e4m3_e5m2", None), ("sparse_e4m3_e5m2", "e4m3"),
                ("dense_i8_4096", "i8")]


def _sparse_problem(name, tb_override, M, N, K, seed=0):
    if name == "dense_i8_4096":
        p = W.make(name, M=M, N=N, K=K, sparse="random", seed_offset=seed)
    else:
        p = W.make(name, M=M, N=N, K=K, seed_offset=seed)
    if tb_override and tb_override != p.tb and tb_override != "i8":
        p.B = p.B.to(torch.float32).to(W.TORCH_DTYPE[tb_override])
        p.tb = tb_override
    if p.C.dtype == torch.float32 and name.startswith("sparse_f16"):
        p.C = torch.randn(p.C.shape, generator=torch.Generator().manual_seed(5))
    return p


@pytest.mark.parametrize("name,tb", SPARSE_CASES)
@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (3, 4, 16), (6, 5, 32)])
def test_sparse_against_exact_rationals(oracle, name, tb, M, N, K):
    p = _sparse_problem(name, tb, M, N, K)
    vals, idx, viol = oracle.compress(W.bits(p.A), p.ta)
    assert viol == 0
    D = oracle.sparse_gemm(vals, idx, p.ta, W.bits(p.B), p.tb, p.C.numpy(), K)
    exact = _exact_gemm(p.A, p.B, p.C)          # on the generator's (dense, masked) A
    if p.ta == "i8":
        assert D.tolist() == [[int(x) for x in row] for row in exact]
        return
    bound = 2 * (K + 1) * 2.0 ** -53 * _abs_sum(p.A, p.B, p.C)
    err = np.array([[abs(Fraction(D[i][j]) - exact[i][j]) for j in range(N)] for i in range(M)])
    assert (err <= bound).all()


@pytest.mark.parametrize("name,tb", SPARSE_CASES)
def test_sparse_equals_dense_on_decompressed(oracle, name, tb):
    M, N, K = 37, 24, 128
    p = _sparse_problem(name, tb, M, N, K, seed=1)
    vals, idx, _ = oracle.compress(W.bits(p.A), p.ta)
    dense_A = oracle.decompress(vals, idx, p.ta, K)
    Ds = oracle.sparse_gemm(vals, idx, p.ta, W.bits(p.B), p.tb, p.C.numpy(), K)
    Dd = oracle.gemm(dense_A, p.ta, W.bits(p.B), p.tb, p.C.numpy())
    # the same non-zero terms in the same K order: identical, not just close
    assert np.array_equal(Ds, Dd)
    rows = [36, 2, 2]
    assert np.array_equal(oracle.sparse_gemm(vals, idx, p.ta, W.bits(p.B), p.tb, p.C.numpy(), K,
                                             rows=rows), Ds[rows])


def test_flop_convention_matches_page_ops_column():
    # "CDNA3 sparse MFMA builtins", section "Instruction throughput": a 16x16x64
    # sparse instruction counts 32768 ops and a 32x32x32 one 65536; dense
    # 32x32x8 f16 on the dense page counts 16384.  Ops = 2*M*N*K, K uncompressed.
    assert W.Problem("x", 16, 16, 64, "e4m3", "e4m3", "f32", None, None, None).flops == 32768
    assert W.Problem("x", 32, 32, 32, "e4m3", "e4m3", "f32", None, None, None).flops == 65536
    assert W.Problem("x", 32, 32, 8, "f16", "f16", "f32", None, None, None).flops == 16384
