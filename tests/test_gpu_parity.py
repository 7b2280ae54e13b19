"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle,
element by element, at sizes that span several tiles and ragged tails.

Tolerances (relative Frobenius error against the f64 oracle): 1e-3 for f16 and
bf16 inputs, 2e-2 for FP8 inputs; i8 -> i32 must be bit-exact.  4:2
compression must be bit-identical to the oracle's.
"""
import numpy as np
import pytest
import torch

from tensor_core_matrix_02_gb300 import mma42
from tensor_core_matrix_02_gb300 import workloads as W

from gpu_helpers import (TOL, assert_half_close, assert_matches, gpu_dense, half_reference, oracle_dense, poisoned_like,
                         ref_sparse, rel_frobenius, wrap_i32)

pytestmark = pytest.mark.gpu

DENSE = {
    "f16": ("dense_f16_128", None, None),
    "bf16": ("dense_bf16_8192", None, None),
    "e4m3xe4m3": ("dense_e4m3_16384", None, None),
    "e4m3xe5m2": ("dense_e4m3_16384", None, "e5m2"),
    "e5m2xe4m3": ("dense_e4m3_16384", "e5m2", None),
    "e5m2xe5m2": ("dense_e4m3_16384", "e5m2", "e5m2"),
    "i8": ("dense_i8_4096", None, None),
    "u8": ("dense_i8_4096", "u8", "u8"),
    "u8xi8": ("dense_i8_4096", "u8", None),
    "i8xu8": ("dense_i8_4096", None, "u8"),
}

# (M, N, K): one tile; the first workload's own shape; ragged in all three
# dimensions over several tiles; a single row; K spanning many pipeline rounds; outputs
# at most 128 wide (128-column blocks of the one-SM kernel), ragged and with K in slices
DENSE_SHAPES = [(128, 256, 128), (128, 128, 256), (300, 528, 208), (1, 16, 16), (257, 784, 1040),
                (640, 512, 4096), (300, 112, 1040), (64, 96, 16384)]


@pytest.mark.parametrize("kind", list(DENSE))
@pytest.mark.parametrize("M,N,K", DENSE_SHAPES)
def test_dense_matches_oracle(oracle, kind, M, N, K):
    name, ta, tb = DENSE[kind]
    p = W.make(name, M=M, N=N, K=K, ta=ta, tb=tb)
    D = gpu_dense(p)
    assert_matches(D, oracle_dense(oracle, p), p.ta, f"{kind} {M}x{N}x{K}")


@pytest.mark.parametrize("kind", ["f16", "bf16", "e4m3xe5m2", "i8"])
def test_dense_closed_forms(kind):
    """A = 0 gives C exactly; A = I gives B + C exactly (every sum has one term)."""
    name, ta, tb = DENSE[kind]
    p = W.make(name, M=256, N=256, K=256, ta=ta, tb=tb)
    p.A = torch.zeros_like(p.A)
    assert torch.equal(gpu_dense(p).cpu(), p.C)
    p.A = torch.eye(256, dtype=torch.float32).to(p.A.dtype)
    D = gpu_dense(p).cpu()
    want = (p.B.to(torch.float64) + p.C.to(torch.float64)).to(p.C.dtype)
    assert torch.equal(D, want)


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_i8_extreme_values_are_exact(monkeypatch, kernel):
    """All -128: every partial sum is as large as the i8 path can make it (a K of 17
    exact chunks of the CTA-pair kernel plus a ragged one); then -128 x 127."""
    monkeypatch.setenv("MMA42_DENSE_KERNEL", kernel)
    M, N, K = 384, 512, 4096 + 256 + 16
    p = W.make("dense_i8_4096", M=M, N=N, K=K)
    p.A = torch.full((M, K), -128, dtype=torch.int8)
    p.B = torch.full((K, N), -128, dtype=torch.int8)
    D = gpu_dense(p).cpu()
    assert torch.equal(D, (p.C.to(torch.int64) + K * 16384).to(torch.int32))
    p.B = torch.full((K, N), 127, dtype=torch.int8)
    D = gpu_dense(p).cpu()
    assert torch.equal(D, (p.C.to(torch.int64) - K * 128 * 127).to(torch.int32))


def near_extreme(t: str, shape, far: int, seed: int) -> torch.Tensor:
    """Mostly `far` (85%), otherwise uniform over the type: chunk sums of large
    magnitude whose low bits are still random."""
    g = torch.Generator().manual_seed(seed)
    lo, hi = (0, 256) if t == "u8" else (-128, 128)
    x = torch.randint(lo, hi, shape, generator=g, dtype=torch.int64)
    x[torch.rand(shape, generator=g) < 0.85] = far
    return x.to(W.TORCH_DTYPE[t])


def chunk_sums_reach(A: torch.Tensor, B: torch.Tensor, chunk: int, shift_a=0, shift_b=0) -> float:
    """Largest |sum over one aligned K chunk| of the (shifted) products, as a power of two."""
    a = A.to(torch.float64) - shift_a
    b = B.to(torch.float64) - shift_b
    top = 0.0
    for k0 in range(0, a.shape[1], chunk):
        top = max(top, float((a[:, k0:k0 + chunk] @ b[k0:k0 + chunk]).abs().max()))
    return np.log2(top)


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("ta,fa,tb,fb", [("i8", -128, "i8", -128), ("i8", 127, "i8", -128), ("u8", 0, "u8", 255)])
def test_i8_chunk_sums_near_the_f32_limit_are_exact(oracle, monkeypatch, kernel, ta, fa, tb, fb):
    """Operands mostly at an extreme value: the exact f32 chunks (1024 K of signed
    products, unsigned operands shifted to signed) reach sums between 2^23 and 2^24
    in magnitude with random low bits, positive and negative, over several chunks
    and a ragged tail.  Bit-exact against the oracle."""
    monkeypatch.setenv("MMA42_DENSE_KERNEL", kernel)
    M, N, K = 256, 384, 3 * 1024 + 512 + 48
    p = W.make("dense_i8_4096", M=M, N=N, K=K, ta=ta, tb=tb)
    p.A = near_extreme(ta, (M, K), fa, 21)
    p.B = near_extreme(tb, (K, N), fb, 22)
    sa, sb = (128 if ta == "u8" else 0), (128 if tb == "u8" else 0)
    assert chunk_sums_reach(p.A, p.B, 1024, sa, sb) > 23.5     # the test reaches the range
    D = gpu_dense(p)
    assert_matches(D, oracle_dense(oracle, p), ta, f"{ta}x{tb} near-extreme {kernel}")


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("ta,va,tb,vb", [("u8", 255, "u8", 255), ("u8", 255, "i8", -128), ("i8", -128, "u8", 255)])
def test_unsigned_extreme_values_are_exact(monkeypatch, kernel, ta, va, tb, vb):
    """The largest products each signedness pair can make, over many exact chunks
    (128 K for unsigned x unsigned, 256 mixed) and a ragged tail."""
    monkeypatch.setenv("MMA42_DENSE_KERNEL", kernel)
    M, N, K = 384, 512, 4096 + 128 + 16
    p = W.make("dense_i8_4096", M=M, N=N, K=K, ta=ta, tb=tb)
    p.A = torch.full((M, K), va, dtype=W.TORCH_DTYPE[ta])
    p.B = torch.full((K, N), vb, dtype=W.TORCH_DTYPE[tb])
    D = gpu_dense(p).cpu()
    assert torch.equal(D, (p.C.to(torch.int64) + K * va * vb).to(torch.int32))


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_i8_sum_wraps_like_i32(monkeypatch, kernel):
    """C near the top of the i32 range plus a positive product wraps modulo 2^32."""
    monkeypatch.setenv("MMA42_DENSE_KERNEL", kernel)
    M, N, K = 256, 256, 512
    p = W.make("dense_i8_4096", M=M, N=N, K=K)
    p.A = torch.full((M, K), -128, dtype=torch.int8)
    p.B = torch.full((K, N), -128, dtype=torch.int8)
    p.C = torch.full((M, N), 2**31 - 1000, dtype=torch.int32)
    D = gpu_dense(p).cpu().numpy().astype(np.int64)
    want = wrap_i32(np.full((M, N), 2**31 - 1000 + K * 16384, dtype=np.int64))
    assert np.array_equal(D, want)


# clamp: D = the exact C + A*B saturated to the i32 range (8-bit integer inputs)

def clamp_ref(exact):
    return np.clip(exact, -(1 << 31), (1 << 31) - 1)


@pytest.mark.parametrize("ta,va,tb,vb,c", [("i8", -128, "i8", -128, (1 << 31) - 1000),
                                           ("i8", -128, "i8", 127, -(1 << 31) + 5),
                                           ("u8", 255, "u8", 255, 0), ("u8", 255, "i8", -128, -(1 << 30))])
@pytest.mark.parametrize("K", [4096 + 16, 70000])
def test_clamp_saturates_exactly(ta, va, tb, vb, c, K):
    """Constant matrices whose exact sums leave (or stay inside) the i32 range,
    with a K that one slice covers and one that needs several (u8 x u8: 33025)."""
    M, N = 64, 128
    A = torch.full((M, K), va, dtype=W.TORCH_DTYPE[ta], device="cuda")
    B = torch.full((K, N), vb, dtype=W.TORCH_DTYPE[tb], device="cuda")
    C = torch.full((M, N), c, dtype=torch.int32, device="cuda")
    D = mma42.mma_gemm(A, B, C, clamp=True)
    assert mma42.mma_sync_status() == 0
    want = clamp_ref(np.full((M, N), c + K * va * vb, dtype=np.int64))
    assert np.array_equal(D.cpu().numpy().astype(np.int64), want)


@pytest.mark.parametrize("ta,tb", [("i8", "i8"), ("u8", "u8"), ("u8", "i8")])
@pytest.mark.parametrize("M,N,K", [(300, 272, 1040), (64, 96, 40000)])
def test_clamp_matches_oracle(oracle, ta, tb, M, N, K):
    """Random inputs and a C near both ends of the i32 range: some outputs
    saturate, the rest equal the exact sum."""
    p = W.make("dense_i8_4096", M=M, N=N, K=K, ta=ta, tb=tb)
    g = torch.Generator().manual_seed(K)
    C = torch.randint(-(1 << 31), (1 << 31) - 1, (M, N), generator=g, dtype=torch.int64).to(torch.int32)
    D = mma42.mma_gemm(p.A.cuda(), p.B.cuda(), C.cuda(), clamp=True)
    assert mma42.mma_sync_status() == 0
    exact = oracle.gemm(W.bits(p.A), ta, W.bits(p.B), tb, C.numpy())
    want = clamp_ref(exact)
    assert (exact != want).any() and (exact == want).any()
    assert np.array_equal(D.cpu().numpy().astype(np.int64), want)


@pytest.mark.parametrize("ta,tb", [("u8", "i8"), ("i8", "u8"), ("u8", "u8")])
def test_clamp_with_k_slices_and_unsigned_operands(oracle, ta, tb):
    """K past the one-slice bound (131008 for the signed-shifted operands): exact i32
    slice partials, the unsigned corrections and C summed in 64 bits, then saturated."""
    M, N, K = 32, 64, 140000
    p = W.make("dense_i8_4096", M=M, N=N, K=K, ta=ta, tb=tb)
    g = torch.Generator().manual_seed(3)
    C = torch.randint(-(1 << 31), (1 << 31) - 1, (M, N), generator=g, dtype=torch.int64).to(torch.int32)
    D = mma42.mma_gemm(p.A.cuda(), p.B.cuda(), C.cuda(), clamp=True)
    assert mma42.mma_sync_status() == 0
    exact = oracle.gemm(W.bits(p.A), ta, W.bits(p.B), tb, C.numpy())
    assert np.array_equal(D.cpu().numpy().astype(np.int64), clamp_ref(exact))
    D = mma42.mma_gemm(p.A.cuda(), p.B.cuda(), C.cuda())             # and wrapping, one slice
    assert np.array_equal(D.cpu().numpy().astype(np.int64), wrap_i32(exact))


# each dense type through both kernels (the CTA-pair one is otherwise only chosen for
# large outputs), at shapes ragged in M, N and K
@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("kind", ["f16", "bf16", "e4m3xe5m2", "i8", "u8", "u8xi8"])
@pytest.mark.parametrize("M,N,K", [(300, 528, 1040), (520, 272, 4160)])
def test_dense_each_kernel_matches_oracle(oracle, monkeypatch, kernel, kind, M, N, K):
    monkeypatch.setenv("MMA42_DENSE_KERNEL", kernel)
    name, ta, tb = DENSE[kind]
    p = W.make(name, M=M, N=N, K=K, ta=ta, tb=tb)
    assert_matches(gpu_dense(p), oracle_dense(oracle, p), p.ta, f"{kernel} {kind} {M}x{N}x{K}")


# the short-K kernel (one CTA per 128 x 128 block, or 128 x 64 for 16-bit operands,
# all of a block's operands in flight at once): 1, 2 and 4 k-blocks, a ragged K,
# several ragged blocks, and in place, at both block widths
@pytest.mark.parametrize("bn", ["64", "128"])
@pytest.mark.parametrize("kind", ["f16", "bf16", "e4m3xe5m2", "e5m2xe4m3"])
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (1000, 704, 208), (1000, 704, 512), (33, 48, 16),
                                   (256, 320, 128), (200, 144, 64)])
def test_small_kernel_matches_oracle(oracle, monkeypatch, kind, M, N, K, bn):
    if bn == "64" and kind.startswith("e"):
        pytest.skip("FP8 blocks are 128 columns wide (one 128-byte row of B)")
    monkeypatch.setenv("MMA42_DENSE_KERNEL", "small")
    monkeypatch.setenv("MMA42_SMALL_BN", bn)
    name, ta, tb = DENSE[kind]
    if K > 256 and kind in ("f16", "bf16"):
        K = 256                                   # the 16-bit kernel holds 4 x 64 K
    p = W.make(name, M=M, N=N, K=K, ta=ta, tb=tb)
    ref = oracle_dense(oracle, p)
    assert_matches(gpu_dense(p), ref, p.ta, f"small bn={bn} {kind} {M}x{N}x{K}")
    C = p.C.cuda()
    mma42.mma_gemm(p.A.cuda(), p.B.cuda(), C, C)
    assert mma42.mma_sync_status() == 0
    assert_matches(C, ref, p.ta, f"small bn={bn} {kind} {M}x{N}x{K} in place")


# half-precision C and D (f16 x f16 -> f16, bf16 x bf16 -> bf16): the f64 oracle's
# result rounded to the output type by the oracle's quantisation, then the usual
# relative Frobenius bound (the two roundings differ by one unit in rare ties)
HALF = {"f16": "dense_f16_128", "bf16": "dense_bf16_8192"}


def half_case(kind, M, N, K):
    p = W.make(HALF[kind], M=M, N=N, K=K)
    C = p.C.to(W.TORCH_DTYPE[kind])
    return p, C


@pytest.mark.parametrize("kind", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", DENSE_SHAPES)
def test_dense_half_output_matches_oracle(oracle, kind, M, N, K):
    p, C = half_case(kind, M, N, K)
    D = mma42.mma_gemm(p.A.cuda(), p.B.cuda(), C.cuda(), torch.full_like(C.cuda(), float("nan")))
    assert mma42.mma_sync_status() == 0
    assert D.dtype == C.dtype
    assert_half_close(D, half_reference(oracle, p, C, kind), f"{kind} out {M}x{N}x{K}")


@pytest.mark.parametrize("kind", ["f16", "bf16"])
@pytest.mark.parametrize("ksplit", [None, "3"])
def test_dense_half_output_split_k_and_in_place(oracle, monkeypatch, kind, ksplit):
    """Few blocks and a long K: K slices reduced in f32, rounded once; then D = C in place."""
    if ksplit:
        monkeypatch.setenv("MMA42_KSPLIT", ksplit)
    p, C = half_case(kind, 300, 272, 8256)
    want = half_reference(oracle, p, C, kind)
    Cd = C.cuda()
    D1 = mma42.mma_gemm(p.A.cuda(), p.B.cuda(), Cd)
    assert_half_close(D1, want, f"{kind} out split {ksplit}")
    mma42.mma_gemm(p.A.cuda(), p.B.cuda(), Cd, Cd)
    assert mma42.mma_sync_status() == 0
    assert torch.equal(Cd, D1), "in place must give the same bits"


@pytest.mark.parametrize("kind", ["f16", "bf16"])
def test_dense_half_output_zero_A_gives_C(kind):
    p, C = half_case(kind, 256, 512, 256)
    A = torch.zeros_like(p.A).cuda()
    D = mma42.mma_gemm(A, p.B.cuda(), C.cuda())
    assert torch.equal(D.cpu(), C)


def test_dense_K_zero_copies_C():
    p = W.make("dense_bf16_8192", M=64, N=64, K=16)
    A = torch.empty((64, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    C = p.C.cuda()
    D = mma42.mma_gemm(A, B, C, poisoned_like(C))
    assert torch.equal(D.cpu(), p.C)


def test_dense_in_place_D_equals_C(oracle):
    p = W.make("dense_bf16_8192", M=384, N=512, K=320)
    ref = oracle_dense(oracle, p)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    mma42.mma_gemm(A, B, C, C)
    assert mma42.mma_sync_status() == 0
    assert_matches(C, ref, "bf16", "in place")


# (workload, ta, tb, environment): every kernel and split path that writes D
IN_PLACE = {
    "bf16 pair": ("dense_bf16_8192", None, None, {"MMA42_DENSE_KERNEL": "pair"}),
    "bf16 single": ("dense_bf16_8192", None, None, {"MMA42_DENSE_KERNEL": "single"}),
    "bf16 split-K": ("dense_bf16_8192", None, None, {"MMA42_DENSE_KERNEL": "pair", "MMA42_KSPLIT": "3"}),
    "bf16 tail split": ("dense_bf16_8192", None, None, {"MMA42_DENSE_KERNEL": "pair", "MMA42_TAIL_SPLIT": "2"}),
    "e4m3": ("dense_e4m3_16384", None, "e5m2", {"MMA42_DENSE_KERNEL": "pair"}),
    "i8 pair": ("dense_i8_4096", None, None, {"MMA42_DENSE_KERNEL": "pair"}),
    "i8 single": ("dense_i8_4096", None, None, {"MMA42_DENSE_KERNEL": "single"}),
    "i8 tail split": ("dense_i8_4096", None, None, {"MMA42_DENSE_KERNEL": "pair", "MMA42_TAIL_SPLIT": "3"}),
    "u8": ("dense_i8_4096", "u8", "u8", {}),
}


@pytest.mark.parametrize("case", list(IN_PLACE))
def test_dense_in_place_matches_out_of_place(monkeypatch, case):
    """D = C in place gives the same bits as a separate D (ragged shape, several blocks)."""
    name, ta, tb, env = IN_PLACE[case]
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    p = W.make(name, M=300, N=528, K=1040, ta=ta, tb=tb)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    D = mma42.mma_gemm(A, B, C, poisoned_like(C))
    mma42.mma_gemm(A, B, C, C)
    assert mma42.mma_sync_status() == 0
    assert torch.equal(C, D)


@pytest.mark.parametrize("kind", ["f16_random", "e4m3xe5m2", "i8_random", "u8_random"])
def test_sparse_in_place_matches_out_of_place(kind):
    p = sparse_problem(kind, 300, 272, 1024)
    vals, idx = mma42.sparse42_compress(p.A.cuda())
    B, C = p.B.cuda(), p.C.cuda()
    D = mma42.sparse42_gemm(vals, idx, B, C, poisoned_like(C))
    mma42.sparse42_gemm(vals, idx, B, C, C)
    assert mma42.mma_sync_status() == 0
    assert torch.equal(C, D)


@pytest.mark.parametrize("case", ["clamp", "f16 out", "bf16 out"])
def test_K_zero_copies_C_for_the_options(case):
    if case == "clamp":
        A = torch.empty((64, 0), dtype=torch.int8, device="cuda")
        B = torch.empty((0, 64), dtype=torch.int8, device="cuda")
        C = torch.randint(-100, 100, (64, 64), dtype=torch.int32, device="cuda")
        D = mma42.mma_gemm(A, B, C, clamp=True)
    else:
        dt = torch.float16 if case == "f16 out" else torch.bfloat16
        A = torch.empty((64, 0), dtype=dt, device="cuda")
        B = torch.empty((0, 64), dtype=dt, device="cuda")
        C = torch.randn((64, 64), device="cuda").to(dt)
        D = mma42.mma_gemm(A, B, C)
    assert torch.equal(D, C)


def test_sparse_K_zero_and_empty_rows():
    vals = torch.empty((64, 0), dtype=torch.float16, device="cuda")
    idx = torch.empty((64, 0), dtype=torch.uint8, device="cuda")
    B = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    C = torch.randn((64, 64), device="cuda")
    assert torch.equal(mma42.sparse42_gemm(vals, idx, B, C), C)
    vals = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    idx = torch.empty((0, 16), dtype=torch.uint8, device="cuda")
    B = torch.zeros((128, 64), dtype=torch.float16, device="cuda")
    assert mma42.sparse42_gemm(vals, idx, B, torch.empty((0, 64), device="cuda")).shape == (0, 64)


@pytest.mark.parametrize("entry", ["compress", "prune", "quantize_prune"])
def test_empty_compression_clears_the_count(entry):
    count = torch.full((1,), 123, dtype=torch.int32, device="cuda")
    if entry == "compress":
        mma42.sparse42_compress(torch.empty((0, 64), dtype=torch.float16, device="cuda"), count)
    elif entry == "prune":
        mma42.sparse42_prune(torch.empty((0, 64), dtype=torch.float16, device="cuda"), count)
    else:
        mma42.sparse42_quantize_prune(torch.empty((0, 64), device="cuda"), torch.float8_e4m3fn, count)
    assert int(count.item()) == 0


def test_quantize_empty_is_a_no_op():
    y = mma42.mma_quantize(torch.empty(0, device="cuda"), torch.bfloat16)
    assert y.numel() == 0


def test_dense_empty_is_a_no_op():
    A = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    C = torch.empty((0, 64), dtype=torch.float32, device="cuda")
    assert mma42.mma_gemm(A, B, C).shape == (0, 64)


def test_dense_split_k_skinny_shape(oracle):
    """Few output tiles and a long K: the K-split path and its fixed-order reduction."""
    p = W.make("dense_bf16_skinny", M=256, N=512, K=16384)
    D1 = gpu_dense(p)
    assert_matches(D1, oracle_dense(oracle, p), "bf16", "split-K")
    D2 = gpu_dense(p)
    assert torch.equal(D1, D2), "split-K result must not depend on timing"


@pytest.mark.parametrize("kind", ["bf16", "e4m3xe5m2"])
@pytest.mark.parametrize("ksplit", [None, "3", "7"])
def test_pair_split_k_matches_oracle(oracle, monkeypatch, kind, ksplit):
    """The CTA-pair kernel with K cut into slices (planned, or forced to uneven
    counts over a ragged K): f32 partials, then the fixed-order reduction."""
    monkeypatch.setenv("MMA42_DENSE_KERNEL", "pair")
    if ksplit:
        monkeypatch.setenv("MMA42_KSPLIT", ksplit)
    name, ta, tb = DENSE[kind]
    p = W.make(name, M=300, N=528, K=8256, ta=ta, tb=tb)
    D1 = gpu_dense(p)
    assert_matches(D1, oracle_dense(oracle, p), p.ta, f"pair split {ksplit} {kind}")
    assert torch.equal(D1, gpu_dense(p)), "split-K result must not depend on timing"


# ----------------------------------------------------------------- compression

COMPRESS = [("sparse_f16_keep02", None), ("sparse_f16_random", None), ("sparse_e4m3_e5m2", None),
            ("sparse_e4m3_e5m2", "e5m2"), ("sparse_f16_random", "bf16"), ("dense_i8_4096", "i8"),
            ("dense_i8_4096", "u8")]


@pytest.mark.parametrize("name,ta", COMPRESS)
@pytest.mark.parametrize("M,K", [(1, 32), (300, 512), (129, 4096)])
def test_compress_bit_identical_to_oracle(oracle, name, ta, M, K):
    if ta in ("i8", "u8"):
        p = W.make(name, M=M, N=16, K=K, sparse="random", ta=ta)
    else:
        p = W.make(name, M=M, N=16, K=K, ta=ta)
    viol = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx = mma42.sparse42_compress(p.A.cuda(), viol)
    ov, oi, on = oracle.compress(W.bits(p.A), p.ta)
    assert np.array_equal(W.bits(vals.cpu()), ov)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert int(viol.item()) == on == 0


def test_compress_special_groups(oracle):
    """Padding, signed zero, NaN/inf and over-full groups follow the oracle's readings."""
    groups = [[0, 3, 0, 5], [0, 0, 0, 7], [4, 0, 0, 0], [0, 0, 0, 0], [-0.0, 2, 0, 0],
              [1, 0, 2, 3], [0, float("inf"), 0, float("nan")], [1, 2, 3, 4]]
    row = [x for g in groups for x in g]
    A = torch.tensor([row] * 5, dtype=torch.float32).to(torch.float16)
    viol = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx = mma42.sparse42_compress(A.cuda(), viol)
    ov, oi, on = oracle.compress(W.bits(A), "f16")
    assert np.array_equal(W.bits(vals.cpu()), ov)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert int(viol.item()) == on == 2 * 5


def test_compress_check_raises_on_dense_input():
    """A that breaks the 4:2 contract is reported as MMA_ERR_NOT_SPARSE when asked."""
    p = W.make("dense_bf16_8192", M=64, N=16, K=128)          # dense: most groups hold 4 non-zeros
    with pytest.raises(mma42.MmaError) as info:
        mma42.sparse42_compress(p.A.cuda(), check=True)
    assert info.value.status == "MMA_ERR_NOT_SPARSE"
    q = W.make("sparse_f16_random", M=64, N=16, K=128)
    mma42.sparse42_compress(q.A.cuda(), check=True)           # a 4:2 matrix passes


# ------------------------------------------------------------------ pruning

PRUNE = [("dense_f16_128", None), ("dense_bf16_8192", None), ("dense_e4m3_16384", None),
         ("dense_e4m3_16384", "e5m2"), ("dense_i8_4096", None), ("dense_i8_4096", "u8")]


@pytest.mark.parametrize("name,ta", PRUNE)
@pytest.mark.parametrize("M,K", [(1, 32), (300, 512), (129, 4096)])
def test_prune_bit_identical_to_oracle(oracle, name, ta, M, K):
    """Dense A pruned to 4:2 by magnitude: vals, idx and the dropped-group count as the oracle."""
    p = W.make(name, M=M, N=16, K=K, ta=ta)
    dropped = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx = mma42.sparse42_prune(p.A.cuda(), dropped)
    ov, oi, on = oracle.prune(W.bits(p.A), p.ta)
    assert np.array_equal(W.bits(vals.cpu()), ov)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert int(dropped.item()) == on


def test_prune_special_groups(oracle):
    """Ties, signed zeros, infinity and NaN follow the oracle's reading."""
    inf, nan = float("inf"), float("nan")
    groups = [[1, 1, 1, 1], [0, 2, -2, 0], [3, -3, 3, 3], [0, 0, 0, 0], [1, inf, nan, 2], [-inf, 7, 1, 0],
              [0.5, -0.25, 0.75, -1], [0, -0.0, 0, 4], [-0.0, -0.0, -0.0, -0.0], [nan, nan, 1, -inf]]
    row = [x for g in groups for x in g]
    for t in ("f16", "bf16", "e5m2", "e4m3"):
        A = torch.tensor([row + [0.0] * 24] * 3, dtype=torch.float32).to(W.TORCH_DTYPE[t])
        vals, idx = mma42.sparse42_prune(A.cuda())
        ov, oi, _ = oracle.prune(W.bits(A), t)
        assert np.array_equal(W.bits(vals.cpu()), ov), t
        assert np.array_equal(idx.cpu().numpy(), oi), t


@pytest.mark.parametrize("name,ta", COMPRESS)
def test_prune_equals_compress_on_4_2_input(name, ta):
    if ta in ("i8", "u8"):
        p = W.make(name, M=200, N=16, K=1024, sparse="random", ta=ta)
    else:
        p = W.make(name, M=200, N=16, K=1024, ta=ta)
    A = p.A.cuda()
    cv, ci = mma42.sparse42_compress(A)
    pv, pi = mma42.sparse42_prune(A)
    assert torch.equal(cv.view(torch.uint8), pv.view(torch.uint8)) and torch.equal(ci, pi)


@pytest.mark.parametrize("name", ["dense_bf16_8192", "dense_i8_4096"])
def test_prune_then_sparse_gemm_matches_oracle(oracle, name):
    p = W.make(name, M=300, N=272, K=1024)
    vals, idx = mma42.sparse42_prune(p.A.cuda())
    D = mma42.sparse42_gemm(vals, idx, p.B.cuda(), p.C.cuda(), poisoned_like(p.C.cuda()))
    assert mma42.mma_sync_status() == 0
    ov, oi, _ = oracle.prune(W.bits(p.A), p.ta)
    ref = ref_sparse(oracle, ov, oi, p.ta, W.bits(p.B), p.tb, p.C.numpy(), p.K)
    assert_matches(D, ref, p.ta, f"prune + sparse {name}")


# ------------------------------------------------------------- quantisation

@pytest.mark.parametrize("t", ["f16", "bf16", "e4m3", "e5m2"])
@pytest.mark.parametrize("n", [1, 3, 4099, 70001])
def test_quantize_bit_identical_to_oracle(oracle, t, n):
    """f32 -> t on the GPU equals the oracle bit for bit (NaN by class), over
    normal, tiny, huge and special values and ragged lengths."""
    g = torch.Generator().manual_seed(n)
    x = torch.randn(n, generator=g) * torch.tensor([1e-6, 1e-2, 1.0, 1e3, 1e6, 1e38])[torch.randint(0, 6, (n,), generator=g)]
    special = torch.tensor([float("inf"), float("-inf"), float("nan"), 0.0, -0.0, 448.0, 464.0, 65520.0, -3.4e38])
    x[: min(n, special.numel())] = special[: min(n, special.numel())]
    y = mma42.mma_quantize(x.cuda(), W.TORCH_DTYPE[t])
    got = W.bits(y.cpu()).astype(np.int64)
    want = oracle.quantize(x.numpy(), t).astype(np.int64)
    nan_in = np.isnan(x.numpy())
    assert np.array_equal(got[~nan_in], want[~nan_in])
    assert torch.isnan(y.cpu().to(torch.float32)[torch.from_numpy(nan_in)]).all()


@pytest.mark.parametrize("t", ["f16", "bf16", "e4m3", "e5m2"])
@pytest.mark.parametrize("M,K", [(1, 32), (300, 512), (129, 4096)])
def test_quantize_prune_equals_oracle_composition(oracle, t, M, K):
    """The fused pass equals pruning the quantised matrix (both oracle steps pinned)."""
    g = torch.Generator().manual_seed(M + K)
    A = torch.randn((M, K), generator=g) * torch.tensor([1e-3, 1.0, 300.0, 1e5])[torch.randint(0, 4, (M, K), generator=g)]
    A[0, :8] = torch.tensor([float("inf"), -1.0, 2.0, 2.0, 0.0, -0.0, 1e-30, 5.0])
    dropped = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx = mma42.sparse42_quantize_prune(A.cuda(), W.TORCH_DTYPE[t], dropped)
    q = oracle.quantize(A.numpy(), t)
    ov, oi, on = oracle.prune(q, t)
    assert np.array_equal(W.bits(vals.cpu()), ov)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert int(dropped.item()) == on


def test_compress_keep02_index_constants():
    """The page's keep-{0,2} index constants: 0x88 per byte, 0x8888 per 16 bits."""
    p = W.make("sparse_e4m3_e5m2", M=64, N=16, K=256, sparse="keep02")
    A = p.A.to(torch.float32)
    A[:, 0::4] = 1.0
    A[:, 2::4] = -2.0
    vals, idx = mma42.sparse42_compress(A.to(torch.float8_e4m3fn).cuda())
    assert (idx.cpu() == 0x88).all()
    assert (idx.cpu().view(torch.int16) == np.int16(np.uint16(0x8888).view(np.int16))).all()


# ------------------------------------------------------------------ sparse GEMM

SPARSE = {
    "f16_keep02": ("sparse_f16_keep02", None, None),
    "f16_random": ("sparse_f16_random", None, None),
    "bf16_random": ("sparse_bf16_8192", None, None),
    "i8_random": ("sparse_i8_8192", None, None),
    "u8_random": ("sparse_i8_8192", "u8", "u8"),
    "u8xi8_random": ("sparse_i8_8192", "u8", "i8"),
    "i8xu8_random": ("sparse_i8_8192", "i8", "u8"),
    "e4m3xe5m2": ("sparse_e4m3_e5m2", None, None),
    "e4m3xe4m3": ("sparse_e4m3_e5m2", None, "e4m3"),
    "e5m2xe4m3": ("sparse_e4m3_e5m2", "e5m2", "e4m3"),
    "e5m2xe5m2": ("sparse_e4m3_e5m2", "e5m2", None),
}
SPARSE_SHAPES = [(128, 128, 128), (128, 128, 256), (300, 272, 384), (1, 16, 128), (257, 400, 1024),
                 (512, 384, 4096)]


def sparse_problem(kind, M, N, K):
    name, ta, tb = SPARSE[kind]
    p = W.make(name, M=M, N=N, K=K, ta=ta, tb=tb)
    if p.C.abs().max() == 0:          # a zero C would hide a dropped C term
        p.C = torch.randn(p.C.shape, generator=torch.Generator().manual_seed(7))
    return p


@pytest.mark.parametrize("kind", list(SPARSE))
@pytest.mark.parametrize("M,N,K", SPARSE_SHAPES)
def test_sparse_matches_oracle(oracle, kind, M, N, K):
    p = sparse_problem(kind, M, N, K)
    vals, idx = mma42.sparse42_compress(p.A.cuda())
    B, C = p.B.cuda(), p.C.cuda()
    D = mma42.sparse42_gemm(vals, idx, B, C, poisoned_like(C))
    assert mma42.mma_sync_status() == 0
    ov, oi, _ = oracle.compress(W.bits(p.A), p.ta)
    ref = ref_sparse(oracle, ov, oi, p.ta, W.bits(p.B), p.tb, p.C.numpy(), K)
    assert_matches(D, ref, p.ta, f"sparse {kind} {M}x{N}x{K}")


@pytest.mark.parametrize("kind", ["f16_random", "bf16_random", "e4m3xe5m2"])
def test_sparse_equals_dense_on_decompressed(kind):
    """sparse42_gemm(compress(A)) against mma_gemm on the same (4:2) A."""
    p = sparse_problem(kind, 384, 512, 2048)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    vals, idx = mma42.sparse42_compress(A)
    Ds = mma42.sparse42_gemm(vals, idx, B, C)
    Dd = mma42.mma_gemm(A, B, C)
    assert mma42.mma_sync_status() == 0
    err = rel_frobenius(Ds.cpu().numpy(), Dd.cpu().numpy().astype(np.float64))
    assert err <= TOL[p.ta] / 4


@pytest.mark.parametrize("kind", ["i8_random", "u8_random", "u8xi8_random", "i8xu8_random"])
def test_sparse_i8_equals_dense_bit_exact(kind):
    """sparse42_gemm(compress(A)) == mma_gemm(A) exactly for 8-bit integers (both exact paths)."""
    p = sparse_problem(kind, 384, 512, 4096)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    vals, idx = mma42.sparse42_compress(A)
    Ds = mma42.sparse42_gemm(vals, idx, B, C)
    Dd = mma42.mma_gemm(A, B, C)
    assert mma42.mma_sync_status() == 0
    assert torch.equal(Ds.cpu(), Dd.cpu())


def test_sparse_i8_extreme_values_are_exact():
    """Every kept value -128 against B = -128 (the largest chunk sums the exact i8
    path allows) over several chunks and a ragged output, then against B = 127."""
    M, N, K = 300, 272, 4096 + 1024 + 128
    p = sparse_problem("i8_random", M, N, K)
    A = torch.where(p.A != 0, torch.full_like(p.A, -128), p.A)
    vals, idx = mma42.sparse42_compress(A.cuda())
    C = p.C.cuda()
    for bval in (-128, 127):
        B = torch.full((K, N), bval, dtype=torch.int8, device="cuda")
        D = mma42.sparse42_gemm(vals, idx, B, C)
        kept = (A != 0).sum(dim=1, keepdim=True).to(torch.int64)       # 2 per group of four
        want = (p.C.to(torch.int64) + kept * (-128 * bval)).to(torch.int32)
        assert torch.equal(D.cpu(), want)


@pytest.mark.parametrize("ta,fa,tb,fb", [("i8", -128, "i8", -128), ("i8", 127, "i8", -128), ("u8", 255, "u8", 255),
                                         ("i8", -128, "u8", 0)])
def test_sparse_i8_chunk_sums_near_the_f32_limit_are_exact(oracle, ta, fa, tb, fb):
    """Kept values and B mostly at an extreme value: the exact f32 chunks (2048
    logical K for a signed A, 1024 for an unsigned one; an unsigned B runs shifted
    to signed, B - 128) reach sums between 2^23 and 2^24 in magnitude with random
    low bits.  Bit-exact against the oracle."""
    M, N, K = 256, 272, 2 * 2048 + 1024 + 128
    kind = {("i8", "i8"): "i8_random", ("u8", "u8"): "u8_random", ("i8", "u8"): "i8xu8_random"}[(ta, tb)]
    p = sparse_problem(kind, M, N, K)
    far = near_extreme(ta, (M, K), fa, 23)
    A = torch.where(p.A != 0, far, torch.zeros_like(far))
    A = torch.where(A == 0, torch.ones_like(A), A) * (p.A != 0)   # kept values stay non-zero
    B = near_extreme(tb, (K, N), fb, 24)
    chunk = 2048 if ta == "i8" else 1024
    assert chunk_sums_reach(A, B, chunk, shift_b=128 if tb == "u8" else 0) > 23.5
    vals, idx = mma42.sparse42_compress(A.cuda())
    D = mma42.sparse42_gemm(vals, idx, B.cuda(), p.C.cuda())
    assert mma42.mma_sync_status() == 0
    ov, oi, viol = oracle.compress(W.bits(A), ta)
    assert viol == 0
    ref = oracle.sparse_gemm(ov, oi, ta, W.bits(B), tb, p.C.numpy(), K)
    assert_matches(D, ref, ta, f"sparse {ta}x{tb} near-extreme")


def test_sparse_single_tile_identity_B():
    """B = I: D equals the expanded A exactly, which pins the index decoding."""
    M = N = K = 128
    p = sparse_problem("f16_random", M, N, K)
    B = torch.eye(K, dtype=torch.float32).to(torch.float16)
    C = torch.zeros(M, N)
    vals, idx = mma42.sparse42_compress(p.A.cuda())
    D = mma42.sparse42_gemm(vals, idx, B.cuda(), C.cuda())
    assert torch.equal(D.cpu(), p.A.to(torch.float32))
