"""Pins of the CPU oracle against facts that do not come from the oracle.

The oracle computes C[i][j] = Σ_k A[i][k]·B[j][k] (C = A·Bᵀ, fp16 operands,
"SASS-Level Kernel Generation for Blackwell", section "The numbers", Setup).
Each test below checks it against something independent: numpy's own fp16
decoding, exact integer arithmetic, an independent fp64 matmul, exact rational
arithmetic, identity and permutation matrices, and closed-form sums. Together
they catch a dropped term, a wrong sign or index, a transposed operand, an
off-by-one in K and a reader that strays into padding.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_fp16_gemm_02_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

# Tiny shapes: every dimension in 1..64, non-multiples of every tile, primes.
TINY_SHAPES = [(1, 1, 1), (1, 1, 64), (64, 64, 64), (3, 5, 7), (17, 1, 33), (1, 29, 2),
               (63, 62, 61), (31, 64, 1), (8, 16, 24), (64, 1, 17), (2, 3, 64), (47, 53, 59),
               (33, 9, 40), (5, 64, 13), (64, 64, 1), (11, 13, 48)]


def _f64(x):
    return x.astype(np.float64)


def test_f16_decoder_all_bit_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits], dtype=np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # The sign of zero is kept.
    assert np.signbit(oracle.f16_to_f64(0x8000)) and not np.signbit(oracle.f16_to_f64(0))


def test_hand_computed_example():
    # 2×3 times (2×3)ᵀ, worked by hand: [[1,2,3],[4,5,6]]·[[7,8,9],[1,0,-1]]ᵀ.
    A = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.float16)
    B = np.array([[7, 8, 9], [1, 0, -1]], dtype=np.float16)
    C = oracle.gemm_f64(A, B)
    assert C.tolist() == [[50.0, -2.0], [122.0, -2.0]]


@pytest.mark.parametrize("M,N,K", TINY_SHAPES)
def test_integer_inputs_exact(M, N, K):
    A, B = inputs.gemm_operands(M, N, K, seed=7, kind="int")
    ref = A.astype(np.int64) @ B.astype(np.int64).T  # exact integer arithmetic
    C = oracle.gemm_f64(A, B)
    assert np.array_equal(C, ref.astype(np.float64))


@pytest.mark.parametrize("M,N,K", TINY_SHAPES)
def test_uniform_inputs_vs_independent_matmul(M, N, K):
    A, B = inputs.gemm_operands(M, N, K, seed=11, kind="uniform")
    C, Cabs = oracle.gemm_f64(A, B, with_abs=True)
    ref = _f64(A) @ _f64(B).T
    ref_abs = np.abs(_f64(A)) @ np.abs(_f64(B)).T
    # Two fp64 sums of the same exact products differ by at most ~K·eps·Σ|ab|.
    bound = 4 * K * np.finfo(np.float64).eps * ref_abs + 1e-300
    assert np.all(np.abs(C - ref) <= bound)
    assert np.all(np.abs(Cabs - ref_abs) <= bound)


def test_exact_rational_small():
    A, B = inputs.gemm_operands(4, 3, 9, seed=3, kind="uniform")
    C = oracle.gemm_f64(A, B)
    for i in range(4):
        for j in range(3):
            exact = sum(Fraction(float(A[i, k])) * Fraction(float(B[j, k])) for k in range(9))
            # At most 9 roundings of a value of magnitude ≤ 9: well inside 1e-14.
            assert abs(Fraction(C[i, j]) - exact) <= Fraction(1, 10 ** 14)


@pytest.mark.parametrize("K", [1, 7, 64, 65])
def test_identity_gives_transpose(K):
    # A = I (M = K): C[i][j] = B[j][i], i.e. C = Bᵀ exactly.
    _, B = inputs.gemm_operands(K, 5, K, seed=5, kind="uniform")
    A = np.eye(K, dtype=np.float16)
    C = oracle.gemm_f64(A, B)
    assert np.array_equal(C, _f64(B).T)


def test_permutation_matrix():
    K = 37
    perm = np.random.default_rng(0).permutation(K)
    A = np.zeros((K, K), dtype=np.float16)
    A[np.arange(K), perm] = 1
    _, B = inputs.gemm_operands(K, 6, K, seed=9, kind="uniform")
    C = oracle.gemm_f64(A, B)
    # Row i of A picks column perm[i]: C[i][j] = B[j][perm[i]].
    assert np.array_equal(C, _f64(B)[:, perm].T)


@pytest.mark.parametrize("K", [1, 2, 3, 64, 100, 1000])
def test_closed_form_all_ones(K):
    A = np.ones((3, K), dtype=np.float16)
    B = np.ones((4, K), dtype=np.float16)
    assert np.all(oracle.gemm_f64(A, B) == K)


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6, 300, 301, 302])
def test_closed_form_mod3(K):
    # A = 1, B[j][k] = (k mod 3) − 1: each run of three k sums to 0, and a
    # remainder of one or two terms adds −1 (−1, or −1 + 0).
    A = np.ones((2, K), dtype=np.float16)
    B = np.tile(((np.arange(K) % 3) - 1).astype(np.float16), (3, 1))
    expect = 0.0 if K % 3 == 0 else -1.0
    assert np.all(oracle.gemm_f64(A, B) == expect)


def test_closed_form_separable_catches_transpose():
    # A[i][k] = (i mod 5) − 2 and B[j][k] = (j mod 7) − 3 for every k:
    # C[i][j] = K·((i mod 5) − 2)·((j mod 7) − 3). Swapping the roles of A and B
    # (or of i and j) gives a different matrix for these M ≠ N.
    M, N, K = 10, 14, 33
    A = np.tile(((np.arange(M) % 5) - 2).astype(np.float16)[:, None], (1, K))
    B = np.tile(((np.arange(N) % 7) - 3).astype(np.float16)[:, None], (1, K))
    expect = K * np.outer((np.arange(M) % 5) - 2, (np.arange(N) % 7) - 3)
    assert np.array_equal(oracle.gemm_f64(A, B), expect.astype(np.float64))


def test_k_dependent_pattern_catches_index_errors():
    # A[i][k] = ((i + k) mod 5) − 2, B[j][k] = ((2j + k) mod 3) − 1, summed by
    # plain Python integers.
    M, N, K = 6, 7, 23
    A = np.array([[((i + k) % 5) - 2 for k in range(K)] for i in range(M)], dtype=np.float16)
    B = np.array([[((2 * j + k) % 3) - 1 for k in range(K)] for j in range(N)], dtype=np.float16)
    C = oracle.gemm_f64(A, B)
    for i in range(M):
        for j in range(N):
            assert C[i, j] == sum((((i + k) % 5) - 2) * (((2 * j + k) % 3) - 1) for k in range(K))


def test_padding_past_k_is_never_read():
    # Columns K..ld-1 hold fp16 NaN; any read of them would poison C.
    M, N, K = 9, 11, 13
    A, B = inputs.gemm_operands(M, N, K, seed=2, kind="uniform", lda=24, ldb=16, pad="nan")
    assert np.isnan(A[:, K:].astype(np.float32)).all()
    C = oracle.gemm_f64(A, B, K=K)
    assert np.isfinite(C).all()
    ref = _f64(A[:, :K]) @ _f64(B[:, :K]).T
    assert np.allclose(C, ref, rtol=1e-13, atol=1e-13)


def test_k_zero_is_empty_sum():
    A = np.zeros((3, 8), dtype=np.float16)
    B = np.zeros((2, 8), dtype=np.float16)
    assert np.array_equal(oracle.gemm_f64(A, B, K=0), np.zeros((3, 2)))


def test_select_matches_full():
    M, N, K = 40, 50, 30
    A, B = inputs.gemm_operands(M, N, K, seed=4, kind="uniform")
    full, full_abs = oracle.gemm_f64(A, B, with_abs=True)
    rows = np.array([0, 3, 39, 17])
    cols = np.array([49, 0, 8])
    sel, sel_abs = oracle.gemm_f64_select(A, B, rows, cols, with_abs=True)
    assert np.array_equal(sel, full[np.ix_(rows, cols)])
    assert np.array_equal(sel_abs, full_abs[np.ix_(rows, cols)])
    assert np.array_equal(oracle.gemm_f64_select(A, B, None, cols), full[:, cols])


def test_thread_count_does_not_change_result():
    A, B = inputs.gemm_operands(70, 30, 200, seed=8, kind="uniform")
    one = oracle.gemm_f64(A, B, nthreads=1)
    many = oracle.gemm_f64(A, B, nthreads=7)
    assert np.array_equal(one, many)


def test_signed_extremes():
    # fp16 extremes: 65504² fits fp64 exactly; subnormal products stay exact.
    A = np.array([[65504, -65504, 2 ** -24]], dtype=np.float16)
    B = np.array([[65504, 65504, 2 ** -24], [1, 1, 1]], dtype=np.float16)
    C = oracle.gemm_f64(A, B)
    assert C[0, 0] == 65504.0 * 65504 - 65504.0 * 65504 + 2.0 ** -48
    assert C[0, 1] == 2.0 ** -24
