"""Pins of the oracle's bf16 operands and 16-bit roundings (CPU only).

The oracle decodes bf16 from its bit fields and rounds fp64 sums to fp16 or
bf16 from the formats' definitions (wgemm_oracle.c). These tests hold each
piece against something other than itself: numpy's reinterpretation of a bf16
pattern as the upper half of an fp32, numpy's float64 → float16 cast, torch's
float32 → bfloat16 cast, exact midpoints between neighbouring values (ties to
even), and exact integer arithmetic.
"""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_02_gb300 import inputs

ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def np_bf16_decode(bits: np.ndarray) -> np.ndarray:
    """numpy's reading of bf16 patterns: the upper 16 bits of an fp32."""
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def test_bf16_decoder_matches_fp32_upper_half_for_all_patterns():
    got = oracle.bf16_to_f64_array(ALL)
    ref = np_bf16_decode(ALL)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def finite_positive(fmt):
    """Ascending finite positive values of a 16-bit format, and their patterns."""
    if fmt == "f16":
        bits = np.arange(1, 0x7C00, dtype=np.uint16)
        vals = bits.view(np.float16).astype(np.float64)
    else:
        bits = np.arange(1, 0x7F80, dtype=np.uint16)
        vals = np_bf16_decode(bits)
    return bits, vals


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_encoder_is_identity_on_representable_values(fmt):
    bits, vals = finite_positive(fmt)
    assert np.array_equal(oracle.round_f64(vals, fmt), bits)
    assert np.array_equal(oracle.round_f64(-vals, fmt), bits | np.uint16(0x8000))
    z = oracle.round_f64(np.array([0.0, -0.0]), fmt)
    assert z.tolist() == [0, 0x8000]


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_encoder_rounds_midpoints_to_even_and_neighbours_to_nearest(fmt):
    bits, vals = finite_positive(fmt)
    lo, hi = vals[:-1], vals[1:]
    mid = (lo + hi) / 2  # exact: both are far coarser than fp64
    even = np.where(bits[:-1] % 2 == 0, bits[:-1], bits[1:])
    assert np.array_equal(oracle.round_f64(mid, fmt), even)
    above = np.nextafter(mid, np.inf)
    below = np.nextafter(mid, -np.inf)
    assert np.array_equal(oracle.round_f64(above, fmt), bits[1:])
    assert np.array_equal(oracle.round_f64(below, fmt), bits[:-1])
    # Below the least subnormal: half of it rounds to zero (tie, 0 is even),
    # anything above half rounds up to it.
    least = vals[0]
    assert oracle.round_f64(np.array([least / 2]), fmt)[0] == 0
    assert oracle.round_f64(np.array([np.nextafter(least / 2, 1)]), fmt)[0] == 1


@pytest.mark.parametrize("fmt,max_bits,inf_bits", [("f16", 0x7BFF, 0x7C00),
                                                   ("bf16", 0x7F7F, 0x7F80)])
def test_encoder_overflow_threshold(fmt, max_bits, inf_bits):
    bits, vals = finite_positive(fmt)
    vmax = vals[-1]
    assert bits[-1] == max_bits
    ulp = vmax - vals[-2]
    edge = vmax + ulp / 2  # the tie goes to the even neighbour: infinity
    # 1.5·vmax lies in the binade just above the largest one, with fraction
    # bits set: it must still become infinity, not a pattern of that binade.
    got = oracle.round_f64(np.array([vmax, np.nextafter(edge, 0), edge, 1.5 * vmax, 4 * vmax,
                                     np.inf, -edge]), fmt)
    assert got.tolist() == [max_bits, max_bits, inf_bits, inf_bits, inf_bits, inf_bits,
                            inf_bits | 0x8000]
    nan = oracle.round_f64(np.array([np.nan]), fmt)[0]
    assert (nan & inf_bits) == inf_bits and (nan & ~np.uint16(0xFC00 if fmt == "f16"
                                                               else 0xFF80)) != 0


def test_f16_encoder_matches_numpy_cast():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(200_000) * np.exp2(rng.uniform(-30, 17, 200_000))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.round_f64(x, "f16"), ref)


def test_bf16_encoder_matches_torch_on_fp32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-120, 120, 200_000)))
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_f64(x.astype(np.float64), "bf16"), ref)


@pytest.mark.parametrize("M,N,K", [(3, 5, 7), (17, 1, 33), (64, 64, 64), (47, 53, 59)])
def test_bf16_gemm_exact_on_integers(M, N, K):
    A, B = inputs.gemm_operands(M, N, K, seed=9, kind="int", lda=K + 8, ldb=K + 16,
                                dtype="bf16")
    Ai = np_bf16_decode(A[:, :K]).astype(np.int64)
    Bi = np_bf16_decode(B[:, :K]).astype(np.int64)
    assert set(np.unique(Ai)) <= {-2, -1, 0, 1, 2}
    got = oracle.gemm_f64(A, B, K=K)
    assert np.array_equal(got, (Ai @ Bi.T).astype(np.float64))


def test_bf16_gemm_against_independent_fp64_matmul():
    M, N, K = 33, 29, 97
    A, B = inputs.gemm_operands(M, N, K, seed=4, kind="uniform", dtype="bf16")
    Ad, Bd = np_bf16_decode(A), np_bf16_decode(B)
    C, Cabs = oracle.gemm_f64(A, B, with_abs=True)
    ref = Ad @ Bd.T
    # Products are exact; two fp64 sums of K terms differ by at most 2·K·eps·Σ|ab|.
    assert np.all(np.abs(C - ref) <= 2 * K * np.finfo(np.float64).eps * Cabs)
    assert np.allclose(Cabs, np.abs(Ad) @ np.abs(Bd).T, rtol=1e-12, atol=0)


def test_bf16_gemm_identity_and_nan_padding():
    K = 37
    _, B = inputs.gemm_operands(K, 5, K, seed=5, kind="uniform", dtype="bf16")
    eye = inputs.bf16_bits_rne(np.eye(K))
    assert np.array_equal(oracle.gemm_f64(eye, B), np_bf16_decode(B).T)
    A, B = inputs.gemm_operands(9, 11, 13, seed=2, kind="uniform", lda=24, ldb=16, pad="nan",
                                dtype="bf16")
    assert np.isfinite(oracle.gemm_f64(A, B, K=13)).all()


def test_bf16_select_equals_full():
    A, B = inputs.gemm_operands(40, 50, 70, seed=6, kind="uniform", dtype="bf16")
    full = oracle.gemm_f64(A, B)
    rows, cols = np.array([0, 7, 39]), np.array([1, 2, 49])
    assert np.array_equal(oracle.gemm_f64_select(A, B, rows, cols), full[np.ix_(rows, cols)])


def test_mixed_operand_types_rejected():
    A = inputs.matrix(4, 8, 1, 0)
    B = inputs.matrix(4, 8, 1, 1, dtype="bf16")
    with pytest.raises(TypeError):
        oracle.gemm_f64(A, B)


def test_fused_epilogue_equals_one_gemm_over_concatenated_k():
    """alpha·A·Bᵀ + beta·A2·B2ᵀ + bias = [alpha·A | beta·A2 | 1]·[B | B2 | bias]ᵀ
    (concatenation along K): the epilogue's definition pinned against the
    GEMM definition itself, exact on small integers."""
    M, N, K1, K2 = 23, 17, 40, 24
    alpha, beta = 2.0, -3.0
    A, B = inputs.gemm_operands(M, N, K1, seed=11, kind="int")
    A2, B2 = inputs.gemm_operands(M, N, K2, seed=12, kind="int")
    bias = (np.arange(N) % 7 - 3).astype(np.float64)
    C = oracle.gemm_f64(A, B)
    Cin = oracle.gemm_f64(A2, B2)
    D = oracle.epilogue_f64(C, alpha, beta, Cin, bias)
    Acat = np.concatenate([(alpha * A.astype(np.float64)).astype(np.float16),
                           (beta * A2.astype(np.float64)).astype(np.float16),
                           np.ones((M, 1), dtype=np.float16)], axis=1)
    Bcat = np.concatenate([B, B2, bias.astype(np.float16)[:, None]], axis=1)
    assert np.array_equal(D, oracle.gemm_f64(Acat, Bcat))
    # beta = 0 never reads Cin; no bias adds nothing
    assert np.array_equal(oracle.epilogue_f64(C, 1.0, 0.0, None, None), C)


def test_decode_array_matches_scalar_decoders():
    bits = np.arange(0, 1 << 16, 97, dtype=np.uint32).astype(np.uint16)
    f = oracle.decode_array(bits, "f16")
    b = oracle.decode_array(bits, "bf16")
    sf = np.array([oracle.f16_to_f64(int(x)) for x in bits])
    sb = np.array([oracle.bf16_to_f64(int(x)) for x in bits])
    assert np.array_equal(np.isnan(f), np.isnan(sf)) and np.array_equal(f[~np.isnan(f)],
                                                                        sf[~np.isnan(sf)])
    assert np.array_equal(np.isnan(b), np.isnan(sb)) and np.array_equal(b[~np.isnan(b)],
                                                                        sb[~np.isnan(sb)])
