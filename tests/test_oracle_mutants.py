"""The oracle's pins catch plausible mistakes.

Copies of the oracle's C source with one planted mistake each (a dropped term,
a wrong sign, a transposed operand, a swapped leading dimension, a wrong fp16
or bf16 exponent bias or field width, a subnormal decoded as normal, a thread
writing the wrong row, Cabs losing its absolute value, bf16 operands decoded
as fp16, a 16-bit rounding that ties away, truncates, keeps a bit too many,
mis-rounds subnormals or overflows late) are compiled on the CPU, and the same
checks the pins in test_oracle.py and test_oracle_types.py make are run on
each mutant: every mutant must fail at least one of them, and the unmodified
source must pass them all.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from dense_fp16_gemm_02_gb300 import inputs

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                          "wgemm_oracle.c")

# (name, text in the source, replacement)
MUTANTS = [
    ("drops the last k term", "for (int64_t k = 0; k < j->K; ++k)\n                s += a[k] * b[k];",
     "for (int64_t k = 0; k + 1 < j->K; ++k)\n                s += a[k] * b[k];"),
    ("subtracts instead of adds", "s += a[k] * b[k];", "s -= a[k] * b[k];"),
    ("transposes B (reads column k of row j from the wrong place)",
     "Bd[c * K + k] = decode(B[jrow * ldb + k]);",
     "Bd[c * K + k] = decode(B[(k % (jrow + 1)) * ldb + (jrow % (K > 0 ? K : 1))]);"),
    ("uses ldb for A", "a[k] = j->decode(j->A[i * j->lda + k]);",
     "a[k] = j->decode(j->A[i * j->ldb + k]);"),
    ("exponent bias off by one", "ldexp((double)(1024 + fraction), exponent - 25)",
     "ldexp((double)(1024 + fraction), exponent - 24)"),
    ("subnormals decoded as normals", "v = ldexp((double)fraction, -24);",
     "v = ldexp((double)(1024 + fraction), -25);"),
    ("writes row r + 1", "j->C[r * j->ldc + c] = s;",
     "j->C[((r + 1) % j->n_rows) * j->ldc + c] = s;"),
    ("drops the sign bit", "return sign ? -v : v;", "return v;"),
    ("Cabs without absolute values", "sa += fabs(a[k]) * fabs(b[k]);", "sa += a[k] * b[k];"),
    ("reads one column past K", "for (int64_t k = 0; k < K; ++k)\n            Bd[c * K + k]",
     "for (int64_t k = 0; k < K; ++k)\n            Bd[c * K + k] = (k + 1 < K) ? decode(B[jrow * ldb + k + 1]) : 0;\n        for (int64_t k = 0; k < 0; ++k)\n            Bd[c * K + k]"),
    ("bf16 exponent bias off by one", "ldexp((double)(128 + fraction), exponent - 134)",
     "ldexp((double)(128 + fraction), exponent - 133)"),
    ("bf16 fraction field one bit wide", "const int fraction = h & 0x7F;",
     "const int fraction = h & 0xFF;"),
    ("bf16 operands decoded as fp16",
     "ab_type == ORACLE_BF16 ? oracle_bf16_to_f64 : oracle_f16_to_f64",
     "ab_type == ORACLE_BF16 ? oracle_f16_to_f64 : oracle_f16_to_f64"),
    ("rounding ties away from zero",
     "if (rest > 0.5 || (rest == 0.5 && fmod(fl, 2.0) == 1.0))", "if (rest >= 0.5)"),
    ("rounding truncates", "if (rest > 0.5 || (rest == 0.5 && fmod(fl, 2.0) == 1.0))",
     "if (rest > 1.0)"),
    ("bf16 rounding keeps one bit too many", "return round_to_format(x, 8, 8);",
     "return round_to_format(x, 9, 8);"),
    ("subnormals rounded at their own binade", "if (E < emin)\n        E = emin;",
     "if (E < emin - 100)\n        E = emin;"),
    ("overflow one binade late", "if (E > emax)\n        return", "if (E > emax + 1)\n        return"),
]


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o",
                    str(lib), str(src), "-lm"], check=True)
    L = ctypes.CDLL(str(lib))
    i64, p = ctypes.c_int64, ctypes.c_void_p
    L.oracle_gemm_f64.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int]
    L.oracle_gemm_f64.restype = ctypes.c_int
    L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_f16_to_f64.restype = ctypes.c_double
    L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f64.restype = ctypes.c_double
    L.oracle_gemm_f64_t.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int,
                                    ctypes.c_int]
    L.oracle_gemm_f64_t.restype = ctypes.c_int
    L.oracle_round_f64.argtypes = [p, p, i64, ctypes.c_int]
    L.oracle_round_f64.restype = ctypes.c_int
    return L


def _gemm(L, A, B, K=None, with_abs=False, nthreads=3):
    M, N = A.shape[0], B.shape[0]
    K = A.shape[1] if K is None else K
    C = np.zeros((M, N))
    Cabs = np.zeros((M, N)) if with_abs else None
    ptr = lambda x: None if x is None else x.ctypes.data_as(ctypes.c_void_p)
    rc = L.oracle_gemm_f64(ptr(A), ptr(B), ptr(C), ptr(Cabs), M, N, K, A.strides[0] // 2,
                           B.strides[0] // 2, N, nthreads)
    assert rc >= 0
    return (C, Cabs) if with_abs else C


def _pins(L):
    """The pins of test_oracle.py, restated compactly; returns the failures."""
    failed = []
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([L.oracle_f16_to_f64(int(b)) for b in bits])
    ok = np.isnan(ref)
    if not (np.array_equal(np.isnan(got), ok) and np.array_equal(got[~ok], ref[~ok])):
        failed.append("decoder")
    for (M, N, K) in [(3, 5, 7), (17, 1, 33), (64, 64, 64), (47, 53, 59)]:
        A, B = inputs.gemm_operands(M, N, K, seed=7, kind="int", lda=K + 8, ldb=K + 16)
        exact = A[:, :K].astype(np.int64) @ B[:, :K].astype(np.int64).T
        if not np.array_equal(_gemm(L, A, B, K=K), exact.astype(np.float64)):
            failed.append(f"integer {M}x{N}x{K}")
            break
    A, B = inputs.gemm_operands(9, 11, 13, seed=2, kind="uniform")
    C, Cabs = _gemm(L, A, B, with_abs=True)
    if not np.allclose(np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)).T, Cabs,
                       rtol=1e-12, atol=0):
        failed.append("abs term")
    K = 37
    _, B = inputs.gemm_operands(K, 5, K, seed=5, kind="uniform")
    if not np.array_equal(_gemm(L, np.eye(K, dtype=np.float16), B), B.astype(np.float64).T):
        failed.append("identity")
    M, N, K = 10, 14, 33
    A = np.tile(((np.arange(M) % 5) - 2).astype(np.float16)[:, None], (1, K))
    B = np.tile(((np.arange(N) % 7) - 3).astype(np.float16)[:, None], (1, K))
    if not np.array_equal(_gemm(L, A, B),
                          (K * np.outer((np.arange(M) % 5) - 2, (np.arange(N) % 7) - 3))
                          .astype(np.float64)):
        failed.append("separable")
    A, B = inputs.gemm_operands(9, 11, 13, seed=2, kind="uniform", lda=24, ldb=16, pad="nan")
    if not np.isfinite(_gemm(L, A, B, K=13)).all():
        failed.append("padding")
    failed += _type_pins(L)
    return failed


def _np_bf16(bits):
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _round(L, x, kind):
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    assert L.oracle_round_f64(x.ctypes.data_as(ctypes.c_void_p),
                              out.ctypes.data_as(ctypes.c_void_p), x.size, kind) == 0
    return out


def _type_pins(L):
    """The pins of test_oracle_types.py, restated compactly."""
    failed = []
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = _np_bf16(bits)
    got = np.array([L.oracle_bf16_to_f64(int(b)) for b in bits])
    ok = np.isnan(ref)
    if not (np.array_equal(np.isnan(got), ok) and np.array_equal(got[~ok], ref[~ok])):
        failed.append("bf16 decoder")
    for kind, top in ((1, 0x7C00), (2, 0x7F80)):
        b = np.arange(1, top, dtype=np.uint16)
        v = b.view(np.float16).astype(np.float64) if kind == 1 else _np_bf16(b)
        if not np.array_equal(_round(L, v, kind), b):
            failed.append(f"encoder identity {kind}")
        mid = (v[:-1] + v[1:]) / 2
        even = np.where(b[:-1] % 2 == 0, b[:-1], b[1:])
        if not np.array_equal(_round(L, mid, kind), even):
            failed.append(f"encoder ties {kind}")
        if not np.array_equal(_round(L, np.nextafter(mid, np.inf), kind), b[1:]):
            failed.append(f"encoder above midpoints {kind}")
        edge = v[-1] + (v[-1] - v[-2]) / 2
        if _round(L, np.array([edge]), kind)[0] != top or \
                _round(L, np.array([1.5 * v[-1]]), kind)[0] != top or \
                _round(L, np.array([np.nextafter(edge, 0)]), kind)[0] != top - 1:
            failed.append(f"encoder overflow {kind}")
    M, N, K = 17, 13, 33
    A, B = inputs.gemm_operands(M, N, K, seed=9, kind="int", lda=K + 8, ldb=K + 16, dtype="bf16")
    exact = _np_bf16(A[:, :K]).astype(np.int64) @ _np_bf16(B[:, :K]).astype(np.int64).T
    C = np.zeros((M, N))
    ptr = lambda x: x.ctypes.data_as(ctypes.c_void_p)
    rc = L.oracle_gemm_f64_t(ptr(A), ptr(B), ptr(C), None, M, N, K, A.strides[0] // 2,
                             B.strides[0] // 2, N, 2, 2)
    if rc < 0 or not np.array_equal(C, exact.astype(np.float64)):
        failed.append("bf16 integer gemm")
    return failed


def test_unmodified_oracle_passes_every_pin(tmp_path):
    L = _build(tmp_path, "clean", open(ORACLE_SRC).read())
    assert _pins(L) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(ORACLE_SRC).read()
    assert old in text, f"mutation site not found: {name}"
    L = _build(tmp_path, "mutant", text.replace(old, new, 1))
    assert _pins(L), f"no pin caught the planted mistake: {name}"
