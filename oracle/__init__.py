"""CPU oracle for C = A·Bᵀ (fp16 or bf16 in, fp64 accumulation), loaded through ctypes.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline / reference arm use it. The GEMM library never imports it, and it
imports nothing from the GEMM library.

The arithmetic lives in `wgemm_oracle.c` (plain C, built with gcc by
`oracle.build_oracle()`); this file only marshals numpy arrays. fp16 matrices
are numpy float16 arrays; bf16 matrices are numpy uint16 arrays of bf16 bit
patterns (numpy has no bf16 type).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wgemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    # -ffp-contract=off: every product and sum is a separate IEEE operation.
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_gemm_f64_select_t.argtypes = [p, p, p, i64, p, i64, i64, i64, i64, p, p,
                                                     i64, ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_f64_select_t.restype = ctypes.c_int
            lib.oracle_gemm_f64_t.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64,
                                              ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_f64_t.restype = ctypes.c_int
            lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
            lib.oracle_f64_to_f16.restype = ctypes.c_uint16
            lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
            lib.oracle_round_f64.argtypes = [p, p, i64, ctypes.c_int]
            lib.oracle_round_f64.restype = ctypes.c_int
            lib.oracle_decode_array.argtypes = [p, p, i64, ctypes.c_int]
            lib.oracle_decode_array.restype = ctypes.c_int
            lib.oracle_gemm_f64.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm_f64.restype = ctypes.c_int
            lib.oracle_gemm_f64_select.argtypes = [p, p, p, i64, p, i64, i64, i64, i64, p, p, i64,
                                                   ctypes.c_int]
            lib.oracle_gemm_f64_select.restype = ctypes.c_int
            lib.oracle_hardware_threads.argtypes = []
            lib.oracle_hardware_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


F16, BF16 = 1, 2  # operand / rounding types of the C entry points


def _operand_type(x: np.ndarray) -> int:
    """float16 arrays hold fp16 values; uint16 arrays hold bf16 bit patterns."""
    if x.dtype == np.float16:
        return F16
    if x.dtype == np.uint16:
        return BF16
    raise TypeError("operands must be float16 (fp16) or uint16 (bf16 bit patterns)")


def _as_rows(x: np.ndarray, name: str) -> np.ndarray:
    if x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D array")
    _operand_type(x)
    if x.strides[1] != 2 or x.strides[0] % 2:
        raise ValueError(f"{name} must have unit column stride")
    return x


def _types(A: np.ndarray, B: np.ndarray) -> int:
    t = _operand_type(A)
    if _operand_type(B) != t:
        raise TypeError("A and B must have the same element type")
    return t


def f16_to_f64(bits: int) -> float:
    """Decode one fp16 bit pattern (the oracle's own decoder)."""
    return _load().oracle_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    """Decode one bf16 bit pattern (the oracle's own decoder)."""
    return _load().oracle_bf16_to_f64(bits)


def decode_array(bits: np.ndarray, kind: str) -> np.ndarray:
    """Decode an array of fp16 ("f16") or bf16 ("bf16") bit patterns with the
    oracle's decoders."""
    t = {"f16": F16, "bf16": BF16}[kind]
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.empty(flat.shape, dtype=np.float64)
    if _load().oracle_decode_array(_ptr(flat), _ptr(out), flat.size, t) != 0:
        raise RuntimeError("oracle_decode_array failed")
    return out.reshape(np.shape(bits))


def bf16_to_f64_array(bits: np.ndarray) -> np.ndarray:
    """Decode an array of bf16 bit patterns with the oracle's decoder."""
    return decode_array(bits, "bf16")


def epilogue_f64(C: np.ndarray, alpha: float, beta: float = 0.0, Cin: np.ndarray | None = None,
                 bias: np.ndarray | None = None) -> np.ndarray:
    """The fused epilogue's definition in fp64 on the oracle's sum C:
    D = alpha·C + beta·Cin + bias[None, :] (Cin as values, bias per column).
    It follows no passage of the pages, which measure the plain product; it
    is the declared contract of the library's fused entry point."""
    D = float(alpha) * C
    if beta != 0.0:
        D = D + float(beta) * np.asarray(Cin, dtype=np.float64)
    if bias is not None:
        D = D + np.asarray(bias, dtype=np.float64)[None, :]
    return D


def round_f64(x: np.ndarray, to: str) -> np.ndarray:
    """x rounded to fp16 ("f16") or bf16 ("bf16"), to nearest with ties to
    even; returns the uint16 bit patterns."""
    kind = {"f16": F16, "bf16": BF16}[to]
    xs = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(xs.shape, dtype=np.uint16)
    if _load().oracle_round_f64(_ptr(xs), _ptr(out), xs.size, kind) != 0:
        raise RuntimeError("oracle_round_f64 failed")
    return out


def hardware_threads() -> int:
    return _load().oracle_hardware_threads()


def gemm_f64(A: np.ndarray, B: np.ndarray, K: int | None = None, with_abs: bool = False,
             nthreads: int = 0):
    """C = A[:, :K]·B[:, :K]ᵀ in fp64 (and |A|·|B|ᵀ if with_abs).

    A is M×lda and B is N×ldb, both fp16 (float16) or both bf16 (uint16 bit
    patterns), row-major, lda, ldb ≥ K; columns past K are never read.
    Returns C, or (C, Cabs).
    """
    A = _as_rows(A, "A")
    B = _as_rows(B, "B")
    t = _types(A, B)
    M, N = A.shape[0], B.shape[0]
    K = A.shape[1] if K is None else K
    lda, ldb = A.strides[0] // 2, B.strides[0] // 2
    if K > A.shape[1] or K > B.shape[1]:
        raise ValueError("K exceeds an operand's columns")
    C = np.zeros((M, N), dtype=np.float64)
    Cabs = np.zeros((M, N), dtype=np.float64) if with_abs else None
    if t == F16:
        rc = _load().oracle_gemm_f64(_ptr(A), _ptr(B), _ptr(C), _ptr(Cabs), M, N, K, lda, ldb, N,
                                     nthreads)
    else:
        rc = _load().oracle_gemm_f64_t(_ptr(A), _ptr(B), _ptr(C), _ptr(Cabs), M, N, K, lda, ldb,
                                       N, nthreads, t)
    if rc < 0:
        raise RuntimeError(f"oracle_gemm_f64 failed ({rc})")
    return (C, Cabs) if with_abs else C


def gemm_f64_select(A: np.ndarray, B: np.ndarray, rows: np.ndarray | None,
                    cols: np.ndarray | None, K: int | None = None, with_abs: bool = False,
                    nthreads: int = 0):
    """C[rows][:, cols] of A·Bᵀ in fp64 (None = every row / column)."""
    A = _as_rows(A, "A")
    B = _as_rows(B, "B")
    t = _types(A, B)
    K = A.shape[1] if K is None else K
    lda, ldb = A.strides[0] // 2, B.strides[0] // 2
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = A.shape[0] if r is None else len(r)
    nc = B.shape[0] if c is None else len(c)
    if r is not None and len(r) and (r.min() < 0 or r.max() >= A.shape[0]):
        raise IndexError("row index out of range")
    if c is not None and len(c) and (c.min() < 0 or c.max() >= B.shape[0]):
        raise IndexError("column index out of range")
    C = np.zeros((nr, nc), dtype=np.float64)
    Cabs = np.zeros((nr, nc), dtype=np.float64) if with_abs else None
    rc = _load().oracle_gemm_f64_select_t(_ptr(A), _ptr(B), _ptr(r), nr, _ptr(c), nc, K, lda,
                                          ldb, _ptr(C), _ptr(Cabs), nc, nthreads, t)
    if rc < 0:
        raise RuntimeError(f"oracle_gemm_f64_select failed ({rc})")
    return (C, Cabs) if with_abs else C
