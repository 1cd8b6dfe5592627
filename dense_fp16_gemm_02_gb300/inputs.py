"""Seeded synthetic inputs for C = A·Bᵀ (A: M×K, B: N×K, row-major; fp16, or
bf16 given as uint16 bit patterns).

This module holds no GEMM arithmetic. It is the one piece that both the CUDA
path (tests, bench) and the CPU oracle are fed from, so that both see the same
matrices.

Generator. A counter-based SplitMix64 stream (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014; the constants are the
ones of Vigna's public-domain splitmix64.c):

    mix64(z):  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9
               z ^= z >> 27; z *= 0x94D049BB133111EB
               z ^= z >> 31
    key        = mix64(seed · 2^16 + tensor_id)
    h(i)       = mix64(key + (i + 1) · 0x9E3779B97F4A7C15)     (mod 2^64)

`i` is the logical row-major index row·cols + col, independent of the leading
dimension. With key = 0, h(0) is the first output of SplitMix64 seeded with 0.

Values.
* "uniform": u = (h >> 11) · 2^-53 in [0, 1), x = 2u − 1, rounded to fp16
  with round-to-nearest-even (numpy's float64 → float16 cast keeps fp16
  subnormals).
* "int": v = ((h >> 32) · 5) >> 32, x = v − 2 in {−2, …, 2} (exact in fp16).
* dtype "bf16": the same x (the uniform draw 2u − 1 before any rounding, or
  the integer), rounded to bf16 with round-to-nearest-even: with
  x = m · 2^e, m in [0.5, 1), the significand m · 2^8 is rounded to an integer
  (numpy's rint: ties to even) and scaled back; the result is exact in fp32,
  whose upper 16 bits are the bf16 pattern.

The pages measured on integers in [−3, 3] from a hash of the index
("SASS-Level Kernel Generation for Blackwell", How we measured); the
workloads here use uniform[−1, 1] fp16 plus a {−2..2} integer copy.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK = (1 << 64) - 1

# fp16 and bf16 quiet NaNs, used to poison padding columns so that a reader
# that strays past K is caught.
F16_NAN_BITS = 0x7E00
BF16_NAN_BITS = 0x7FC0


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2^64)."""
    z &= _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> int:
    return mix64_int(seed * (1 << 16) + tensor_id)


def hash_stream(key: int, start: int, count: int) -> np.ndarray:
    """h(i) for i in [start, start + count), as uint64."""
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + idx * _GAMMA)


def _draws(h: np.ndarray, kind: str) -> np.ndarray:
    """The values before rounding to the element type, as float64."""
    if kind == "uniform":
        u = (h >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        return 2.0 * u - 1.0
    if kind == "int":
        with np.errstate(over="ignore"):
            v = ((h >> np.uint64(32)) * np.uint64(5)) >> np.uint64(32)
        return (v.astype(np.int64) - 2).astype(np.float64)
    raise ValueError(f"unknown value kind {kind!r}")


def bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """float64 values (|x| within fp32's normal range or 0) rounded to bf16,
    to nearest with ties to even; returns the uint16 bit patterns."""
    m, e = np.frexp(x)
    y = np.ldexp(np.rint(m * 256.0), e - 8)  # 8 significant bits, exact in fp32
    return (y.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _values(h: np.ndarray, kind: str, dtype: str) -> np.ndarray:
    x = _draws(h, kind)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        return bf16_bits_rne(x)
    raise ValueError(f"unknown element type {dtype!r}")


def matrix(rows: int, cols: int, seed: int, tensor_id: int, kind: str = "uniform",
           ld: int | None = None, pad: str = "zero",
           chunk_elems: int = 1 << 22, dtype: str = "f16") -> np.ndarray:
    """A rows×ld array whose first `cols` columns hold the seeded stream:
    float16 for dtype "f16", uint16 bf16 bit patterns for dtype "bf16".

    Columns [cols, ld) are padding: zeros (pad="zero") or NaN (pad="nan").
    The stream index of element (r, c) is r·cols + c, so the values do not
    depend on `ld`.
    """
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("ld < cols")
    if dtype not in ("f16", "bf16"):
        raise ValueError(f"unknown element type {dtype!r}")
    out = np.empty((rows, ld), dtype=np.float16 if dtype == "f16" else np.uint16)
    if ld > cols:
        if pad == "nan":
            out[:, cols:].view(np.uint16)[...] = F16_NAN_BITS if dtype == "f16" else BF16_NAN_BITS
        else:
            out[:, cols:] = 0
    if rows == 0 or cols == 0:
        return out
    key = stream_key(seed, tensor_id)
    rows_per_chunk = max(1, chunk_elems // cols)

    def fill(r0: int) -> None:
        r1 = min(rows, r0 + rows_per_chunk)
        h = hash_stream(key, r0 * cols, (r1 - r0) * cols)
        out[r0:r1, :cols] = _values(h, kind, dtype).reshape(r1 - r0, cols)

    starts = range(0, rows, rows_per_chunk)
    if len(starts) == 1:
        fill(0)
    else:  # chunks are independent; numpy releases the GIL inside them
        with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, starts))
    return out


def gemm_operands(M: int, N: int, K: int, seed: int, kind: str = "uniform",
                  lda: int | None = None, ldb: int | None = None,
                  pad: str = "zero", dtype: str = "f16") -> tuple[np.ndarray, np.ndarray]:
    """The A (M×lda) and B (N×ldb) operands of one problem (tensor ids 0 and
    1), fp16 or bf16 (bit patterns)."""
    A = matrix(M, K, seed, 0, kind, lda, pad, dtype=dtype)
    B = matrix(N, K, seed, 1, kind, ldb, pad, dtype=dtype)
    return A, B


def sample_indices(n: int, count: int, seed: int, tensor_id: int) -> np.ndarray:
    """`count` distinct sorted indices in [0, n) that always include 0 and n−1.

    Used to check large problems on a sampled set of rows and columns.
    """
    if count >= n:
        return np.arange(n, dtype=np.int64)
    h = hash_stream(stream_key(seed, tensor_id), 0, 4 * count + 64)
    picked = {0, n - 1}
    for v in (h % np.uint64(n)).astype(np.int64):
        if len(picked) >= count:
            break
        picked.add(int(v))
    j = 0
    while len(picked) < count:  # only for pathological collisions
        picked.add(j)
        j += 1
    return np.array(sorted(picked), dtype=np.int64)
