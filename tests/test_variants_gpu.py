"""GPU parity of the adjacent element types: bf16 operands, and fp16 / bf16 C.

Same kernels as the fp16 → fp32 product (bf16 operands change only the MMA
instruction descriptor and the tensor maps; a 16-bit C changes the epilogue),
held against the CPU oracle on the same seeded inputs:
* integer inputs in {-2..2}: bit-exact. Every partial sum is an integer below
  2^24, so the fp32 accumulator is the exact sum, and a 16-bit C is that exact
  sum rounded once to nearest-even — the oracle's rounding of its fp64 sum.
* uniform[-1, 1] inputs: |C − C_ref| ≤ 2e-3·(|A|·|B|ᵀ) + 1e-6, plus for a
  16-bit C half a unit in the last place of the 16-bit result (the final
  rounding).
"""
import re

import numpy as np
import pytest
import torch

import oracle
from config_names import plain_16bit, plain_fp32
from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-3, 1e-6
DP = wgemm.MODE_DATA_PARALLEL
TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build_oracle()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return wgemm.load()


def ceil8(k):
    return (k + 7) // 8 * 8


def operands(M, N, K, seed, kind, ab):
    return inputs.gemm_operands(M, N, K, seed=seed, kind=kind, lda=ceil8(K), ldb=ceil8(K),
                                pad="nan", dtype=ab)


def upload(x: np.ndarray, ab: str) -> torch.Tensor:
    if ab == "f16":
        return torch.from_numpy(x).cuda()
    return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)


def run(A, B, K, ab, c, config=None, mode=-1, C=None):
    dA, dB = upload(A, ab), upload(B, ab)
    if C is None:  # row pitch a multiple of 16 bytes, as the TMA epilogue needs
        M, N = A.shape[0], B.shape[0]
        C = torch.empty((M, ceil8(N)), dtype=TORCH[c], device="cuda")[:, :N]
    out = wgemm.gemm(dA[:, :K], dB[:, :K], C, config=config, mode=mode)
    status = wgemm.wgemm_check(torch.cuda.current_stream().cuda_stream)
    assert status == 0, (status, wgemm.wgemm_last_device_error())
    return out


def host_values(C: torch.Tensor, c: str):
    """(values as float64, bit patterns or None) of a result tensor."""
    if c == "f32":
        return C.cpu().numpy().astype(np.float64), None
    bits = C.cpu().view(torch.int16).numpy().view(np.uint16)
    if c == "f16":
        return bits.view(np.float16).astype(np.float64), bits
    with np.errstate(invalid="ignore"):
        vals = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return vals, bits


def half_ulp(x: np.ndarray, c: str) -> np.ndarray:
    """Half a unit in the last place of a 16-bit format at magnitude |x|."""
    if c == "f32":
        return np.zeros_like(x)
    p, emin = (11, -14) if c == "f16" else (8, -126)
    _, e2 = np.frexp(np.abs(x))
    E = np.maximum(e2 - 1, emin)
    return np.ldexp(0.5, E - (p - 1))


def check(C, A, B, K, kind, c, what, rows=None, cols=None):
    vals, bits = host_values(C, c)
    if rows is not None or cols is not None:
        vals = vals[np.ix_(rows, cols)] if rows is not None and cols is not None else (
            vals[rows, :] if rows is not None else vals[:, cols])
        if bits is not None:
            bits = bits[np.ix_(rows, cols)] if rows is not None and cols is not None else (
                bits[rows, :] if rows is not None else bits[:, cols])
    if kind == "int":
        ref = oracle.gemm_f64_select(A, B, rows, cols, K=K)
        if c == "f32":
            bad = np.argwhere(vals != ref)
        else:
            bad = np.argwhere(bits != oracle.round_f64(ref, c))
        assert bad.size == 0, f"{what}: {len(bad)} mismatches, first {bad[:5].tolist()}"
    else:
        ref, ref_abs = oracle.gemm_f64_select(A, B, rows, cols, K=K, with_abs=True)
        err = np.abs(vals - ref)
        bound = RTOL * ref_abs + ATOL + half_ulp(np.maximum(np.abs(ref), np.abs(vals)), c)
        ok = err <= bound
        assert ok.all(), f"{what}: {(~ok).sum()} outside tolerance, max excess " \
                         f"{(err - bound).max()}"


def names_by_width():
    """Plain (not fused) configurations: (fp32 C, 16-bit C)."""
    names = [n for n in wgemm.config_names() if "_ab" not in n]
    return ([n for n in names if not n.endswith("_h")], [n for n in names if n.endswith("_h")])


# ------------------------------------------------------------------ bf16 operands, fp32 C

@pytest.mark.parametrize("name", plain_fp32())
def test_bf16_inputs_every_fp32_config(name):
    M, N, K = 600, 1100, 300
    for kind in ("int", "uniform"):
        A, B = operands(M, N, K, 500 + plain_fp32().index(name), kind, "bf16")
        C = run(A, B, K, "bf16", "f32", config=name, mode=DP)
        check(C, A, B, K, kind, "f32", f"{name} bf16 {kind}")


def test_bf16_inputs_split_and_stream_k():
    fp32, _ = names_by_width()
    M, N, K = 300, 520, 1000
    A, B = operands(M, N, K, 77, "int", "bf16")
    for name in [n for n in fp32 if n.endswith("_tma") and not re.match(r"g\dm2_", n)]:
        cid = wgemm.config_id(name)
        for mode, splits in ((wgemm.MODE_SPLIT_K, 3), (wgemm.MODE_STREAM_K, 1)):
            dA, dB = upload(A, "bf16"), upload(B, "bf16")
            C = torch.empty((M, N), dtype=torch.float32, device="cuda")
            rc = wgemm.wgemm_gemm_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                                         wgemm.WGEMM_BF16, wgemm.WGEMM_F32, M, N, K,
                                         dA.stride(0), dB.stride(0), N, cid, mode, splits, None)
            assert rc == 0
            assert wgemm.wgemm_check(None) == 0
            check(C, A, B, K, "int", "f32", f"{name} bf16 mode {mode}")


# ------------------------------------------------------------------ 16-bit C

@pytest.mark.parametrize("c", ["f16", "bf16"])
@pytest.mark.parametrize("name", plain_16bit())
def test_16bit_output_every_config(name, c):
    M, N, K = 600, 1100, 300
    for ab in ("f16", "bf16"):
        for kind in ("int", "uniform"):
            A, B = operands(M, N, K, 700 + plain_16bit().index(name), kind, ab)
            C = run(A, B, K, ab, c, config=name, mode=DP)
            check(C, A, B, K, kind, c, f"{name} {ab}->{c} {kind}")


@pytest.mark.parametrize("name", plain_16bit())
def test_16bit_output_multi_round(name):
    # More tiles than workers, ragged edges; integer sums up to ±544 so bf16 C
    # rounds (8 significant bits): both sides round the same exact sum.
    M, N, K = 2600, 7000, 136
    A, B = operands(M, N, K, 900 + plain_16bit().index(name), "int", "bf16")
    ref = oracle.round_f64(oracle.gemm_f64(A, B, K=K), "bf16")
    for _ in range(2):
        C = run(A, B, K, "bf16", "bf16", config=name, mode=DP)
        _, bits = host_values(C, "bf16")
        bad = np.argwhere(bits != ref)
        assert bad.size == 0, f"{name}: {len(bad)} mismatches, first {bad[:5].tolist()}"


@pytest.mark.parametrize("ab,c", [("bf16", "f32"), ("f16", "f16"), ("bf16", "bf16"),
                                  ("f16", "bf16"), ("bf16", "f16")])
def test_default_path_every_type_pair(ab, c):
    M, N, K = 1000, 1500, 520
    for kind in ("int", "uniform"):
        A, B = operands(M, N, K, 31, kind, ab)
        C = run(A, B, K, ab, c)
        check(C, A, B, K, kind, c, f"default {ab}->{c} {kind}")


def test_typed_shorthands():
    M, N, K = 300, 520, 200
    A, B = operands(M, N, K, 41, "int", "bf16")
    dA, dB = upload(A, "bf16"), upload(B, "bf16")
    Af, Bf = operands(M, N, K, 42, "int", "f16")
    dAf, dBf = upload(Af, "f16"), upload(Bf, "f16")
    ld = ceil8(K)
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert wgemm.wgemm_bf16f32(dA.data_ptr(), dB.data_ptr(), C32.data_ptr(), M, N, K, ld, ld, N,
                               None) == 0
    Cbf = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert wgemm.wgemm_bf16bf16(dA.data_ptr(), dB.data_ptr(), Cbf.data_ptr(), M, N, K, ld, ld, N,
                                None) == 0
    Ch = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert wgemm.wgemm_f16f16(dAf.data_ptr(), dBf.data_ptr(), Ch.data_ptr(), M, N, K, ld, ld, N,
                              None) == 0
    assert wgemm.wgemm_check(None) == 0
    check(C32, A, B, K, "int", "f32", "bf16f32")
    check(Cbf, A, B, K, "int", "bf16", "bf16bf16")
    check(Ch, Af, Bf, K, "int", "f16", "f16f16")


def test_16bit_unaligned_c_rows():
    # ldc = N + 1: rows 2-byte aligned only. The default path stores from
    # registers; a forced TMA-epilogue configuration is refused.
    M, N, K = 300, 517, 200
    A, B = operands(M, N, K, 51, "int", "f16")
    full = torch.full((M, N + 1), -7.0, dtype=torch.float16, device="cuda")
    C = full[:, :N]
    run(A, B, K, "f16", "f16", C=C)
    check(C, A, B, K, "int", "f16", "unaligned ldc")
    assert torch.all(full[:, N] == -7.0)
    dA, dB = upload(A, "f16"), upload(B, "f16")
    cid = wgemm.config_id("g2_256x256_s6_a2_tma_h")
    rc = wgemm.wgemm_gemm_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), wgemm.WGEMM_F16,
                                 wgemm.WGEMM_F16, M, N, K, ceil8(K), ceil8(K), N + 1, cid, DP, 1,
                                 None)
    assert rc == -2


def test_16bit_k_zero_and_width_errors():
    M, N = 130, 64  # 16-bit rows of 128 bytes: TMA-aligned, so only the width decides
    C = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    dA = torch.zeros((M, 8), dtype=torch.bfloat16, device="cuda")
    dB = torch.zeros((N, 8), dtype=torch.bfloat16, device="cuda")
    assert wgemm.wgemm_bf16bf16(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, 0, 8, 8, N,
                                None) == 0
    assert wgemm.wgemm_check(None) == 0
    assert torch.all(C.view(torch.int16) == 0)
    fp32_id = wgemm.config_id("g2_256x256_s6_a2_tma")
    h_id = wgemm.config_id("g2_256x256_s6_a2_tma_h")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    args = (dA.data_ptr(), dB.data_ptr())
    assert wgemm.wgemm_gemm_config(*args, C.data_ptr(), wgemm.WGEMM_BF16, wgemm.WGEMM_BF16, M, N,
                                   8, 8, 8, N, fp32_id, DP, 1, None) == -6
    assert wgemm.wgemm_gemm_config(*args, C32.data_ptr(), wgemm.WGEMM_BF16, wgemm.WGEMM_F32, M,
                                   N, 8, 8, 8, N, h_id, DP, 1, None) == -6
    assert wgemm.wgemm_gemm_config(*args, C.data_ptr(), wgemm.WGEMM_BF16, wgemm.WGEMM_BF16, M, N,
                                   8, 8, 8, N, h_id, wgemm.MODE_SPLIT_K, 2, None) == -6
    assert wgemm.wgemm_check(None) == 0


@pytest.mark.parametrize("ab,c", [("bf16", "bf16"), ("bf16", "f32"), ("f16", "f16")])
def test_4096_cubed_sampled(ab, c):
    n = 4096
    A, B = inputs.gemm_operands(n, n, n, seed=4000, kind="uniform", dtype=ab)
    C = run(A, B, n, ab, c)
    rows = inputs.sample_indices(n, 64, 5, 2)
    cols = inputs.sample_indices(n, 64, 5, 3)
    check(C, A, B, n, "uniform", c, f"4096^3 {ab}->{c} rows", rows=rows)
    check(C, A, B, n, "uniform", c, f"4096^3 {ab}->{c} cols", cols=cols)
    del C
    torch.cuda.empty_cache()
