"""GPU parity past 2^31 elements: C, A or B holding more elements than a
signed 32-bit index reaches, so every address the kernels and the host form
must be 64-bit. Checked against the CPU oracle on sampled rows and columns
that include those past the 2^31-element boundary, exact on integer inputs
(every partial sum is an integer below 2^24 in magnitude; "SASS-Level Kernel
Generation for Blackwell", section "The numbers": C = A·Bᵀ, fp16 in, fp32
accumulation and output).

The sizes: C of 139264 × 16384 fp32 (2.28·10^9 elements, 9.1 GB), and A or
B of 40000 × 65536 fp16 (2.62·10^9 elements, 5.2 GB)."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

pytestmark = pytest.mark.gpu

TWO31 = 1 << 31


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build_oracle()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return wgemm.load()


def pick(n: int, boundary: int, seed: int) -> np.ndarray:
    """Sorted distinct indices in [0, n): both ends, both sides of
    `boundary` (the first index whose elements lie past 2^31), and a sample."""
    fixed = set(range(0, 4)) | set(range(n - 4, n))
    fixed |= {i for i in range(boundary - 4, boundary + 4) if 0 <= i < n}
    sampled = inputs.sample_indices(n, 16, seed=seed, tensor_id=7)
    return np.array(sorted(fixed | {int(i) for i in sampled}), dtype=np.int64)


def check_status():
    rc = wgemm.wgemm_check(torch.cuda.current_stream().cuda_stream)
    assert rc == 0, (rc, wgemm.wgemm_last_device_error())


def exact(got: np.ndarray, ref: np.ndarray, what: str):
    bad = np.argwhere(got.astype(np.float64) != ref)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first {bad[:5].tolist()}"


@pytest.mark.parametrize("config", [None, "g1_128x256_s4_a2_direct", "g2_256x256_s6_a2_tma"])
def test_c_past_2_31_elements(lib, config):
    # The default choice, a register-store epilogue and a TMA-store epilogue.
    M, N, K = 139264, 16384, 64
    assert M * N > TWO31
    A, B = inputs.gemm_operands(M, N, K, seed=77, kind="int")
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    wgemm.gemm(dA, dB, C, config=config)
    check_status()
    rows = pick(M, TWO31 // N, seed=1)
    got = C.index_select(0, torch.from_numpy(rows).cuda()).cpu().numpy()
    del C, dA, dB
    torch.cuda.empty_cache()
    exact(got, oracle.gemm_f64(A[rows], B, K=K), f"C past 2^31 elements, config {config}")


@pytest.mark.parametrize("side", ["A", "B"])
def test_operand_past_2_31_elements(lib, side):
    # The default choice (the rule's, for this off-table shape).
    big, small, K = 40000, 512, 65536
    M, N = (big, small) if side == "A" else (small, big)
    assert big * K > TWO31
    A, B = inputs.gemm_operands(M, N, K, seed=78, kind="int")
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = wgemm.gemm(dA, dB)
    check_status()
    got = C.cpu().numpy()
    del C, dA, dB
    torch.cuda.empty_cache()
    if side == "A":
        rows, cols = pick(M, TWO31 // K, seed=2), np.arange(N)
    else:
        rows, cols = pick(M, 0, seed=3), pick(N, TWO31 // K, seed=4)
    exact(got[np.ix_(rows, cols)], oracle.gemm_f64(A[rows], B[cols], K=K),
          f"{side} past 2^31 elements")
