"""The allocation-free split-K entry point against the existing one and the oracle.

wgemm_f16f32_splitk_noalloc is for callers that may not allocate device
memory while they run; its split-K flags sit in a fixed array inside the
library image instead of a workspace the library allocates. This file runs
last, so a failure here leaves every other test already run. It passes on its
own in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-3, 1e-6
SPLIT = 1
CONFIG = "g2_512x256_s4_a1_tma"


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build_oracle()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return wgemm.load()


def _both(A, B, M, N, K, splits):
    """Two no-alloc calls in a row, and the existing entry point on the same
    operands with the same configuration and split."""
    h = torch.cuda.current_stream().cuda_stream
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    lda, ldb = A.shape[1], B.shape[1]
    outs = []
    for _ in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        rc = wgemm.wgemm_f16f32_splitk_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N,
                                               K, lda, ldb, N, splits, h)
        assert rc == 0, wgemm.STATUS_NAMES.get(rc, rc)
        assert wgemm.wgemm_check(h) == 0, wgemm.wgemm_last_device_error()
        outs.append(C.cpu().numpy().astype(np.float64))
    ref = torch.full((M, N), float("nan"), device="cuda")
    rc = wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), ref.data_ptr(), M, N, K, lda,
                                   ldb, N, wgemm.config_id(CONFIG), SPLIT, splits, h)
    assert rc == 0
    assert wgemm.wgemm_check(h) == 0
    return outs, ref.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K,splits", [(1024, 1024, 8192, 9), (300, 700, 2000, 3),
                                          (256, 512, 640, 1)])
def test_noalloc_matches_existing_entry_point(M, N, K, splits):
    for kind in ("int", "uniform"):
        A, B = inputs.gemm_operands(M, N, K, seed=M + splits, kind=kind)
        outs, ref = _both(A, B, M, N, K, splits)
        exact, exact_abs = oracle.gemm_f64(A, B, with_abs=True)
        if kind == "int":
            # Exact arithmetic: both entry points and the oracle agree exactly.
            assert np.array_equal(ref, exact)
            for got in outs:
                assert np.array_equal(got, ref)
                assert np.array_equal(got, exact)
        else:
            # Within the tolerance the other tests use: against the other
            # entry point, and against the oracle's fp64 sum.
            bound = RTOL * exact_abs + ATOL
            for got in outs:
                assert np.all(np.abs(got - ref) <= bound)
                assert np.all(np.abs(got - exact) <= bound)


def test_noalloc_rejects_problems_beyond_its_array():
    # 8192 × 8192 with 9 splits needs 32 · 16 · 2 · 9 = 9216 words: fits;
    # 16384 × 16384 with 9 splits needs 64 · 32 · 2 · 9 = 36864 > 16384 words.
    M = N = 16384
    K = 1024
    rc = wgemm.wgemm_f16f32_splitk_noalloc(1 << 20, 1 << 20, 1 << 20, M, N, K, K, K, N, 9, None)
    assert rc == -8
    before = wgemm.wgemm_workspace_bytes()
    A, B = inputs.gemm_operands(256, 512, 640, seed=1, kind="int")
    outs, ref = _both(A, B, 256, 512, 640, 2)
    assert np.array_equal(outs[1], ref)
    assert np.array_equal(outs[1], oracle.gemm_f64(A, B))
    assert wgemm.wgemm_workspace_bytes() == before  # the no-alloc calls took no workspace
