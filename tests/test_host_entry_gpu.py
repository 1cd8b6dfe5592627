"""GPU parity of wgemm_f16f32_host (A, B and C in host memory, uploads and
downloads pipelined with row panels of A and blocks of B's rows) against the
CPU oracle:
exact on integer inputs, |C − C_ref| ≤ 2e-3·(|A|·|B|ᵀ) + 1e-6 on uniform
inputs ("SASS-Level Kernel Generation for Blackwell", section "The numbers",
the setup paragraph: C = A·Bᵀ, fp16 in, fp32 accumulation and output)."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-3, 1e-6


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build_oracle()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    lib = wgemm.load()
    yield lib
    lib.wgemm_debug_set_host_panels(0)
    lib.wgemm_debug_set_host_blocks(0)


def host_call(A, B, M, N, K, lda, ldb, ldc, stream=None, sentinel=np.nan):
    """A (M×lda), B (N×ldb) fp16 numpy with pitches; C comes back M×ldc with
    the columns past N untouched (sentinel)."""
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.full((M, ldc), sentinel, dtype=torch.float32).pin_memory()
    na, nb, nc = wgemm.host_device_elems(M, N, K)
    dA = torch.empty(max(na, 1), dtype=torch.float16, device="cuda")
    dB = torch.empty(max(nb, 1), dtype=torch.float16, device="cuda")
    dC = torch.empty(max(nc, 1), dtype=torch.float32, device="cuda")
    s = stream or torch.cuda.current_stream()
    rc = wgemm.wgemm_f16f32_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), M, N, K, lda, ldb,
                                 ldc, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), s.cuda_stream)
    return rc, hC, (dA, dB, dC, hA, hB), s


def finish(rc, s):
    assert rc == 0, wgemm.status_string(rc)
    s.synchronize()
    status = wgemm.wgemm_check(s.cuda_stream)
    assert status == 0, (status, wgemm.wgemm_last_device_error())


def check(hC, A, B, M, N, K, kind, what):
    got = hC.numpy()[:, :N].astype(np.float64)
    if kind == "int":
        ref = oracle.gemm_f64(A, B, K=K)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, f"{what}: {len(bad)} mismatches, first {bad[:5].tolist()}"
    else:
        ref, ref_abs = oracle.gemm_f64(A, B, K=K, with_abs=True)
        err = np.abs(got - ref)
        assert (err <= RTOL * ref_abs + ATOL).all(), f"{what}: outside tolerance"


@pytest.mark.parametrize("panels,blocks", [(0, 0), (2, 0), (4, 0), (0, 2), (3, 2), (3, 4)])
@pytest.mark.parametrize("kind", ["int", "uniform"])
def test_host_buffers_with_panels(lib, kind, panels, blocks):
    # Host pitches above the row lengths; K not a multiple of 8 (device
    # pitch 528); N not a multiple of 4 (device pitch 780); with 4 panels the
    # rows split 256 + 256 + 256 + 232, with 2 blocks the columns 512 + 265
    # (the second block's C starts 512 floats into each device row), with 4
    # blocks 256 + 256 + 256 + 9 (two before A, two after).
    M, N, K = 1000, 777, 521
    lda, ldb, ldc = K + 3, K + 11, N + 5
    A, B = inputs.gemm_operands(M, N, K, seed=41 + panels + 10 * blocks, kind=kind, lda=lda,
                                ldb=ldb)
    assert lib.wgemm_debug_set_host_panels(panels) >= 0
    assert lib.wgemm_debug_set_host_blocks(blocks) >= 0
    try:
        rc, hC, keep, s = host_call(A, B, M, N, K, lda, ldb, ldc)
        finish(rc, s)
    finally:
        lib.wgemm_debug_set_host_panels(0)
        lib.wgemm_debug_set_host_blocks(0)
    check(hC, A, B, M, N, K, kind, f"host buffers, {panels} panels, {blocks} blocks")
    assert np.isnan(hC.numpy()[:, N:]).all(), "columns past N were written"


@pytest.mark.parametrize("blocks", [0, 4])
def test_host_buffers_default_panels_at_8192(lib, blocks):
    # The rule's own split: min(A, C) = 128 MiB gives eight panels of 1024
    # rows; B (128 MiB) stays one block unless the hook asks for four, the
    # split the rule gives a B of 512 MiB (16384³).
    M = N = K = 8192
    assert lib.wgemm_debug_host_panel_rows(M, N, K) == 1024
    assert lib.wgemm_debug_host_block_cols(N, K) == 8192
    A, B = inputs.gemm_operands(M, N, K, seed=43 + blocks, kind="int")
    assert lib.wgemm_debug_set_host_blocks(blocks) >= 0
    try:
        rc, hC, keep, s = host_call(A, B, M, N, K, K, K, N)
        finish(rc, s)
    finally:
        lib.wgemm_debug_set_host_blocks(0)
    rows = np.r_[0:32, 1008:1056, 4080:4112, 7152:7200, 8160:8192]  # seams between panels
    ref = oracle.gemm_f64(A[rows], B, K=K)
    got = hC.numpy()[rows].astype(np.float64)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"


def test_host_buffers_k_zero_and_empty(lib):
    M, N = 300, 260
    A = np.zeros((M, 8), dtype=np.float16)
    B = np.zeros((N, 8), dtype=np.float16)
    rc, hC, keep, s = host_call(A, B, M, N, 0, 8, 8, N, sentinel=7.0)
    finish(rc, s)
    assert (hC.numpy() == 0).all()  # the empty sum
    rc, hC, keep, s = host_call(A, B, 0, N, 8, 8, 8, N, sentinel=7.0)
    assert rc == 0


def test_host_buffers_on_two_streams_at_once(lib):
    shapes = [(2048, 1536, 1024), (1536, 2048, 2048)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    runs = []
    for i, ((M, N, K), st) in enumerate(zip(shapes, streams)):
        A, B = inputs.gemm_operands(M, N, K, seed=50 + i, kind="int")
        runs.append((host_call(A, B, M, N, K, K, K, N, stream=st), A, B, M, N, K))
    for (rc, hC, keep, s), A, B, M, N, K in runs:
        finish(rc, s)
        check(hC, A, B, M, N, K, "int", f"{M}x{N}x{K} on its own stream")


def test_gemm_from_host_helper(lib):
    M, N, K = 700, 900, 640
    A, B = inputs.gemm_operands(M, N, K, seed=60, kind="int")
    C = wgemm.gemm_from_host(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory())
    torch.cuda.current_stream().synchronize()
    check(C, A, B, M, N, K, "int", "gemm_from_host")


def test_host_buffer_argument_errors(lib):
    z = torch.zeros(64, dtype=torch.float16, device="cuda")
    h = torch.zeros(64, dtype=torch.float16).pin_memory()
    c = torch.zeros(64, dtype=torch.float32).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    call = wgemm.wgemm_f16f32_host
    assert call(h.data_ptr(), h.data_ptr(), c.data_ptr(), 4, 4, 8, 7, 8, 4, z.data_ptr(),
                z.data_ptr(), z.data_ptr(), s) == -1  # lda < K
    assert call(h.data_ptr(), h.data_ptr(), c.data_ptr(), 4, 4, 8, 8, 8, 4, z.data_ptr() + 2,
                z.data_ptr(), z.data_ptr(), s) == -2  # device A off 16 bytes


def test_host_buffers_split_k_shape(lib):
    # The table runs 1024×1024×65536 as split-K 9: through the host call it
    # stays one launch (one panel, one block, even with the hooks asking for
    # more), with the K split, exact on integers.
    M, N, K = 1024, 1024, 65536
    assert wgemm.wgemm_select(M, N, K)[1] == 1  # split-K
    A, B = inputs.gemm_operands(M, N, K, seed=44, kind="int")
    assert lib.wgemm_debug_set_host_panels(4) >= 0
    assert lib.wgemm_debug_set_host_blocks(2) >= 0
    try:
        rc, hC, keep, s = host_call(A, B, M, N, K, K, K, N)
        finish(rc, s)
    finally:
        lib.wgemm_debug_set_host_panels(0)
        lib.wgemm_debug_set_host_blocks(0)
    check(hC, A, B, M, N, K, "int", "split-K shape through the host call")


def test_host_buffers_pageable_and_with_pdl(lib):
    # Pageable host memory (plain numpy arrays) works, only without overlap;
    # programmatic dependent launch on does not change the result.
    M, N, K = 1500, 900, 700
    A, B = inputs.gemm_operands(M, N, K, seed=70, kind="int")
    C = np.full((M, N), np.nan, dtype=np.float32)
    na, nb, nc = wgemm.host_device_elems(M, N, K)
    dA = torch.empty(na, dtype=torch.float16, device="cuda")
    dB = torch.empty(nb, dtype=torch.float16, device="cuda")
    dC = torch.empty(nc, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    prev = wgemm.wgemm_set_pdl(True)
    try:
        assert lib.wgemm_debug_set_host_panels(3) >= 0
        rc = wgemm.wgemm_f16f32_host(A.ctypes.data, B.ctypes.data, C.ctypes.data, M, N, K, K, K,
                                     N, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                                     s.cuda_stream)
        finish(rc, s)
    finally:
        lib.wgemm_debug_set_host_panels(0)
        wgemm.wgemm_set_pdl(bool(prev))
    check(torch.from_numpy(C), A, B, M, N, K, "int", "pageable host buffers, PDL on")
