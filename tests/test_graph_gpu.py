"""The product call inside a CUDA graph: captured after one warm-up call (which
sets up the configuration, its tensor-map encoder and, for K-split plans,
the flag workspace), replayed twice, and checked against the CPU oracle
(exact on integer inputs: "SASS-Level Kernel Generation for Blackwell",
section "The numbers", C = A·Bᵀ with fp16 in and fp32 out)."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build_oracle()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return wgemm.load()


# A data-parallel single-CTA tile, a pair tile, and a shape the rule runs as
# split-K outside a capture (inside one it takes a data-parallel plan).
SHAPES = [(1024, 1024, 1024), (2048, 1536, 1024), (1024, 1024, 16384)]


def test_calls_captured_in_a_graph_and_replayed():
    cases = []
    for i, (M, N, K) in enumerate(SHAPES):
        A, B = inputs.gemm_operands(M, N, K, seed=80 + i, kind="int")
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        C = torch.full((M, N), float("nan"), device="cuda")
        cases.append((M, N, K, A, B, dA, dB, C))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for M, N, K, A, B, dA, dB, C in cases:  # warm-up outside the capture
            assert wgemm.wgemm_f16f32(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K,
                                      N, s.cuda_stream) == 0
    s.synchronize()
    for *_, C in cases:
        C.fill_(float("nan"))
    assert wgemm.wgemm_select(1024, 1024, 16384)[1] == 1  # split-K outside a capture
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        h = torch.cuda.current_stream().cuda_stream
        for M, N, K, A, B, dA, dB, C in cases:
            rc = wgemm.wgemm_f16f32(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K, N,
                                    h)
            assert rc == 0, wgemm.status_string(rc)
        # A K split forced inside the capture is refused, and nothing is enqueued.
        M, N, K, A, B, dA, dB, C = cases[2]
        cid = wgemm.config_id("g2_256x256_s6_a2_tma")
        assert wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K,
                                         K, N, cid, 1, 4, h) == -6
        assert wgemm.wgemm_f16f32_splitk_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M,
                                                 N, K, K, K, N, 4, h) == -6
    torch.cuda.synchronize()
    for rep in range(2):
        for *_, C in cases:
            C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert wgemm.wgemm_check(torch.cuda.current_stream().cuda_stream) == 0
        for M, N, K, A, B, dA, dB, C in cases:
            got = C.cpu().numpy().astype(np.float64)
            ref = oracle.gemm_f64(A, B)
            bad = np.argwhere(got != ref)
            assert bad.size == 0, f"{M}x{N}x{K} replay {rep}: {len(bad)} mismatches"


def test_host_buffer_call_captured_in_a_graph(lib):
    # The host-buffer call's copy streams join the capture through its events:
    # the replayed graph uploads, computes in panels and downloads.
    M, N, K = 1200, 1000, 640
    A, B = inputs.gemm_operands(M, N, K, seed=90, kind="int")
    hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    na, nb, nc = wgemm.host_device_elems(M, N, K)
    dA = torch.empty(na, dtype=torch.float16, device="cuda")
    dB = torch.empty(nb, dtype=torch.float16, device="cuda")
    dC = torch.empty(nc, dtype=torch.float32, device="cuda")
    call = lambda h: wgemm.wgemm_f16f32_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), M, N,
                                             K, K, K, N, dA.data_ptr(), dB.data_ptr(),
                                             dC.data_ptr(), h)
    assert lib.wgemm_debug_set_host_panels(3) >= 0
    assert lib.wgemm_debug_set_host_blocks(4) >= 0
    try:
        s = torch.cuda.Stream()
        assert call(s.cuda_stream) == 0  # warm-up outside the capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            assert call(torch.cuda.current_stream().cuda_stream) == 0
    finally:
        lib.wgemm_debug_set_host_panels(0)
        lib.wgemm_debug_set_host_blocks(0)
    for rep in range(2):
        hC.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = hC.numpy().astype(np.float64)
        bad = np.argwhere(got != oracle.gemm_f64(A, B))
        assert bad.size == 0, f"replay {rep}: {len(bad)} mismatches"
