"""Programmatic dependent launch keeps stream order (GPU).

With PDL on, a wgemm kernel may be scheduled before the previous kernel on the
stream has finished; it must still read only the previous kernel's finished
output. Two checks, launched back to back with no synchronisation between the
calls:
* a chain X_{i+1} = X_i · P_iᵀ with fp16 C, each call reading the previous
  call's output as A, where P_i are permutation matrices (X_{i+1} is X_i with
  its columns permuted, so values never grow and the exact result is the
  composed permutation of X_0). Every intermediate buffer starts as NaN: a read
  that ran ahead of its producer would carry NaN or stale values into the end.
* repeated split-K calls into one C with alternating inputs: each call zeroes
  C and adds partial tiles; a call that started before the previous one had
  finished its adds would leave a mixture. The last result must be exact.
"""
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
    lib = wgemm.load()
    prev = wgemm.wgemm_set_pdl(True)
    yield lib
    wgemm.wgemm_set_pdl(bool(prev))


def permutation_matrix(n, seed):
    perm = np.random.default_rng(seed).permutation(n)
    P = np.zeros((n, n), dtype=np.float16)
    P[np.arange(n), perm] = 1  # row j of P selects column perm[j]: (X·Pᵀ)[:, j] = X[:, perm[j]]
    return P, perm


@pytest.mark.parametrize("config", [None, "g2_256x256_s6_a2_tma_h", "g2_256x256_s6_a2_direct_clc_h",
                                    "g2_512x256_s4_a1_tma_h", "g1_128x128_s6_a2_tma_h"])
def test_chain_reads_previous_output(config):
    M, N, L = 1000, 512, 24
    X0 = inputs.matrix(M, N, 61, 0, "int")
    perms = [permutation_matrix(N, 100 + i) for i in range(L)]
    dP = [torch.from_numpy(P).cuda() for P, _ in perms]
    bufs = [torch.from_numpy(X0).cuda()] + [
        torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for _ in range(L)]
    torch.cuda.synchronize()
    cid = -1 if config is None else wgemm.config_id(config)
    for i in range(L):
        if cid < 0:
            rc = wgemm.wgemm_gemm(bufs[i].data_ptr(), dP[i].data_ptr(), bufs[i + 1].data_ptr(),
                                  wgemm.WGEMM_F16, wgemm.WGEMM_F16, M, N, N, N, N, N, None)
        else:
            rc = wgemm.wgemm_gemm_config(bufs[i].data_ptr(), dP[i].data_ptr(),
                                         bufs[i + 1].data_ptr(), wgemm.WGEMM_F16,
                                         wgemm.WGEMM_F16, M, N, N, N, N, N, cid, 0, 1, None)
        assert rc == 0
    assert wgemm.wgemm_check(None) == 0
    expect = X0.astype(np.float64)
    for _, perm in perms:
        expect = expect[:, perm]
    got = bufs[L].cpu().numpy().astype(np.float64)
    assert np.array_equal(got, expect)
    # the first step against the oracle too (the permutation reading of P)
    ref1 = oracle.gemm_f64(X0, perms[0][0])
    assert np.array_equal(bufs[1].cpu().numpy().astype(np.float64), ref1)


def test_back_to_back_split_k_into_one_c():
    M, N, K, reps = 512, 1024, 4096, 16
    pairs = [inputs.gemm_operands(M, N, K, seed=70 + j, kind="int") for j in range(2)]
    dev = [(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()) for A, B in pairs]
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    cid = wgemm.config_id("g2_512x256_s4_a1_tma")
    for r in range(reps):
        dA, dB = dev[r % 2]
        rc = wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K,
                                       N, cid, wgemm.MODE_SPLIT_K, 8, None)
        assert rc == 0
    assert wgemm.wgemm_check(None) == 0
    A, B = pairs[(reps - 1) % 2]
    assert np.array_equal(C.cpu().numpy().astype(np.float64), oracle.gemm_f64(A, B))


def test_pdl_and_plain_calls_interleave():
    # PDL calls after a torch kernel that writes the operand: the GEMM must see
    # the torch kernel's result (an ordinary kernel triggers its dependents
    # only at completion).
    M, N, K = 640, 520, 256
    A, B = inputs.gemm_operands(M, N, K, seed=80, kind="int")
    dA = torch.full((M, K), float("nan"), dtype=torch.float16, device="cuda")
    dB = torch.from_numpy(B).cuda()
    hA = torch.from_numpy(A).cuda()
    for _ in range(8):
        dA.fill_(float("nan"))
        dA.copy_(hA)
        C = wgemm.gemm(dA, dB)
    assert wgemm.wgemm_check(None) == 0
    assert np.array_equal(C.cpu().numpy().astype(np.float64), oracle.gemm_f64(A, B))
