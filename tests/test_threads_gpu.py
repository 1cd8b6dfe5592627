"""Several host threads calling the library at once, each on its own stream:
the device-pointer call (the per-shape choice), a forced split-K call and
the host-buffer call, interleaved. The library's shared state (per-device
set-up, the per-stream flag workspaces, the host-buffer copy streams) must
keep every result exact against the CPU oracle on integer inputs
("SASS-Level Kernel Generation for Blackwell", section "The numbers":
C = A·Bᵀ, fp16 in, fp32 accumulation and output)."""
import threading

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

pytestmark = pytest.mark.gpu

THREADS, ROUNDS = 4, 4
SHAPES = {
    "default": (600, 700, 520),
    "split_k": (256, 512, 8192),
    "host": (700, 500, 640),
}
SPLIT_CONFIG, SPLIT_MODE, SPLITS = "g1_128x256_s4_a2_tma", 1, 4


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build_oracle()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return wgemm.load()


def test_threads_on_their_own_streams(lib):
    # Operands per (thread, round, kind), generated before the threads start.
    work = {}
    for t in range(THREADS):
        for r in range(ROUNDS):
            for j, (kind, (M, N, K)) in enumerate(SHAPES.items()):
                work[t, r, kind] = inputs.gemm_operands(M, N, K, seed=300 + 37 * t + 7 * r + j,
                                                        kind="int")
    # One call of each kind first, outside the threads (per-device set-up).
    for kind, (M, N, K) in SHAPES.items():
        A, B = work[0, 0, kind]
        if kind == "host":
            hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
            wgemm.gemm_from_host(hA, hB)
            torch.cuda.synchronize()
        else:
            cfg = dict(config=SPLIT_CONFIG, mode=SPLIT_MODE, splits=SPLITS) if kind == "split_k" else {}
            wgemm.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), **cfg)
    torch.cuda.synchronize()

    results, errors = {}, []

    def worker(t):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            keep = []  # host operands stay untouched until the stream is done
            with torch.cuda.stream(s):
                for r in range(ROUNDS):
                    for kind, (M, N, K) in SHAPES.items():
                        A, B = work[t, r, kind]
                        if kind == "host":
                            hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
                            keep += [hA, hB]
                            C = wgemm.gemm_from_host(hA, hB, stream=s)
                        else:
                            cfg = (dict(config=SPLIT_CONFIG, mode=SPLIT_MODE, splits=SPLITS)
                                   if kind == "split_k" else {})
                            C = wgemm.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(),
                                           stream=s, **cfg)
                        results[t, r, kind] = C
            s.synchronize()
            rc = wgemm.wgemm_check(s.cuda_stream)
            if rc != 0:
                errors.append((t, rc, wgemm.wgemm_last_device_error()))
        except Exception as e:  # reported below, on the main thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a thread did not finish"
    assert not errors, errors
    assert len(results) == THREADS * ROUNDS * len(SHAPES)
    for (t, r, kind), C in results.items():
        A, B = work[t, r, kind]
        got = (C if not C.is_cuda else C.cpu()).numpy().astype(np.float64)
        bad = np.argwhere(got != oracle.gemm_f64(A, B))
        assert bad.size == 0, f"thread {t} round {r} {kind}: {len(bad)} mismatches"
