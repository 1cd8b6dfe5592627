"""GPU parity of the fused epilogue D = alpha·A·Bᵀ + beta·Cin + bias[column].

Every fused configuration ("_ab": fp32 D, "_ab_h": 16-bit D), against the
oracle's sum and its epilogue definition on the same seeded inputs:
* integer inputs, integer alpha, beta, Cin and bias: every value the kernel
  forms in fp32 is an integer below 2^24, so fp32 D is bit-exact and a 16-bit
  D is the exact value rounded once to nearest-even, bit for bit;
* uniform inputs and real alpha, beta, bias: |D − D_ref| within
  |alpha|·(2e-3·(|A|·|B|ᵀ) + 1e-6), plus the two fp32 roundings of the
  epilogue's fused multiply-adds (2^-23 of |alpha·C| + |beta·Cin| + |bias|
  each), plus half a unit in the last place of a 16-bit D.
Also: D computed in place over Cin, beta = 0 with no Cin, no bias, K = 0,
many tiles per worker, and the argument checks of the fused entry point.
The reduce-add configurations ("_tma_ab1") serve only the in-place form
D += alpha·A·Bᵀ + bias (beta = 1, fp32 D): they add alpha·sum + bias into
D's old values with TMA reduce-adds, two fp32 roundings as in the general
form, so the same bounds hold.
"""
import numpy as np
import pytest
import torch

import oracle
from config_names import compiled_config_names
from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-3, 1e-6
TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
WT = {"f16": wgemm.WGEMM_F16, "bf16": wgemm.WGEMM_BF16, "f32": wgemm.WGEMM_F32}


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build_oracle()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return wgemm.load()


def ceil8(k):
    return (k + 7) // 8 * 8


def fused_names(width):
    """The Cin-ring fused configurations of one D width."""
    names = [n for n in compiled_config_names() if "_direct_ab" in n]
    return [n for n in names if n.endswith("_h") == (width == 16)]


def reduce_names():
    """The reduce-add fused configurations (in place, beta = 1, fp32 D)."""
    return [n for n in compiled_config_names() if "_tma_ab" in n]


def by_width(cs):
    """(D type, configuration) pairs: every fused configuration of each D type's width."""
    return [(c, n) for c in cs for n in fused_names(32 if c == "f32" else 16)]


def upload(x: np.ndarray, ab: str) -> torch.Tensor:
    if ab == "f16":
        return torch.from_numpy(x).cuda()
    return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)


def to_dev_c(vals: np.ndarray, c: str, ld: int) -> torch.Tensor:
    """A C-typed device matrix holding `vals` (exactly representable), pitch ld."""
    M, N = vals.shape
    t = torch.zeros((M, ld), dtype=TORCH[c], device="cuda")[:, :N]
    t.copy_(torch.from_numpy(vals.astype(np.float32)).cuda().to(TORCH[c]))
    return t


def host_values(D: torch.Tensor, c: str):
    if c == "f32":
        return D.cpu().numpy().astype(np.float64), None
    bits = D.cpu().view(torch.int16).numpy().view(np.uint16)
    return oracle.decode_array(bits, c), bits


def half_ulp(x, c):
    if c == "f32":
        return np.zeros_like(x)
    p, emin = (11, -14) if c == "f16" else (8, -126)
    _, e2 = np.frexp(np.abs(x))
    return np.ldexp(0.5, np.maximum(e2 - 1, emin) - (p - 1))


def run_fused(A, B, K, ab, c, alpha, beta, cin_vals, bias_vals, config=None, in_place=False,
              ldd=None):
    M, N = A.shape[0], B.shape[0]
    ldd = ldd or ceil8(N)
    dA, dB = upload(A, ab), upload(B, ab)
    Cin = None if cin_vals is None else to_dev_c(cin_vals, c, ldd)
    D = Cin if in_place else torch.full((M, ldd), float("nan"), dtype=TORCH[c],
                                        device="cuda")[:, :N]
    bias = None if bias_vals is None else torch.from_numpy(
        bias_vals.astype(np.float32)).cuda()
    out = wgemm.gemm_ex(dA[:, :K], dB[:, :K], D, Cin=Cin, bias=bias, alpha=alpha, beta=beta,
                        config=config)
    status = wgemm.wgemm_check(torch.cuda.current_stream().cuda_stream)
    assert status == 0, (status, wgemm.wgemm_last_device_error())
    return out


def check(D, A, B, K, kind, c, alpha, beta, cin_vals, bias_vals, what):
    vals, bits = host_values(D, c)
    if kind == "int":
        ref = oracle.epilogue_f64(oracle.gemm_f64(A, B, K=K), alpha, beta, cin_vals, bias_vals)
        bad = np.argwhere(vals != ref) if c == "f32" else np.argwhere(bits != oracle.round_f64(ref, c))
        assert bad.size == 0, f"{what}: {len(bad)} mismatches, first {bad[:5].tolist()}"
        return
    C, Cabs = oracle.gemm_f64(A, B, K=K, with_abs=True)
    ref = oracle.epilogue_f64(C, alpha, beta, cin_vals, bias_vals)
    mag = np.abs(alpha * C)
    if beta != 0.0:
        mag = mag + np.abs(beta * cin_vals)
    if bias_vals is not None:
        mag = mag + np.abs(bias_vals)[None, :]
    bound = (abs(alpha) * (RTOL * Cabs + ATOL) + 2.0 * 2.0 ** -23 * mag
             + half_ulp(np.maximum(np.abs(ref), np.abs(vals)), c))
    err = np.abs(vals - ref)
    ok = err <= bound
    assert ok.all(), f"{what}: {(~ok).sum()} outside tolerance, max excess {(err - bound).max()}"


def epilogue_operands(M, N, kind, seed, c):
    """Cin values and bias exactly representable in the C type."""
    if kind == "int":
        cin = inputs.matrix(M, N, seed, 5, "int").astype(np.float64)
        bias = (np.arange(N) % 11 - 5).astype(np.float64)
        return cin, bias, 2.0, -3.0
    cin = inputs.matrix(M, N, seed, 5, "uniform").astype(np.float64)
    if c == "bf16":
        cin = oracle.decode_array(inputs.bf16_bits_rne(cin), "bf16")
    bias = inputs.matrix(1, N, seed, 6, "uniform").astype(np.float64).ravel()
    return cin, bias, 0.75, -0.5


@pytest.mark.parametrize("c,name", by_width(["f32", "f16", "bf16"]))
def test_every_fused_config(c, name):
    idx = fused_names(32 if c == "f32" else 16).index(name)
    M, N, K = 600, 1100, 300
    for ab in ("f16", "bf16"):
        for kind in ("int", "uniform"):
            A, B = inputs.gemm_operands(M, N, K, seed=40 + idx, kind=kind, lda=ceil8(K),
                                        ldb=ceil8(K), pad="nan", dtype=ab)
            cin, bias, alpha, beta = epilogue_operands(M, N, kind, 41 + idx, c)
            D = run_fused(A, B, K, ab, c, alpha, beta, cin, bias, config=name)
            check(D, A, B, K, kind, c, alpha, beta, cin, bias, f"{name} {ab}->{c} {kind}")


@pytest.mark.parametrize("c,name", by_width(["f32", "bf16"]))
def test_fused_multi_round_in_place(c, name):
    # More tiles than workers, ragged edges, D written over Cin.
    idx = fused_names(32 if c == "f32" else 16).index(name)
    M, N, K = 2600, 7000, 136
    A, B = inputs.gemm_operands(M, N, K, seed=50 + idx, kind="int", lda=ceil8(K), ldb=ceil8(K))
    cin, bias, alpha, beta = epilogue_operands(M, N, "int", 51 + idx, c)
    D = run_fused(A, B, K, "f16", c, alpha, beta, cin, bias, config=name, in_place=True)
    check(D, A, B, K, "int", c, alpha, beta, cin, bias, f"{name} in place")


@pytest.mark.parametrize("c", ["f32", "f16", "bf16"])
def test_default_choice_and_partial_epilogues(c):
    M, N, K = 1000, 1500, 520
    A, B = inputs.gemm_operands(M, N, K, seed=60, kind="int")
    cin, bias, alpha, beta = epilogue_operands(M, N, "int", 61, c)
    # full epilogue, default configuration
    D = run_fused(A, B, K, "f16", c, alpha, beta, cin, bias)
    check(D, A, B, K, "int", c, alpha, beta, cin, bias, "default")
    # beta = 0: Cin is not read (none given)
    D = run_fused(A, B, K, "f16", c, alpha, 0.0, None, bias)
    check(D, A, B, K, "int", c, alpha, 0.0, None, bias, "beta 0")
    # no bias
    D = run_fused(A, B, K, "f16", c, alpha, beta, cin, None)
    check(D, A, B, K, "int", c, alpha, beta, cin, None, "no bias")
    # alpha = 1, beta = 0, no bias: the plain product
    D = run_fused(A, B, K, "f16", c, 1.0, 0.0, None, None)
    check(D, A, B, K, "int", c, 1.0, 0.0, None, None, "plain")


def test_fused_k_zero():
    M, N = 300, 260
    dA = torch.zeros((M, 8), dtype=torch.float16, device="cuda")
    dB = torch.zeros((N, 8), dtype=torch.float16, device="cuda")
    cin, bias, alpha, beta = epilogue_operands(M, N, "int", 70, "f32")
    Cin = to_dev_c(cin, "f32", N)
    bias_t = torch.from_numpy(bias.astype(np.float32)).cuda()
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    wgemm.gemm_ex(dA[:, :0], dB[:, :0], D, Cin=Cin, bias=bias_t, alpha=alpha, beta=beta)
    assert wgemm.wgemm_check(None) == 0
    assert np.array_equal(D.cpu().numpy().astype(np.float64), beta * cin + bias[None, :])


def test_fused_argument_checks():
    M, N, K = 256, 264, 64
    dA = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    dB = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    D = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    base = torch.zeros((M, N + 1), dtype=torch.float32, device="cuda")
    Cin_odd = base[:, :N]  # row pitch N + 1 floats: not a multiple of 16 bytes
    F16, F32 = wgemm.WGEMM_F16, wgemm.WGEMM_F32
    a = (dA.data_ptr(), dB.data_ptr(), D.data_ptr())
    assert wgemm.wgemm_gemm_ex(*a, Cin_odd.data_ptr(), None, 1.0, 1.0, F16, F32, M, N, K, K, K,
                               N, N + 1, None) == -2
    assert wgemm.wgemm_gemm_ex(*a, None, None, 1.0, 1.0, F16, F32, M, N, K, K, K, N, N,
                               None) == -1               # beta != 0 without Cin
    assert wgemm.wgemm_gemm_ex(*a, D.data_ptr(), None, float("inf"), 1.0, F16, F32, M, N, K, K,
                               K, N, N, None) == -1
    plain = wgemm.config_id("g2_256x256_s6_a2_direct")
    assert wgemm.wgemm_gemm_ex_config(*a, D.data_ptr(), None, 2.0, 1.0, F16, F32, M, N, K, K, K,
                                      N, N, plain, None) == -6
    fused_h = fused_names(16)[0]
    assert wgemm.wgemm_gemm_ex_config(*a, D.data_ptr(), None, 2.0, 1.0, F16, F32, M, N, K, K, K,
                                      N, N, wgemm.config_id(fused_h), None) == -6
    # a fused configuration through the plain entry point
    assert wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), M, N, K, K, K,
                                     N, wgemm.config_id(fused_names(32)[0]), 0, 1, None) == -6
    assert wgemm.wgemm_check(None) == 0


@pytest.mark.parametrize("name", reduce_names())
def test_every_reduce_config_in_place(name):
    idx = reduce_names().index(name)
    M, N, K = 600, 1100, 300
    for ab in ("f16", "bf16"):
        for kind in ("int", "uniform"):
            A, B = inputs.gemm_operands(M, N, K, seed=80 + idx, kind=kind, lda=ceil8(K),
                                        ldb=ceil8(K), pad="nan", dtype=ab)
            cin, bias, alpha, _ = epilogue_operands(M, N, kind, 81 + idx, "f32")
            for b in (bias, None):
                D = run_fused(A, B, K, ab, "f32", alpha, 1.0, cin, b, config=name,
                              in_place=True)
                check(D, A, B, K, kind, "f32", alpha, 1.0, cin, b,
                      f"{name} {ab} {kind} bias={b is not None}")


@pytest.mark.parametrize("name", reduce_names())
def test_reduce_multi_round(name):
    # More tiles than workers, ragged edges: every tile is added exactly once.
    idx = reduce_names().index(name)
    M, N, K = 2600, 7000, 136
    A, B = inputs.gemm_operands(M, N, K, seed=90 + idx, kind="int", lda=ceil8(K), ldb=ceil8(K))
    cin, bias, alpha, _ = epilogue_operands(M, N, "int", 91 + idx, "f32")
    D = run_fused(A, B, K, "f16", "f32", alpha, 1.0, cin, bias, config=name, in_place=True)
    check(D, A, B, K, "int", "f32", alpha, 1.0, cin, bias, f"{name} multi-round")


def test_reduce_configs_only_in_place_with_unit_beta():
    M, N, K = 256, 256, 64
    dA = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    dB = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    D = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    other = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    F16, F32 = wgemm.WGEMM_F16, wgemm.WGEMM_F32
    cid = wgemm.config_id(reduce_names()[0])
    a = (dA.data_ptr(), dB.data_ptr(), D.data_ptr())
    # beta != 1, Cin elsewhere, and no Cin: not the in-place form
    assert wgemm.wgemm_gemm_ex_config(*a, D.data_ptr(), None, 1.0, 2.0, F16, F32, M, N, K, K, K,
                                      N, N, cid, None) == -6
    assert wgemm.wgemm_gemm_ex_config(*a, other.data_ptr(), None, 1.0, 1.0, F16, F32, M, N, K,
                                      K, K, N, N, cid, None) == -6
    assert wgemm.wgemm_gemm_ex_config(*a, None, None, 2.0, 0.0, F16, F32, M, N, K, K, K, N, N,
                                      cid, None) == -6
    # a 16-bit D
    Dh = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    assert wgemm.wgemm_gemm_ex_config(dA.data_ptr(), dB.data_ptr(), Dh.data_ptr(),
                                      Dh.data_ptr(), None, 1.0, 1.0, F16, wgemm.WGEMM_F16, M, N,
                                      K, K, K, N, N, cid, None) == -6
    # the in-place form runs
    assert wgemm.wgemm_gemm_ex_config(*a, D.data_ptr(), None, 1.0, 1.0, F16, F32, M, N, K, K, K,
                                      N, N, cid, None) == 0
    assert wgemm.wgemm_check(None) == 0


def test_in_place_default_choice():
    M, N, K = 1000, 1500, 520
    A, B = inputs.gemm_operands(M, N, K, seed=95, kind="int")
    cin, bias, alpha, _ = epilogue_operands(M, N, "int", 96, "f32")
    D = run_fused(A, B, K, "f16", "f32", alpha, 1.0, cin, bias, in_place=True)
    check(D, A, B, K, "int", "f32", alpha, 1.0, cin, bias, "in place, default choice")
    cid, mode, splits = wgemm.wgemm_select(M, N, K, c_type=wgemm.WGEMM_F32, fused=2)
    assert wgemm.config_fused(cid) == 1 and mode == 0 and splits == 1
