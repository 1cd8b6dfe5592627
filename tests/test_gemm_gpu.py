"""GPU parity: the CUDA path through the C-ABI against the CPU oracle.

Acceptance (for C = A·Bᵀ, fp16 in, fp32 accumulation and output, "SASS-Level
Kernel Generation for Blackwell", section "The numbers"):
* integer-valued inputs in {-2..2}: exact. Every product is exact and every
  partial sum is an integer of magnitude ≤ 4K ≤ 2^18 < 2^24, so any fp32
  accumulation order, on the tensor cores or in L2 reduce-adds, is exact.
  Compared as values (+0 == -0).
* uniform[-1, 1] fp16 inputs: |C − C_ref| ≤ 2e-3·(|A|·|B|ᵀ)_ij + 1e-6 elementwise.

Small cases run every configuration and every K-decomposition at sizes that
span several tiles with ragged edges. The full-size cases of the workloads run
the default per-shape choice (the launch the bench times) and are checked
element by element over the whole of C, except 8192³ and 16384³, which are
checked on 256 sampled rows and columns (the workload's own rule).
"""
import re

import numpy as np
import pytest
import torch

import oracle
from config_names import plain_fp32
from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-3, 1e-6
DP, SPLIT, STREAM, HYBRID, ZERO_FIRST = 0, 1, 2, 3, 4


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build_oracle()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return wgemm.load()


def ceil8(k: int) -> int:
    return (k + 7) // 8 * 8


def operands(M, N, K, seed, kind):
    """Seeded operands with leading dimensions padded to a multiple of 8
    (the TMA row-stride rule); the padding columns hold fp16 NaN."""
    return inputs.gemm_operands(M, N, K, seed=seed, kind=kind, lda=ceil8(K), ldb=ceil8(K),
                                pad="nan")


def upload(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x).cuda()


def run(A, B, K, config=None, mode=-1, splits=1, C=None):
    """C = A[:, :K]·B[:, :K]ᵀ on the GPU; A, B numpy fp16 with ld ≥ K."""
    dA, dB = upload(A), upload(B)
    out = wgemm.gemm(dA[:, :K], dB[:, :K], C, config=config, mode=mode, splits=splits)
    status = wgemm.wgemm_check(torch.cuda.current_stream().cuda_stream)
    assert status == 0, (status, wgemm.wgemm_last_device_error())
    return out


def assert_exact(got: np.ndarray, ref: np.ndarray, what=""):
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first {bad[:5].tolist()}"


def assert_tol(got: np.ndarray, ref: np.ndarray, ref_abs: np.ndarray, what=""):
    err = np.abs(got - ref)
    bound = RTOL * ref_abs + ATOL
    ok = err <= bound
    rel = float((err / np.maximum(np.abs(ref), 1e-30)).max()) if ref.size else 0.0
    assert ok.all(), f"{what}: {(~ok).sum()} outside tolerance, max excess {(err - bound).max()}"
    return rel


def check_full(A, B, K, kind, what, **kw):
    C = run(A, B, K, **kw).cpu().numpy().astype(np.float64)
    if kind == "int":
        assert_exact(C, oracle.gemm_f64(A, B, K=K), what)
    else:
        ref, ref_abs = oracle.gemm_f64(A, B, K=K, with_abs=True)
        assert_tol(C, ref, ref_abs, what)


def configs(suffix=""):
    """Plain fp32-output configurations whose name ends with `suffix`."""
    return [n for n in wgemm.config_names()
            if n.endswith(suffix) and not n.endswith("_h") and "_ab" not in n]


def is_multicast(name: str) -> bool:
    """A cluster of MMA groups sharing an operand tile (g?m2_ or g?r2_)."""
    return re.match(r"g\d[mr]2_", name) is not None


def k_split_configs():
    """Configurations that run split-K and stream-K: TMA epilogue, no column
    multicast (row-multicast clusters run them as one worker)."""
    return [n for n in configs("_tma") if not re.match(r"g\dm2_", n)]


# ---------------------------------------------------------------- every configuration


@pytest.mark.parametrize("kind", ["int", "uniform"])
@pytest.mark.parametrize("name", plain_fp32())
def test_every_config_ragged(name, kind):
    # 3 tile rows and 3 tile columns for the largest tiles, all edges ragged,
    # K a non-multiple of the 64-wide k-block.
    M, N, K = 600, 1100, 300
    A, B = operands(M, N, K, 100 + plain_fp32().index(name), kind)
    check_full(A, B, K, kind, f"{name} {kind}", config=name, mode=DP)


@pytest.mark.parametrize("name", plain_fp32())
def test_every_config_multi_round(name):
    # More tiles than co-resident workers for every configuration (≥ 2 tiles
    # per worker even for the 512×256 pair tile: 11 × 14 = 154 tiles over at
    # most 76 pairs), so each CTA alternates accumulators and crosses tiles;
    # ragged last tile row and column, K not a multiple of 64. Exact on
    # integer inputs; run twice to catch state left over between launches.
    M, N, K = 2600, 7000, 136
    A, B = operands(M, N, K, 300 + plain_fp32().index(name), "int")
    ref = oracle.gemm_f64(A, B, K=K)
    for _ in range(2):
        C = run(A, B, K, config=name, mode=DP).cpu().numpy().astype(np.float64)
        assert_exact(C, ref, f"{name} multi-round")


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_split_k_every_tma_config(splits):
    M, N, K = 300, 700, 2000
    for kind in ("int", "uniform"):
        A, B = inputs.gemm_operands(M, N, K, seed=7 + splits, kind=kind)
        for name in k_split_configs():
            check_full(A, B, K, kind, f"{name} split {splits} {kind}", config=name, mode=SPLIT,
                       splits=splits)


def test_stream_k_every_tma_config():
    M, N, K = 520, 1100, 3000
    for kind in ("int", "uniform"):
        A, B = inputs.gemm_operands(M, N, K, seed=21, kind=kind)
        for name in k_split_configs():
            check_full(A, B, K, kind, f"{name} stream-K {kind}", config=name, mode=STREAM)


def test_stream_k_zero_first_every_tma_config():
    # Stream-K with zeroing first: ragged edges, K not a multiple of 64; more
    # tiles than workers too (the 256-wide tiles at 2600 × 3000); twice, to
    # cross the flag epochs.
    for (M, N, K) in ((520, 1100, 3000), (2600, 3000, 700)):
        for kind in ("int", "uniform"):
            A, B = operands(M, N, K, 23, kind)
            for name in k_split_configs():
                for _ in range(2):
                    check_full(A, B, K, kind, f"{name} stream-K zero first {M}x{N}x{K} {kind}",
                               config=name, mode=ZERO_FIRST)


@pytest.mark.parametrize("held", [1, 2])
def test_hybrid_every_tma_config(held):
    # Whole waves of tiles data parallel and the rest by stream-K: more tiles
    # than workers for the pair 256-wide tiles (11 × 12 = 132 over 76 pairs)
    # and the single-CTA ones (21 × 12 over 152); ragged edges, K not a
    # multiple of 64. Fewer tiles than workers (the 512-wide pair tiles) runs
    # plain stream-K. Twice, to cross the flag epochs.
    M, N, K = 2600, 3000, 700
    for kind in ("int", "uniform"):
        A, B = operands(M, N, K, 31 + held, kind)
        for name in k_split_configs():
            for _ in range(2):
                check_full(A, B, K, kind, f"{name} hybrid {held} {kind}", config=name,
                           mode=HYBRID, splits=held)


def test_split_and_stream_equal_data_parallel_on_integers():
    # Exact arithmetic: every decomposition of K gives the same C, bit for bit.
    M, N, K = 256, 512, 4096
    A, B = inputs.gemm_operands(M, N, K, seed=5, kind="int")
    name = "g2_512x256_s4_a1_tma"
    base = run(A, B, K, config=name, mode=DP).cpu().numpy()
    for mode, s in ((SPLIT, 2), (SPLIT, 9), (STREAM, 1), (HYBRID, 1), (ZERO_FIRST, 1)):
        other = run(A, B, K, config=name, mode=mode, splits=s).cpu().numpy()
        assert np.array_equal(base, other), (mode, s)


def test_repeated_calls_share_flag_workspace():
    # Monotone epochs: flags are never reset between calls; alternate modes and
    # shapes on one stream and check every result.
    shapes = [(300, 700, 2000, SPLIT, 3), (520, 1100, 3000, STREAM, 1),
              (256, 512, 4096, SPLIT, 9), (300, 700, 2000, STREAM, 1),
              (520, 1100, 3000, ZERO_FIRST, 1)]
    for rep in range(3):
        for M, N, K, mode, s in shapes:
            A, B = inputs.gemm_operands(M, N, K, seed=rep, kind="int")
            C = run(A, B, K, config="g2_512x128_s4_a2_tma", mode=mode, splits=s)
            assert_exact(C.cpu().numpy().astype(np.float64), oracle.gemm_f64(A, B), "repeat")
    assert wgemm.wgemm_workspace_bytes() > 0


def test_k_split_calls_on_several_streams_at_once():
    """K-split grids wait on flags raised by other CTAs of the same grid, so
    the library launches them cooperatively: a grid starts only once all its
    CTAs fit. Here split-K, stream-K and zero-first stream-K calls, each
    filling most of the GPU, are enqueued on three streams at once, with no
    ordering between them, several rounds; every result is exact and no wait
    expires."""
    M, N, K = 1024, 1024, 8192
    A, B = inputs.gemm_operands(M, N, K, seed=17, kind="int")
    ref = oracle.gemm_f64(A, B)
    dA, dB = upload(A), upload(B)
    cid = wgemm.config_id("g2_512x256_s4_a1_tma")
    streams = [torch.cuda.Stream() for _ in range(3)]
    plans = [(SPLIT, 9), (STREAM, 1), (ZERO_FIRST, 1)]
    torch.cuda.synchronize()
    outs = []
    for rnd in range(4):
        for s, (mode, sp) in zip(streams, plans):
            C = torch.full((M, N), float("nan"), device="cuda")
            C.record_stream(s)
            outs.append((mode, C))
        for (mode, C), s, (_, sp) in zip(outs[-3:], streams, plans):
            s.wait_stream(torch.cuda.current_stream())
            rc = wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K,
                                           K, K, N, cid, mode, sp, s.cuda_stream)
            assert rc == 0
    for s in streams:
        assert wgemm.wgemm_check(s.cuda_stream) == 0, wgemm.wgemm_last_device_error()
    for mode, C in outs:
        assert_exact(C.cpu().numpy().astype(np.float64), ref, f"mode {mode} on its own stream")


def test_k_split_without_cooperative_launch():
    """The profiling hook launches K-split grids plainly (for Nsight Compute,
    which runs kernels alone); on an otherwise idle GPU the results stay
    exact, and the default is restored."""
    lib = wgemm.load()
    M, N, K = 1024, 1024, 8192
    A, B = inputs.gemm_operands(M, N, K, seed=19, kind="int")
    ref = oracle.gemm_f64(A, B)
    assert lib.wgemm_debug_set_cooperative(0) == 1
    try:
        for mode, sp in ((SPLIT, 9), (STREAM, 1), (ZERO_FIRST, 1)):
            C = run(A, B, K, config="g2_512x256_s4_a1_tma", mode=mode, splits=sp)
            assert_exact(C.cpu().numpy().astype(np.float64), ref, f"plain launch, mode {mode}")
    finally:
        assert lib.wgemm_debug_set_cooperative(1) == 0


def test_device_timeout_is_reported_and_context_survives():
    # Failure detection without a GPU fault: the split-K waiters are told to
    # wait for a flag value that nothing writes. Their bounded waits run out
    # (2 s), the kernel records the timeout and tears down normally; the host
    # reads it from the status word, and the next call works.
    lib = wgemm.load()
    M, N, K = 256, 512, 640
    A, B = inputs.gemm_operands(M, N, K, seed=8, kind="int")
    dA, dB = upload(A), upload(B)
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    h = torch.cuda.current_stream().cuda_stream
    cid = wgemm.config_id("g2_512x256_s4_a1_tma")
    assert lib.wgemm_debug_set_flag_wait_skew(1) == 0
    try:
        rc = wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K,
                                       N, cid, SPLIT, 2, h)
        assert rc == 0
        assert wgemm.wgemm_check(h) == -5
        err = wgemm.wgemm_last_device_error()
        assert err["code"] == -5 and err["site"] == 0x23  # epilogue, split-K flag wait
    finally:
        assert lib.wgemm_debug_set_flag_wait_skew(0) == 0
    assert lib.wgemm_debug_set_flag_wait_skew(-1) == -1
    C = run(A, B, K, config="g2_512x256_s4_a1_tma", mode=SPLIT, splits=2)
    assert_exact(C.cpu().numpy().astype(np.float64), oracle.gemm_f64(A, B), "after timeout")


# ---------------------------------------------------------------- edge cases


def test_k_zero_writes_zeros():
    C = torch.full((37, 53), float("nan"), device="cuda")
    A = torch.zeros((37, 8), dtype=torch.float16, device="cuda")
    B = torch.zeros((53, 8), dtype=torch.float16, device="cuda")
    wgemm.gemm(A[:, :0], B[:, :0], C)
    assert wgemm.wgemm_check(torch.cuda.current_stream().cuda_stream) == 0
    assert torch.all(C == 0)


def test_empty_m_or_n_is_noop():
    A = torch.ones((0, 64), dtype=torch.float16, device="cuda")
    B = torch.ones((5, 64), dtype=torch.float16, device="cuda")
    C = wgemm.gemm(A, B)
    assert C.shape == (0, 5)
    rc = wgemm.wgemm_f16f32(0, 0, 0, 4, 0, 64, 64, 64, 4, None)
    assert rc == 0


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 300, 7), (300, 1, 64), (17, 33, 65),
                                   (128, 256, 64), (256, 512, 128)])
def test_tiny_and_exact_tile_shapes(M, N, K):
    lda = ldb = ((K + 7) // 8) * 8
    names = ["g1_128x64_s8_a2_direct", "g2_256x256_s6_a2_direct", None]
    if N % 4 == 0:  # a contiguous C allows the TMA epilogue
        names += ["g1_128x256_s4_a2_tma", "g2_256x256_s6_a2_tma", "g2_512x256_s4_a1_tma"]
    for name in names:
        A, B = inputs.gemm_operands(M, N, K, seed=3, kind="int", lda=lda, ldb=ldb)
        check_full(A, B, K, "int", f"{name} {M}x{N}x{K}", config=name,
                   mode=DP if name else -1)


def test_padding_past_k_never_read():
    # lda, ldb > K with fp16 NaN in the padding: TMA must stop at K.
    M, N, K = 200, 300, 100
    A, B = inputs.gemm_operands(M, N, K, seed=9, kind="uniform", lda=136, ldb=112, pad="nan")
    for name in ("g1_128x256_s4_a2_tma", "g2_256x256_s6_a2_direct", "g2_512x128_s4_a2_tma"):
        check_full(A, B, K, "uniform", name, config=name, mode=DP)


@pytest.mark.parametrize("extra_rows", [0, 17])
def test_row_multicast_second_group_past_m(extra_rows):
    """Row multicast: the second MMA group of a cluster tile needs no rows of
    C when M ends inside (or at the end of) the first group's rows, but its
    producer still loads and multicasts its half of the B slice, which the
    first group reads. M = one group's rows (+ a ragged 17 more rows, which
    puts the second group of the last tile partly in range), N ragged over
    several cluster tiles, K several k-blocks with a ragged tail; exact on
    integers."""
    names = [n for n in configs() if re.match(r"g\dr2_", n)]
    assert names, "row-multicast configurations are compiled"
    for name in names:
        bn = int(name.split("_")[1].split("x")[1]) // 2  # tile rows = 2 groups of BN
        M, N, K = bn + extra_rows, 900, 200
        A, B = operands(M, N, K, 41, "int")
        check_full(A, B, K, "int", f"{name} M={M}", config=name, mode=DP)


def test_unaligned_c_rows_use_register_stores():
    # N = 53: rows of a contiguous C are not 16-byte aligned; the default
    # choice stores from registers and the result is still exact.
    for M, N, K in ((37, 53, 72), (700, 1531, 200), (1600, 1999, 64)):
        A, B = operands(M, N, K, 31, "int")
        check_full(A, B, K, "int", f"unaligned C {M}x{N}x{K}")


def test_ldc_padding_untouched():
    M, N, K = 130, 260, 96
    A, B = inputs.gemm_operands(M, N, K, seed=4, kind="int")
    for name in ("g1_128x256_s4_a2_direct", "g2_256x256_s6_a2_tma"):
        Cfull = torch.full((M, 300), -7.0, device="cuda")
        run(A, B, K, config=name, mode=DP, C=Cfull[:, :N])
        got = Cfull.cpu().numpy()
        assert np.all(got[:, N:] == -7.0)
        assert_exact(got[:, :N].astype(np.float64), oracle.gemm_f64(A, B), name)


def test_side_stream():
    M, N, K = 300, 400, 500
    A, B = operands(M, N, K, 12, "int")
    s = torch.cuda.Stream()
    dA, dB = upload(A), upload(B)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        C = wgemm.gemm(dA[:, :K], dB[:, :K])
        assert wgemm.wgemm_check(s.cuda_stream) == 0
    assert_exact(C.cpu().numpy().astype(np.float64), oracle.gemm_f64(A, B, K=K), "side stream")


def test_argument_errors_on_gpu():
    A = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    assert wgemm.wgemm_f16f32(A.data_ptr() + 2, A.data_ptr(), C.data_ptr(), 8, 8, 8, 64, 64, 64,
                              None) == -2
    assert wgemm.wgemm_f16f32(A.data_ptr(), A.data_ptr(), C.data_ptr(), 8, 8, 8, 4, 64, 64,
                              None) == -1
    assert wgemm.wgemm_f16f32_config(A.data_ptr(), A.data_ptr(), C.data_ptr(), 8, 8, 8, 64, 64,
                                     64, 999, 0, 1, None) == -6
    direct = wgemm.config_id("g2_256x256_s6_a2_direct")
    assert wgemm.wgemm_f16f32_config(A.data_ptr(), A.data_ptr(), C.data_ptr(), 64, 64, 64, 64,
                                     64, 64, direct, SPLIT, 2, None) == -6
    # A TMA epilogue forced on a C whose rows are not 16-byte aligned.
    tma = wgemm.config_id("g2_256x256_s6_a2_tma")
    assert wgemm.wgemm_f16f32_config(A.data_ptr(), A.data_ptr(), C.data_ptr() + 4, 8, 8, 8, 64,
                                     64, 64, tma, 0, 1, None) == -2
    assert wgemm.wgemm_f16f32_config(A.data_ptr(), A.data_ptr(), C.data_ptr(), 8, 6, 8, 64,
                                     64, 6, tma, 0, 1, None) == -2


# ---------------------------------------------------------------- the workloads at full size

WORKLOADS = [
    # (M, N, K, kinds): every element of C against the oracle. The integer
    # copies (exact) are the pages' check; uniform inputs within the bound.
    (1024, 1024, 1024, ("int", "uniform")),
    (1536, 1536, 1536, ("uniform",)),
    (2048, 2048, 2048, ("uniform",)),
    (3072, 1280, 2048, ("uniform",)),
    (4096, 4096, 1024, ("uniform",)),
    (4096, 4096, 4096, ("uniform",)),
    (8192, 2048, 4096, ("uniform",)),
    (1024, 1024, 65536, ("int", "uniform")),
    (2048, 2048, 16384, ("int", "uniform")),
]


def check_sampled(A, B, C: torch.Tensor, M, N, K, kind, n_sample, seed, what):
    rows = inputs.sample_indices(M, n_sample, seed, 2)
    cols = inputs.sample_indices(N, n_sample, seed, 3)
    Ch = C.cpu().numpy().astype(np.float64)
    # Full rows R (every column) and full columns J (every row).
    for sel_rows, sel_cols, got in ((rows, None, Ch[rows, :]), (None, cols, Ch[:, cols])):
        if kind == "int":
            ref = oracle.gemm_f64_select(A, B, sel_rows, sel_cols)
            assert_exact(got, ref, what)
        else:
            ref, ref_abs = oracle.gemm_f64_select(A, B, sel_rows, sel_cols, with_abs=True)
            assert_tol(got, ref, ref_abs, what)


@pytest.mark.parametrize("M,N,K,kinds", WORKLOADS)
def test_workload_default_path(M, N, K, kinds):
    for kind in kinds:
        A, B = inputs.gemm_operands(M, N, K, seed=1000 + M + N + K, kind=kind)
        C = run(A, B, K)
        got = C.cpu().numpy().astype(np.float64)
        del C
        torch.cuda.empty_cache()
        if kind == "int":
            assert_exact(got, oracle.gemm_f64(A, B), f"{M}x{N}x{K} int")
        else:
            ref, ref_abs = oracle.gemm_f64(A, B, with_abs=True)
            assert_tol(got, ref, ref_abs, f"{M}x{N}x{K}")


@pytest.mark.parametrize("n", [8192, 16384])
def test_large_compute_bound_sampled(n):
    # 256 sampled rows and 256 sampled columns: the full 256×256 block C[R, J],
    # plus, at 8192, the full rows R.
    A, B = inputs.gemm_operands(n, n, n, seed=2000 + n, kind="uniform")
    C = run(A, B, n)
    rows = inputs.sample_indices(n, 256, 5, 2)
    cols = inputs.sample_indices(n, 256, 5, 3)
    Ch = C.cpu().numpy()
    ref, ref_abs = oracle.gemm_f64_select(A, B, rows, cols, with_abs=True)
    assert_tol(Ch[np.ix_(rows, cols)].astype(np.float64), ref, ref_abs, f"{n}^3 block")
    if n == 8192:
        ref, ref_abs = oracle.gemm_f64_select(A, B, rows[:64], None, with_abs=True)
        assert_tol(Ch[rows[:64], :].astype(np.float64), ref, ref_abs, f"{n}^3 rows")
    del C
    torch.cuda.empty_cache()


# Off-table shapes: the per-shape rule picks from the measured rates, with
# operand pitches on and off 32-byte sectors.
OFF_TABLE = [
    (3000, 5000, 3000, 3000),   # rows 6000 B apart: 16 bytes off a sector
    (777, 1999, 5003, 5008),
    (2500, 7000, 2500, 2504),
    (5000, 700, 12000, 12000),
    (1000, 8000, 4096, 4096),
    (1536, 1536, 32768, 32768),  # long K, 36 pair tiles: the rule takes split-K
    (768, 3072, 24576, 24576),
]


def test_rule_k_split_choices():
    """The rule takes split-K where few tiles meet a long K (measured 12-16 %
    faster than the best data-parallel kernel at these shapes) and never
    stream-K, whose k-loop runs slower than its model assumes."""
    for M, N, K in ((1536, 1536, 32768), (768, 3072, 24576)):
        cid, mode, splits = wgemm.wgemm_select(M, N, K, K, K)
        assert mode == SPLIT and splits >= 2, (M, N, K, wgemm.config_names()[cid], mode)
    for M, N, K, pitch in OFF_TABLE:
        assert wgemm.wgemm_select(M, N, K, pitch, pitch)[1] in (DP, SPLIT)


def test_rule_long_calls_take_cluster_launch_control():
    """Off-table calls predicted at 0.5 ms or more take the 512-column
    cluster-launch-control tile (back to back, under the power cap, it ran
    2-5 % faster than the rule's lone-call choice at 12288³ and
    8192×8192×16384); shorter ones keep the lone-call rule."""
    names = wgemm.config_names()
    for M, N, K in ((12288, 12288, 12288), (8192, 8192, 16384), (16384, 16384, 8192)):
        cid, mode, splits = wgemm.wgemm_select(M, N, K)
        assert mode == DP and names[cid] == "g2_512x256_s4_a1_tma_clc", (M, N, K, names[cid])
    cid, mode, _ = wgemm.wgemm_select(12288, 12288, 12288)
    A, B = inputs.gemm_operands(12288, 12288, 12288, seed=3100, kind="int")
    C = run(A, B, 12288)
    check_sampled(A, B, C, 12288, 12288, 12288, "int", 32, 93, f"12288³ via {names[cid]}")
    del C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,N,K,pitch", OFF_TABLE)
def test_off_table_rule_sampled(M, N, K, pitch):
    cid, mode, splits = wgemm.wgemm_select(M, N, K, pitch, pitch)
    assert 0 <= cid < len(wgemm.config_names()) and mode in (0, 1, 2) and splits >= 1
    A, B = inputs.gemm_operands(M, N, K, seed=3000 + M + N + K, kind="uniform", lda=pitch,
                                ldb=pitch)
    C = run(A, B, K)
    check_sampled(A, B, C, M, N, K, "uniform", 32, 91,
                  f"{M}x{N}x{K} pitch {pitch} via {wgemm.config_names()[cid]} mode {mode}")
    del C
    torch.cuda.empty_cache()
