"""The seeded input generator: published SplitMix64 outputs, ranges, determinism."""
import numpy as np

from dense_fp16_gemm_02_gb300 import inputs


def test_splitmix64_published_first_outputs():
    # SplitMix64 seeded with state 0 starts 0xE220A8397B1DCDAF,
    # 0x6E789E6AA1B965F4, 0x06C45D188009454F; the counter form with key 0 is
    # the same sequence.
    h = inputs.hash_stream(0, 0, 3)
    assert [int(x) for x in h] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert int(inputs.hash_stream(0, 2, 1)[0]) == 0x06C45D188009454F


def test_uniform_range_and_rounding():
    A = inputs.matrix(64, 257, seed=1, tensor_id=0, kind="uniform")
    x = A.astype(np.float64)
    assert x.min() >= -1.0 and x.max() <= 1.0
    assert abs(x.mean()) < 0.02 and 0.3 < x.std() < 0.65
    # The fp16 values are the RNE rounding of 2u − 1 computed in fp64.
    h = inputs.hash_stream(inputs.stream_key(1, 0), 0, 257)
    u = (h >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    assert np.array_equal(A[0].view(np.uint16), (2 * u - 1).astype(np.float16).view(np.uint16))


def test_int_values():
    A = inputs.matrix(128, 100, seed=2, tensor_id=1, kind="int")
    vals, counts = np.unique(A.astype(np.int64), return_counts=True)
    assert vals.tolist() == [-2, -1, 0, 1, 2]
    assert counts.min() > 0.15 * A.size


def test_deterministic_and_independent_of_ld_and_chunking():
    a = inputs.matrix(33, 40, seed=5, tensor_id=0)
    b = inputs.matrix(33, 40, seed=5, tensor_id=0, ld=48, pad="nan", chunk_elems=7)
    assert np.array_equal(a.view(np.uint16), b[:, :40].view(np.uint16))
    assert np.all(b[:, 40:].view(np.uint16) == inputs.F16_NAN_BITS)
    c = inputs.matrix(33, 40, seed=5, tensor_id=1)
    assert not np.array_equal(a, c)


def test_sample_indices():
    idx = inputs.sample_indices(8192, 256, seed=3, tensor_id=2)
    assert len(idx) == 256 and idx[0] == 0 and idx[-1] == 8191
    assert np.all(np.diff(idx) > 0)
    assert np.array_equal(inputs.sample_indices(10, 256, 3, 2), np.arange(10))


def test_bf16_values_are_the_draws_rounded_to_nearest_even():
    """bf16 operands hold the same seeded draws as fp16 ones, each rounded to
    the nearest bf16 (numpy's reading of the pattern as an fp32's upper half;
    ties to the even pattern)."""
    rows, cols = 64, 257
    bits = inputs.matrix(rows, cols, 5, 0, "uniform", dtype="bf16")
    h = inputs.hash_stream(inputs.stream_key(5, 0), 0, rows * cols)
    x = 2.0 * ((h >> np.uint64(11)).astype(np.float64) * 2.0 ** -53) - 1.0
    v = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64).ravel()
    up = (((bits.astype(np.uint32) + 1) << np.uint32(16)).view(np.float32)
          .astype(np.float64).ravel())
    dn = (((bits.astype(np.uint32) - 1) << np.uint32(16)).view(np.float32)
          .astype(np.float64).ravel())
    err = np.abs(x - v)
    assert np.all(err <= np.abs(x - up)) and np.all(err <= np.abs(x - dn))
    tie = (err == np.abs(x - up)) | (err == np.abs(x - dn))
    assert np.all(bits.ravel()[tie] % 2 == 0)
    # the fp16 copy rounds the same draws: the two differ by under one bf16 step
    f16 = inputs.matrix(rows, cols, 5, 0, "uniform").astype(np.float64).ravel()
    assert np.all(np.abs(f16 - v) <= np.abs(v) * 2.0 ** -7 + 2.0 ** -24)


def test_bf16_integers_and_padding():
    bits = inputs.matrix(20, 30, 3, 1, "int", ld=40, pad="nan", dtype="bf16")
    v = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    assert np.array_equal(v[:, :30], inputs.matrix(20, 30, 3, 1, "int").astype(np.float32))
    assert np.all(bits[:, 30:] == inputs.BF16_NAN_BITS)
