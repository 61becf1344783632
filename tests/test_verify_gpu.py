"""M-row speculative verify (w4g128_gemm_verify, 1 <= M <= 16) against the fp64
oracle, plus exact cases and row consistency."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, check_against_oracle, run  # noqa: E402


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 12, 16])
@pytest.mark.parametrize("K,N", [(128, 16), (640, 80), (1152, 208), (4096, 4096)])
def test_verify_matches_oracle(M, K, N):
    mat = DevMatrix(K, N, matrix_id=N + M)
    x = synth.x(SEED, 1000 + M, M, K)
    check_against_oracle(run(mat, x, verify=True), x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", [(5120, 6144), (6144, 5120), (5120, 34816), (17408, 5120)])
def test_verify_projection_shapes_m8(K, N):
    mat = DevMatrix(K, N, matrix_id=N + 8)
    x = synth.x(SEED, 2000 + K, 8, K)
    check_against_oracle(run(mat, x), x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [8, 16])
def test_verify_exact_integer_case_bit_exact(M):
    rng = np.random.default_rng(31)
    O = oracle.Oracle()
    K, N = 1024, 144
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    codes = O.pack_canonical(q)
    s = np.full((K // 128, N), 0x3F80, np.uint16)
    m = np.full((K // 128, N), 0xC100, np.uint16)  # -8.0
    x = (rng.integers(-4, 5, size=(M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y = run(DevMatrix(K, N, codes, s, m), x)
    y_ref, _ = O.gemm(x, codes, s, m)
    expect = np.array([O.bf16_rn(v) for v in y_ref.ravel()], dtype=np.uint16).reshape(M, N)
    assert np.array_equal(y, expect)


@pytest.mark.gpu
def test_verify_identical_rows_give_identical_outputs():
    K, N = 2048, 512
    mat = DevMatrix(K, N, matrix_id=4)
    x1 = synth.x(SEED, 4, 1, K)
    x = np.repeat(x1, 8, axis=0)
    y = run(mat, x)
    for r in range(1, 8):
        assert np.array_equal(y[r], y[0])


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", [(128, 16), (640, 80), (1152, 208), (5120, 6144), (17408, 5120)])
def test_verify_rows_bitwise_equal_single_row_verify(K, N):
    """Row m of an M-row verify equals a verify of row m alone (M = 1), bit for
    bit, for every M in 1..16 (both the one-tile and the two-tile MMA): the
    exact speculative-decoding property."""
    mat = DevMatrix(K, N, matrix_id=6 + K)
    x16 = synth.x(SEED, 6 + N, 16, K)
    single = [run(mat, x16[m:m + 1], verify=True)[0] for m in range(16)]
    for M in range(1, 17):
        yM = run(mat, x16[:M], verify=True)
        for m in range(M):
            assert np.array_equal(yM[m], single[m]), (M, m)


@pytest.mark.gpu
def test_verify_deterministic():
    K, N = 5120, 6144
    mat = DevMatrix(K, N, matrix_id=8)
    x = synth.x(SEED, 8, 8, K)
    assert np.array_equal(run(mat, x), run(mat, x))


def _wide_range_x(rng, M, K):
    """bf16 bits of x whose magnitudes span 2^-100 .. 2^100 within and across
    groups and rows; group 1 of every row is all zeros, and row 1 (when
    present) is a single large value per group."""
    mag = np.exp2(rng.integers(-100, 101, size=(M, K)).astype(np.float64))
    x = (rng.standard_normal((M, K)) * mag).astype(np.float32)
    x[:, 128:256] = 0.0
    if M > 1:
        x[1] = 0.0
        x[1, ::128] = 3.0e20
    return (x.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 2, 8, 16])
def test_wide_dynamic_range_x(M):
    """The kernels carry x into fp16 with one power of two per (group, row);
    values far below a group's largest, zero groups and huge values must all
    stay within the bound (M = 1 also through w4g128_gemv)."""
    K, N = 1024, 208
    mat = DevMatrix(K, N, matrix_id=77)
    x = _wide_range_x(np.random.default_rng(5 + M), M, K)
    check_against_oracle(run(mat, x), x, mat.codes, mat.scales, mat.mins)
    if M == 1:
        check_against_oracle(run(mat, x, verify=True), x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", [(5120, 6144), (17408, 5120)])
def test_verify_projection_shapes_m16(K, N):
    """Sixteen draft rows (two MMA x tiles) on full layer shapes."""
    mat = DevMatrix(K, N, matrix_id=N + 16)
    x = synth.x(SEED, 2100 + K, 16, K)
    check_against_oracle(run(mat, x), x, mat.codes, mat.scales, mat.mins)
