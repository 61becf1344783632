"""w4g128_quantize on the GPU against the quantizer oracle, bit for bit: codes,
scales and minimums are integer decisions both sides take with the same fp32
operations.  Also: determinism, a full-size projection on sampled columns,
and the chain quantize -> pack -> GEMV / verify against the GEMM oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import oracle  # noqa: E402
from gpu_helpers import DevMatrix, check_against_oracle, run, to_dev, to_host  # noqa: E402


def weights(kind, K, N, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        v = rng.standard_normal((K, N)) * 0.02
    elif kind == "heavy":
        v = rng.standard_t(3, size=(K, N)) * 0.01
    elif kind == "outliers":
        v = rng.standard_normal((K, N)) * 0.02
        rows = rng.integers(0, K, size=N)
        v[rows, np.arange(N)] = rng.choice([-1.0, 1.0], size=N) * 0.4
    elif kind == "constant_groups":
        v = np.repeat(rng.standard_normal((K // 128, N)), 128, axis=0)
    else:
        raise KeyError(kind)
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def quantize_gpu(wbits, search):
    K, N = wbits.shape
    wd = to_dev(wbits)
    codes = torch.empty((K // 8) * N, dtype=torch.int32, device="cuda")
    scales = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
    mins = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
    w.w4g128_quantize(wd, K, N, search, codes, scales, mins)
    torch.cuda.synchronize()
    return (to_host(codes, np.uint32).reshape(K // 8, N), to_host(scales, np.uint16).reshape(K // 128, N),
            to_host(mins, np.uint16).reshape(K // 128, N))


@pytest.mark.gpu
@pytest.mark.parametrize("search", [0, 1])
@pytest.mark.parametrize("kind", ["normal", "heavy", "outliers", "constant_groups"])
@pytest.mark.parametrize("K,N", [(128, 16), (256, 48), (640, 80), (1024, 208), (4096, 4096)])
def test_quantize_bit_exact_vs_oracle(K, N, kind, search):
    wb = weights(kind, K, N, seed=K + N)
    c, s, m = quantize_gpu(wb, search)
    rc, rs, rm, _ = oracle.Oracle().quantize(wb, search)
    assert np.array_equal(c, rc)
    assert np.array_equal(s, rs)
    assert np.array_equal(m, rm)


@pytest.mark.gpu
def test_quantize_deterministic():
    wb = weights("heavy", 1024, 1024, seed=11)
    a = quantize_gpu(wb, 1)
    b = quantize_gpu(wb, 1)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.gpu
def test_quantize_full_size_sampled_columns():
    """The fused gate+up shape (5120 x 34816) on the GPU; the oracle quantises
    sampled columns (groups are per column, so a column slice is exact)."""
    K, N = 5120, 34816
    wb = weights("heavy", K, N, seed=12)
    c, s, m = quantize_gpu(wb, 1)
    cols = np.unique(np.concatenate([[0, 1, N - 1], np.random.default_rng(13).integers(0, N, 40)]))
    rc, rs, rm, _ = oracle.Oracle().quantize(np.ascontiguousarray(wb[:, cols]), 1)
    assert np.array_equal(c[:, cols], rc)
    assert np.array_equal(s[:, cols], rs)
    assert np.array_equal(m[:, cols], rm)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8])
def test_quantize_pack_gemv_chain(M):
    """Quantised on the GPU, packed, streamed: the GEMV / verify result is
    within the bound of the oracle's product on the same quantised weights."""
    K, N = 2048, 1040
    wb = weights("outliers", K, N, seed=14)
    c, s, m = quantize_gpu(wb, 1)
    mat = DevMatrix(K, N, c, s, m)
    x = (np.random.default_rng(15).standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y = run(mat, x, verify=(M > 1))
    check_against_oracle(y, x, c, s, m)


@pytest.mark.gpu
def test_quantize_rejects_bad_arguments():
    dummy = torch.empty(1 << 16, dtype=torch.int32, device="cuda")
    with pytest.raises(w.W4G128Error):
        w.w4g128_quantize(dummy, 100, 16, 0, dummy, dummy, dummy)  # K % 128
    with pytest.raises(w.W4G128Error):
        w.w4g128_quantize(dummy, 128, 16, 2, dummy, dummy, dummy)  # search flag
