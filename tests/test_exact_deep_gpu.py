"""Bit-exact integer cases on the deep split-K paths.

With integer activations x in {-4..4}, every scale 1 and every minimum -8 (or
0), each product, group sum, segment sum and fold of the kernels is an exact
fp32 integer (all below 2^24), so the GPU output must be bf16_rn of the fp64
oracle's exact y, bit for bit.  A fold that drops, repeats or reorders a
split-K slot, a segment or group placed in the wrong matrix, or a misindexed
partial changes some output by at least one unit and is caught here, however
many segments a quad has (the tolerance tests alone could miss such a
mistake at large K).  Covered: K = 17408 and 65536 (34 and 128 segments per
quad) through w4g128_gemv and w4g128_gemm_verify at 8 and 16 rows; a decode
step of more than 8 matrices (the large descriptor table); both forms of the
M >= 2 fold (per quad, and per streaming warp from the schedule or from the
warps' records); the residual add + RMS norm at K = 17408 (h bit-exact).
The full-size cases generate the random codes on the device and copy them
back for the oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import oracle  # noqa: E402
from gpu_helpers import (MINUS_EIGHT, ONE, DevMatrix, exact_bits, int_x, run, to_dev, to_host,  # noqa: E402
                         workspace)


def exact_matrix(K, N, matrix_id, mn=MINUS_EIGHT):
    return DevMatrix(K, N, matrix_id=matrix_id, device_fill=True, const_meta=(ONE, mn), keep_host=True)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8, 16])
@pytest.mark.parametrize("K,N", [(17408, 5120), (65536, 208)])
def test_exact_large_k(K, N, M):
    O = oracle.Oracle()
    mat = exact_matrix(K, N, 3100 + K // 128)
    x = int_x(np.random.default_rng(K + M), M, K)
    y_ref, _ = O.gemm(x, mat.codes, mat.scales, mat.mins)
    expect = exact_bits(y_ref, O)
    assert np.array_equal(run(mat, x, verify=(M > 1)), expect)
    if M == 1:  # the verify arithmetic at one row gives the same bits
        assert np.array_equal(run(mat, x, verify=True), expect)


def decode_step(mats, xs_bits, M, verify=False):
    xs = [to_dev(x) for x in xs_bits]
    ys = [torch.empty(M * m.N, dtype=torch.int16, device="cuda") for m in mats]
    descs = [(m.packed, x, y, m.K, m.N) for m, x, y in zip(mats, xs, ys)]
    ws = torch.empty(w.w4g128_decode_step_workspace_bytes(descs, M), dtype=torch.uint8, device="cuda")
    (w.w4g128_verify_step if verify else w.w4g128_decode_step)(descs, M, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    return [to_host(y, np.uint16).reshape(M, m.N) for m, y in zip(mats, ys)]


# eleven matrices: more than the 8-descriptor kernel holds, with ragged quads,
# ragged segments, one-quad and one-segment matrices, and deep quads
MANY = [(17408, 1024), (128, 16), (640, 80), (4096, 4096), (1152, 208), (65536, 64), (384, 48),
        (6144, 5120), (2048, 1008), (5120, 960), (256, 4096)]


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8, 16])
def test_exact_decode_step_many_matrices(M):
    O = oracle.Oracle()
    rng = np.random.default_rng(50 + M)
    mats = [exact_matrix(K, N, 3200 + i, mn=(MINUS_EIGHT if i % 2 == 0 else 0)) for i, (K, N) in enumerate(MANY)]
    xs = [int_x(rng, M, K) for K, _ in MANY]
    ys = decode_step(mats, xs, M, verify=(M == 8))
    for i, (mat, x, y) in enumerate(zip(mats, xs, ys)):
        y_ref, _ = O.gemm(x, mat.codes, mat.scales, mat.mins)
        assert np.array_equal(y, exact_bits(y_ref, O)), MANY[i]


# 3168 quads: the M >= 4 call folds per streaming warp from the warps' records
# (see test_reduce_forms_gpu.py); each matrix alone folds per quad
PER_WARP = [(4096, 131072), (1024, 65536), (5120, 6144)]


@pytest.mark.gpu
@pytest.mark.parametrize("M", [4, 8, 16])
def test_exact_per_warp_fold_several_matrices(M):
    O = oracle.Oracle()
    rng = np.random.default_rng(60 + M)
    mats = [exact_matrix(K, N, 3300 + i) for i, (K, N) in enumerate(PER_WARP)]
    xs = [int_x(rng, M, K) for K, _ in PER_WARP]
    ys = decode_step(mats, xs, M)
    for mat, x, y in zip(mats, xs, ys):
        y_ref, _ = O.gemm(x, mat.codes, mat.scales, mat.mins)
        expect = exact_bits(y_ref, O)
        assert np.array_equal(y, expect)
        assert np.array_equal(run(mat, x, verify=True), expect)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8, 16])
def test_exact_lm_head(M):
    """The 5120 x 248320 lm_head (3880 quads: per-warp fold from the schedule
    at M >= 4; tickets and the CTA-end fold at M = 1)."""
    O = oracle.Oracle()
    K, N = 5120, 248320
    mat = exact_matrix(K, N, 3400)
    x = int_x(np.random.default_rng(70 + M), M, K)
    y_ref, _ = O.gemm(x, mat.codes, mat.scales, mat.mins)
    assert np.array_equal(run(mat, x, verify=(M > 1)), exact_bits(y_ref, O))


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8, 16])
def test_exact_add_rmsnorm_deep_k(M):
    """The residual add folded into 34-segment quads: h = bf16(residual + y)
    is an exact integer sum, so h must be bf16_rn of the oracle's h."""
    O = oracle.Oracle()
    K, N = 17408, 5120
    rng = np.random.default_rng(80 + M)
    mat = exact_matrix(K, N, 3500)
    x = int_x(rng, M, K)
    res = int_x(rng, M, N, lo=-64, hi=64)
    gam = np.full(N, ONE, np.uint16)
    h = torch.empty(M * N, dtype=torch.int16, device="cuda")
    out = torch.empty(M * N, dtype=torch.int16, device="cuda")
    ws = workspace(M, K, N)
    w.w4g128_gemm_add_rmsnorm(mat.packed, to_dev(x), to_dev(res), to_dev(gam), 1e-6, h, out, M, K, N,
                              int(M > 1), ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    y_ref, _ = O.gemm(x, mat.codes, mat.scales, mat.mins)
    h_ref, _ = O.add_rmsnorm(y_ref, res, gam, 1e-6)
    h_bits = exact_bits(h_ref, O)
    assert np.array_equal(to_host(h, np.uint16).reshape(M, N), h_bits)
    # the norm reads the rounded h: out within one bf16 ulp of the definition
    # applied to it
    _, out_ref = O.add_rmsnorm(oracle.bf16_bits_to_f64(h_bits), np.zeros((M, N), np.uint16), gam, 1e-6)
    err = np.abs(oracle.bf16_bits_to_f64(to_host(out, np.uint16).reshape(M, N)) - out_ref)
    assert np.all(err <= O.bf16_ulp_array(out_ref))
