"""The product folded into the residual add and RMS norm
(w4g128_gemm_add_rmsnorm) against the fp64 oracle: h within the product's
bound, out within the bound the norm carries it to (oracle.norm_bounds); an
exact integer case where h is bit-exact and out within one bf16 ulp; h equal
bit for bit to the plain call's y when the residual is -0; in-place update;
determinism; rows of the verify arithmetic independent of M; degenerate rows."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, bf16_to_f64, run, to_dev, to_host, workspace  # noqa: E402

EPS = 1e-6


def fused(mat, x_bits, res_bits, gam_bits, eps=EPS, verify=0, in_place=False):
    """(h bits, out bits), each [M][N]."""
    M = x_bits.shape[0]
    x, res, gam = to_dev(x_bits), to_dev(res_bits), to_dev(gam_bits)
    h = res if in_place else torch.empty(M * mat.N, dtype=torch.int16, device="cuda")
    out = torch.empty(M * mat.N, dtype=torch.int16, device="cuda")
    ws = workspace(M, mat.K, mat.N)
    w.w4g128_gemm_add_rmsnorm(mat.packed, x, res, gam, eps, h, out, M, mat.K, mat.N, verify, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    return to_host(h, np.uint16).reshape(M, mat.N), to_host(out, np.uint16).reshape(M, mat.N)


def inputs(mat, M, sid):
    x = synth.x(SEED, 3000 + sid, M, mat.K)
    res = synth.x(SEED, 4000 + sid, M, mat.N)
    gam = synth.norm_weight(SEED, 5000 + sid, mat.N)
    return x, res, gam


def check(mat, x, res, gam, h, out, eps=EPS):
    O = oracle.Oracle()
    y_ref, a = O.gemm(x, mat.codes, mat.scales, mat.mins)
    h_ref, out_ref = O.add_rmsnorm(y_ref, res, gam, eps)
    dh, dout = oracle.norm_bounds(h_ref, out_ref, a, gam, eps, O)
    eh = np.abs(bf16_to_f64(h) - h_ref)
    eo = np.abs(bf16_to_f64(out) - out_ref)
    assert np.all(eh <= dh), f"h: {np.sum(eh > dh)} outside, worst {np.max(eh / dh)}"
    assert np.all(eo <= dout), f"out: {np.sum(eo > dout)} outside, worst {np.max(eo / dout)}"
    return float(np.max(eh / dh)), float(np.max(eo / dout))


@pytest.mark.gpu
@pytest.mark.parametrize("verify", [0, 1])
@pytest.mark.parametrize("M", [1, 2, 5, 8, 16])
@pytest.mark.parametrize("K,N", [(128, 16), (640, 80), (1152, 208), (4096, 4096)])
def test_add_rmsnorm_matches_oracle(K, N, M, verify):
    mat = DevMatrix(K, N, matrix_id=7 * N + M)
    x, res, gam = inputs(mat, M, N + M)
    h, out = fused(mat, x, res, gam, verify=verify)
    check(mat, x, res, gam, h, out)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("K,N", [(6144, 5120), (17408, 5120)])
def test_add_rmsnorm_projection_shapes(K, N, M):
    """The two projections a norm follows in a decoder layer (attention output
    and MLP down), at full size."""
    mat = DevMatrix(K, N, matrix_id=K + M)
    x, res, gam = inputs(mat, M, K + M)
    h, out = fused(mat, x, res, gam)
    check(mat, x, res, gam, h, out)


def exact_case(rng, K, N, M):
    """Integer x in {-1, 0, 1} (sparse), weights q - 8, small integer residuals:
    every h is an integer the fp32 product reaches exactly, and a bf16."""
    O = oracle.Oracle()
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    codes = O.pack_canonical(q)
    s = np.full((K // 128, N), 0x3F80, np.uint16)  # 1.0
    m = np.full((K // 128, N), 0xC100, np.uint16)  # -8.0
    xv = rng.choice([-1.0, 0.0, 1.0], p=[0.03, 0.94, 0.03], size=(M, K)).astype(np.float32)
    x = (xv.view(np.uint32) >> 16).astype(np.uint16)
    rv = rng.integers(-16, 17, size=(M, N)).astype(np.float32)
    res = (rv.view(np.uint32) >> 16).astype(np.uint16)
    return codes, s, m, x, res


@pytest.mark.gpu
@pytest.mark.parametrize("eps", [0.0, 1e-6, 1.0, 1000.0])
@pytest.mark.parametrize("M,verify", [(1, 0), (1, 1), (3, 0), (8, 1)])
def test_add_rmsnorm_exact_integer_case(M, verify, eps):
    """h bit-exact; out within one bf16 ulp of the fp64 definition."""
    rng = np.random.default_rng(77 + M)
    O = oracle.Oracle()
    K, N = 1024, 144
    codes, s, m, x, res = exact_case(rng, K, N, M)
    gam = synth.norm_weight(SEED, 6000 + M, N)
    h, out = fused(DevMatrix(K, N, codes, s, m), x, res, gam, eps=eps, verify=verify)
    y_ref, _ = O.gemm(x, codes, s, m)
    h_ref, out_ref = O.add_rmsnorm(y_ref, res, gam, eps)
    h_bits = np.array([O.bf16_rn(v) for v in h_ref.ravel()], dtype=np.uint16).reshape(M, N)
    assert np.array_equal(bf16_to_f64(h_bits), h_ref), "the case must keep h on bf16 values"
    assert np.array_equal(h, h_bits)
    err = np.abs(bf16_to_f64(out) - out_ref)
    assert np.all(err <= O.bf16_ulp_array(out_ref)), f"worst {np.max(err / O.bf16_ulp_array(out_ref))} ulp"


@pytest.mark.gpu
@pytest.mark.parametrize("M,verify", [(1, 0), (1, 1), (4, 0), (8, 1)])
@pytest.mark.parametrize("K,N", [(640, 80), (5120, 6144)])
def test_h_is_the_product_when_residual_is_negative_zero(K, N, M, verify):
    """-0 + v == v for every fp32 v, so h must equal the plain call's y bit for bit."""
    mat = DevMatrix(K, N, matrix_id=11 + N)
    x, _, gam = inputs(mat, M, 17)
    res = np.full((M, N), 0x8000, np.uint16)
    h, _ = fused(mat, x, res, gam, verify=verify)
    y = run(mat, x, verify=bool(verify))
    assert np.array_equal(h, y)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8])
def test_in_place_and_deterministic(M):
    K, N = 5120, 6144
    mat = DevMatrix(K, N, matrix_id=23)
    x, res, gam = inputs(mat, M, 23)
    h1, o1 = fused(mat, x, res, gam)
    h2, o2 = fused(mat, x, res, gam)
    h3, o3 = fused(mat, x, res, gam, in_place=True)
    assert np.array_equal(h1, h2) and np.array_equal(o1, o2)
    assert np.array_equal(h1, h3) and np.array_equal(o1, o3)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", [(640, 80), (17408, 5120)])
def test_verify_rows_independent_of_m(K, N):
    """With the verify arithmetic, row m of h and out equals the one-row call on
    row m (the norm's order depends on N alone), for 8 and 16 rows."""
    mat = DevMatrix(K, N, matrix_id=29)
    x, res, gam = inputs(mat, 16, 29)
    h8, o8 = fused(mat, x, res, gam, verify=1)
    for r in (0, 3, 7, 8, 15):
        h1, o1 = fused(mat, x[r:r + 1], res[r:r + 1], gam, verify=1)
        assert np.array_equal(h1[0], h8[r]) and np.array_equal(o1[0], o8[r])


@pytest.mark.gpu
@pytest.mark.parametrize("K,N,M,verify", [(128, 40960, 1, 0), (256, 40960, 1, 1), (128, 10240, 8, 0),
                                          (384, 9216, 2, 1)])
def test_add_rmsnorm_wide_rows(K, N, M, verify):
    """Wide rows: many 1024-column slices per row, each computing the row's
    mean square itself."""
    mat = DevMatrix(K, N, matrix_id=37 + M)
    x, res, gam = inputs(mat, M, 37 + M)
    h, out = fused(mat, x, res, gam, verify=verify)
    check(mat, x, res, gam, h, out)


@pytest.mark.gpu
def test_degenerate_rows():
    """x = 0 and residual = 0: h = 0, out = 0 for eps > 0, and NaN for eps = 0
    (0 / 0, as the definition gives)."""
    K, N, M = 256, 48, 2
    mat = DevMatrix(K, N, matrix_id=31)
    x = np.zeros((M, K), np.uint16)
    res = np.zeros((M, N), np.uint16)
    gam = synth.norm_weight(SEED, 31, N)
    h, out = fused(mat, x, res, gam, eps=1e-6)
    assert np.all(bf16_to_f64(h) == 0) and np.all(bf16_to_f64(out) == 0)
    _, out0 = fused(mat, x, res, gam, eps=0.0)
    _, ref0 = oracle.Oracle().add_rmsnorm(np.zeros((M, N)), res, gam, 0.0)
    assert np.all(np.isnan(ref0)) and np.all(np.isnan(bf16_to_f64(out0)))


@pytest.mark.gpu
@pytest.mark.parametrize("M", [4, 8, 16])
def test_add_rmsnorm_with_the_per_warp_fold(M):
    """2560 quads of 2 segments: more quads than streaming warps and than one
    wave of per-quad reduce CTAs, so the split quads are folded per warp with
    the residual added there.  h with a -0 residual is the plain call's y bit
    for bit; at M = 4 h and out are also checked against the oracle."""
    K, N = 1024, 163840
    mat = DevMatrix(K, N, matrix_id=900 + M)
    x, res, gam = inputs(mat, M, 900 + M)
    zero = np.full((M, N), 0x8000, np.uint16)
    h0, _ = fused(mat, x, zero, gam, verify=1)
    assert np.array_equal(h0, run(mat, x, verify=True))
    if M == 4:
        h, out = fused(mat, x, res, gam, verify=1)
        check(mat, x, res, gam, h, out)
