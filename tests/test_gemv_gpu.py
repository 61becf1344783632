"""M = 1 decode GEMV (w4g128_gemv) against the fp64 oracle, element by element,
plus the exact cases, determinism, the column-prefix slice, and the lm_head
and the largest N at full size, every output."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, check_against_oracle, run, to_dev, to_host, workspace  # noqa: E402

# Shapes spanning one tile, ragged quads (N % 64 != 0), ragged segments
# (K/128 % 4 != 0), several tiles and split-K.
EDGE = [(128, 16), (128, 64), (256, 16), (640, 80), (1152, 208), (2048, 4080), (384, 1008)]
# The 27B-class projection shapes and the small square case.
FULL = [(4096, 4096), (5120, 6144), (6144, 5120), (5120, 34816), (17408, 5120)]


def f32_bits_to_bf16_trunc(a):
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", EDGE + FULL)
def test_gemv_matches_oracle(K, N):
    mat = DevMatrix(K, N, matrix_id=N)
    x = synth.x(SEED, N, 1, K)
    y = run(mat, x)
    check_against_oracle(y, x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
def test_gemv_exact_integer_case_bit_exact():
    """x in {-4..4}, scale 1, min 0 or -8: every partial sum is an exact fp32
    integer, so y must equal bf16_rn(exact y) bit for bit."""
    rng = np.random.default_rng(21)
    O = oracle.Oracle()
    for K, N, mn in [(1024, 128, 0.0), (768, 80, -8.0), (4096, 256, -8.0)]:
        q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
        codes = O.pack_canonical(q)
        s = np.full((K // 128, N), 0x3F80, np.uint16)
        m = np.full((K // 128, N), f32_bits_to_bf16_trunc(mn), np.uint16)
        x = f32_bits_to_bf16_trunc(rng.integers(-4, 5, size=(1, K)).astype(np.float32))
        y = run(DevMatrix(K, N, codes, s, m), x)
        y_ref, _ = O.gemm(x, codes, s, m)
        expect = np.array([O.bf16_rn(v) for v in y_ref.ravel()], dtype=np.uint16).reshape(1, N)
        assert np.array_equal(y, expect)


@pytest.mark.gpu
def test_gemv_one_hot_rows_bit_exact():
    """x = e_k: y_n = bf16(min + q_kn * scale), exactly, for a sample of rows k."""
    K, N = 1024, 96
    mat = DevMatrix(K, N, matrix_id=5)
    O = oracle.Oracle()
    q = O.unpack_canonical(mat.codes)
    s = oracle.bf16_bits_to_f64(mat.scales)
    mn = oracle.bf16_bits_to_f64(mat.mins)
    for k in [0, 1, 7, 8, 9, 15, 16, 63, 64, 127, 128, 200, 511, 1023]:
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y = run(mat, x)
        w_k = mn[k // 128] + q[k].astype(np.float64) * s[k // 128]
        expect = np.array([O.bf16_rn(v) for v in w_k], dtype=np.uint16)
        assert np.array_equal(y[0], expect), k


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", [(5120, 6144), (17408, 5120), (1152, 208)])
def test_gemv_deterministic_and_equal_to_verify_m1(K, N):
    """gemv is bitwise run-to-run deterministic, within the bound, and bit for
    bit gemm_verify at M = 1 (one arithmetic serves every M)."""
    mat = DevMatrix(K, N, matrix_id=3)
    x = synth.x(SEED, 3, 1, K)
    y1, y2 = run(mat, x), run(mat, x)
    y3 = run(mat, x, verify=True)
    assert np.array_equal(y1, y2) and np.array_equal(y1, y3)
    check_against_oracle(y1, x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
def test_gemv_column_prefix_slice():
    """The first N' = 64*Q' columns of a packed matrix are a valid packed matrix."""
    K, N = 2048, 1024
    mat = DevMatrix(K, N, matrix_id=9)
    x = synth.x(SEED, 9, 1, K)
    full = run(mat, x)
    for Np in (64, 128, 576, 960):
        xd = to_dev(x)
        y = torch.empty(Np, dtype=torch.int16, device="cuda")
        ws = workspace(1, K, Np)
        w.w4g128_gemv(mat.packed, xd, y, K, Np, ws)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(y, np.uint16), full[0, :Np])


@pytest.mark.gpu
@pytest.mark.parametrize("scale_exp", [-100, -40, -20, 20, 40, 100])
def test_gemv_activation_magnitudes(scale_exp):
    K, N = 1024, 128
    mat = DevMatrix(K, N, matrix_id=13)
    xf = (synth.x(SEED, 13, 1, K).astype(np.uint32) << 16).view(np.float32) * np.float32(2.0**scale_exp)
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)
    check_against_oracle(run(mat, x), x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
def test_gemv_small_workspace_rejected():
    K, N = 512, 64
    mat = DevMatrix(K, N)
    x = to_dev(synth.x(SEED, 0, 1, K))
    y = torch.empty(N, dtype=torch.int16, device="cuda")
    nb = w.w4g128_workspace_bytes(1, K, N)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    with pytest.raises(w.W4G128Error) as ei:
        w.w4g128_gemv(mat.packed, x, y, K, N, ws, ws_bytes=nb - 1)
    assert ei.value.status == 4


@pytest.mark.gpu
def test_gemv_leaves_neighbours_untouched():
    K, N = 640, 80
    mat = DevMatrix(K, N, matrix_id=2)
    x = to_dev(synth.x(SEED, 2, 1, K))
    guard = torch.full((N + 2048,), 0x5A5A, dtype=torch.int16, device="cuda")
    y = guard[1024:1024 + N]
    w.w4g128_gemv(mat.packed, x, y, K, N, workspace(1, K, N))
    torch.cuda.synchronize()
    g = guard.cpu().numpy()
    assert np.all(g[:1024] == 0x5A5A) and np.all(g[1024 + N:] == 0x5A5A)


@pytest.mark.gpu
def test_lm_head_full_size_every_output():
    """K = 5120 lm_head at full size (device-generated weights), M = 1 (gemv)
    and M = 8 (verify): every one of the 248320 columns against the oracle;
    its first 131072 columns called as a prefix view give the same bits."""
    K, N, Np = 5120, 248320, 131072
    mat = DevMatrix(K, N, matrix_id=100, device_fill=True, keep_host=True)
    mat.free_canonical()
    for M in (1, 8):
        x = synth.x(SEED, 100 + M, M, K)
        y = run(mat, x)
        check_against_oracle(y, x, mat.codes, mat.scales, mat.mins)
        xd = to_dev(x)
        yp = torch.empty(M * Np, dtype=torch.int16, device="cuda")
        ws = workspace(M, K, Np)
        if M == 1:
            w.w4g128_gemv(mat.packed, xd, yp, K, Np, ws)
        else:
            w.w4g128_gemm_verify(mat.packed, xd, yp, M, K, Np, ws)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(yp, np.uint16).reshape(M, Np), y[:, :Np])


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8])
def test_largest_k(M):
    """K = 65536, the largest K the boundary accepts (512 groups, 128 segments
    per quad), with a ragged last quad: every output against the oracle."""
    K, N = 65536, 208
    mat = DevMatrix(K, N, matrix_id=101)
    x = synth.x(SEED, 101 + M, M, K)
    check_against_oracle(run(mat, x, verify=(M > 1)), x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
def test_largest_n_every_output():
    """N = 2^24, the largest N the boundary accepts (262,144 quads, 1.07 GB
    packed at K = 128), device-generated; every output at M = 1 (gemv) and
    M = 8 (verify)."""
    K, N = 128, 1 << 24
    mat = DevMatrix(K, N, matrix_id=102, device_fill=True, keep_host=True)
    mat.free_canonical()
    for M in (1, 8):
        x = synth.x(SEED, 102 + M, M, K)
        y = run(mat, x, verify=(M > 1))
        check_against_oracle(y, x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", [(4096, 4096), (17408, 5120), (1152, 208), (5120, 248320)])
def test_local_and_prep_paths_agree(K, N):
    """An M = 1 call builds its activation packages inside each streaming CTA
    when x is 16-byte aligned (and the CTAs' working sets fit in shared
    memory), else through the prep kernel; with x only 4-byte aligned the
    call takes the prep path.  Both paths give the same bits, within the
    bound, through w4g128_gemv and through a two-matrix decode step."""
    mat = DevMatrix(K, N, matrix_id=K + 7)
    x = synth.x(SEED, K + 7, 1, K)
    xa = to_dev(x)
    buf = torch.zeros(K + 8, dtype=torch.int16, device="cuda")
    xm = buf[2:2 + K]  # 4 bytes past a 16-byte boundary
    xm.copy_(xa.view(-1))
    assert xm.data_ptr() % 16 == 4
    ys = []
    for xd in (xa, xm):
        y = torch.empty(N, dtype=torch.int16, device="cuda")
        ws = workspace(1, K, N)
        w.w4g128_gemv(mat.packed, xd, y, K, N, ws)
        torch.cuda.synchronize()
        assert w.w4g128_workspace_status(ws) == 0
        ys.append(to_host(y, np.uint16))
    assert np.array_equal(ys[0], ys[1])
    check_against_oracle(ys[0].reshape(1, N), x, mat.codes, mat.scales, mat.mins)
    small = DevMatrix(640, 80, matrix_id=K + 8)
    xs = synth.x(SEED, K + 8, 1, 640)
    for xd in (xa, xm):
        y = torch.empty(N, dtype=torch.int16, device="cuda")
        y2 = torch.empty(80, dtype=torch.int16, device="cuda")
        descs = [(mat.packed, xd, y, K, N), (small.packed, to_dev(xs), y2, 640, 80)]
        ws = torch.empty(w.w4g128_decode_step_workspace_bytes(descs, 1), dtype=torch.uint8, device="cuda")
        w.w4g128_decode_step(descs, 1, ws)
        torch.cuda.synchronize()
        assert w.w4g128_workspace_status(ws) == 0
        assert np.array_equal(to_host(y, np.uint16), ys[0])
        assert np.array_equal(to_host(y2, np.uint16), run(small, xs)[0])
