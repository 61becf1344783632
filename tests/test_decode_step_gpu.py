"""Multi-matrix weight stream (w4g128_decode_step): every output bitwise equal to
a separate call on the same matrix, every output within the oracle bound, and
the whole 27B-class decode step (64 layers x 6 projections + lm_head, 14.04 GB)
checked on every output."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, canonical_from_device, check_against_oracle, run, to_dev, to_host  # noqa: E402,E501

LAYER = [(5120, 6144), (5120, 6144), (5120, 6144), (6144, 5120), (5120, 34816), (17408, 5120)]


def decode_step(mats, xs, M):
    ys = [torch.empty(M * m.N, dtype=torch.int16, device="cuda") for m in mats]
    descs = [(m.packed, x, y, m.K, m.N) for m, x, y in zip(mats, xs, ys)]
    nb = w.w4g128_decode_step_workspace_bytes(descs, M)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    w.w4g128_decode_step(descs, M, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    return [to_host(y, np.uint16).reshape(M, m.N) for m, y in zip(mats, ys)]


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 2, 8, 11, 16])
def test_decode_step_equals_separate_calls(M):
    shapes = [(128, 16), (640, 80), (4096, 4096), (1152, 208), (2048, 1024), (384, 48)]
    mats = [DevMatrix(K, N, matrix_id=200 + i) for i, (K, N) in enumerate(shapes)]
    xh = [synth.x(SEED, 300 + i, M, K) for i, (K, N) in enumerate(shapes)]
    ys = decode_step(mats, [to_dev(x) for x in xh], M)
    for mat, x, y in zip(mats, xh, ys):
        assert np.array_equal(y, run(mat, x, M=M, verify=(M > 1)))
        check_against_oracle(y, x, mat.codes, mat.scales, mat.mins)


def verify_step(mats, xs, M):
    ys = [torch.empty(M * m.N, dtype=torch.int16, device="cuda") for m in mats]
    descs = [(m.packed, x, y, m.K, m.N) for m, x, y in zip(mats, xs, ys)]
    nb = w.w4g128_decode_step_workspace_bytes(descs, M)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    w.w4g128_verify_step(descs, M, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    return [to_host(y, np.uint16).reshape(M, m.N) for m, y in zip(mats, ys)]


@pytest.mark.gpu
def test_verify_step_rows_equal_single_row_verify():
    """w4g128_verify_step: at M = 1 each output equals gemm_verify(M = 1) on
    its matrix; at M = 8 row m equals the M = 1 step on row m; at every M it
    equals w4g128_decode_step -- all bit for bit, and within the bound."""
    shapes = [(128, 16), (640, 80), (4096, 4096), (1152, 208), (384, 48), (17408, 5120)]
    mats = [DevMatrix(K, N, matrix_id=400 + i) for i, (K, N) in enumerate(shapes)]
    x8 = [synth.x(SEED, 500 + i, 8, K) for i, (K, N) in enumerate(shapes)]
    y8 = verify_step(mats, [to_dev(x) for x in x8], 8)
    d8 = decode_step(mats, [to_dev(x) for x in x8], 8)
    for a, b in zip(y8, d8):
        assert np.array_equal(a, b)
    for m in range(8):
        y1 = verify_step(mats, [to_dev(x[m:m + 1]) for x in x8], 1)
        for a, b in zip(y1, decode_step(mats, [to_dev(x[m:m + 1]) for x in x8], 1)):
            assert np.array_equal(a, b)
        for mat, x, a, b in zip(mats, x8, y1, y8):
            assert np.array_equal(a[0], b[m]), m
            if m == 0:
                assert np.array_equal(a, run(mat, x[:1], verify=True))
                check_against_oracle(a, x[:1], mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
def test_decode_step_single_matrix_equals_gemv():
    mat = DevMatrix(6144, 5120, matrix_id=77)
    x = synth.x(SEED, 77, 1, 6144)
    (y,) = decode_step([mat], [to_dev(x)], 1)
    assert np.array_equal(y, run(mat, x))


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8])
def test_full_decode_step_every_output(M):
    """64 layers x (q, k, v, o, gate+up, down) + the 248320-row lm_head, one
    call; every output of all 385 matrices against the oracle (each matrix's
    canonical arrays regenerated on the device and copied back in turn)."""
    shapes = LAYER * 64 + [(5120, 248320)]
    mats = []
    for i, (K, N) in enumerate(shapes):
        m = DevMatrix(K, N, matrix_id=10000 + i, device_fill=True)
        m.free_canonical()
        mats.append(m)
    total = sum(m.nbytes for m in mats)
    assert total == 14044774400
    xh = [synth.x(SEED, 20000 + i, M, K) for i, (K, N) in enumerate(shapes)]
    ys = decode_step(mats, [to_dev(x) for x in xh], M)
    del mats
    torch.cuda.empty_cache()
    for i, (K, N) in enumerate(shapes):
        c, s, mn = canonical_from_device(K, N, 10000 + i)
        check_against_oracle(ys[i], xh[i], c, s, mn)


@pytest.mark.gpu
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M", [1, 8])
def test_decode_step_host_buffers(M, pinned):
    """w4g128_decode_step_host: x moved in from host memory, the matrices
    streamed, y moved back -- one call (pinned buffers through the library's
    upload and download kernels, pageable ones through copy-engine copies);
    y equals w4g128_decode_step's bit for bit, also through the prepared
    DecodeStep (run_host) twice in a row with new activations."""
    shapes = [(5120, 6144), (6144, 5120), (640, 80)]
    mats = [DevMatrix(K, N, matrix_id=1200 + i) for i, (K, N) in enumerate(shapes)]
    xoff = np.cumsum([0] + [M * K for K, _ in shapes])
    yoff = np.cumsum([0] + [M * N for _, N in shapes])
    x_dev = torch.zeros(int(xoff[-1]), dtype=torch.int16, device="cuda")
    y_dev = torch.zeros(int(yoff[-1]), dtype=torch.int16, device="cuda")
    x_host = torch.empty(int(xoff[-1]), dtype=torch.int16)
    y_host = torch.empty(int(yoff[-1]), dtype=torch.int16)
    if pinned:
        x_host, y_host = x_host.pin_memory(), y_host.pin_memory()
    descs = [(m.packed, x_dev[xoff[i]:xoff[i + 1]], y_dev[yoff[i]:yoff[i + 1]], K, N)
             for i, (m, (K, N)) in enumerate(zip(mats, shapes))]
    ws = torch.empty(w.w4g128_decode_step_workspace_bytes(descs, M), dtype=torch.uint8, device="cuda")
    step = w.DecodeStep(descs, M, ws, x_host=x_host, x_dev=x_dev, y_host=y_host, y_dev=y_dev)
    for rep in range(3):
        xh = [synth.x(SEED, 1300 + 10 * rep + i, M, K) for i, (K, _) in enumerate(shapes)]
        x_host.copy_(torch.from_numpy(np.concatenate([x.ravel() for x in xh]).view(np.int16)))
        if rep == 0:
            w.w4g128_decode_step_host(descs, M, x_host, x_dev, x_dev.numel() * 2, y_host, y_dev, y_dev.numel() * 2, ws)
        else:
            step.run_host()
        torch.cuda.synchronize()
        assert w.w4g128_workspace_status(ws) == 0
        got = y_host.numpy().view(np.uint16).copy()
        expect = decode_step(mats, [to_dev(x) for x in xh], M)
        for i in range(len(shapes)):
            assert np.array_equal(got[yoff[i]:yoff[i + 1]].reshape(M, -1), expect[i])


@pytest.mark.gpu
@pytest.mark.parametrize("units", [5, 256 * 152 + 1, 256 * 152 * 16 + 3, 256 * 152 * 16 * 2 + 256 * 7 + 9])
def test_decode_step_host_moves_whole_ranges(units):
    """The upload and download kernels move every 16-byte unit of the ranges
    they are given, whatever the count: part of one CTA, just over one unit
    per thread on every SM, and over one and two rounds of the loads each
    thread keeps in flight.  The x range holds (the start of) one matrix's x
    and arbitrary bytes after it; the y range holds that matrix's y and bytes
    the step does not write.  After the call x_dev equals x_host and y_host
    equals y_dev over the whole ranges, and the matrix's y is the plain step's."""
    K, N, M = 640, 80, 1
    mat = DevMatrix(K, N, matrix_id=1400)
    nx = units * 8  # int16 elements, 16 bytes a unit
    ny = max(units * 8, M * N)
    ny += (-ny) % 8
    rng = np.random.default_rng(units)
    x_host = torch.from_numpy(rng.integers(-2**15, 2**15, nx, dtype=np.int16)).pin_memory()
    xh = synth.x(SEED, 1401, M, K).ravel().view(np.int16)
    head = min(nx, M * K)  # the tiny range covers only the start of x; the rest of x_dev stays zero
    x_host[:head].copy_(torch.from_numpy(xh[:head]))
    y_fill = rng.integers(-2**15, 2**15, ny, dtype=np.int16)
    y_dev = torch.from_numpy(y_fill).cuda()
    x_dev = torch.zeros(max(nx, M * K), dtype=torch.int16, device="cuda")
    y_host = torch.zeros(ny, dtype=torch.int16).pin_memory()
    descs = [(mat.packed, x_dev[:M * K], y_dev[:M * N], K, N)]
    ws = torch.empty(w.w4g128_decode_step_workspace_bytes(descs, M), dtype=torch.uint8, device="cuda")
    w.w4g128_decode_step_host(descs, M, x_host, x_dev, nx * 2, y_host, y_dev, ny * 2, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    assert torch.equal(x_dev[:nx].cpu(), x_host)
    assert torch.equal(y_host, y_dev.cpu())
    assert np.array_equal(y_fill[M * N:], y_host.numpy()[M * N:])
    expect = decode_step([mat], [x_dev[:M * K].clone()], M)[0]  # the plain step on the x the call moved in
    assert np.array_equal(y_host.numpy()[:M * N].view(np.uint16).reshape(M, N), expect)
