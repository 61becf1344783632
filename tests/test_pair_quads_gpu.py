"""Quads split over a two-CTA thread-block cluster (M = 1, one matrix of 11
to 32 segments per quad whose quads fit twice on the SMs and leave few of
them idle): CTA 2q streams
the first half of quad q's 512-row segments, CTA 2q + 1 the rest, and the
first CTA folds all of the quad's segment sums, in segment order, from its
shared memory.

Checked: the schedule takes that path for these shapes and no other; every
output is within the oracle's bound; the exact-integer case is bf16_rn of
the oracle bit for bit (a segment sum dropped, repeated or placed in the
wrong slot changes an output by at least one unit); the outputs are bitwise
those of the same matrix streamed through the multi-matrix schedule (other
CTAs, other folds, the same summation order) and through the package-kernel
path that an x only 4-byte aligned takes; back-to-back calls on one stream
without synchronisation; the residual add + RMS norm entry point's h."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import (MINUS_EIGHT, ONE, SEED, DevMatrix, check_against_oracle, exact_bits, int_x, run,  # noqa: E402
                         to_dev, to_host, workspace)

# (K, N): segments per quad S = ceil(K / 512), quads NQ = ceil(N / 64)
SHAPES = [
    (5632, 2432),    # S 11 (6 + 5), NQ 38
    (8192, 4096),    # S 16, NQ 64
    (11392, 4080),   # S 23 (12 + 11; the last segment one group), NQ 64, the last quad 3 tiles
    (10240, 3072),   # S 20 (10 warps per CTA), NQ 48
    (16384, 4864),   # S 32 (16 warps per CTA), NQ 76: every SM
]


def schedule(K, N):
    return w.w4g128_schedule([(None, None, None, K, N)], 1)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", SHAPES)
def test_schedule_pairs_quads(K, N):
    S, NQ = -(-K // 512), -(-N // 64)
    s = schedule(K, N)
    assert s["local"] == 1 and s["pair_quads"] == 1, s
    assert s["ctas"] == 2 * NQ and s["cta_warps"] == -(-S // 2) and s["second_pass"] == 0, s
    assert s["items"] == NQ * S and s["workspace_bytes"] == w.w4g128_workspace_bytes(1, K, N)


@pytest.mark.gpu
def test_schedule_other_shapes_do_not_pair():
    assert schedule(4096, 4096)["pair_quads"] == 0            # one CTA holds a quad of 8 segments
    assert schedule(8192, 8192)["pair_quads"] == 0            # more quads than the pairs the SMs hold
    assert schedule(17408, 4096)["pair_quads"] == 0           # 34 segments
    assert schedule(8192, 1024)["pair_quads"] == 0            # too few quads
    assert schedule(16384, 2432)["pair_quads"] == 0           # half the SMs idle behind 16-item CTAs
    assert w.w4g128_schedule([(None, None, None, 8192, 4096)] * 2, 1)["pair_quads"] == 0
    assert w.w4g128_schedule([(None, None, None, 8192, 4096)], 8)["pair_quads"] == 0


def multi_matrix(mat, x_bits):
    """mat's y through a two-matrix decode step (the multi-matrix schedule)."""
    other = DevMatrix(256, 48, matrix_id=2999)
    xs = [to_dev(x_bits).view(-1), to_dev(synth.x(SEED, 2998, 1, 256)).view(-1)]
    ys = [torch.empty(mat.N, dtype=torch.int16, device="cuda"), torch.empty(48, dtype=torch.int16, device="cuda")]
    descs = [(mat.packed, xs[0], ys[0], mat.K, mat.N), (other.packed, xs[1], ys[1], 256, 48)]
    assert w.w4g128_schedule(descs, 1)["pair_quads"] == 0
    ws = torch.empty(w.w4g128_decode_step_workspace_bytes(descs, 1), dtype=torch.uint8, device="cuda")
    w.w4g128_decode_step(descs, 1, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    return to_host(ys[0], np.uint16).reshape(1, mat.N)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", SHAPES)
def test_pairs_match_oracle_and_multi_matrix_path(K, N):
    mat = DevMatrix(K, N, matrix_id=2900 + K // 128 + N)
    x = synth.x(SEED, 2901 + K, 1, K)
    y = run(mat, x)
    check_against_oracle(y, x, mat.codes, mat.scales, mat.mins)
    assert np.array_equal(y, multi_matrix(mat, x))
    assert np.array_equal(run(mat, x, verify=True), y)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", SHAPES)
def test_pair_shapes_with_misaligned_x(K, N):
    """x only 4-byte aligned: the call takes the package-kernel path over the
    balanced split (paired quads leave a warp without an item when the
    segment count is odd, which that path's ticket count does not allow) and
    gives the aligned call's bits."""
    mat = DevMatrix(K, N, matrix_id=3050 + K // 128)
    xb = synth.x(SEED, 3051 + K, 1, K)
    buf = torch.zeros(K + 8, dtype=torch.int16, device="cuda")
    xm = buf[2:2 + K]  # 4 bytes past a 16-byte boundary
    xm.copy_(to_dev(xb).view(-1))
    sch = w.w4g128_schedule([(None, xm, None, K, N)], 1)
    assert sch["local"] == 0 and sch["pair_quads"] == 0, sch
    assert sch["ctas"] * sch["cta_warps"] <= sch["items"] + sch["cta_warps"], sch
    y = torch.empty(N, dtype=torch.int16, device="cuda")
    ws = workspace(1, K, N)
    w.w4g128_gemv(mat.packed, xm, y, K, N, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    assert np.array_equal(to_host(y, np.uint16).reshape(1, N), run(mat, xb))


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", SHAPES)
def test_pairs_exact_integer(K, N):
    O = oracle.Oracle()
    mat = DevMatrix(K, N, matrix_id=2950 + K // 128, device_fill=True, const_meta=(ONE, MINUS_EIGHT),
                    keep_host=True)
    x = int_x(np.random.default_rng(K + N), 1, K)
    y_ref, _ = O.gemm(x, mat.codes, mat.scales, mat.mins)
    assert np.array_equal(run(mat, x), exact_bits(y_ref, O))


@pytest.mark.gpu
def test_pairs_back_to_back():
    """Calls on two shapes and fresh activations, issued back to back on one
    stream and one workspace with no synchronisation, each equal to the same
    call made alone."""
    shapes = [(8192, 4096), (11392, 4080)]
    mats = [DevMatrix(K, N, matrix_id=2970 + i) for i, (K, N) in enumerate(shapes)]
    nb = max(w.w4g128_workspace_bytes(1, K, N) for K, N in shapes)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    calls = []
    for r in range(6):
        m = mats[r % 2]
        xb = synth.x(SEED, 2980 + r, 1, m.K)
        calls.append((m, xb, to_dev(xb).view(-1), torch.empty(m.N, dtype=torch.int16, device="cuda")))
    for m, _, x, y in calls:
        w.w4g128_gemv(m.packed, x, y, m.K, m.N, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    for m, xb, _, y in calls:
        assert np.array_equal(to_host(y, np.uint16).reshape(1, m.N), run(m, xb))


@pytest.mark.gpu
def test_pairs_fused_norm_h():
    """The residual add + RMS norm call with a zero residual: h is the plain
    product's y bit for bit (h = bf16(0 + the fp32 fold))."""
    K, N = 8192, 4096
    mat = DevMatrix(K, N, matrix_id=2990)
    xb = synth.x(SEED, 2991, 1, K)
    x = to_dev(xb)
    res = torch.zeros(N, dtype=torch.int16, device="cuda")
    gam = to_dev(synth.norm_weight(SEED, 2992, N))
    h = torch.empty(N, dtype=torch.int16, device="cuda")
    out = torch.empty(N, dtype=torch.int16, device="cuda")
    ws = workspace(1, K, N)
    w.w4g128_gemm_add_rmsnorm(mat.packed, x, res, gam, 1e-6, h, out, 1, K, N, 0, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    assert np.array_equal(to_host(h, np.uint16).reshape(1, N), run(mat, xb))
