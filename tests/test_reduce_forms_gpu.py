"""The two forms of the M >= 2 split-K fold: a call folds per quad unless it
has more quads than streaming warps and than one wave of per-quad reduce
CTAs, and then per streaming warp (one matrix: from the schedule; several:
from the warps' records).  Both fold a quad's segment partials in segment
order, so the outputs are bitwise equal whichever form a call takes; and every
output is within the oracle bound."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, check_against_oracle, run, to_dev, to_host, workspace  # noqa: E402

# 2048 + 1024 + 96 = 3168 quads: more than the 2432 (M <= 8) or 1216 (M > 8)
# streaming warps a 152-SM GPU holds, and than one wave of per-quad reduce
# CTAs at M >= 4, so the call folds per warp from the warps' records; alone,
# each matrix folds per quad (at M = 16 the first folds per warp from the
# schedule).
SHAPES = [(4096, 131072), (1024, 65536), (5120, 6144)]


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
@pytest.mark.parametrize("M", [4, 8, 16])
def test_per_warp_fold_several_matrices(M):
    mats = [DevMatrix(K, N, matrix_id=600 + i, device_fill=True, keep_host=True) for i, (K, N) in enumerate(SHAPES)]
    for m in mats:
        m.free_canonical()
    xh = [synth.x(SEED, 700 + i, M, K) for i, (K, N) in enumerate(SHAPES)]
    ys = decode_step(mats, [to_dev(x) for x in xh], M)
    for mat, x, y in zip(mats, xh, ys):
        assert np.array_equal(y, run(mat, x, M=M, verify=True))
        check_against_oracle(y, x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [4, 8, 16])
def test_per_warp_fold_one_matrix_equals_prefix_view(M):
    """The lm_head shape (3880 quads) folds per warp; its first 131072 columns
    called as a prefix view (2048 quads) fold per quad at M <= 8: the same
    bits; every output within the bound."""
    K, N, Np = 5120, 248320, 131072
    mat = DevMatrix(K, N, matrix_id=610, device_fill=True, keep_host=True)
    mat.free_canonical()
    x = synth.x(SEED, 611, M, K)
    full = run(mat, x, M=M, verify=True)
    xd = to_dev(x)
    y = torch.empty(M * Np, dtype=torch.int16, device="cuda")
    ws = workspace(M, K, Np)
    w.w4g128_gemm_verify(mat.packed, xd, y, M, K, Np, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    assert np.array_equal(to_host(y, np.uint16).reshape(M, Np), full[:, :Np])
    check_against_oracle(full, x, mat.codes, mat.scales, mat.mins)
