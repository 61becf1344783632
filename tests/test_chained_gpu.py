"""Dependent calls back to back on one stream, without synchronising: each
call's prep kernel is launched early behind the previous kernel and must wait
for it before it reads x or touches the workspace.  The output of call n is
the input of call n + 1 (the shapes chain K -> N -> K ...), one workspace is
shared, and the chain is replayed from a CUDA graph too; every result must be
bitwise the result of separately synchronised calls."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, to_dev, to_host  # noqa: E402

# each call's K is the previous call's N, so y of one call is x of the next;
# sizes span few quads to many, split and owned quads
CHAIN = [(1024, 4096), (4096, 1024), (1024, 2048), (2048, 4096), (4096, 1024), (1024, 1024)]
assert all(CHAIN[i + 1][0] == CHAIN[i][1] for i in range(len(CHAIN) - 1))


def _call(mat, x, y, M, ws, verify, stream=None):
    if M == 1 and not verify:
        w.w4g128_gemv(mat.packed, x, y, mat.K, mat.N, ws, stream=stream)
    else:
        w.w4g128_gemm_verify(mat.packed, x, y, M, mat.K, mat.N, ws, stream=stream)


def _run_chain(mats, x0, M, verify, sync_each, ws, graph=False):
    bufs = [x0] + [torch.empty(M * m.N, dtype=torch.int16, device="cuda") for m in mats]
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream().cuda_stream
            for i, m in enumerate(mats):
                _call(m, bufs[i], bufs[i + 1], M, ws, verify, stream=cs)
        g.replay()
    else:
        for i, m in enumerate(mats):
            _call(m, bufs[i], bufs[i + 1], M, ws, verify)
            if sync_each:
                torch.cuda.synchronize()
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    return [to_host(b, np.uint16).copy() for b in bufs[1:]]


@pytest.mark.gpu
@pytest.mark.parametrize("M,verify", [(1, False), (1, True), (8, True), (16, True)])
def test_dependent_chain_equals_synchronised_calls(M, verify):
    mats = [DevMatrix(K, N, matrix_id=500 + i) for i, (K, N) in enumerate(CHAIN)]
    x0 = to_dev(synth.x(SEED, 600 + M, M, CHAIN[0][0]))
    nb = max(w.w4g128_workspace_bytes(M, K, N) for K, N in CHAIN)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ref = _run_chain(mats, x0, M, verify, True, ws)
    got = _run_chain(mats, x0, M, verify, False, ws)
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)
    got_g = _run_chain(mats, x0, M, verify, False, ws, graph=True)
    for a, b in zip(ref, got_g):
        assert np.array_equal(a, b)


@pytest.mark.gpu
def test_norm_output_feeds_next_call():
    """The residual add + RMS norm's out is the next projection's x, h its
    residual: the whole chain back to back equals synchronised calls."""
    K = N = 2048
    mats = [DevMatrix(K, N, matrix_id=700 + i) for i in range(3)]
    gam = to_dev(synth.norm_weight(SEED, 701, N))
    x0 = to_dev(synth.x(SEED, 702, 1, K))
    r0 = to_dev(synth.x(SEED, 703, 1, N))
    ws = torch.empty(w.w4g128_workspace_bytes(1, K, N), dtype=torch.uint8, device="cuda")

    def chain(sync_each):
        x, res = x0, r0.clone()
        outs = []
        for m in mats:
            out = torch.empty(N, dtype=torch.int16, device="cuda")
            w.w4g128_gemm_add_rmsnorm(m.packed, x, res, gam, 1e-6, res, out, 1, K, N, 0, ws)  # h in place
            if sync_each:
                torch.cuda.synchronize()
            outs.append(out)
            x = out
        torch.cuda.synchronize()
        assert w.w4g128_workspace_status(ws) == 0
        return [to_host(o, np.uint16).copy() for o in outs] + [to_host(res, np.uint16).copy()]

    ref = chain(True)
    got = chain(False)
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)
