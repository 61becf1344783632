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
from gpu_helpers import SEED, DevMatrix, check_against_oracle, to_dev, to_host  # noqa: E402

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


@pytest.mark.gpu
def test_many_plans_interleaved():
    """More distinct (shapes, M) calls than the library's per-thread plan cache
    holds, interleaved and repeated: every repeat gives the first pass's bits,
    so no cached plan carries state from another call."""
    shapes = [(4096, 4096), (5120, 6144), (1152, 208), (17408, 1024), (640, 80), (2048, 4080)]
    mats = [DevMatrix(K, N, matrix_id=950 + i) for i, (K, N) in enumerate(shapes)]
    calls = [(i, M) for M in (1, 8, 2, 16) for i in range(len(shapes))]
    first = {}
    for rep in range(2):
        for i, M in calls:
            mat = mats[i]
            x = synth.x(SEED, 960 + i, M, mat.K)
            xd = to_dev(x)
            y = torch.empty(M * mat.N, dtype=torch.int16, device="cuda")
            ws = torch.empty(w.w4g128_workspace_bytes(M, mat.K, mat.N), dtype=torch.uint8, device="cuda")
            if M == 1:
                w.w4g128_gemv(mat.packed, xd, y, mat.K, mat.N, ws)
            else:
                w.w4g128_gemm_verify(mat.packed, xd, y, M, mat.K, mat.N, ws)
            torch.cuda.synchronize()
            assert w.w4g128_workspace_status(ws) == 0
            out = to_host(y, np.uint16).reshape(M, mat.N)
            if rep == 0:
                check_against_oracle(out, x, mat.codes, mat.scales, mat.mins)
                first[(i, M)] = out
            else:
                assert np.array_equal(out, first[(i, M)]), (shapes[i], M)


@pytest.mark.gpu
def test_graph_replays_complete_every_boundary_fold():
    """M = 1 calls fold the quads that straddle two streaming CTAs in a kernel
    behind the streaming kernel, and leave no state in the workspace that a
    later call depends on.  A CUDA graph of three calls replayed three times,
    with every y cleared between replays, must give the eager results each
    time (state carried from one replay to the next -- such as a counter the
    previous replay completed -- would leave quads unwritten)."""
    shapes = [(17408, 5120), (4096, 4096), (5120, 6144)]
    mats = [DevMatrix(K, N, matrix_id=970 + i) for i, (K, N) in enumerate(shapes)]
    xs = [to_dev(synth.x(SEED, 980 + i, 1, K)) for i, (K, _) in enumerate(shapes)]
    ys = [torch.empty(N, dtype=torch.int16, device="cuda") for _, N in shapes]
    wss = [torch.empty(w.w4g128_workspace_bytes(1, K, N), dtype=torch.uint8, device="cuda") for K, N in shapes]
    for m, x, y, ws in zip(mats, xs, ys, wss):
        w.w4g128_gemv(m.packed, x, y, m.K, m.N, ws)
    torch.cuda.synchronize()
    eager = [to_host(y, np.uint16).copy() for y in ys]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream().cuda_stream
        for m, x, y, ws in zip(mats, xs, ys, wss):
            w.w4g128_gemv(m.packed, x, y, m.K, m.N, ws, stream=cs)
    for rep in range(3):
        for y in ys:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for ws in wss:
            assert w.w4g128_workspace_status(ws) == 0
        for i, y in enumerate(ys):
            assert np.array_equal(to_host(y, np.uint16), eager[i]), (rep, shapes[i])
