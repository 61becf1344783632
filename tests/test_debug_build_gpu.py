"""The range-checked build (libw4g128_debug.so, compiled with W4G128_DEBUG):
every global access the kernels derive from the schedule -- weight and
package copies, x staging, partial slots, tickets, y -- is checked against
its buffer, and a failed check is recorded as W4G128_ERR_INTERNAL in the
status word (the access is skipped; nothing traps).  A spread of calls
covering every kernel path (CTA-local M = 1, quads split over a two-CTA
cluster, the prep-kernel path at M = 1
and M >= 2, both reduce forms, many matrices, the fused norm, the
workspace-free entry point) must pass every check, give the release
library's bits, and leave guard bytes around each y and each workspace
untouched."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, to_dev, to_host  # noqa: E402

GUARD = 4096  # bytes of 0x5A on each side
E_INTERNAL = 8


def guarded(nbytes):
    """A device buffer of nbytes between two guard regions: (whole, view)."""
    whole = torch.full((nbytes + 2 * GUARD,), 0x5A, dtype=torch.uint8, device="cuda")
    return whole, whole[GUARD:GUARD + nbytes]


def guards_intact(whole):
    h = whole.cpu().numpy()
    return bool(np.all(h[:GUARD] == 0x5A) and np.all(h[-GUARD:] == 0x5A))


def status(L, ws):
    out = ctypes.c_int(0)
    assert L.w4g128_workspace_status(ws.data_ptr(), ctypes.byref(out), None) == 0
    return out.value


def stream_call(L, mats, xs, M, kind="step"):
    """decode_step over (mat, x) pairs through library L; returns (ys, status, guards ok)."""
    ys_w = [guarded(2 * M * m.N) for m in mats]
    arr = w._matrices([(m.packed, x, yv.data_ptr(), m.K, m.N) for m, x, (_, yv) in zip(mats, xs, ys_w)])
    nb = L.w4g128_decode_step_workspace_bytes(arr, len(mats), M)
    ws_w, ws = guarded(nb)
    st = torch.cuda.current_stream().cuda_stream
    if kind == "gemv":
        rc = L.w4g128_gemv(mats[0].packed.data_ptr(), xs[0].data_ptr(), ys_w[0][1].data_ptr(), mats[0].K,
                           mats[0].N, ws.data_ptr(), nb, st)
    elif kind == "verify":
        rc = L.w4g128_gemm_verify(mats[0].packed.data_ptr(), xs[0].data_ptr(), ys_w[0][1].data_ptr(), M,
                                  mats[0].K, mats[0].N, ws.data_ptr(), nb, st)
    else:
        rc = L.w4g128_decode_step(arr, len(mats), M, ws.data_ptr(), nb, st)
    assert rc == 0, w.w4g128_status_string(rc)
    torch.cuda.synchronize()
    ok = all(guards_intact(yw) for yw, _ in ys_w) and guards_intact(ws_w)
    ys = [to_host(yv, np.uint16).reshape(M, m.N).copy() for (_, yv), m in zip(ys_w, mats)]
    return ys, status(L, ws), ok


CASES = [
    ("gemv local", [(17408, 5120)], 1, "gemv", False),
    ("gemv prep path (x 4-byte aligned)", [(5120, 6144)], 1, "gemv", True),
    ("gemv largest K", [(65536, 208)], 1, "gemv", False),
    ("gemv paired quads", [(8192, 4096)], 1, "gemv", False),
    ("gemv paired quads, odd and ragged segments, ragged quad", [(11392, 4080)], 1, "gemv", False),
    ("gemv paired quads, 16 warps", [(16384, 4864)], 1, "gemv", False),
    ("verify M=2", [(6144, 5120)], 2, "verify", False),
    ("verify M=8", [(17408, 5120)], 8, "verify", False),
    ("verify M=16", [(5120, 6144)], 16, "verify", False),
    ("lm_head M=1", [(5120, 248320)], 1, "gemv", False),
    ("lm_head M=8 per-warp fold", [(5120, 248320)], 8, "verify", False),
    ("layer step M=1", [(5120, 6144)] * 3 + [(6144, 5120), (5120, 34816), (17408, 5120)], 1, "step", False),
    ("layer step M=8", [(5120, 6144)] * 3 + [(6144, 5120), (5120, 34816), (17408, 5120)], 8, "step", False),
    ("eleven matrices M=1", [(17408, 1024), (128, 16), (640, 80), (4096, 4096), (1152, 208), (65536, 64),
                             (384, 48), (6144, 5120), (2048, 1008), (5120, 960), (256, 4096)], 1, "step", False),
    ("eleven matrices M=8", [(17408, 1024), (128, 16), (640, 80), (4096, 4096), (1152, 208), (65536, 64),
                             (384, 48), (6144, 5120), (2048, 1008), (5120, 960), (256, 4096)], 8, "step", False),
    ("per-warp records M=8", [(4096, 131072), (1024, 65536), (5120, 6144)], 8, "step", False),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,shapes,M,kind,misalign", CASES, ids=[c[0] for c in CASES])
def test_debug_build_checks_pass_and_match_release(name, shapes, M, kind, misalign):
    D, R = w.lib_debug(), w.lib()
    mats = [DevMatrix(K, N, matrix_id=1500 + i, device_fill=True) for i, (K, N) in enumerate(shapes)]
    xs = []
    for i, (K, _) in enumerate(shapes):
        x = to_dev(synth.x(SEED, 1600 + i, M, K)).view(-1)
        if misalign:
            buf = torch.zeros(x.numel() + 8, dtype=torch.int16, device="cuda")
            xm = buf[2:2 + x.numel()]
            xm.copy_(x)
            x = xm
        xs.append(x)
    yd, sd, okd = stream_call(D, mats, xs, M, kind)
    yr, sr, okr = stream_call(R, mats, xs, M, kind)
    assert sd == 0, f"{name}: a range check failed (status {sd})"
    assert sr == 0 and okd and okr, name
    for a, b in zip(yd, yr):
        assert np.array_equal(a, b), name


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8])
def test_debug_build_fused_norm(M):
    D, R = w.lib_debug(), w.lib()
    K, N = 17408, 5120
    mat = DevMatrix(K, N, matrix_id=1700, device_fill=True)
    x = to_dev(synth.x(SEED, 1701, M, K))
    res = to_dev(synth.x(SEED, 1702, M, N))
    gam = to_dev(synth.norm_weight(SEED, 1703, N))
    outs = []
    for L in (D, R):
        hw, h = guarded(2 * M * N)
        ow, o = guarded(2 * M * N)
        nb = L.w4g128_workspace_bytes(M, K, N)
        wsw, ws = guarded(nb)
        rc = L.w4g128_gemm_add_rmsnorm(mat.packed.data_ptr(), x.data_ptr(), res.data_ptr(), gam.data_ptr(), 1e-6,
                                       h.data_ptr(), o.data_ptr(), M, K, N, int(M > 1), ws.data_ptr(), nb,
                                       torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert status(L, ws) == 0
        assert guards_intact(hw) and guards_intact(ow) and guards_intact(wsw)
        outs.append((to_host(h, np.uint16).copy(), to_host(o, np.uint16).copy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


@pytest.mark.gpu
def test_debug_build_noalloc():
    D, R = w.lib_debug(), w.lib()
    K, N = 5120, 6144
    mat = DevMatrix(K, N, matrix_id=1710, device_fill=True)
    x = to_dev(synth.x(SEED, 1711, 1, K))
    ys = []
    for L in (D, R):
        yw, y = guarded(2 * N)
        assert L.w4g128_gemv_noalloc(mat.packed.data_ptr(), x.data_ptr(), y.data_ptr(), K, N,
                                     torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        st = ctypes.c_int(-1)
        assert L.w4g128_noalloc_status(ctypes.byref(st), None) == 0 and st.value == 0
        assert guards_intact(yw)
        ys.append(to_host(y, np.uint16).copy())
    assert np.array_equal(ys[0], ys[1])
