"""Failure detection on the GPU without a fault: every device-side wait of the
library is bounded.  w4g128_selftest_wait runs the library's bounded flag wait
on a workspace word that nothing writes, with a 1 ms limit: the wait must run
out, the kernel must record W4G128_ERR_TIMEOUT in the status word and return
on its own, and the context and the workspace must stay usable -- a normal
call on the same workspace afterwards succeeds and is correct."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, check_against_oracle, to_dev, to_host  # noqa: E402

E_TIMEOUT = 7


@pytest.mark.gpu
def test_bounded_wait_runs_out_and_the_workspace_stays_usable():
    K, N = 5120, 6144
    mat = DevMatrix(K, N, matrix_id=41)
    nb = max(w.w4g128_workspace_bytes(1, K, N), w.SELFTEST_WS_BYTES)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    w.w4g128_selftest_wait(ws, 1_000_000, 0)   # nothing sets the flag: 1 ms, then give up
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert w.w4g128_workspace_status(ws) == E_TIMEOUT
    assert waited < 1.0
    w.w4g128_selftest_wait(ws, 1_000_000, 1)   # flag set: no timeout
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    w.w4g128_selftest_wait(ws, 1_000_000, 0)   # leave a timeout behind, then a real call
    x = synth.x(SEED, 41, 1, K)
    y = torch.empty(N, dtype=torch.int16, device="cuda")
    w.w4g128_gemv(mat.packed, to_dev(x), y, K, N, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    check_against_oracle(to_host(y, np.uint16).reshape(1, N), x, mat.codes, mat.scales, mat.mins)


@pytest.mark.gpu
def test_timeout_limit_is_respected():
    """A 50 ms limit waits about that long (the kernel gives up on its own)."""
    ws = torch.empty(w.SELFTEST_WS_BYTES, dtype=torch.uint8, device="cuda")
    w.w4g128_selftest_wait(ws, 1000, 0)  # warm-up launch
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    w.w4g128_selftest_wait(ws, 50_000_000, 0)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    assert w.w4g128_workspace_status(ws) == E_TIMEOUT
    assert 45.0 <= ms <= 500.0, ms
