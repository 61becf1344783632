"""The no-workspace GEMV entry point (w4g128_gemv_noalloc).

Some callers cannot give the library a device workspace because they must
not allocate device memory -- plugin hooks of another runtime that owns the
memory budget, fixed-pool servers, latency-critical threads that must not call
cudaMalloc.  This entry point keeps its scratch in a fixed array inside the
library.  The test calls it through the C ABI several times in a row and
checks every output against the regular w4g128_gemv (same tolerance as the
parity tests, and in fact the same bits), so stale scratch contents from one
call cannot leak into the next.  It lives in its own file so that it runs last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, to_dev, to_host, workspace  # noqa: E402


def noalloc(mat, x_bits):
    y = torch.empty(mat.N, dtype=torch.int16, device="cuda")
    rc = w.lib().w4g128_gemv_noalloc(mat.packed.data_ptr(), to_dev(x_bits).data_ptr(), y.data_ptr(),
                                     mat.K, mat.N, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, w.w4g128_status_string(rc)
    torch.cuda.synchronize()
    return to_host(y, np.uint16)


def regular(mat, x_bits):
    y = torch.empty(mat.N, dtype=torch.int16, device="cuda")
    w.w4g128_gemv(mat.packed, to_dev(x_bits), y, mat.K, mat.N, workspace(1, mat.K, mat.N))
    torch.cuda.synchronize()
    return to_host(y, np.uint16)


@pytest.mark.gpu
def test_noalloc_matches_gemv_on_consecutive_calls():
    O = oracle.Oracle()
    # split-K everywhere (tickets and partials live in the scratch), then a
    # different shape, then the first shape again with new activations
    cases = [(DevMatrix(5120, 6144, matrix_id=501), 1), (DevMatrix(17408, 5120, matrix_id=502), 2)]
    cases.append((cases[0][0], 3))
    for mat, xid in cases:
        x = synth.x(SEED, 600 + xid, 1, mat.K)
        y_new = noalloc(mat, x)
        y_ref = regular(mat, x)
        _, a = O.gemm(x, mat.codes, mat.scales, mat.mins)
        ok, _ = oracle.accept(oracle.bf16_bits_to_f64(y_new)[None, :],
                              oracle.bf16_bits_to_f64(y_ref)[None, :], a, O)
        assert ok.all()
        assert np.array_equal(y_new, y_ref)


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_the_scratch():
    # K = 65536, N = 65536 needs far more than the fixed scratch; the call must
    # fail before launching anything, so the pointers are never dereferenced.
    fake = 1 << 20
    rc = w.lib().w4g128_gemv_noalloc(fake, fake, fake, 65536, 65536, None)
    assert rc == 4  # W4G128_ERR_WORKSPACE
    assert w.w4g128_workspace_bytes(1, 65536, 65536) > (16 << 20)
