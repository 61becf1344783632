"""The no-workspace GEMV entry point (w4g128_gemv_noalloc).

Some callers cannot give the library a device workspace because they must
not allocate device memory -- plugin hooks of another runtime that owns the
memory budget, fixed-pool servers, latency-critical threads that must not call
cudaMalloc.  This entry point keeps its scratch in a fixed array inside the
library.  The test calls it through the C ABI several times in a row, with
and without synchronising between calls, and checks every output against the
fp64 oracle (same tolerance as the parity tests) and bit for bit against the
regular w4g128_gemv, so stale scratch contents from one call cannot leak into
the next.  It lives in its own file so that it runs last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, to_dev, to_host, workspace  # noqa: E402


def noalloc(mat, x_bits, sync=True):
    y = torch.empty(mat.N, dtype=torch.int16, device="cuda")
    xd = to_dev(x_bits)
    rc = w.lib().w4g128_gemv_noalloc(mat.packed.data_ptr(), xd.data_ptr(), y.data_ptr(),
                                     mat.K, mat.N, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, w.w4g128_status_string(rc)
    if not sync:
        return y, xd
    torch.cuda.synchronize()
    assert w.w4g128_noalloc_status() == 0
    return to_host(y, np.uint16)


def regular(mat, x_bits):
    y = torch.empty(mat.N, dtype=torch.int16, device="cuda")
    w.w4g128_gemv(mat.packed, to_dev(x_bits), y, mat.K, mat.N, workspace(1, mat.K, mat.N))
    torch.cuda.synchronize()
    return to_host(y, np.uint16)


@pytest.mark.gpu
def test_noalloc_matches_gemv_on_consecutive_calls():
    """Against the fp64 oracle (the bound of the parity tests) and bit for bit
    against w4g128_gemv, on calls in a row that reuse the scratch."""
    O = oracle.Oracle()
    # split-K everywhere (tickets and partials live in the scratch), then a
    # different shape, then the first shape again with new activations
    cases = [(DevMatrix(5120, 6144, matrix_id=501), 1), (DevMatrix(17408, 5120, matrix_id=502), 2)]
    cases.append((cases[0][0], 3))
    for mat, xid in cases:
        x = synth.x(SEED, 600 + xid, 1, mat.K)
        y_new = noalloc(mat, x)
        y_ref, a = O.gemm(x, mat.codes, mat.scales, mat.mins)
        ok, _ = oracle.accept(oracle.bf16_bits_to_f64(y_new)[None, :], y_ref, a, O)
        assert ok.all()
        assert np.array_equal(y_new, regular(mat, x))


@pytest.mark.gpu
def test_noalloc_back_to_back_without_synchronising():
    """Four calls on one stream with no synchronisation between them (one on
    the paired-quad schedule, each quad on a two-CTA cluster): each
    call's first kernel waits for the previous call before it rewrites the
    shared scratch, so every output is still bitwise w4g128_gemv's."""
    mats = [DevMatrix(5120, 6144, matrix_id=511), DevMatrix(8192, 4096, matrix_id=514),  # paired quads
            DevMatrix(6144, 5120, matrix_id=512), DevMatrix(1152, 208, matrix_id=513)]
    xs = [synth.x(SEED, 620 + i, 1, m.K) for i, m in enumerate(mats)]
    pending = [noalloc(m, x, sync=False) for m, x in zip(mats, xs)]
    torch.cuda.synchronize()
    assert w.w4g128_noalloc_status() == 0
    for m, x, (y, _) in zip(mats, xs, pending):
        assert np.array_equal(to_host(y, np.uint16), regular(m, x))


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_the_scratch():
    # K = 65536, N = 65536 needs far more than the fixed scratch; the call must
    # fail before launching anything, so the pointers are never dereferenced.
    fake = 1 << 20
    rc = w.lib().w4g128_gemv_noalloc(fake, fake, fake, 65536, 65536, None)
    assert rc == 4  # W4G128_ERR_WORKSPACE
    assert w.w4g128_workspace_bytes(1, 65536, 65536) > (16 << 20)
