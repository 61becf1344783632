"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every function the headers declare, and rejects bad arguments
synchronously, before anything is launched."""
import ctypes

import pytest

import int4_weight_only_g128_gb300 as w

E_INVALID, E_SHAPE, E_ALIGN, E_WS, E_CUDA, E_DEVICE, E_TIMEOUT = 1, 2, 3, 4, 5, 6, 7


@pytest.fixture(scope="module")
def L():
    return w.lib()


def test_every_header_symbol_is_exported(L):
    names = w.exported_symbols()
    assert len(names) == 21
    for n in names:
        assert hasattr(L, n), n


def test_packed_bytes_exact():
    assert w.w4g128_packed_bytes(4096, 4096) == 4096 * 4096 // 2 + 4 * 32 * 4096 == 8912896
    assert w.w4g128_packed_bytes(5120, 248320) == 675430400
    assert w.w4g128_packed_bytes(5120, 131072) == 356515840
    assert w.w4g128_packed_bytes(17408, 5120) == 47349760
    for K, N in [(128, 16), (5120, 34816)]:
        assert w.w4g128_packed_bytes(K, N) * 32 == K * N * 17
    for K, N in [(100, 16), (128, 8), (0, 16), (128, 0), (128, 24), (65536 + 128, 16)]:
        assert w.w4g128_packed_bytes(K, N) == 0


def test_status_strings():
    for s in range(9):
        assert isinstance(w.w4g128_status_string(s), str) and w.w4g128_status_string(s)
    assert "unknown" in w.w4g128_status_string(99)


FAKE = 0x10000  # a 16-byte-aligned non-null address that is never dereferenced on these paths


def test_gemv_argument_errors(L):
    assert L.w4g128_gemv(None, FAKE, FAKE, 128, 16, FAKE, 1 << 20, None) == E_INVALID
    assert L.w4g128_gemv(FAKE, FAKE, FAKE, 100, 16, FAKE, 1 << 20, None) == E_SHAPE
    assert L.w4g128_gemv(FAKE, FAKE, FAKE, 128, 24, FAKE, 1 << 20, None) == E_SHAPE
    assert L.w4g128_gemv(FAKE + 8, FAKE, FAKE, 128, 16, FAKE, 1 << 20, None) == E_ALIGN
    assert L.w4g128_gemv(FAKE, FAKE + 2, FAKE, 128, 16, FAKE, 1 << 20, None) == E_ALIGN
    assert L.w4g128_gemv(FAKE, FAKE, FAKE, 128, 16, FAKE + 4, 1 << 20, None) == E_ALIGN
    assert L.w4g128_gemv(FAKE, FAKE, FAKE, 128, 16, None, 1 << 20, None) == E_INVALID


def test_verify_argument_errors(L):
    for M in (0, 17, -1):
        assert L.w4g128_gemm_verify(FAKE, FAKE, FAKE, M, 128, 16, FAKE, 1 << 20, None) == E_INVALID


def test_add_rmsnorm_argument_errors(L):
    F, G, H, O, R = FAKE, FAKE + 0x1000, FAKE + 0x2000, FAKE + 0x3000, FAKE + 0x4000

    def call(packed=F, x=F + 0x800, res=R, gam=G, eps=1e-6, h=H, out=O, M=1, K=128, N=16, verify=0, ws=F):
        return L.w4g128_gemm_add_rmsnorm(packed, x, res, gam, eps, h, out, M, K, N, verify, ws, 1 << 20, None)

    assert call(res=None) == E_INVALID
    assert call(gam=None) == E_INVALID
    assert call(out=None) == E_INVALID
    assert call(h=None) == E_INVALID
    assert call(eps=-1.0) == E_INVALID
    assert call(eps=float("nan")) == E_INVALID
    assert call(eps=float("inf")) == E_INVALID
    assert call(verify=2) == E_INVALID
    assert call(out=H) == E_INVALID          # out is h
    assert call(out=R) == E_INVALID          # out is the residual
    assert call(x=H) == E_INVALID            # h is x
    assert call(M=17) == E_INVALID
    assert call(N=24) == E_SHAPE
    assert call(gam=G + 2) == E_ALIGN
    assert call(res=R + 2) == E_ALIGN
    assert call(out=O + 2) == E_ALIGN
    assert call(h=H + 2) == E_ALIGN


def test_decode_step_argument_errors(L):
    mats = (w._Matrix * 2)()
    mats[0] = w._Matrix(FAKE, FAKE, FAKE, 128, 16)
    mats[1] = w._Matrix(FAKE, FAKE, FAKE, 256, 48)
    assert L.w4g128_decode_step(mats, 0, 1, FAKE, 1 << 20, None) == E_INVALID
    assert L.w4g128_decode_step(mats, 513, 1, FAKE, 1 << 20, None) == E_INVALID
    assert L.w4g128_decode_step(None, 1, 1, FAKE, 1 << 20, None) == E_INVALID
    mats[1] = w._Matrix(FAKE, FAKE, FAKE, 256, 40)
    assert L.w4g128_decode_step(mats, 2, 1, FAKE, 1 << 20, None) == E_SHAPE
    mats[1] = w._Matrix(FAKE, FAKE, None, 256, 48)
    assert L.w4g128_decode_step(mats, 2, 1, FAKE, 1 << 20, None) == E_INVALID


def test_schedule_argument_errors(L):
    mats = (w._Matrix * 2)()
    mats[0] = w._Matrix(None, None, None, 128, 16)
    mats[1] = w._Matrix(None, None, None, 256, 48)
    out = (ctypes.c_longlong * 8)()
    assert L.w4g128_schedule(None, 1, 1, out, 8) == E_INVALID
    assert L.w4g128_schedule(mats, 0, 1, out, 8) == E_INVALID
    assert L.w4g128_schedule(mats, 513, 1, out, 8) == E_INVALID
    assert L.w4g128_schedule(mats, 2, 0, out, 8) == E_INVALID
    assert L.w4g128_schedule(mats, 2, 17, out, 8) == E_INVALID
    assert L.w4g128_schedule(mats, 2, 1, None, 8) == E_INVALID
    assert L.w4g128_schedule(mats, 2, 1, out, 0) == E_INVALID
    mats[1] = w._Matrix(None, None, None, 200, 48)
    assert L.w4g128_schedule(mats, 2, 1, out, 8) == E_SHAPE
    with open(w._INCLUDE + "/w4g128.h") as f:
        assert "#define W4G128_SCHEDULE_FIELDS %d" % w.SCHEDULE_FIELDS in f.read()


def test_pack_argument_errors(L):
    assert L.w4g128_pack(None, FAKE, FAKE, 128, 16, FAKE, None) == E_INVALID
    assert L.w4g128_pack(FAKE, FAKE, FAKE, 128, 17, FAKE, None) == E_SHAPE
    assert L.w4g128_pack(FAKE, FAKE, FAKE, 128, 16, FAKE + 4, None) == E_ALIGN
    assert L.w4g128_unpack(FAKE, 128, 16, FAKE, FAKE + 1, FAKE, None) == E_ALIGN


def test_probe_argument_errors(L):
    assert L.w4g128_probe_read(None, 16, FAKE, None) == E_INVALID
    assert L.w4g128_probe_read(FAKE, 15, FAKE, None) == E_SHAPE
    assert L.w4g128_probe_copy(FAKE, FAKE + 8, 16, None) == E_ALIGN


def test_workspace_queries_reject_bad_shapes(L):
    assert w.w4g128_workspace_bytes(0, 128, 16) == 0
    assert w.w4g128_workspace_bytes(1, 127, 16) == 0
    assert w.w4g128_decode_step_workspace_bytes([(FAKE, FAKE, FAKE, 128, 15)], 1) == 0


def test_no_device_is_reported_not_faked():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = w.lib()
    assert L.w4g128_gemv(FAKE, FAKE, FAKE, 128, 16, FAKE, 1 << 20, None) == E_DEVICE
    assert L.w4g128_pack(FAKE, FAKE, FAKE, 128, 16, FAKE, None) == E_DEVICE
    assert L.w4g128_gemm_add_rmsnorm(FAKE, FAKE + 0x800, FAKE + 0x1000, FAKE + 0x2000, 1e-6, FAKE + 0x1000,
                                     FAKE + 0x3000, 1, 128, 16, 0, FAKE, 1 << 20, None) == E_DEVICE
    assert w.w4g128_workspace_bytes(1, 128, 16) == 0
    mats = (w._Matrix * 1)()
    mats[0] = w._Matrix(None, None, None, 128, 16)
    out = (ctypes.c_longlong * 8)()
    assert L.w4g128_schedule(mats, 1, 1, out, 8) == E_DEVICE


def test_error_raises_in_binding():
    with pytest.raises(w.W4G128Error) as ei:
        w.w4g128_gemv(FAKE, FAKE, FAKE, 100, 16, FAKE, ws_bytes=1 << 20, stream=0)
    assert ei.value.status == E_SHAPE
    assert ctypes.sizeof(w._Matrix) == 32


def test_selftest_argument_errors(L):
    assert L.w4g128_selftest_wait(None, 512, 1000, 0, None) == E_INVALID
    assert L.w4g128_selftest_wait(FAKE, 512, 1000, 2, None) == E_INVALID
    assert L.w4g128_selftest_wait(FAKE, 512, 0, 0, None) == E_INVALID
    assert L.w4g128_selftest_wait(FAKE, 512, 3_000_000_000, 0, None) == E_INVALID
    assert L.w4g128_selftest_wait(FAKE + 8, 512, 1000, 0, None) == E_ALIGN
    assert L.w4g128_selftest_wait(FAKE, 511, 1000, 0, None) == E_WS
    assert L.w4g128_noalloc_status(None, None) == E_INVALID


_FAULT_CHILD = """
import sys
sys.path.insert(0, {root!r})
import int4_weight_only_g128_gb300 as w
L = w.lib()
F = 0x10000
mats = (w._Matrix * 1)()
mats[0] = w._Matrix(F, F, F, 128, 16)
print(L.w4g128_gemv(F, F, F, 128, 16, F, 1 << 20, None),
      L.w4g128_gemm_verify(F, F, F, 8, 128, 16, F, 1 << 20, None),
      L.w4g128_decode_step(mats, 1, 1, F, 1 << 20, None),
      L.w4g128_gemm_add_rmsnorm(F, F + 0x800, F + 0x1000, F + 0x2000, 1e-6, F + 0x1000, F + 0x3000, 1, 128, 16,
                                0, F, 1 << 20, None),
      L.w4g128_gemv_noalloc(F, F, F, 128, 16, None),
      L.w4g128_pack(F, F, F, 128, 16, F, None),
      L.w4g128_selftest_wait(F, 512, 1000, 0, None),
      L.w4g128_gemv(F, F, F, 100, 16, F, 1 << 20, None))
"""


@pytest.mark.parametrize("mode,status", [("launch", E_CUDA), ("workspace", E_WS)])
def test_host_fault_hook(mode, status):
    """W4G128_FAULT makes every compute entry point return the injected error
    after argument validation and before touching the device (no GPU needed);
    argument errors still come first."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, W4G128_FAULT=mode)
    out = subprocess.run([sys.executable, "-c", _FAULT_CHILD.format(root=root)], env=env, capture_output=True,
                         text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    codes = [int(v) for v in out.stdout.split()]
    assert codes[:-1] == [status] * 7
    assert codes[-1] == E_SHAPE


def test_decode_step_host_argument_errors(L):
    mats = (w._Matrix * 1)()
    mats[0] = w._Matrix(FAKE, FAKE, FAKE, 128, 16)
    assert L.w4g128_decode_step_host(mats, 1, 1, None, FAKE, 16, FAKE, FAKE, 16, FAKE, 1 << 20, None) == E_INVALID
    assert L.w4g128_decode_step_host(mats, 1, 1, FAKE, FAKE, 16, FAKE, None, 16, FAKE, 1 << 20, None) == E_INVALID
    assert L.w4g128_decode_step_host(mats, 0, 1, FAKE, FAKE, 16, FAKE, FAKE, 16, FAKE, 1 << 20, None) == E_INVALID
    mats[0] = w._Matrix(FAKE, FAKE, FAKE, 128, 24)
    assert L.w4g128_decode_step_host(mats, 1, 1, FAKE, FAKE, 16, FAKE, FAKE, 16, FAKE, 1 << 20, None) == E_SHAPE


def test_debug_library_exports_every_symbol():
    """The range-checked build (W4G128_DEBUG) loads beside the release one and
    exports the same entry points, with the same argument checks."""
    D = w.lib_debug()
    for n in w.exported_symbols():
        assert hasattr(D, n), n
    assert D.w4g128_gemv(FAKE, FAKE, FAKE, 100, 16, FAKE, 1 << 20, None) == E_SHAPE
