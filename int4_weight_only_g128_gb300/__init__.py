"""Python binding of libw4g128, the int4-g128 weight-streaming GEMV for GB300.

Argument marshalling only: every function forwards to the C entry point of
the same name in ``include/*.h``; every step of the computation runs in the
library's CUDA kernels.  Tensors are passed as device pointers taken from
``torch.Tensor.data_ptr()`` (plain integers are accepted as raw pointers), and
the stream defaults to torch's current CUDA stream.  There is no CPU fallback:
if the library cannot be built or loaded, the first call raises.
"""
import ctypes
import os

__all__ = [
    "W4G128Error", "lib", "lib_debug", "exported_symbols",
    "w4g128_status_string", "w4g128_packed_bytes", "w4g128_pack", "w4g128_unpack", "w4g128_quantize",
    "w4g128_workspace_bytes", "w4g128_gemv", "w4g128_gemm_verify",
    "w4g128_decode_step_workspace_bytes", "w4g128_decode_step", "w4g128_verify_step", "w4g128_workspace_status",
    "w4g128_probe_read", "w4g128_probe_copy", "w4g128_probe_sink_bytes", "w4g128_gemv_noalloc",
    "w4g128_noalloc_status", "w4g128_selftest_wait", "w4g128_gemm_add_rmsnorm", "w4g128_decode_step_host",
    "w4g128_schedule", "DecodeStep",
    "MAX_M", "MAX_MATRICES", "SELFTEST_WS_BYTES", "SCHEDULE_FIELDS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_INCLUDE = os.path.join(os.path.dirname(_HERE), "include")
MAX_M = 16          # W4G128_MAX_M
MAX_MATRICES = 512  # W4G128_MAX_MATRICES
SELFTEST_WS_BYTES = 512  # W4G128_SELFTEST_WS_BYTES
SCHEDULE_FIELDS = 8  # W4G128_SCHEDULE_FIELDS

_lib = None


class W4G128Error(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({w4g128_status_string(status)})")


class _Matrix(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("K", ctypes.c_int), ("N", ctypes.c_int)]


def exported_symbols():
    """Names of every function the public headers (include/*.h) declare."""
    names = []
    for fn in sorted(os.listdir(_INCLUDE)):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(_INCLUDE, fn)) as f:
            for line in f:
                line = line.strip()
                if line.startswith("W4G128_API") and "(" in line:
                    names.append(line.split("(")[0].split()[-1].lstrip("*"))
    return names


_lib_debug = None


def lib():
    """Load libw4g128.so (building it in-tree if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    from . import build as _build
    path = _build.LIB
    if not os.path.exists(path):
        _build.build()
    _lib = _declare(ctypes.CDLL(path))
    return _lib


def lib_debug():
    """Load libw4g128_debug.so, the range-checked build of the same sources
    (W4G128_DEBUG: every global access derived from the schedule is checked,
    a failure recorded as W4G128_ERR_INTERNAL in the status word); for tests.
    Call its functions directly (the wrappers below use lib())."""
    global _lib_debug
    if _lib_debug is not None:
        return _lib_debug
    from . import build as _build
    path = _build.LIB_DEBUG
    if not os.path.exists(path):
        _build.build(debug=True)
    _lib_debug = _declare(ctypes.CDLL(path))
    return _lib_debug


def _declare(L):
    """Argument and result types of every entry point."""
    p, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.w4g128_status_string.restype = ctypes.c_char_p
    L.w4g128_status_string.argtypes = [i]
    L.w4g128_packed_bytes.restype = sz
    L.w4g128_packed_bytes.argtypes = [i, i]
    L.w4g128_pack.restype = i
    L.w4g128_pack.argtypes = [p, p, p, i, i, p, p]
    L.w4g128_unpack.restype = i
    L.w4g128_unpack.argtypes = [p, i, i, p, p, p, p]
    L.w4g128_quantize.restype = i
    L.w4g128_quantize.argtypes = [p, i, i, i, p, p, p, p]
    L.w4g128_workspace_bytes.restype = sz
    L.w4g128_workspace_bytes.argtypes = [i, i, i]
    L.w4g128_gemv.restype = i
    L.w4g128_gemv.argtypes = [p, p, p, i, i, p, sz, p]
    L.w4g128_gemm_verify.restype = i
    L.w4g128_gemm_verify.argtypes = [p, p, p, i, i, i, p, sz, p]
    L.w4g128_decode_step_workspace_bytes.restype = sz
    L.w4g128_decode_step_workspace_bytes.argtypes = [ctypes.POINTER(_Matrix), i, i]
    L.w4g128_decode_step.restype = i
    L.w4g128_decode_step.argtypes = [ctypes.POINTER(_Matrix), i, i, p, sz, p]
    L.w4g128_workspace_status.restype = i
    L.w4g128_workspace_status.argtypes = [p, ctypes.POINTER(ctypes.c_int), p]
    L.w4g128_probe_read.restype = i
    L.w4g128_probe_read.argtypes = [p, sz, p, p]
    L.w4g128_probe_copy.restype = i
    L.w4g128_probe_copy.argtypes = [p, p, sz, p]
    L.w4g128_probe_sink_bytes.restype = sz
    L.w4g128_probe_sink_bytes.argtypes = []
    L.w4g128_decode_step_host.restype = i
    L.w4g128_decode_step_host.argtypes = [ctypes.POINTER(_Matrix), i, i, p, p, sz, p, p, sz, p, sz, p]
    L.w4g128_verify_step.restype = i
    L.w4g128_verify_step.argtypes = [ctypes.POINTER(_Matrix), i, i, p, sz, p]
    L.w4g128_gemv_noalloc.restype = i
    L.w4g128_gemv_noalloc.argtypes = [p, p, p, i, i, p]
    L.w4g128_noalloc_status.restype = i
    L.w4g128_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int), p]
    L.w4g128_selftest_wait.restype = i
    L.w4g128_selftest_wait.argtypes = [p, sz, ctypes.c_ulonglong, i, p]
    L.w4g128_gemm_add_rmsnorm.restype = i
    L.w4g128_gemm_add_rmsnorm.argtypes = [p, p, p, p, ctypes.c_float, p, p, i, i, i, i, p, sz, p]
    L.w4g128_schedule.restype = i
    L.w4g128_schedule.argtypes = [ctypes.POINTER(_Matrix), i, i, ctypes.POINTER(ctypes.c_longlong), i]
    return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    return t.numel() * t.element_size()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, rc):
    if rc != 0:
        raise W4G128Error(fn, rc)


def w4g128_status_string(status):
    return lib().w4g128_status_string(int(status)).decode()


def w4g128_packed_bytes(K, N):
    return int(lib().w4g128_packed_bytes(K, N))


def w4g128_pack(codes, scales, mins, K, N, packed, stream=None):
    _check("w4g128_pack", lib().w4g128_pack(_ptr(codes), _ptr(scales), _ptr(mins), K, N, _ptr(packed),
                                            _stream(stream)))


def w4g128_unpack(packed, K, N, codes, scales, mins, stream=None):
    _check("w4g128_unpack", lib().w4g128_unpack(_ptr(packed), K, N, _ptr(codes), _ptr(scales), _ptr(mins),
                                                _stream(stream)))


def w4g128_quantize(w, K, N, search, codes, scales, mins, stream=None):
    """bf16 weights [K][N] -> canonical codes, scales, mins (search: 0 RTN, 1 range search)."""
    _check("w4g128_quantize", lib().w4g128_quantize(_ptr(w), K, N, int(search), _ptr(codes), _ptr(scales),
                                                    _ptr(mins), _stream(stream)))


def w4g128_workspace_bytes(M, K, N):
    return int(lib().w4g128_workspace_bytes(M, K, N))


def w4g128_gemv(packed, x, y, K, N, ws, ws_bytes=None, stream=None):
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("w4g128_gemv", lib().w4g128_gemv(_ptr(packed), _ptr(x), _ptr(y), K, N, _ptr(ws), wb, _stream(stream)))


def w4g128_gemm_verify(packed, x, y, M, K, N, ws, ws_bytes=None, stream=None):
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("w4g128_gemm_verify", lib().w4g128_gemm_verify(_ptr(packed), _ptr(x), _ptr(y), M, K, N, _ptr(ws), wb,
                                                          _stream(stream)))


def _matrices(mats):
    arr = (_Matrix * len(mats))()
    for i, (packed, x, y, K, N) in enumerate(mats):
        arr[i] = _Matrix(_ptr(packed), _ptr(x), _ptr(y), K, N)
    return arr


def w4g128_decode_step_workspace_bytes(mats, M):
    """mats: sequence of (packed, x, y, K, N)."""
    arr = _matrices(mats)
    return int(lib().w4g128_decode_step_workspace_bytes(arr, len(mats), M))


def w4g128_decode_step(mats, M, ws, ws_bytes=None, stream=None):
    """mats: sequence of (packed, x, y, K, N); one persistent launch for all."""
    arr = _matrices(mats)
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("w4g128_decode_step", lib().w4g128_decode_step(arr, len(mats), M, _ptr(ws), wb, _stream(stream)))


def w4g128_verify_step(mats, M, ws, ws_bytes=None, stream=None):
    """decode_step with the verify (warp-MMA) arithmetic at every M, M = 1 included."""
    arr = _matrices(mats)
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("w4g128_verify_step", lib().w4g128_verify_step(arr, len(mats), M, _ptr(ws), wb, _stream(stream)))


def w4g128_schedule(mats, M):
    """The schedule a decode_step of mats (sequence of (packed, x, y, K, N);
    only K, N and x are read, pointers may be None) takes at M rows: a dict
    of the W4G128_SCHEDULE_FIELDS values."""
    arr = _matrices(mats)
    out = (ctypes.c_longlong * SCHEDULE_FIELDS)()
    _check("w4g128_schedule", lib().w4g128_schedule(arr, len(mats), M, out, SCHEDULE_FIELDS))
    keys = ("local", "ctas", "cta_warps", "second_pass", "pair_quads", "ring_depth", "workspace_bytes", "items")
    return dict(zip(keys, (int(v) for v in out)))


def w4g128_gemm_add_rmsnorm(packed, x, residual, gamma, eps, h, out, M, K, N, verify, ws, ws_bytes=None,
                            stream=None):
    """h = residual + x W (bf16, one rounding), out = gamma h / rms(h) per row."""
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("w4g128_gemm_add_rmsnorm",
           lib().w4g128_gemm_add_rmsnorm(_ptr(packed), _ptr(x), _ptr(residual), _ptr(gamma), float(eps), _ptr(h),
                                         _ptr(out), M, K, N, int(verify), _ptr(ws), wb, _stream(stream)))


def w4g128_workspace_status(ws, stream=None):
    out = ctypes.c_int(0)
    _check("w4g128_workspace_status", lib().w4g128_workspace_status(_ptr(ws), ctypes.byref(out), _stream(stream)))
    return out.value


def w4g128_probe_sink_bytes():
    return int(lib().w4g128_probe_sink_bytes())


def w4g128_probe_read(buf, nbytes, sink, stream=None):
    _check("w4g128_probe_read", lib().w4g128_probe_read(_ptr(buf), nbytes, _ptr(sink), _stream(stream)))


def w4g128_probe_copy(src, dst, nbytes, stream=None):
    _check("w4g128_probe_copy", lib().w4g128_probe_copy(_ptr(src), _ptr(dst), nbytes, _stream(stream)))


def w4g128_gemv_noalloc(packed, x, y, K, N, stream=None):
    """w4g128_gemv without a workspace argument: for callers that must not
    allocate device memory (see include/w4g128.h)."""
    _check("w4g128_gemv_noalloc", lib().w4g128_gemv_noalloc(_ptr(packed), _ptr(x), _ptr(y), K, N,
                                                            _stream(stream)))


def w4g128_noalloc_status(stream=None):
    """Status word the last w4g128_gemv_noalloc call on this device left."""
    out = ctypes.c_int(0)
    _check("w4g128_noalloc_status", lib().w4g128_noalloc_status(ctypes.byref(out), _stream(stream)))
    return out.value


def w4g128_selftest_wait(ws, limit_ns, set_flag, ws_bytes=None, stream=None):
    """Diagnostic: a bounded device wait on a flag of `ws` (see include/w4g128.h)."""
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("w4g128_selftest_wait", lib().w4g128_selftest_wait(_ptr(ws), wb, int(limit_ns), int(set_flag),
                                                              _stream(stream)))


def w4g128_decode_step_host(mats, M, x_host, x_dev, x_bytes, y_host, y_dev, y_bytes, ws, ws_bytes=None,
                            stream=None):
    """decode_step with the activations copied from / to host buffers in the same call."""
    arr = _matrices(mats)
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("w4g128_decode_step_host",
           lib().w4g128_decode_step_host(arr, len(mats), M, _ptr(x_host), _ptr(x_dev), x_bytes, _ptr(y_host),
                                         _ptr(y_dev), y_bytes, _ptr(ws), wb, _stream(stream)))


class DecodeStep:
    """A decode step whose arguments are marshalled once: the descriptor
    array and the pointers are fixed, so each call is one C call.

    mats: sequence of (packed, x, y, K, N); ws: the workspace.  ``run`` calls
    w4g128_decode_step, ``run_host`` w4g128_decode_step_host with the host
    and device buffers given here."""

    def __init__(self, mats, M, ws, stream=None, x_host=None, x_dev=None, y_host=None, y_dev=None):
        self._keep = (mats, ws, x_host, x_dev, y_host, y_dev)  # the buffers outlive the step
        self._arr = _matrices(mats)
        self._n = len(mats)
        self._M = M
        self._ws = _ptr(ws)
        self._wb = _nbytes(ws)
        self._stream = _stream(stream)
        self._xh, self._xd = _ptr(x_host), _ptr(x_dev)
        self._xb = 0 if x_host is None else _nbytes(x_host)
        self._yh, self._yd = _ptr(y_host), _ptr(y_dev)
        self._yb = 0 if y_host is None else _nbytes(y_host)
        self._fn = lib().w4g128_decode_step
        self._fn_host = lib().w4g128_decode_step_host

    def run(self):
        rc = self._fn(self._arr, self._n, self._M, self._ws, self._wb, self._stream)
        if rc != 0:
            raise W4G128Error("w4g128_decode_step", rc)

    def run_host(self):
        rc = self._fn_host(self._arr, self._n, self._M, self._xh, self._xd, self._xb, self._yh, self._yd, self._yb,
                           self._ws, self._wb, self._stream)
        if rc != 0:
            raise W4G128Error("w4g128_decode_step_host", rc)
