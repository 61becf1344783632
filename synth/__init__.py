"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This package holds no arithmetic of the int4-g128 method: it draws the
canonical inputs (codes, scales, mins, x) from counter-based SplitMix64
streams.  ``synth.c`` is the host generator; ``synth_dev.cu`` fills the large
weight arrays straight into device memory with bit-identical values.

Workload recipe (one matrix of shape K x N, M activation rows):
  codes  uint32 [K/8][N]    uniform 4-bit codes, 8 per word, code k = 8j+i in
                            bits 4i..4i+3 of word j
  scales bf16   [K/128][N]  U(0.002, 0.02) rounded to bf16
  mins   bf16   [K/128][N]  -8 * scale * (1 + U(-0.1, 0.1)) rounded to bf16
  x      bf16   [M][K]      N(0, 1) rounded to bf16
Each (seed, matrix_id) pair names independent streams for the four arrays.

For the residual add + RMS norm call: the residual [M][N] is drawn like x
(N(0, 1), its own stream id) and the norm weight gamma [N] is
1 + 0.25 N(0, 1), cut to bf16 (norm_weight).
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_HOST_SO = os.path.join(_BUILD, "libsynth.so")
_DEV_SO = os.path.join(_BUILD, "libsynth_dev.so")

_host = None
_dev = None


def build_host():
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "synth.c")
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                           "-std=c11", "-o", _HOST_SO, src, "-lm"])


def build_dev():
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "synth_dev.cu")
    subprocess.check_call(["nvcc", "-O2", "-shared", "-Xcompiler", "-fPIC", "-fmad=false",
                           "-gencode", "arch=compute_103a,code=sm_103a", "-o", _DEV_SO, src])


def _needs(so, src):
    return (not os.path.exists(so)) or os.path.getmtime(so) < os.path.getmtime(src)


def host():
    global _host
    if _host is None:
        if _needs(_HOST_SO, os.path.join(_HERE, "synth.c")):
            build_host()
        lib = ctypes.CDLL(_HOST_SO)
        u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_key.restype = u64
        lib.synth_key.argtypes = [u64, u64, ctypes.c_uint32]
        lib.synth_draw.restype = u64
        lib.synth_draw.argtypes = [u64, u64]
        lib.synth_bf16_rn.restype = ctypes.c_uint16
        lib.synth_bf16_rn.argtypes = [ctypes.c_double]
        lib.synth_codes.argtypes = [u64, u64, i64, p]
        lib.synth_meta.argtypes = [u64, u64, i64, p, p]
        lib.synth_x.argtypes = [u64, u64, i64, p]
        lib.synth_columns.argtypes = [u64, u64, ctypes.c_int, ctypes.c_int, p, ctypes.c_int, p, p, p]
        _host = lib
    return _host


def dev():
    global _dev
    if _dev is None:
        if _needs(_DEV_SO, os.path.join(_HERE, "synth_dev.cu")):
            build_dev()
        lib = ctypes.CDLL(_DEV_SO)
        u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_dev_codes.restype = ctypes.c_int
        lib.synth_dev_codes.argtypes = [u64, u64, i64, p, p]
        lib.synth_dev_meta.restype = ctypes.c_int
        lib.synth_dev_meta.argtypes = [u64, u64, i64, p, p, p]
        _dev = lib
    return _dev


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def codes(seed, matrix_id, K, N):
    """Canonical codes uint32 [K/8][N]."""
    out = np.empty((K // 8, N), dtype=np.uint32)
    host().synth_codes(seed, matrix_id, out.size, _ptr(out))
    return out


def meta(seed, matrix_id, K, N):
    """(scales, mins) as uint16 bf16 bit patterns, each [K/128][N]."""
    s = np.empty((K // 128, N), dtype=np.uint16)
    m = np.empty((K // 128, N), dtype=np.uint16)
    host().synth_meta(seed, matrix_id, s.size, _ptr(s), _ptr(m))
    return s, m


def x(seed, matrix_id, M, K):
    """Activations as uint16 bf16 bit patterns [M][K]."""
    out = np.empty((M, K), dtype=np.uint16)
    host().synth_x(seed, matrix_id, out.size, _ptr(out))
    return out


def matrix(seed, matrix_id, K, N):
    """(codes, scales, mins) of one K x N matrix."""
    c = codes(seed, matrix_id, K, N)
    s, m = meta(seed, matrix_id, K, N)
    return c, s, m


def columns(seed, matrix_id, K, N, cols):
    """The canonical inputs restricted to the listed columns of a K x N matrix."""
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int32))
    nc = cols.size
    c = np.empty((K // 8, nc), dtype=np.uint32)
    s = np.empty((K // 128, nc), dtype=np.uint16)
    m = np.empty((K // 128, nc), dtype=np.uint16)
    host().synth_columns(seed, matrix_id, K, N, _ptr(cols), nc, _ptr(c), _ptr(s), _ptr(m))
    return c, s, m


def bf16_rn(value):
    """Round a double to bf16 bits (round to nearest, ties to even)."""
    return int(host().synth_bf16_rn(float(value)))


def fill_device(seed, matrix_id, K, N, codes_ptr, scales_ptr, mins_ptr, stream=0):
    """Fill device buffers with the same values codes()/meta() return."""
    lib = dev()
    rc = lib.synth_dev_codes(seed, matrix_id, (K // 8) * N, codes_ptr, stream)
    if rc != 0:
        raise RuntimeError(f"synth_dev_codes failed with CUDA error {rc}")
    rc = lib.synth_dev_meta(seed, matrix_id, (K // 128) * N, scales_ptr, mins_ptr, stream)
    if rc != 0:
        raise RuntimeError(f"synth_dev_meta failed with CUDA error {rc}")


def norm_weight(seed, stream_id, N):
    """RMS-norm weight gamma [N] as bf16 bits: 1 + 0.25 N(0, 1), truncated to bf16."""
    z = x(seed, stream_id, 1, N)[0].astype(np.uint32) << 16
    g = (1.0 + 0.25 * z.view(np.float32).astype(np.float64)).astype(np.float32)
    return (g.view(np.uint32) >> 16).astype(np.uint16)
