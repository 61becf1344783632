"""fp64 CPU oracle for the int4-g128 weight-streaming GEMV.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product package
(``int4_weight_only_g128_gb300``) never imports it, and the two share no code.

The oracle is plain C (``oracle.c``) computing the definition of the method in
fp64: dequantise w = min + q*scale per 128-row group (Token Rush README,
"Quantization" section), then y = x . w summed in ascending k.  See the header
comment of ``oracle.c`` for the passages it follows and the readings it takes.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SRC = os.path.join(_HERE, "oracle.c")

_libs = {}


def so_path(mutant=0):
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant=0):
    """Compile the oracle (or one of its planted-mistake mutants) with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    out = so_path(mutant)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", f"-DORACLE_MUTANT={mutant}", "-o", out, _SRC, "-lm"]
    subprocess.check_call(cmd)
    return out


def _load(mutant=0):
    if mutant in _libs:
        return _libs[mutant]
    path = so_path(mutant)
    if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        build(mutant)
    lib = ctypes.CDLL(path)
    p, i = ctypes.c_void_p, ctypes.c_int
    lib.oracle_bf16_value.restype = ctypes.c_double
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_rn.restype = ctypes.c_uint16
    lib.oracle_bf16_rn.argtypes = [ctypes.c_double]
    lib.oracle_bf16_rn_array.argtypes = [p, ctypes.c_size_t, p]
    lib.oracle_bf16_ulp.restype = ctypes.c_double
    lib.oracle_bf16_ulp.argtypes = [ctypes.c_double]
    lib.oracle_pack_canonical.argtypes = [p, i, i, p]
    lib.oracle_unpack_canonical.argtypes = [p, i, i, p]
    lib.oracle_gemm.argtypes = [i, i, i, p, p, p, p, p, p, i]
    lib.oracle_max_threads.restype = i
    lib.oracle_packed_bytes.restype = ctypes.c_size_t
    lib.oracle_packed_bytes.argtypes = [i, i]
    lib.oracle_pack_tiled.argtypes = [p, p, p, i, i, p]
    lib.oracle_unpack_tiled.argtypes = [p, i, i, p, p, p]
    lib.oracle_quantize.argtypes = [p, i, i, i, p, p, p, p]
    lib.oracle_add_rmsnorm.argtypes = [i, i, p, p, p, ctypes.c_double, p, p]
    _libs[mutant] = lib
    return lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


QUANT_CANDIDATES = 21


class Oracle:
    """ctypes view of one build of the oracle (mutant 0 is the real one)."""

    def __init__(self, mutant=0):
        self.lib = _load(mutant)
        self.mutant = mutant

    # bf16
    def bf16_value(self, bits):
        return self.lib.oracle_bf16_value(int(bits))

    def bf16_rn(self, v):
        return int(self.lib.oracle_bf16_rn(float(v)))

    def bf16_rn_array(self, v):
        """bf16_rn of every element: uint16 bits, same shape."""
        v, vp = _c(v, np.float64)
        out = np.empty(v.shape, dtype=np.uint16)
        self.lib.oracle_bf16_rn_array(vp, v.size, out.ctypes.data_as(ctypes.c_void_p))
        return out

    def bf16_ulp(self, v):
        return self.lib.oracle_bf16_ulp(float(v))

    def bf16_ulp_array(self, v):
        """Vectorised bf16_ulp: 2^(max(floor(log2|v|), -126) - 7), 2^-133 at 0."""
        a = np.abs(np.asarray(v, dtype=np.float64))
        _, e = np.frexp(a)                    # a = f * 2^e, f in [0.5, 1): floor(log2 a) = e - 1
        ex = np.maximum(e.astype(np.int64) - 1, -126)
        return np.where(a > 0, np.ldexp(1.0, ex - 7), np.ldexp(1.0, -133))

    # canonical codes
    def pack_canonical(self, q):
        q, qp = _c(q, np.uint8)
        K, N = q.shape
        out = np.empty((K // 8, N), dtype=np.uint32)
        self.lib.oracle_pack_canonical(qp, K, N, out.ctypes.data_as(ctypes.c_void_p))
        return out

    def unpack_canonical(self, codes):
        codes, cp = _c(codes, np.uint32)
        K, N = codes.shape[0] * 8, codes.shape[1]
        out = np.empty((K, N), dtype=np.uint8)
        self.lib.oracle_unpack_canonical(cp, K, N, out.ctypes.data_as(ctypes.c_void_p))
        return out

    # dequantise-then-multiply
    def gemm(self, x, codes, scales, mins, nthreads=0):
        """Return (y, a): y[M][N] in fp64 and a[M][N] = sum_k |x w|."""
        x, xp = _c(x, np.uint16)
        codes, cp = _c(codes, np.uint32)
        scales, sp = _c(scales, np.uint16)
        mins, mp = _c(mins, np.uint16)
        M, K = x.shape
        N = codes.shape[1]
        assert codes.shape == (K // 8, N) and scales.shape == (K // 128, N) == mins.shape
        y = np.empty((M, N), dtype=np.float64)
        a = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_gemm(M, K, N, xp, cp, sp, mp, y.ctypes.data_as(ctypes.c_void_p),
                             a.ctypes.data_as(ctypes.c_void_p), int(nthreads))
        return y, a

    def max_threads(self):
        return int(self.lib.oracle_max_threads())

    # tiled device layout
    def packed_bytes(self, K, N):
        return int(self.lib.oracle_packed_bytes(K, N))

    def pack_tiled(self, codes, scales, mins):
        codes, cp = _c(codes, np.uint32)
        scales, sp = _c(scales, np.uint16)
        mins, mp = _c(mins, np.uint16)
        K, N = codes.shape[0] * 8, codes.shape[1]
        out = np.empty(self.packed_bytes(K, N), dtype=np.uint8)
        self.lib.oracle_pack_tiled(cp, sp, mp, K, N, out.ctypes.data_as(ctypes.c_void_p))
        return out

    def unpack_tiled(self, packed, K, N):
        packed, pp = _c(packed, np.uint8)
        codes = np.empty((K // 8, N), dtype=np.uint32)
        scales = np.empty((K // 128, N), dtype=np.uint16)
        mins = np.empty((K // 128, N), dtype=np.uint16)
        self.lib.oracle_unpack_tiled(pp, K, N, codes.ctypes.data_as(ctypes.c_void_p),
                                     scales.ctypes.data_as(ctypes.c_void_p),
                                     mins.ctypes.data_as(ctypes.c_void_p))
        return codes, scales, mins


def accept(y_gpu, y_ref, a, oracle=None):
    """Per-element acceptance |y_gpu - y_ref| <= 4e-3*a + ulp_bf16(y_ref).

    Returns (ok_mask, ratio) where ratio = |err| / bound (<= 1 passes)."""
    o = oracle or Oracle()
    bound = 4e-3 * np.asarray(a, dtype=np.float64) + o.bf16_ulp_array(y_ref)
    err = np.abs(np.asarray(y_gpu, dtype=np.float64) - np.asarray(y_ref, dtype=np.float64))
    return err <= bound, err / bound


def bf16_bits_to_f64(bits):
    """uint16 bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _quantize(self, w, search):
    """Quantise bf16 weights w[K][N] (bits) to the canonical format.

    Returns (codes [K/8][N] uint32, scales [K/128][N] bf16 bits,
    mins [K/128][N] bf16 bits, errs [K/128][N][21] float32), where errs holds
    every candidate's squared error (only the first is filled when search is
    False: round-to-nearest alone)."""
    w, wp = _c(w, np.uint16)
    K, N = w.shape
    assert K % 128 == 0
    codes = np.empty((K // 8, N), dtype=np.uint32)
    scales = np.empty((K // 128, N), dtype=np.uint16)
    mins = np.empty((K // 128, N), dtype=np.uint16)
    errs = np.zeros((K // 128, N, QUANT_CANDIDATES), dtype=np.float32)
    self.lib.oracle_quantize(wp, K, N, int(bool(search)), codes.ctypes.data_as(ctypes.c_void_p),
                             scales.ctypes.data_as(ctypes.c_void_p), mins.ctypes.data_as(ctypes.c_void_p),
                             errs.ctypes.data_as(ctypes.c_void_p))
    return codes, scales, mins, errs


Oracle.quantize = _quantize


def _add_rmsnorm(self, y, residual, gamma, eps):
    """Residual add and RMS norm of the product rows (oracle_add_rmsnorm).

    y: [M][N] fp64 product (from ``gemm``), residual: [M][N] bf16 bits,
    gamma: [N] bf16 bits.  Returns (h, out), both [M][N] fp64 and unrounded:
    h = residual + y, out = gamma * h / sqrt(mean_n(h^2) + eps)."""
    y, yp = _c(y, np.float64)
    residual, rp = _c(residual, np.uint16)
    gamma, gp = _c(gamma, np.uint16)
    M, N = y.shape
    assert residual.shape == (M, N) and gamma.shape == (N,)
    h = np.empty((M, N), dtype=np.float64)
    out = np.empty((M, N), dtype=np.float64)
    self.lib.oracle_add_rmsnorm(M, N, yp, rp, gp, float(eps), h.ctypes.data_as(ctypes.c_void_p),
                                out.ctypes.data_as(ctypes.c_void_p))
    return h, out


Oracle.add_rmsnorm = _add_rmsnorm


def norm_bounds(h_ref, out_ref, a, gamma, eps, oracle=None, mutant=0):
    """Acceptance bounds for the fused residual add + RMS norm.

    h: the product's bound carried over, |h_gpu - h_ref| <= dh = 4e-3*a +
    ulp_bf16(h_ref) (the GPU adds the residual to its fp32 product and rounds
    once to bf16).  out: the GPU normalises its own bf16 h, so each h_j may be
    off by dh_j; with ms = mean(h_ref^2) + eps the mean square moves by at
    most D = mean(2|h_ref| dh + dh^2), the reciprocal root by the relative
    rho = 1/sqrt(1 - D/ms) - 1 (plus 2^-20 for the fp32 sum, root and
    products), and
        |out_gpu - out_ref| <= |gamma| r (1 + rho) dh + |out_ref| rho + ulp_bf16(out_ref),
    r = 1/sqrt(ms).  Returns (dh, dout); rows whose D reaches ms get an
    infinite bound (no information left).

    mutant (negative controls for the pins only): 1 drops the |out_ref| rho
    term, 2 drops the (1 + rho) factor of the first term, 3 drops the factor 2
    in D."""
    o = oracle or Oracle()
    h_ref = np.asarray(h_ref, dtype=np.float64)
    out_ref = np.asarray(out_ref, dtype=np.float64)
    g = np.abs(bf16_bits_to_f64(gamma))[None, :]
    dh = 4e-3 * np.asarray(a, dtype=np.float64) + o.bf16_ulp_array(h_ref)
    ms = np.mean(h_ref * h_ref, axis=1, keepdims=True) + float(eps)
    two = 1.0 if mutant == 3 else 2.0
    D = np.mean(two * np.abs(h_ref) * dh + dh * dh, axis=1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        rho = np.where(D < ms, 1.0 / np.sqrt(np.maximum(1.0 - D / ms, 1e-300)) - 1.0, np.inf) + 2.0 ** -20
        r = 1.0 / np.sqrt(ms)
    first = g * r * dh if mutant == 2 else g * r * (1.0 + rho) * dh
    with np.errstate(invalid="ignore"):
        second = 0.0 if mutant == 1 else np.abs(out_ref) * rho
    dout = first + second + o.bf16_ulp_array(out_ref)
    # rows with no information left: infinite everywhere (0 * inf would be NaN)
    dout = np.where(np.isinf(rho), np.inf, dout)
    return dh, dout


def accept_norm(h_gpu, out_gpu, h_ref, out_ref, a, gamma, eps, oracle=None):
    """Per-element acceptance of the residual add + RMS norm call: h within
    dh and out within dout of norm_bounds.  Returns (ok_h, ok_out)."""
    dh, dout = norm_bounds(h_ref, out_ref, a, gamma, eps, oracle)
    ok_h = np.abs(np.asarray(h_gpu, dtype=np.float64) - h_ref) <= dh
    ok_out = np.abs(np.asarray(out_gpu, dtype=np.float64) - out_ref) <= dout
    return ok_h, ok_out
