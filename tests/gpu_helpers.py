"""Helpers for the GPU parity tests: device buffers for one int4-g128 matrix,
built from the shared seeded generator, and calls through the C ABI."""
import numpy as np
import torch

import int4_weight_only_g128_gb300 as w
import oracle
import synth

SEED = 20260001


def to_dev(a):
    """numpy uint16/uint32/uint8 -> CUDA tensor of the same bits."""
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32, np.dtype(np.uint8): np.uint8}[a.dtype]
    return torch.from_numpy(a.view(view)).cuda()


def to_host(t, dtype):
    """CUDA tensor -> numpy array reinterpreted as `dtype`."""
    return t.cpu().numpy().view(dtype)


def bf16_to_f64(bits):
    return oracle.bf16_bits_to_f64(bits)


class DevMatrix:
    """Canonical inputs on the device plus their packed form.

    device_fill: the canonical arrays are generated on the device (same values
    as the host generator); const_meta = (scale bits, min bits) then replaces
    every scale and min by those constants; keep_host copies the canonical
    arrays back to the host for the oracle."""

    def __init__(self, K, N, codes=None, scales=None, mins=None, seed=SEED, matrix_id=0, device_fill=False,
                 const_meta=None, keep_host=False):
        self.K, self.N = K, N
        if device_fill:
            self.codes_d = torch.empty((K // 8) * N, dtype=torch.int32, device="cuda")
            self.scales_d = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
            self.mins_d = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
            synth.fill_device(seed, matrix_id, K, N, self.codes_d.data_ptr(), self.scales_d.data_ptr(),
                              self.mins_d.data_ptr(), torch.cuda.current_stream().cuda_stream)
            if const_meta is not None:
                self.scales_d.fill_(int(np.uint16(const_meta[0]).view(np.int16)))
                self.mins_d.fill_(int(np.uint16(const_meta[1]).view(np.int16)))
            self.codes = self.scales = self.mins = None
            if keep_host:
                self.codes = to_host(self.codes_d, np.uint32).reshape(K // 8, N)
                self.scales = to_host(self.scales_d, np.uint16).reshape(K // 128, N)
                self.mins = to_host(self.mins_d, np.uint16).reshape(K // 128, N)
        else:
            if codes is None:
                codes, scales, mins = synth.matrix(seed, matrix_id, K, N)
            self.codes, self.scales, self.mins = codes, scales, mins
            self.codes_d, self.scales_d, self.mins_d = to_dev(codes), to_dev(scales), to_dev(mins)
        self.nbytes = w.w4g128_packed_bytes(K, N)
        self.packed = torch.empty(self.nbytes, dtype=torch.uint8, device="cuda")
        w.w4g128_pack(self.codes_d, self.scales_d, self.mins_d, K, N, self.packed)

    def free_canonical(self):
        self.codes_d = self.scales_d = self.mins_d = None


def canonical_from_device(K, N, matrix_id, seed=SEED):
    """The canonical (codes, scales, mins) of one seeded matrix, generated on
    the device (bit-identical to the host generator) and copied back: the
    fast way to hand a multi-GB weight set to the oracle."""
    codes = torch.empty((K // 8) * N, dtype=torch.int32, device="cuda")
    scales = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
    mins = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
    synth.fill_device(seed, matrix_id, K, N, codes.data_ptr(), scales.data_ptr(), mins.data_ptr(),
                      torch.cuda.current_stream().cuda_stream)
    return (to_host(codes, np.uint32).reshape(K // 8, N), to_host(scales, np.uint16).reshape(K // 128, N),
            to_host(mins, np.uint16).reshape(K // 128, N))


def workspace(M, K, N):
    nb = w.w4g128_workspace_bytes(M, K, N)
    assert nb > 0
    return torch.empty(nb, dtype=torch.uint8, device="cuda")


def run(mat, x_bits, M=None, verify=None):
    """y bits [M][N] for x bits [M][K] (gemv when M == 1 unless verify=True)."""
    M = x_bits.shape[0] if M is None else M
    x = to_dev(x_bits)
    y = torch.empty(M * mat.N, dtype=torch.int16, device="cuda")
    ws = workspace(M, mat.K, mat.N)
    if M == 1 and not verify:
        w.w4g128_gemv(mat.packed, x, y, mat.K, mat.N, ws)
    else:
        w.w4g128_gemm_verify(mat.packed, x, y, M, mat.K, mat.N, ws)
    torch.cuda.synchronize()
    assert w.w4g128_workspace_status(ws) == 0
    return to_host(y, np.uint16).reshape(M, mat.N)


# "Passes but sloppy" ceiling.  Beyond the final rounding of the fp32 sum to
# bf16 (at most half a bf16 ulp), the error a correct kernel accumulates is
# a small fraction of the target's 4e-3 * sum|x w| allowance; a kernel that
# drops a split-K slot or misplaces a group at large K can still pass the
# allowance there, but not this.
SLOPPY_FRACTION = 0.1


def sloppiness(y, y_ref, a, O):
    """Per element: (|y - y_ref| - ulp(max(|y|, |y_ref|)) / 2)+ / (4e-3 a), the
    accumulated error beyond the output rounding as a fraction of the target's
    allowance (0 where a = 0 and the error is within the rounding)."""
    y = np.asarray(y, dtype=np.float64)
    half_ulp = 0.5 * O.bf16_ulp_array(np.maximum(np.abs(y), np.abs(y_ref)))
    excess = np.maximum(np.abs(y - y_ref) - half_ulp, 0.0)
    allow = 4e-3 * np.asarray(a, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(excess == 0.0, 0.0, excess / allow)


def check_against_oracle(y_bits, x_bits, codes, scales, mins, cols=None, y_ref=None, a=None):
    """Element-wise acceptance against the fp64 oracle (the target's bound and
    the sloppiness ceiling); returns the worst ratio to the bound.  y_ref, a:
    the oracle's result when the caller already has it."""
    O = oracle.Oracle()
    if y_ref is None:
        y_ref, a = O.gemm(x_bits, codes, scales, mins)
    y = bf16_to_f64(y_bits if cols is None else y_bits[:, cols])
    ok, ratio = oracle.accept(y, y_ref, a, O)
    bad = np.argwhere(~ok)
    assert ok.all(), f"{bad.shape[0]} elements outside the bound; first {bad[:5].tolist()}, worst ratio {ratio.max()}"
    sl = sloppiness(y, y_ref, a, O)
    assert sl.max() <= SLOPPY_FRACTION, f"accumulated error {sl.max():.3g} of the allowance at {np.argmax(sl)}"
    return float(ratio.max())


def int_x(rng, M, K, lo=-4, hi=4):
    """bf16 bits of integer activations drawn uniformly from lo..hi."""
    v = rng.integers(lo, hi + 1, size=(M, K)).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


ONE, MINUS_EIGHT = 0x3F80, 0xC100  # bf16 1.0 and -8.0


def exact_bits(y_ref, O=None):
    """bf16 bits the GPU must produce for an exact-integer case: y_ref must be
    integers small enough that every fp32 partial sum is exact."""
    O = O or oracle.Oracle()
    assert np.all(y_ref == np.round(y_ref)) and np.max(np.abs(y_ref)) < 2.0 ** 24
    return O.bf16_rn_array(y_ref)
