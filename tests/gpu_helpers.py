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
    """Canonical inputs on the device plus their packed form."""

    def __init__(self, K, N, codes=None, scales=None, mins=None, seed=SEED, matrix_id=0, device_fill=False):
        self.K, self.N = K, N
        if device_fill:
            self.codes_d = torch.empty((K // 8) * N, dtype=torch.int32, device="cuda")
            self.scales_d = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
            self.mins_d = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
            synth.fill_device(seed, matrix_id, K, N, self.codes_d.data_ptr(), self.scales_d.data_ptr(),
                              self.mins_d.data_ptr(), torch.cuda.current_stream().cuda_stream)
            self.codes = self.scales = self.mins = None
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


def check_against_oracle(y_bits, x_bits, codes, scales, mins, cols=None):
    """Element-wise acceptance against the fp64 oracle; returns the worst ratio."""
    O = oracle.Oracle()
    y_ref, a = O.gemm(x_bits, codes, scales, mins)
    y = bf16_to_f64(y_bits if cols is None else y_bits[:, cols])
    ok, ratio = oracle.accept(y, y_ref, a, O)
    bad = np.argwhere(~ok)
    assert ok.all(), f"{bad.shape[0]} elements outside the bound; first {bad[:5].tolist()}, worst ratio {ratio.max()}"
    return float(ratio.max())
