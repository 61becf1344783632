"""Device packer: bit-exact against the oracle's independent restatement of the
packed layout, exact round trip, exact size, nothing written past the end."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, to_dev, to_host  # noqa: E402

SHAPES = [(128, 16), (256, 32), (384, 48), (640, 80), (1152, 208), (256, 96), (4096, 4096)]


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", SHAPES)
def test_pack_bit_exact_vs_oracle(K, N):
    mat = DevMatrix(K, N, matrix_id=K + N)
    ref = oracle.Oracle().pack_tiled(mat.codes, mat.scales, mat.mins)
    got = mat.packed.cpu().numpy()
    assert got.size == ref.size == K * N * 17 // 32
    assert np.array_equal(got, ref)


@pytest.mark.gpu
def test_pack_random_bits_and_extremes():
    rng = np.random.default_rng(3)
    K, N = 512, 80
    for codes in (rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint32),
                  np.zeros((K // 8, N), np.uint32), np.full((K // 8, N), 0xFFFFFFFF, np.uint32)):
        s = rng.integers(0, 2**16, size=(K // 128, N), dtype=np.uint16)
        m = rng.integers(0, 2**16, size=(K // 128, N), dtype=np.uint16)
        mat = DevMatrix(K, N, codes, s, m)
        assert np.array_equal(mat.packed.cpu().numpy(), oracle.Oracle().pack_tiled(codes, s, m))


@pytest.mark.gpu
def test_pack_writes_nothing_past_the_end():
    K, N = 384, 48
    codes, s, m = synth.matrix(SEED, 1, K, N)
    nb = w.w4g128_packed_bytes(K, N)
    buf = torch.full((nb + 4096,), 0xAB, dtype=torch.uint8, device="cuda")
    w.w4g128_pack(to_dev(codes), to_dev(s), to_dev(m), K, N, buf)
    torch.cuda.synchronize()
    tail = buf[nb:].cpu().numpy()
    assert np.all(tail == 0xAB)


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", [(128, 16), (640, 80), (4096, 4096)])
def test_unpack_round_trip(K, N):
    mat = DevMatrix(K, N, matrix_id=7)
    codes = torch.empty((K // 8) * N, dtype=torch.int32, device="cuda")
    s = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
    m = torch.empty_like(s)
    w.w4g128_unpack(mat.packed, K, N, codes, s, m)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(codes, np.uint32).reshape(K // 8, N), mat.codes)
    assert np.array_equal(to_host(s, np.uint16).reshape(K // 128, N), mat.scales)
    assert np.array_equal(to_host(m, np.uint16).reshape(K // 128, N), mat.mins)


@pytest.mark.gpu
def test_device_generator_matches_host_generator():
    K, N = 1024, 272
    dev = DevMatrix(K, N, matrix_id=11, device_fill=True)
    c, s, m = synth.matrix(SEED, 11, K, N)
    assert np.array_equal(to_host(dev.codes_d, np.uint32).reshape(K // 8, N), c)
    assert np.array_equal(to_host(dev.scales_d, np.uint16).reshape(K // 128, N), s)
    assert np.array_equal(to_host(dev.mins_d, np.uint16).reshape(K // 128, N), m)
