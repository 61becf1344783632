"""The shared seeded input generator (CPU side): determinism, distributions,
column sampling and its double -> bf16 rounding."""
import numpy as np
import pytest

import synth

SEED = 20260001


def test_deterministic_and_seed_sensitive():
    a = synth.matrix(SEED, 3, 256, 64)
    b = synth.matrix(SEED, 3, 256, 64)
    c = synth.matrix(SEED, 4, 256, 64)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    assert not np.array_equal(a[0], c[0])
    assert np.array_equal(synth.x(SEED, 1, 2, 512), synth.x(SEED, 1, 2, 512))


def test_code_distribution_uniform():
    c = synth.codes(SEED, 0, 4096, 256)
    nib = np.stack([(c >> np.uint32(4 * i)) & 0xF for i in range(8)]).ravel()
    counts = np.bincount(nib, minlength=16)
    expected = nib.size / 16
    assert np.all(np.abs(counts - expected) < 6 * np.sqrt(expected))


def test_scale_min_ranges():
    s, m = synth.meta(SEED, 0, 128 * 64, 512)
    sv = (s.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    mv = (m.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert sv.min() >= 0.002 - 1e-4 and sv.max() <= 0.02 + 1e-4
    ratio = mv / (-8.0 * sv)
    assert ratio.min() >= 0.9 - 0.01 and ratio.max() <= 1.1 + 0.01
    assert abs(sv.mean() - 0.011) < 5e-4


def test_x_standard_normal():
    x = synth.x(SEED, 0, 4, 8192)
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(xv.mean()) < 0.03 and abs(xv.std() - 1.0) < 0.03


def test_columns_match_full_matrix():
    K, N = 512, 96
    c, s, m = synth.matrix(SEED, 7, K, N)
    cols = [0, 5, 17, 95, 64]
    cc, ss, mm = synth.columns(SEED, 7, K, N, cols)
    assert np.array_equal(cc, c[:, cols]) and np.array_equal(ss, s[:, cols]) and np.array_equal(mm, m[:, cols])


def test_bf16_rn_against_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(3000), rng.standard_normal(300) * 1e-39,
                           rng.standard_normal(300) * 1e37, [0.0, 1.0, -2.5, 1.00390625, 1.01171875]])
    vals = vals.astype(np.float32)                    # float32-representable doubles
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([synth.bf16_rn(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rn_ties_and_overflow():
    assert synth.bf16_rn(1.0 + 2.0**-8) == 0x3F80          # tie -> even (down)
    assert synth.bf16_rn(1.0 + 3 * 2.0**-8) == 0x3F82      # tie -> even (up)
    assert synth.bf16_rn(1.0 + 2.0**-8 + 2.0**-40) == 0x3F81
    assert synth.bf16_rn(3.5e38) == 0x7F80
    assert synth.bf16_rn(-0.0) == 0x8000
    assert synth.bf16_rn(2.0**-133) == 0x0001
    assert synth.bf16_rn(2.0**-134) == 0x0000               # tie at half the smallest subnormal -> even
