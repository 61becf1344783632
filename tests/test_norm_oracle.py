"""Pins of the residual-add + RMS-norm oracle (oracle_add_rmsnorm), CPU only.

The pages name the step ("partials summed in the norm") without a formula, so
the oracle follows the textbook RMS normalisation after the residual update.
It is pinned by hand-worked rows (tests/golden/rmsnorm_rows.txt), closed
forms (unit mean square with gamma = 1 and eps = 0; a constant row), exact
invariants (power-of-two scaling, sign symmetry), its composition with the
GEMM oracle (x = 0 gives h = residual, residual = 0 gives h = y) and planted
mistakes that must fail.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "rmsnorm_rows.txt")


def bits(a):
    """float -> bf16 bits, for values that are bf16 already."""
    a = np.asarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all(u & 0xFFFF == 0), "not a bf16 value"
    return (u >> 16).astype(np.uint16)


def golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, eps, y, res, gam, h, out = [f.strip() for f in line.split(";")]
        fl = lambda s: np.array([float(v) for v in s.split(",")])
        hx = lambda s: np.array([int(v, 16) for v in s.split(",")], dtype=np.uint16)
        rows.append((name, float(eps), fl(y), hx(res), hx(gam), fl(h), fl(out)))
    return rows


def check_golden(O):
    bad = 0
    for name, eps, y, res, gam, h_exp, out_exp in golden_rows():
        h, out = O.add_rmsnorm(y[None, :], res[None, :], gam, eps)
        bad += not np.allclose(h[0], h_exp, rtol=0, atol=1e-15)
        bad += not np.allclose(out[0], out_exp, rtol=1e-15, atol=1e-15)
    return bad


def test_golden_rows():
    assert len(golden_rows()) == 3
    assert check_golden(oracle.Oracle()) == 0


def random_case(rng, M, N, scale=1.0):
    y = rng.standard_normal((M, N)) * scale
    res = bits(np.round(rng.standard_normal((M, N)) * 64) / 64)
    gam = bits(np.round((1 + 0.25 * rng.standard_normal(N)) * 128) / 128)
    return y, res, gam


def test_unit_mean_square():
    """gamma = 1, eps = 0: every output row has mean square exactly 1 (up to
    fp64 rounding)."""
    O = oracle.Oracle()
    rng = np.random.default_rng(1)
    y, res, _ = random_case(rng, 4, 300)
    _, out = O.add_rmsnorm(y, res, bits(np.ones(300)), 0.0)
    assert np.allclose(np.mean(out * out, axis=1), 1.0, rtol=0, atol=1e-13)


def test_constant_row():
    O = oracle.Oracle()
    c, eps = -2.5, 0.75
    N = 64
    gam = bits(np.full(N, 1.5))
    _, out = O.add_rmsnorm(np.full((1, N), c), bits(np.zeros((1, N))), gam, eps)
    assert np.allclose(out[0], 1.5 * c / np.sqrt(c * c + eps), rtol=1e-15, atol=0)


def test_power_of_two_scaling_and_sign():
    """eps = 0: scaling y and the residual by 2^k leaves out unchanged bit for
    bit; negating both negates out exactly."""
    O = oracle.Oracle()
    rng = np.random.default_rng(2)
    y, res, gam = random_case(rng, 3, 200)
    resf = oracle.bf16_bits_to_f64(res)
    _, out = O.add_rmsnorm(y, res, gam, 0.0)
    for k in (-3, 5):
        _, o2 = O.add_rmsnorm(y * 2.0 ** k, bits(resf * 2.0 ** k), gam, 0.0)
        assert np.array_equal(out, o2)
    _, on = O.add_rmsnorm(-y, bits(-resf), gam, 0.0)
    assert np.array_equal(on, -out)


def test_eps_weight():
    """A large eps dominates: out -> gamma h / sqrt(eps)."""
    O = oracle.Oracle()
    rng = np.random.default_rng(3)
    y, res, gam = random_case(rng, 2, 100, scale=1e-3)
    res = bits(np.zeros((2, 100)))
    h, out = O.add_rmsnorm(y, res, gam, 1e6)
    g = oracle.bf16_bits_to_f64(gam)
    assert np.allclose(out, g * h / 1e3, rtol=1e-9, atol=0)


def test_composition_with_gemm():
    """x = 0: h is the residual itself; residual = 0: h is the GEMM output."""
    O = oracle.Oracle()
    rng = np.random.default_rng(4)
    K, N, M = 256, 48, 2
    codes = O.pack_canonical(rng.integers(0, 16, size=(K, N)).astype(np.uint8))
    scales = bits(np.full((K // 128, N), 2.0 ** -5))
    mins = bits(np.full((K // 128, N), -0.25))
    _, res, gam = random_case(rng, M, N)
    y0, _ = O.gemm(np.zeros((M, K), dtype=np.uint16), codes, scales, mins)
    h, _ = O.add_rmsnorm(y0, res, gam, 1e-6)
    assert np.array_equal(h, oracle.bf16_bits_to_f64(res))
    x = bits(np.round(rng.standard_normal((M, K)) * 8) / 8)
    y, _ = O.gemm(x, codes, scales, mins)
    h, _ = O.add_rmsnorm(y, bits(np.zeros((M, N))), gam, 1e-6)
    assert np.array_equal(h, y)


BOUNDS_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "norm_bounds_rows.txt")


def bounds_rows():
    rows = []
    for line in open(BOUNDS_GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, eps, h, out, gam, a, dh, dout = [f.strip() for f in line.split(";")]
        fl = lambda s: np.array([float(v) for v in s.split(",")])
        hx = lambda s: np.array([int(v, 16) for v in s.split(",")], dtype=np.uint16)
        rows.append((name, float(eps), fl(h), fl(out), hx(gam), fl(a), fl(dh), fl(dout)))
    return rows


def bounds_golden_mismatches(mutant=0):
    O = oracle.Oracle()
    bad = 0
    for name, eps, h, out, gam, a, dh_exp, dout_exp in bounds_rows():
        dh, dout = oracle.norm_bounds(h[None, :], out[None, :], a[None, :], gam, eps, O, mutant=mutant)
        bad += not np.allclose(dh[0], dh_exp, rtol=1e-12, atol=0)
        fin = np.isfinite(dout_exp)
        bad += not np.array_equal(np.isfinite(dout[0]), fin)
        bad += not np.allclose(dout[0][fin], dout_exp[fin], rtol=1e-12, atol=0)
    return bad


def test_bounds_golden_rows():
    """The bound's value on hand-worked rows (tests/golden/norm_bounds_rows.txt)."""
    assert len(bounds_rows()) == 2
    assert bounds_golden_mismatches() == 0


def worst_corner_deviation(h, gam, eps, dh):
    """Largest |out'_n - out_n| over h' in the box |h'_j - h_j| <= dh_j, exact
    in fp64 for each n: out'_n = gamma_n h'_n / sqrt(mean h'^2 + eps) is
    monotone in h'_n's own offset and in the mean square, so the extremes sit
    at h'_n = h_n +- dh_n with every other |h'_j| at its smallest or largest."""
    N = h.size
    g = oracle.bf16_bits_to_f64(gam)
    out = g * h / np.sqrt(np.mean(h * h) + eps)
    lo = np.maximum(np.abs(h) - dh, 0.0) ** 2
    hi = (np.abs(h) + dh) ** 2
    best = np.zeros(N)
    for sign in (1.0, -1.0):
        hn = h + sign * dh
        for total, own in ((lo.sum(), lo), (hi.sum(), hi)):
            o = g * hn / np.sqrt((total - own + hn * hn) / N + eps)
            best = np.maximum(best, np.abs(o - out))
    return best, out


def random_bound_rows(seed, count=150):
    rng = np.random.default_rng(seed)
    for _ in range(count):
        N = int(rng.integers(2, 300))
        eps = float(rng.choice([0.0, 1e-6, 0.5]))
        h = np.round(rng.standard_normal(N) * 64) / 64 * float(rng.choice([1.0, 0.01, 100.0]))
        gam = bits(np.round((1 + 0.25 * rng.standard_normal(N)) * 128) / 128)
        a = np.abs(h) * rng.uniform(1, 40, N) * float(rng.choice([0.1, 1.0, 5.0]))
        yield h, gam, eps, a


def bound_violations(mutant):
    """Over random rows: (elements whose worst-case deviation exceeds the
    bound, largest deviation / (bound - ulp(out)))."""
    O = oracle.Oracle()
    viol, tight = 0, 0.0
    for h, gam, eps, a in random_bound_rows(11):
        g = oracle.bf16_bits_to_f64(gam)
        out = g * h / np.sqrt(np.mean(h * h) + eps)
        dh, dout = oracle.norm_bounds(h[None, :], out[None, :], a[None, :], gam, eps, O, mutant=mutant)
        if not np.all(np.isfinite(dout)):
            continue
        dev, _ = worst_corner_deviation(h, gam, eps, dh[0])
        viol += int(np.sum(dev > dout[0]))
        tight = max(tight, float(np.max(dev / (dout[0] - O.bf16_ulp_array(out)))))
    return viol, tight


def test_bound_is_sound_and_tight():
    """Every h within dh of h_ref moves out by no more than dout (sound), and
    the worst such h comes within 10% of the bound's arithmetic part (tight,
    so a loose bound cannot pass every GPU test unnoticed)."""
    viol, tight = bound_violations(0)
    assert viol == 0
    assert tight > 0.9


@pytest.mark.parametrize("mutant", [1, 2, 3])
def test_planted_bound_mistakes_are_caught(mutant):
    """Dropping the |out| rho term (1), the (1 + rho) factor (2) or the factor
    2 in the mean-square shift (3) fails the hand-worked rows and lets some
    admissible h move out past the bound."""
    assert bounds_golden_mismatches(mutant) >= 1
    viol, _ = bound_violations(mutant)
    assert viol > 0


def test_bound_infinite_where_no_information_is_left():
    """D >= ms: dout is +inf for every element of the row, zero outputs included."""
    O = oracle.Oracle()
    h = np.array([[0.5, 0.0, -0.5]])
    gam = bits(np.ones(3))
    out = oracle.bf16_bits_to_f64(gam)[None, :] * h / np.sqrt(np.mean(h * h))
    _, dout = oracle.norm_bounds(h, out, np.full((1, 3), 1000.0), gam, 0.0, O)
    assert np.all(np.isposinf(dout))


def test_accept_norm_at_the_bound():
    """An output moved to 0.99 of the bound passes, to 1.01 of it fails; the
    same for h."""
    O = oracle.Oracle()
    rng = np.random.default_rng(5)
    y, res, gam = random_case(rng, 2, 64)
    h, out = O.add_rmsnorm(y, res, gam, 1e-6)
    a = np.abs(y) * 10 + 1.0
    dh, dout = oracle.norm_bounds(h, out, a, gam, 1e-6, O)
    assert dh.shape == dout.shape == (2, 64)
    assert np.all(np.isfinite(dout)) and np.all(dout > 0) and np.all(dh > 0)
    sign = np.where(rng.random((2, 64)) < 0.5, -1.0, 1.0)
    ok_h, ok_o = oracle.accept_norm(h + 0.99 * sign * dh, out + 0.99 * sign * dout, h, out, a, gam, 1e-6, O)
    assert ok_h.all() and ok_o.all()
    ok_h, ok_o = oracle.accept_norm(h + 1.01 * sign * dh, out + 1.01 * sign * dout, h, out, a, gam, 1e-6, O)
    assert not ok_h.any() and not ok_o.any()


@pytest.mark.parametrize("mutant", [7, 8, 9])
def test_planted_norm_mistakes_are_caught(mutant):
    """Mean over N - 1 (7), eps dropped (8) and residual not added (9) must
    each fail the hand-worked rows."""
    assert check_golden(oracle.Oracle(mutant)) >= 1
