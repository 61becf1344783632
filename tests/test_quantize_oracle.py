"""Pins of the quantizer oracle (oracle_quantize), CPU only.

The quantizer has no printed worked example on the pages, so it is pinned by
hand-worked groups (tests/golden/quantize_groups.txt), exact closed forms
(weights already on a 16-level grid are recovered exactly; a constant group
has scale 0), invariants (power-of-two homogeneity, monotone codes, the
half-step rounding bound, the range search never worse than
round-to-nearest), the pages' stated purpose of the search (outliers are
clipped), agreement with the GEMM oracle's dequantisation, and planted
mistakes that must fail.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "quantize_groups.txt")


def f32_to_bf16_bits(a):
    """Exact only for values that are bf16 already (the tests build them so)."""
    a = np.asarray(a, dtype=np.float32)
    bits = a.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value is not a bf16"
    return (bits >> 16).astype(np.uint16)


def bf16_to_f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def group_values(name):
    k = np.arange(128)
    if name == "A":
        return -1.0 + (k % 16) / 8.0
    if name == "B":
        return np.full(128, 0.75)
    if name == "C":
        return 6.0 * (k % 2) - 3.0
    raise KeyError(name)


def read_golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, search, words, sc, mn = [p.strip() for p in line.split(";")]
            rows.append((name, int(search), [int(v, 16) for v in words.split(",")], int(sc, 16), int(mn, 16)))
    return rows


def dequant(codes, scales, mins):
    """fp64 weights from the canonical format: w = min + q * scale."""
    O = oracle.Oracle()
    q = O.unpack_canonical(codes).astype(np.float64)
    G = scales.shape[0]
    s = np.repeat(bf16_to_f64(scales), 128, axis=0)
    m = np.repeat(bf16_to_f64(mins), 128, axis=0)
    assert s.shape[0] == 128 * G
    return m + q * s, q


def random_weights(rng, K, N, outliers=False):
    w = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    if outliers:
        idx = rng.integers(0, K, size=N)
        w[idx, np.arange(N)] = (rng.choice([-1.0, 1.0], size=N) * rng.uniform(0.2, 0.5, size=N)).astype(np.float32)
    return (w.view(np.uint32) >> 16).astype(np.uint16)  # truncation: any bf16 bits will do


@pytest.mark.parametrize("row", read_golden(), ids=lambda r: f"{r[0]}-search{r[1]}")
def test_hand_worked_groups(row):
    name, search, words, sc, mn = row
    w = f32_to_bf16_bits(group_values(name)).reshape(128, 1)
    codes, scales, mins, errs = oracle.Oracle().quantize(w, search)
    assert [int(v) for v in codes[:, 0]] == words
    assert int(scales[0, 0]) == sc and int(mins[0, 0]) == mn


@pytest.mark.parametrize("search", [0, 1])
def test_weights_on_a_grid_are_recovered_exactly(search):
    """w = (q - 8) * 2^e with both q = 0 and q = 15 present: the range is
    exactly 15 steps of 2^e, so scale, minimum and every code come back."""
    rng = np.random.default_rng(3)
    K, N = 512, 24
    q = rng.integers(0, 16, size=(K, N))
    q[::128][0] = 0
    q[1::128][0] = 15
    q[0::128, :] = 0
    q[1::128, :] = 15
    e = rng.integers(-20, 4, size=(1, N)).astype(np.float64)
    w = (q - 8.0) * np.exp2(e)
    codes, scales, mins, errs = oracle.Oracle().quantize(f32_to_bf16_bits(w), search)
    dq, qq = dequant(codes, scales, mins)
    assert np.array_equal(qq, q)
    assert np.array_equal(bf16_to_f64(scales), np.repeat(np.exp2(e), K // 128, axis=0))
    assert np.array_equal(bf16_to_f64(mins), np.repeat(-8.0 * np.exp2(e), K // 128, axis=0))
    assert np.all(errs[:, :, 0] == 0.0)


def test_constant_groups_have_zero_scale():
    w = np.zeros((256, 4), dtype=np.float32)
    w[:128] = np.array([0.5, -2.0, 0.0, 1e-3], dtype=np.float32)
    w[128:] = np.array([-0.25, 8.0, 3.0, -1e-3], dtype=np.float32)
    w = (w.view(np.uint32) >> 16).astype(np.uint16)  # bf16 of these values (truncation)
    for search in (0, 1):
        codes, scales, mins, _ = oracle.Oracle().quantize(w, search)
        assert np.all(codes == 0) and np.all(scales == 0)
        assert np.array_equal(mins, w[::128])


@pytest.mark.parametrize("search", [0, 1])
def test_power_of_two_homogeneity(search):
    """Scaling every weight by 2^j scales scale and minimum by 2^j exactly and
    leaves every code (and so the chosen candidate) unchanged."""
    rng = np.random.default_rng(4)
    w = random_weights(rng, 384, 40, outliers=True)
    O = oracle.Oracle()
    c0, s0, m0, _ = O.quantize(w, search)
    for j in (-3, 5):
        wj = (w.astype(np.int32) + (j << 7)).astype(np.uint16)  # exponent shift of a bf16 (no zeros here)
        cj, sj, mj, _ = O.quantize(wj, search)
        assert np.array_equal(cj, c0)
        assert np.array_equal(bf16_to_f64(sj), bf16_to_f64(s0) * 2.0 ** j)
        assert np.array_equal(bf16_to_f64(mj), bf16_to_f64(m0) * 2.0 ** j)


def test_round_to_nearest_half_step_bound_and_monotone_codes():
    """Inside the grid, every weight is at most half a step from its
    dequantised value (nearest rounding), and codes never decrease as the
    weight increases within a group."""
    rng = np.random.default_rng(5)
    w = random_weights(rng, 512, 64)
    codes, scales, mins, _ = oracle.Oracle().quantize(w, 0)
    dq, q = dequant(codes, scales, mins)
    wf = bf16_to_f64(w)
    s = np.repeat(bf16_to_f64(scales), 128, axis=0)
    m = np.repeat(bf16_to_f64(mins), 128, axis=0)
    inside = (wf >= m) & (wf <= m + 15 * s)
    assert inside.mean() > 0.95
    assert np.all(np.abs(wf - dq)[inside] <= 0.5 * s[inside] * (1 + 2.0 ** -10))
    for g in range(4):
        for n in range(64):
            order = np.argsort(wf[128 * g:128 * g + 128, n], kind="stable")
            assert np.all(np.diff(q[128 * g:128 * g + 128, n][order]) >= 0)


def test_range_search_never_worse_and_clips_outliers():
    """The search keeps p = 1 among its candidates, so its squared error is
    never above round-to-nearest; on heavy-tailed weights (Student t, 3
    degrees of freedom) it clips the tails of nearly every group (a narrower
    grid) and lowers the total squared error."""
    rng = np.random.default_rng(6)
    O = oracle.Oracle()
    for heavy in (False, True):
        if heavy:
            wt = (rng.standard_t(3, size=(512, 64)) * 0.01).astype(np.float32)
            w = (wt.view(np.uint32) >> 16).astype(np.uint16)
        else:
            w = random_weights(rng, 512, 64, outliers=True)
        wf = bf16_to_f64(w)
        rtn = O.quantize(w, 0)
        mse = O.quantize(w, 1)
        e_rtn = ((wf - dequant(*rtn[:3])[0]) ** 2).reshape(4, 128, 64).sum(axis=1)
        e_mse = ((wf - dequant(*mse[:3])[0]) ** 2).reshape(4, 128, 64).sum(axis=1)
        assert np.all(e_mse <= e_rtn * (1 + 1e-5))
        if heavy:
            narrower = bf16_to_f64(mse[1]) < bf16_to_f64(rtn[1])
            assert narrower.mean() > 0.8
            assert e_mse.sum() < 0.95 * e_rtn.sum()


def test_chosen_candidate_is_the_minimum_error():
    rng = np.random.default_rng(7)
    w = random_weights(rng, 256, 32, outliers=True)
    codes, scales, mins, errs = oracle.Oracle().quantize(w, 1)
    wf = bf16_to_f64(w)
    e = ((wf - dequant(codes, scales, mins)[0]) ** 2).reshape(2, 128, 32).sum(axis=1)
    # the chosen grid's fp64 error is the smallest candidate error up to fp32 summation
    assert np.allclose(e, errs.min(axis=2), rtol=1e-4, atol=0)


def test_quantized_weights_match_gemm_oracle_dequantisation():
    """One-hot rows through the GEMM oracle return min + q * scale of the
    quantizer's output, within half a step of the original weight."""
    rng = np.random.default_rng(8)
    K, N = 256, 16
    w = random_weights(rng, K, N)
    O = oracle.Oracle()
    codes, scales, mins, _ = O.quantize(w, 1)
    wf = bf16_to_f64(w)
    for k in (0, 5, 127, 128, 200, 255):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y, _ = O.gemm(x, codes, scales, mins)
        s = bf16_to_f64(scales[k // 128])
        assert np.all(np.abs(y[0] - wf[k]) <= 0.5 * s * (1 + 2.0 ** -10) + np.abs(y[0] - wf[k]) * (wf[k] > bf16_to_f64(mins[k // 128]) + 15 * s))


@pytest.mark.parametrize("mutant", [4, 5, 6])
def test_planted_quantizer_mistakes_are_caught(mutant):
    """Round toward zero (4), 16 steps instead of 15 (5) and keeping the worst
    candidate (6) must each fail a pin above."""
    Om = oracle.Oracle(mutant)
    rng = np.random.default_rng(9)
    failures = 0
    # exact-grid recovery
    q = rng.integers(0, 16, size=(256, 8))
    q[0::128, :] = 0
    q[1::128, :] = 15
    w = f32_to_bf16_bits((q - 8.0) * 2.0 ** -6)
    codes, scales, mins, _ = Om.quantize(w, 1)
    failures += not np.array_equal(Om.unpack_canonical(codes), q)
    # half-step bound
    wr = random_weights(rng, 256, 32)
    codes, scales, mins, _ = Om.quantize(wr, 0)
    dq, _ = dequant(codes, scales, mins)
    wf = bf16_to_f64(wr)
    s = np.repeat(bf16_to_f64(scales), 128, axis=0)
    m = np.repeat(bf16_to_f64(mins), 128, axis=0)
    inside = (wf >= m) & (wf <= m + 15 * s)
    failures += not np.all(np.abs(wf - dq)[inside] <= 0.5 * s[inside] * (1 + 2.0 ** -10))
    # search never worse than round-to-nearest
    wo = random_weights(rng, 256, 32, outliers=True)
    wof = bf16_to_f64(wo)
    e_rtn = ((wof - dequant(*Om.quantize(wo, 0)[:3])[0]) ** 2).sum()
    e_mse = ((wof - dequant(*Om.quantize(wo, 1)[:3])[0]) ** 2).sum()
    failures += not (e_mse <= e_rtn * (1 + 1e-5))
    assert failures >= 1
