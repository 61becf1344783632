"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test checks the oracle against a hand-derived value, exact rational
arithmetic, brute force, a mathematical invariant or an independent library
routine, chosen so that a plausible mistake (reversed nibble order, an
off-by-one group, a dropped minimum term, a transposed operand) fails at least
one of them.  The planted-mistake tests at the end build such mutants of the
oracle and check that the pins catch them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def O():
    return oracle.Oracle()


def bf16_bits(values):
    """float values that are exactly bf16 -> bit patterns (asserting exactness)."""
    f = np.asarray(values, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (b >> 16).astype(np.uint16)


def frac_bf16(bits):
    return Fraction(float(oracle.bf16_bits_to_f64(np.uint16(bits))))


def trunc_bf16(values):
    """float32 values truncated to bf16 -> bit patterns (any bf16 is a valid input)."""
    return (np.asarray(values, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def random_problem(rng, M, K, N):
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    G = K // 128
    s_b = trunc_bf16(rng.uniform(0.002, 0.02, size=(G, N)))
    m_b = trunc_bf16(-8.0 * oracle.bf16_bits_to_f64(s_b) * rng.uniform(0.9, 1.1, size=(G, N)))
    x_b = trunc_bf16(rng.standard_normal(size=(M, K)))
    return q, s_b, m_b, x_b


# ---------------------------------------------------------------- canonical codes

def read_canonical_golden():
    rows = []
    with open(os.path.join(GOLDEN, "canonical_words.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            codes, words = line.split(";")
            codes = [int(v) for v in codes.split(",")]
            words = [int(v, 16) for v in words.split(",")]
            rows.append((codes, words))
    return rows


def test_canonical_pack_hand_words(O):
    for codes, words in read_canonical_golden():
        q = np.array(codes, dtype=np.uint8).reshape(-1, 1)
        got = O.pack_canonical(q)
        assert got[:, 0].tolist() == words


def test_canonical_unpack_hand_words(O):
    for codes, words in read_canonical_golden():
        c = np.array(words, dtype=np.uint32).reshape(-1, 1)
        assert O.unpack_canonical(c)[:, 0].tolist() == codes


def test_canonical_round_trip(O):
    rng = np.random.default_rng(1)
    for K, N in [(8, 1), (128, 3), (256, 64)]:
        q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
        assert np.array_equal(O.unpack_canonical(O.pack_canonical(q)), q)
        c = rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint32)
        assert np.array_equal(O.pack_canonical(O.unpack_canonical(c)), c)
    for v in (0, 15):
        q = np.full((128, 4), v, dtype=np.uint8)
        assert np.array_equal(O.unpack_canonical(O.pack_canonical(q)), q)


def test_bits_per_weight_exact(O):
    for K, N in [(128, 16), (4096, 4096), (5120, 6144), (17408, 5120), (5120, 248320)]:
        nbytes = O.packed_bytes(K, N)
        assert Fraction(nbytes * 8, K * N) == Fraction(17, 4)   # 4.25 bits per weight


# ---------------------------------------------------------------- bf16 helpers

def test_bf16_rn_against_torch():
    torch = pytest.importorskip("torch")
    O = oracle.Oracle()
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32),
        (rng.standard_normal(500) * 1e-38).astype(np.float32),   # bf16 subnormal range
        (rng.standard_normal(500) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38], dtype=np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.bf16_rn(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_ulp_closed_form(O):
    assert O.bf16_ulp(1.0) == 2.0**-7
    assert O.bf16_ulp(1.99) == 2.0**-7
    assert O.bf16_ulp(-2.0) == 2.0**-6
    assert O.bf16_ulp(0.0) == 2.0**-133
    assert O.bf16_ulp(2.0**-130) == 2.0**-133
    assert O.bf16_ulp(2.0**100 * 1.5) == 2.0**93
    v = np.array([1.0, 1.99, -2.0, 0.0, 2.0**-130, 3 * 2.0**99])
    assert np.array_equal(O.bf16_ulp_array(v), [O.bf16_ulp(t) for t in v])


# ---------------------------------------------------------------- closed forms

def exact_gemm(q, s_b, m_b, x_b):
    """Exact rational y for tiny problems (brute force in Fractions)."""
    M, K = x_b.shape
    N = q.shape[1]
    xs = [[frac_bf16(x_b[m, k]) for k in range(K)] for m in range(M)]
    y = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        for k in range(K):
            g = k // 128
            w = frac_bf16(m_b[g, n]) + int(q[k, n]) * frac_bf16(s_b[g, n])
            for m in range(M):
                y[m][n] += xs[m][k] * w
    return y


def test_closed_form_constant_codes(O):
    """All codes equal c: y = sum_g (min_g + c*scale_g) * X_g, X_g = sum of x over group g."""
    rng = np.random.default_rng(3)
    K, N, M = 384, 4, 2
    _, s_b, m_b, x_b = random_problem(rng, M, K, N)
    for c in (0, 7, 15):
        q = np.full((K, N), c, dtype=np.uint8)
        y, _ = O.gemm(x_b, O.pack_canonical(q), s_b, m_b)
        for m in range(M):
            X = [sum(frac_bf16(x_b[m, k]) for k in range(128 * g, 128 * g + 128)) for g in range(K // 128)]
            for n in range(N):
                exact = sum((frac_bf16(m_b[g, n]) + c * frac_bf16(s_b[g, n])) * X[g] for g in range(K // 128))
                assert abs(Fraction(y[m, n]) - exact) <= Fraction(1, 10**12) * (1 + abs(exact))


def test_closed_form_zero_scale(O):
    """scale = 0: y = sum_g min_g * X_g, whatever the codes."""
    rng = np.random.default_rng(4)
    K, N, M = 256, 8, 1
    q, _, m_b, x_b = random_problem(rng, M, K, N)
    s_b = np.zeros_like(m_b)
    y, _ = O.gemm(x_b, O.pack_canonical(q), s_b, m_b)
    for n in range(N):
        exact = sum(frac_bf16(m_b[g, n]) * sum(frac_bf16(x_b[0, k]) for k in range(128 * g, 128 * g + 128))
                    for g in range(K // 128))
        assert abs(Fraction(y[0, n]) - exact) <= Fraction(1, 10**12) * (1 + abs(exact))


def test_exact_integer_case(O):
    """min = 0, scale = 1, integer x: y = sum_k x_k q_k is an exact integer."""
    rng = np.random.default_rng(5)
    K, N, M = 1024, 16, 3
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    x_b = bf16_bits(x)
    s_b = np.full((K // 128, N), bf16_bits([1.0])[0], dtype=np.uint16)
    m_b = np.zeros((K // 128, N), dtype=np.uint16)
    y, a = O.gemm(x_b, O.pack_canonical(q), s_b, m_b)
    ref = x.astype(np.int64) @ q.astype(np.int64)
    assert np.array_equal(y, ref.astype(np.float64))
    assert np.array_equal(a, np.abs(x.astype(np.int64)) @ q.astype(np.int64))
    # min = -8 moves every weight by -8 exactly
    m_b8 = np.full_like(m_b, bf16_bits([-8.0])[0])
    y8, _ = O.gemm(x_b, O.pack_canonical(q), s_b, m_b8)
    assert np.array_equal(y8, (x.astype(np.int64) @ (q.astype(np.int64) - 8)).astype(np.float64))


def test_one_hot_rows_pin_layout(O):
    """x = e_k picks row k: y_n = min_g(k),n + q_kn * scale_g(k),n, exactly, for every k."""
    rng = np.random.default_rng(6)
    K, N = 384, 16
    q, s_b, m_b, _ = random_problem(rng, 1, K, N)
    codes = O.pack_canonical(q)
    X = np.zeros((K, K), dtype=np.uint16)
    X[np.arange(K), np.arange(K)] = bf16_bits([1.0])[0]
    y, _ = O.gemm(X, codes, s_b, m_b)
    s = oracle.bf16_bits_to_f64(s_b)
    mn = oracle.bf16_bits_to_f64(m_b)
    for k in range(K):
        expect = mn[k // 128] + q[k].astype(np.float64) * s[k // 128]
        assert np.array_equal(y[k], expect), k


def test_brute_force_tiny(O):
    """Tiny problems against an exact rational triple loop."""
    rng = np.random.default_rng(7)
    for M, K, N in [(1, 128, 1), (3, 128, 8), (8, 256, 2), (2, 128, 64)]:
        q, s_b, m_b, x_b = random_problem(rng, M, K, N)
        y, a = O.gemm(x_b, O.pack_canonical(q), s_b, m_b)
        ex = exact_gemm(q, s_b, m_b, x_b)
        for m in range(M):
            for n in range(N):
                assert abs(Fraction(y[m, n]) - ex[m][n]) <= Fraction(a[m, n]) * Fraction(1, 2**45)


def test_exhaustive_code_patterns(O):
    """Every code value at every nibble position: column n has q_k = (k + n) mod 16."""
    K, N = 128, 16
    q = np.array([[(k + n) % 16 for n in range(N)] for k in range(K)], dtype=np.uint8)
    x = np.arange(1, K + 1, dtype=np.float32)          # exact in bf16 up to 256
    x_b = bf16_bits(x)[None, :]
    s_b = np.full((1, N), bf16_bits([1.0])[0], dtype=np.uint16)
    m_b = np.zeros((1, N), dtype=np.uint16)
    y, _ = O.gemm(x_b, O.pack_canonical(q), s_b, m_b)
    ref = (np.arange(1, K + 1, dtype=np.int64) @ q.astype(np.int64)).astype(np.float64)
    assert np.array_equal(y[0], ref)


# ---------------------------------------------------------------- invariants

def test_power_of_two_homogeneity(O):
    rng = np.random.default_rng(8)
    M, K, N = 2, 512, 32
    q, s_b, m_b, x_b = random_problem(rng, M, K, N)
    codes = O.pack_canonical(q)
    y, _ = O.gemm(x_b, codes, s_b, m_b)
    x = oracle.bf16_bits_to_f64(x_b).astype(np.float32)
    for alpha in (0.25, 2.0, 64.0):
        y2, _ = O.gemm(bf16_bits(x * np.float32(alpha)), codes, s_b, m_b)
        assert np.array_equal(y2, alpha * y)


def test_additivity_disjoint_support(O):
    rng = np.random.default_rng(9)
    K, N = 512, 32
    q, s_b, m_b, x_b = random_problem(rng, 1, K, N)
    codes = O.pack_canonical(q)
    mask = rng.random(K) < 0.5
    x1 = np.where(mask, x_b[0], 0).astype(np.uint16)[None, :]
    x2 = np.where(~mask, x_b[0], 0).astype(np.uint16)[None, :]
    y, a = O.gemm(x_b, codes, s_b, m_b)
    y1, _ = O.gemm(x1, codes, s_b, m_b)
    y2, _ = O.gemm(x2, codes, s_b, m_b)
    assert np.all(np.abs(y - (y1 + y2)) <= 1e-13 * a)


def test_group_permutation_invariance(O):
    """Permuting the 128-row groups of W together with x leaves y unchanged."""
    rng = np.random.default_rng(10)
    M, K, N = 2, 640, 16
    q, s_b, m_b, x_b = random_problem(rng, M, K, N)
    G = K // 128
    perm = rng.permutation(G)
    rows = np.concatenate([np.arange(128 * g, 128 * g + 128) for g in perm])
    y, a = O.gemm(x_b, O.pack_canonical(q), s_b, m_b)
    yp, _ = O.gemm(x_b[:, rows], O.pack_canonical(q[rows]), s_b[perm], m_b[perm])
    assert np.all(np.abs(y - yp) <= 1e-13 * a)


def test_rows_independent(O):
    rng = np.random.default_rng(11)
    M, K, N = 5, 256, 16
    q, s_b, m_b, x_b = random_problem(rng, M, K, N)
    codes = O.pack_canonical(q)
    y, a = O.gemm(x_b, codes, s_b, m_b)
    for m in range(M):
        ym, am = O.gemm(x_b[m:m + 1], codes, s_b, m_b)
        assert np.array_equal(ym[0], y[m]) and np.array_equal(am[0], a[m])


def test_threads_do_not_change_result(O):
    rng = np.random.default_rng(12)
    q, s_b, m_b, x_b = random_problem(rng, 2, 512, 64)
    codes = O.pack_canonical(q)
    y1, a1 = O.gemm(x_b, codes, s_b, m_b, nthreads=1)
    y4, a4 = O.gemm(x_b, codes, s_b, m_b, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(a1, a4)


# ---------------------------------------------------------------- tiled layout

def read_tiled_golden():
    codes, metas = [], []
    with open(os.path.join(GOLDEN, "tiled_positions.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "code":
                codes.append(tuple(int(v) for v in parts[1:]))
            else:
                metas.append((parts[1], int(parts[2]), int(parts[3]), int(parts[4])))
    return codes, metas


def test_tiled_hand_positions(O):
    K, N = 256, 96
    code_rows, meta_rows = read_tiled_golden()
    for k, n, byte, half in code_rows:
        q = np.zeros((K, N), dtype=np.uint8)
        q[k, n] = 0xA
        s = np.zeros((K // 128, N), dtype=np.uint16)
        packed = O.pack_tiled(O.pack_canonical(q), s, s)
        nz = np.nonzero(packed)[0]
        assert nz.tolist() == [byte], (k, n, nz)
        assert packed[byte] == (0xA << (4 * half)), (k, n)
    for kind, g, n, byte in meta_rows:
        s = np.zeros((K // 128, N), dtype=np.uint16)
        m = np.zeros((K // 128, N), dtype=np.uint16)
        (s if kind == "scale" else m)[g, n] = 0xBEEF
        packed = O.pack_tiled(np.zeros((K // 8, N), dtype=np.uint32), s, m)
        nz = np.nonzero(packed)[0]
        assert nz.tolist() == [byte, byte + 1], (kind, g, n, nz)
        assert packed[byte] == 0xEF and packed[byte + 1] == 0xBE


def test_tiled_round_trip_and_size(O):
    rng = np.random.default_rng(13)
    for K, N in [(128, 16), (384, 48), (1024, 64)]:
        c = rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint32)
        s = rng.integers(0, 2**16, size=(K // 128, N), dtype=np.uint16)
        m = rng.integers(0, 2**16, size=(K // 128, N), dtype=np.uint16)
        packed = O.pack_tiled(c, s, m)
        assert packed.size * 32 == K * N * 17        # 4.25 bits per weight, no padding
        c2, s2, m2 = O.unpack_tiled(packed, K, N)
        assert np.array_equal(c, c2) and np.array_equal(s, s2) and np.array_equal(m, m2)


def test_tiled_column_prefix_is_byte_prefix(O):
    """Packing the first N' = 64*Q' columns gives the first bytes of the full packing."""
    rng = np.random.default_rng(14)
    K, N = 256, 208
    c = rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint32)
    s = rng.integers(0, 2**16, size=(K // 128, N), dtype=np.uint16)
    m = rng.integers(0, 2**16, size=(K // 128, N), dtype=np.uint16)
    full = O.pack_tiled(c, s, m)
    for Np in (64, 128, 192):
        pre = O.pack_tiled(c[:, :Np], s[:, :Np], m[:, :Np])
        assert np.array_equal(pre, full[:pre.size])


def test_tiled_quad_is_one_contiguous_run(O):
    """All bytes of the columns of quad q occupy [q*G*4352, (q+1)*G*4352)."""
    K, N = 384, 128
    G = K // 128
    for q in range(N // 64):
        cc = np.zeros((K // 8, N), np.uint32)
        cc[:, 64 * q:64 * q + 64] = 0xFFFFFFFF
        z = np.zeros((G, N), np.uint16)
        packed = O.pack_tiled(cc, z, z)
        nz = np.nonzero(packed)[0]
        assert nz.min() >= q * G * 4352 and nz.max() < (q + 1) * G * 4352


def test_tiled_each_word_holds_two_columns_of_one_lane(O):
    """A column n of tile 0 lives only in the 4 lanes 4*(n%8)+c, in nibbles of parity n//8."""
    K, N = 128, 16
    for n in range(N):
        q = np.zeros((K, N), dtype=np.uint8)
        q[:, n] = 1
        z = np.zeros((1, N), np.uint16)
        packed = O.pack_tiled(O.pack_canonical(q), z, z)
        words = packed[:1024].view(np.uint32).reshape(2, 32, 4)
        lanes = sorted(set(np.nonzero(words)[1].tolist()))
        assert lanes == [4 * (n % 8) + c for c in range(4)]
        expect = 0x01010101 if n < 8 else 0x10101010
        assert np.all(words[:, lanes, :] == expect)


# ---------------------------------------------------------------- planted mistakes

@pytest.mark.parametrize("mutant", [1, 2, 3])
def test_planted_mistakes_are_caught(mutant):
    """Each mutant oracle (reversed nibbles, off-by-one group, dropped min) must
    fail at least one of the pins above."""
    Om = oracle.Oracle(mutant)
    failures = 0
    for test in (test_canonical_unpack_hand_words, test_one_hot_rows_pin_layout,
                 test_closed_form_zero_scale, test_closed_form_constant_codes,
                 test_exact_integer_case, test_brute_force_tiny):
        try:
            test(Om)
        except AssertionError:
            failures += 1
    assert failures >= 1


# ---------------------------------------------------------------- acceptance helper

def test_accept_bound():
    O = oracle.Oracle()
    y_ref = np.array([1.0, 100.0, 0.0])
    a = np.array([10.0, 10.0, 0.0])
    ok, ratio = oracle.accept(y_ref + np.array([0.04, 0.0, 0.0]), y_ref, a, O)
    assert ok.tolist() == [True, True, True]
    ok, _ = oracle.accept(y_ref + np.array([0.04 + 2**-7 + 1e-9, 0.0, 2**-132]), y_ref, a, O)
    assert ok.tolist() == [False, True, False]
    assert ratio.shape == (3,)


def test_synth_inputs_feed_the_oracle():
    """The shared generator's arrays have the shapes the oracle expects."""
    O = oracle.Oracle()
    c, s, m = synth.matrix(20260001, 0, 256, 32)
    x = synth.x(20260001, 0, 2, 256)
    y, a = O.gemm(x, c, s, m)
    assert y.shape == (2, 32) and np.all(a > 0)
