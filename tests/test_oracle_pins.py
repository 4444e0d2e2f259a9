"""Pins for the CPU oracle, against facts that do not come from the oracle's own code.

Each test names what it pins: math.fsum (a correctly rounded library sum), numpy
integer / float64 matmul of the unpacked weights (brute force), closed forms of
the absmean ternarisation of N(0,1) weights, exhaustive enumeration of the 81
valid packed bytes, hand-worked fixtures under tests/golden/, and the symmetry
invariants of the method.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            left, right = line.split("|")
            rows.append((left.split(), right.split()))
    return rows


# ---------------------------------------------------------------- exact sums
def test_exact_sum_matches_fsum_wide_range():
    rng = np.random.default_rng(1)
    for trial in range(20):
        n = int(rng.integers(1, 3000))
        mant = rng.random(n)
        expo = rng.integers(-1074, 1000, size=n)
        v = np.ldexp(mant, expo)
        v = v[np.isfinite(v)]
        assert oracle.exact_sum(v) == math.fsum(v.tolist())


def test_exact_sum_ties_and_subnormals():
    # 1 + 2^-53 is exactly half way between 1 and 1 + 2^-52: ties-to-even gives 1.
    assert oracle.exact_sum([1.0, 2.0 ** -53]) == 1.0
    # a tiny extra term breaks the tie upwards
    assert oracle.exact_sum([1.0, 2.0 ** -53, 2.0 ** -300]) == 1.0 + 2.0 ** -52
    # 1 + 3*2^-53 is half way between 1+2^-52 and 1+2^-51: even mantissa is 1+2^-51
    assert oracle.exact_sum([1.0, 3 * 2.0 ** -53]) == 1.0 + 2.0 ** -51
    tiny = 5e-324
    assert oracle.exact_sum([tiny] * 3) == 3 * tiny
    assert oracle.exact_sum([]) == 0.0
    big = [1e308, 1e-308, 1e308 * 0.5]
    assert oracle.exact_sum(big) == math.fsum(big)


def test_exact_sum_many_equal_terms():
    # 2^20 copies of 0.1 (as double): fsum gives the correctly rounded result.
    v = np.full(1 << 20, 0.1)
    assert oracle.exact_sum(v) == math.fsum(v.tolist())


def test_exact_sum_rejects_bad_input():
    with pytest.raises(oracle.OracleError):
        oracle.exact_sum([1.0, -1.0])
    with pytest.raises(oracle.OracleError):
        oracle.exact_sum([1.0, float("inf")])


# ---------------------------------------------------------------- absmean (O1, O2)
@pytest.mark.parametrize("shape,seed", [((256, 256), 0), ((7, 68), 3), ((1, 4), 5), ((33, 640), 11)])
def test_absmean_is_fsum_mean(shape, seed):
    W = si.weights(*shape, seed=seed)
    gamma, S = oracle.absmean(W)
    ref_S = math.fsum(np.abs(W.astype(np.float64)).ravel().tolist())
    assert S == ref_S
    assert gamma == np.float32(ref_S / W.size)


def test_absmean_zero_fraction_closed_form():
    # W ~ N(0,1): gamma -> E|W| = sqrt(2/pi); t = 0 iff |W| < gamma/2, so the zero
    # fraction -> erf(sqrt(2/pi)/2/sqrt(2)) = 0.31006 ("about 1/3 zeros").
    W, _ = si.gemv_case(1, 256, 256, seed=0)
    packed, gamma = oracle.pack_ternary(W)
    t = oracle.unpack_ternary(packed, 256)
    n = W.size
    p0 = math.erf(math.sqrt(2 / math.pi) / 2 / math.sqrt(2))
    assert abs(p0 - 0.31006) < 1e-5
    sigma = math.sqrt(p0 * (1 - p0) / n)
    assert abs((t == 0).mean() - p0) < 5 * sigma
    g_mean = math.sqrt(2 / math.pi)
    g_sigma = math.sqrt((1 - 2 / math.pi) / n)
    assert abs(float(gamma) - g_mean) < 5 * g_sigma
    # +1 and -1 equally likely
    sig_pm = math.sqrt((1 - p0) / 2 * (1 + p0) / 2 / n)
    assert abs((t == 1).mean() - (1 - p0) / 2) < 5 * sig_pm


def test_constant_weights():
    for c in (0.37, 3.0, 1e-30):
        W = np.full((3, 8), c, np.float32)
        packed, gamma = oracle.pack_ternary(W)
        assert gamma == np.float32(c)
        assert (oracle.unpack_ternary(packed, 8) == 1).all()
        packed, gamma = oracle.pack_ternary(-W)
        assert gamma == np.float32(c)
        assert (oracle.unpack_ternary(packed, 8) == -1).all()


def test_all_zero_weights():
    packed, gamma = oracle.pack_ternary(np.zeros((2, 4), np.float32))
    assert gamma == 0.0
    assert (packed == 0x55).all()


def test_scaling_by_power_of_two():
    W = si.weights(16, 64, seed=4)
    p0, g0 = oracle.pack_ternary(W)
    for k in (-20, -1, 3, 40):
        pk, gk = oracle.pack_ternary(W * np.float32(2.0 ** k))
        assert (pk == p0).all()
        assert gk == np.float32(g0 * np.float32(2.0 ** k))


def test_negated_weights_mirror_codes():
    W = si.weights(9, 36, seed=6)
    p, g = oracle.pack_ternary(W)
    pn, gn = oracle.pack_ternary(-W)
    assert g == gn
    assert (oracle.unpack_ternary(pn, 36) == -oracle.unpack_ternary(p, 36)).all()


def test_round_half_even_on_weights():
    # gamma = mean|W| = 1 for W = [0.5, 1.5, 1.0, 1.0]; 0.5 -> 0 (tie to even), 1.5 -> 2 -> clamp 1
    W = np.array([[0.5, 1.5, -1.0, 1.0]], np.float32)
    packed, gamma = oracle.pack_ternary(W)
    assert gamma == 1.0
    assert oracle.unpack_ternary(packed, 4).tolist() == [[0, 1, -1, 1]]


# ---------------------------------------------------------------- packing (O3)
def _byte_of(ts):
    # pack four t values through the oracle: W = t as floats (gamma <= 1 keeps +-1, 0 stays 0)
    W = np.array([ts], np.float32)
    packed, _ = oracle.pack_ternary(W)
    return int(packed[0, 0])


def test_pack_layout_golden():
    for left, right in _golden_rows("pack_layout.txt"):
        ts = [int(v) for v in left]
        assert _byte_of(ts) == int(right[0], 16), (ts, right)


def test_exhaustive_valid_bytes_round_trip():
    valid = []
    for b in range(256):
        fields = [(b >> (2 * j)) & 3 for j in range(4)]
        if 3 in fields:
            with pytest.raises(oracle.OracleError):
                oracle.unpack_ternary(np.array([[b]], np.uint8), 4)
            continue
        valid.append(b)
        t = oracle.unpack_ternary(np.array([[b]], np.uint8), 4)
        assert t[0].tolist() == [f - 1 for f in fields]
        assert _byte_of(t[0].tolist()) == b
    assert len(valid) == 81


def test_random_round_trip_and_size():
    rng = np.random.default_rng(2)
    for N, K in [(1, 4), (5, 12), (17, 64), (3, 68)]:
        t = rng.integers(-1, 2, size=(N, K)).astype(np.float32)
        packed, _ = oracle.pack_ternary(t)
        assert packed.nbytes == N * K // 4  # 2 bits per weight: 1e9 weights -> 250 MB
        assert (oracle.unpack_ternary(packed, K) == t).all()
    with pytest.raises(oracle.OracleError):
        oracle.pack_ternary(np.zeros((2, 6), np.float32))  # K % 4 != 0


# ---------------------------------------------------------------- activation quant (O4)
def test_act_quant_golden_ties():
    for left, right in _golden_rows("act_quant_ties.txt"):
        x = np.array([float(v) for v in left], np.float32)
        xq, sx, xs = oracle.quant_act(x)
        assert xq[0].tolist() == [int(v) for v in right]
        assert sx[0] == np.abs(x).max()
        assert xs[0] == sum(int(v) for v in right)


# Exact rational arithmetic for re-deriving the hand-worked fixtures: fp32 values as
# Fractions, IEEE round-to-nearest-even onto the fp32 grid, a correctly rounded square root
# (checked against the squares of the neighbouring midpoints) and round-half-even to an
# integer.  None of it comes from the oracle.
def _ex(v):
    return Fraction(float(np.float32(v)))


def _fl32(q):
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    if Fraction(2) ** (e + 1) <= q:
        e += 1
    step = Fraction(1, 2 ** 149) if e < -126 else Fraction(2) ** (e - 23)
    n = q / step
    return sign * _rne(n) * step


def _rne(q):
    f = q.numerator // q.denominator
    r = q - f
    return f + (1 if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1) else 0)


def _next32(v, up):
    return Fraction(float(np.nextafter(np.float32(float(v)), np.float32(np.inf if up else -np.inf))))


def _sqrt32(t):
    c = Fraction(float(np.float32(math.sqrt(float(t)))))
    for cand in (_next32(c, False), c, _next32(c, True)):
        lo, hi = (_next32(cand, False) + cand) / 2, (cand + _next32(cand, True)) / 2
        if lo * lo < t < hi * hi:
            return cand
    raise AssertionError("no fp32 square root found")


def test_act_quant_golden_order():
    """Tokens where fl(fl(x*127)/a) sits exactly on a half-integer: the oracle must take
    the tie to even, and the reciprocal form must land elsewhere (so the fixture tells
    the two orders apart)."""
    for left, right in _golden_rows("act_quant_order.txt"):
        x = np.array([float(v) for v in left], np.float32)
        expect = [int(v) for v in right]
        a = max(abs(_ex(v)) for v in x)
        derived = [_rne(_fl32(_fl32(_ex(v) * 127) / a)) for v in x]
        assert derived == expect  # the fixture agrees with its exact derivation
        recip = _fl32(Fraction(127) / a)
        assert [_rne(_fl32(_ex(v) * recip)) for v in x] != expect
        xq, sx, xs = oracle.quant_act(x)
        assert xq[0].tolist() == expect
        assert sx[0] == np.float32(float(a)) and xs[0] == sum(expect)


def test_rmsnorm_golden_k4():
    """One K = 4 token with every fp32 step of the RMSNorm reading pinned (u bits and x_q),
    re-derived here with exact rationals; the one-rounding inverse and the (x*g)*inv order
    both give a different x_q on it."""
    rows = []
    with open(os.path.join(GOLDEN, "rmsnorm_k4.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([part.split() for part in line.split("|")])
    assert rows
    eps = np.float32(si.RMS_EPS)
    for xs_, gs_, ubits_, q_ in rows:
        x = np.array([float(v) for v in xs_], np.float32)
        g = np.array([float(v) for v in gs_], np.float32)
        ubits = np.array([int(v) for v in ubits_], np.uint32)
        expect = [int(v) for v in q_]
        # exact derivation of the reading
        r = sum(_ex(v) ** 2 for v in x)
        ms = _fl32(r / len(x))
        inv = _fl32(1 / _sqrt32(_fl32(ms + _ex(eps))))
        u = [_fl32(_fl32(_ex(xv) * inv) * _ex(gv)) for xv, gv in zip(x, g)]
        assert [int(np.float32(float(v)).view(np.uint32)) for v in u] == ubits.tolist()
        a = max(abs(v) for v in u)
        assert [_rne(_fl32(_fl32(v * 127) / a)) for v in u] == expect
        # the oracle
        u_o, r_o = oracle.rmsnorm(x, g, eps)
        assert r_o[0] == float(r)
        assert (u_o[0].view(np.uint32) == ubits).all()
        xq, sx, _ = oracle.rmsnorm_quant_act(x, g, eps)
        assert xq[0].tolist() == expect and sx[0] == np.float32(float(a))
        # the other readings differ on this row
        t = np.float32(float(_fl32(ms + _ex(eps))))
        inv_one = np.float32(1.0 / math.sqrt(float(t)))
        for uu in ([np.float32(np.float32(xv * inv_one) * gv) for xv, gv in zip(x, g)],
                   [np.float32(np.float32(xv * gv) * np.float32(float(inv))) for xv, gv in zip(x, g)]):
            aa = max(abs(v) for v in uu)
            alt = [int(np.rint(np.float32(np.float32(v * np.float32(127)) / aa))) for v in uu]
            assert alt != expect


def test_act_quant_invariants():
    x = si.activations(6, 300, seed=9, outliers=True)
    xq, sx, xs = oracle.quant_act(x)
    # the element of largest magnitude maps to exactly +-127
    for m in range(6):
        i = np.argmax(np.abs(x[m]))
        assert abs(int(xq[m, i])) == 127
        assert sx[m] == np.abs(x[m]).max()
    assert (np.abs(xq.astype(int)) <= 127).all()
    assert (xs == xq.astype(np.int64).sum(1)).all()
    for k in (-30, 5):
        xq2, sx2, _ = oracle.quant_act(x * np.float32(2.0 ** k))
        assert (xq2 == xq).all()
        assert (sx2 == sx * np.float32(2.0 ** k)).all()
    xqn, sxn, xsn = oracle.quant_act(-x)
    assert (xqn == -xq).all() and (sxn == sx).all() and (xsn == -xs).all()


def test_act_quant_within_half_step():
    # |x_q - x*127/a| <= 0.5 + fp32 rounding of the quotient
    x = si.activations(4, 1000, seed=10)
    xq, sx, _ = oracle.quant_act(x)
    exact = x.astype(np.float64) * 127.0 / sx[:, None].astype(np.float64)
    assert (np.abs(xq - exact) <= 0.5 + 1e-4).all()


# ---------------------------------------------------------------- RMSNorm (O5)
def test_rmsnorm_against_float64_definition():
    x = si.activations(3, 2560, seed=12)
    g = si.rms_gain(2560, seed=12)
    u, r = oracle.rmsnorm(x, g, si.RMS_EPS)
    for m in range(3):
        x64 = x[m].astype(np.float64)
        assert r[m] == math.fsum((x64 * x64).tolist())
        ref = x64 / np.sqrt(np.mean(x64 * x64) + si.RMS_EPS) * g.astype(np.float64)
        assert np.allclose(u[m], ref, rtol=1e-6, atol=0)


# ---------------------------------------------------------------- int GEMV + dequant (O6, O7)
def _dense_reference(packed, gamma, xq, sx, K):
    t = oracle.unpack_ternary(packed, K).astype(np.int64)
    acc = xq.astype(np.int64) @ t.T
    Wd = t.astype(np.float64) * float(gamma)
    xd = xq.astype(np.float64) * (sx.astype(np.float64)[:, None] / 127.0)
    return acc, xd @ Wd.T


@pytest.mark.parametrize("M,N,K,seed", [(1, 256, 256, 0), (3, 7, 68, 1), (16, 33, 64, 2),
                                        (2, 1, 4, 3), (5, 64, 640, 4)])
def test_matmul_against_brute_force(M, N, K, seed):
    W, x = si.gemv_case(M, N, K, seed=seed, outliers=(seed % 2 == 1))
    packed, gamma = oracle.pack_ternary(W)
    xq, sx, _ = oracle.quant_act(x)
    y, acc = oracle.ternary_matmul(packed, gamma, xq, sx)
    acc_ref, y_dense = _dense_reference(packed, gamma, xq, sx, K)
    assert (acc == acc_ref).all()
    # y is the fp32 rounding of a value within a few double ulps of the dense result
    assert np.all(np.abs(y.astype(np.float64) - y_dense) <= 6.0e-8 * np.abs(y_dense) + 1e-37)


def test_matmul_exhaustive_k4():
    rows = []
    for b in range(256):
        if 3 not in [(b >> (2 * j)) & 3 for j in range(4)]:
            rows.append(b)
    packed = np.array(rows, np.uint8)[:, None]            # 81 rows, K = 4
    t = np.array([[((b >> (2 * j)) & 3) - 1 for j in range(4)] for b in rows], np.int64)
    grid = [-128, -127, -1, 0, 1, 127]
    xq = np.array(np.meshgrid(grid, grid, grid, grid)).reshape(4, -1).T.astype(np.int8)
    sx = np.ones(len(xq), np.float32)
    y, acc = oracle.ternary_matmul(packed, np.float32(1.0), xq, sx)
    assert (acc == xq.astype(np.int64) @ t.T).all()


def test_matmul_one_hot():
    W = si.weights(12, 64, seed=21)
    packed, gamma = oracle.pack_ternary(W)
    t = oracle.unpack_ternary(packed, 64)
    for k in (0, 5, 63):
        xq = np.zeros((1, 64), np.int8)
        xq[0, k] = 127
        _, acc = oracle.ternary_matmul(packed, gamma, xq, np.ones(1, np.float32))
        assert (acc[0] == 127 * t[:, k].astype(np.int32)).all()


def test_matmul_invariants():
    W, x = si.gemv_case(4, 40, 128, seed=8)
    W[3] = 0.0  # an all-zero weight row
    packed, gamma = oracle.pack_ternary(W)
    xq, sx, _ = oracle.quant_act(x)
    y, acc = oracle.ternary_matmul(packed, gamma, xq, sx)
    assert (acc[:, 3] == 0).all() and (y[:, 3] == 0).all()
    # -W gives -y bitwise
    pn, gn = oracle.pack_ternary(-W)
    yn, _ = oracle.ternary_matmul(pn, gn, xq, sx)
    assert (yn == -y).all()  # float equality: bitwise except +0 / -0 of zero rows
    # -x gives -y; 2x gives 2y exactly
    xqn, sxn, _ = oracle.quant_act(-x)
    yx, _ = oracle.ternary_matmul(packed, gamma, xqn, sxn)
    assert (yx == -y).all()
    xq2, sx2, _ = oracle.quant_act(2 * x)
    y2, _ = oracle.ternary_matmul(packed, gamma, xq2, sx2)
    assert (y2 == 2 * y).all()


def test_matmul_all_core_build_is_identical():
    """The all-core (OpenMP over output rows) build of the integer product used for the
    CPU baseline returns the same accumulators and outputs bit for bit."""
    W, x = si.gemv_case(5, 301, 640, seed=31, outliers=True)
    p, g = oracle.pack_ternary(W)
    q, s, _ = oracle.quant_act(x)
    y1, a1 = oracle.ternary_matmul(p, g, q, s)
    y2, a2 = oracle.ternary_matmul(p, g, q, s, openmp=True)
    assert (a1 == a2).all() and (y1.view(np.uint32) == y2.view(np.uint32)).all()
    assert oracle.threads(openmp=False) == 1 and oracle.threads(openmp=True) >= 1
    bad = p.copy()
    bad[7, 3] |= 0x30  # a code 3 in row 7
    with pytest.raises(oracle.OracleError):
        oracle.ternary_matmul(bad, g, q, s, openmp=True)


def test_matmul_rejects_invalid_code():
    packed = np.array([[0xFF]], np.uint8)
    with pytest.raises(oracle.OracleError):
        oracle.ternary_matmul(packed, np.float32(1), np.ones((1, 4), np.int8), np.ones(1, np.float32))
