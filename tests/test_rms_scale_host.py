"""Integer RMSNorm scale of the kernels, run on the host and pinned to exact arithmetic.

The kernels form 1 / sqrt(fl32(fl64(S) / K) + eps) from the exact sum of squares S
without double-precision instructions: S is rounded to 53 bits, the division by K is an
invariant-integer multiplication carried 32 bits past the quotient, and the two
roundings of the double-precision formula are applied to the integers.  The same
__host__ __device__ code is compiled for the host here and compared with Python's
exact rationals (Fraction), its correctly rounded int / int and float / float
division, and numpy's IEEE fp32 conversion, square root and divide.  No oracle code
is involved.
"""
import os
import random
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "host_progs", "rms_scale_check.cu")
EPS_BITS = int(np.float32(1e-6).view(np.uint32))


@pytest.fixture(scope="module")
def prog(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("rsc") / "rms_scale_check")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a", SRC, "-o", out],
                   check=True, capture_output=True)
    return out


def run(prog, cases):
    text = "".join(f"{hi} {lo} {E} {K} {eb} {sh}\n" for hi, lo, E, K, eb, sh in cases)
    res = subprocess.run([prog], input=text, capture_output=True, text=True, check=True).stdout.split("\n")
    return [tuple(int(v) for v in line.split()) for line in res if line.strip()]


def expected(hi, lo, E, K, eps_bits, sh):
    v = (hi << 64) | lo
    if v == 0:
        ms = np.float32(0.0)
        m = e = None
    else:
        S = Fraction(v) * Fraction(2) ** (2 * E - 364)
        R = float(S)                      # correctly rounded to double
        m, e = None, None
        mant, ex = np.frexp(R)            # R = mant 2^ex, 0.5 <= mant < 1
        m, e = int(mant * 2 ** 53), int(ex) - 53
        with np.errstate(over="ignore"):
            ms = np.float32(R / K)        # double division, then fp32 rounding
    eps = np.array([eps_bits], dtype=np.uint32).view(np.float32)[0]
    with np.errstate(divide="ignore"):
        inv = np.float32(1.0) / np.sqrt(np.float32(ms + eps))
    shifted = v >> sh
    exact = (shifted << sh) == v
    return m, e, int(np.float32(ms).view(np.uint32)), int(np.float32(inv).view(np.uint32)), shifted, exact


def check(prog, cases):
    got = run(prog, cases)
    assert len(got) == len(cases)
    for c, g in zip(cases, got):
        m, e, msb, invb, shifted, exact = expected(*c)
        gm, ge, gms, ginv, shi, slo, sex = g
        if m is not None:
            # fl64(S) = m 2^e; the program may return m = 2^53 with e one lower
            assert Fraction(gm) * Fraction(2) ** ge == Fraction(m) * Fraction(2) ** e, c
            assert 2 ** 52 <= gm <= 2 ** 53, c
        assert gms == msb, (c, hex(gms), hex(msb))
        assert ginv == invb, (c, hex(ginv), hex(invb))
        assert (shi << 64) | slo == shifted and bool(sex) == exact, c


def test_random_sums_all_magnitudes(prog):
    rng = random.Random(20261202)
    cases = []
    for _ in range(4000):
        K = rng.choice([rng.randrange(1, 65533), 4 * rng.randrange(1, 16384), 2560, 6912, 28672, 1 << rng.randrange(0, 17)])
        nb = rng.randrange(1, 128)
        v = rng.getrandbits(nb) | (1 << (nb - 1))
        # aim the quotient anywhere from below the fp32 subnormals to above its range
        target = rng.randrange(-175, 140)
        E = (target + 364 + K.bit_length() - nb) // 2 + rng.randrange(-2, 3)
        E = max(1, min(254, E))
        cases.append((v >> 64, v & (2 ** 64 - 1), E, K, EPS_BITS, rng.randrange(0, 130)))
    check(prog, cases)


def test_midpoints_and_double_rounding(prog):
    """Quotients exactly on an fp32 midpoint, and a hair to either side (the double
    rounding can land on the midpoint and then round to even)."""
    rng = random.Random(7)
    cases = []
    for _ in range(1500):
        K = rng.choice([3, 7, 2560, 6912, 65532, rng.randrange(1, 65533)])
        f = rng.randrange(1 << 23, 1 << 24)           # fp32 significand
        k = rng.randrange(-170, 100)                  # exponent of its last bit
        # S = K (f + 1/2) 2^k (+ a tiny offset), as an integer times 2^(2E - 364)
        E = max(1, min(254, (k - 8 + 364) // 2))
        base = 2 * E - 364
        num = Fraction(K) * (Fraction(2 * f + 1, 2)) * Fraction(2) ** k / Fraction(2) ** base
        off = rng.choice([0, 0, 1, -1, 2 ** rng.randrange(0, 40), -(2 ** rng.randrange(0, 40))])
        v = int(num) + off
        if v <= 0 or v >= 2 ** 128:
            continue
        cases.append((v >> 64, v & (2 ** 64 - 1), E, K, EPS_BITS, 0))
    check(prog, cases)


def test_edges(prog):
    top = 2 ** 128 - 1
    cases = [
        (0, 0, 1, 2560, EPS_BITS, 5),                 # zero sum: ms = 0, scale = 1/sqrt(eps)
        (0, 1, 1, 1, EPS_BITS, 0),                    # smallest sum: underflows to 0
        (top >> 64, top & (2 ** 64 - 1), 254, 1, EPS_BITS, 1),    # overflows fp32: ms = inf, scale 0
        (top >> 64, top & (2 ** 64 - 1), 254, 65532, EPS_BITS, 127),
        (0, (1 << 53) - 1, 254, 3, EPS_BITS, 128),    # sh = 128 clears the sum
        (1 << 40, 12345, 100, 2560, 0, 64),           # eps = 0
    ]
    # the fp32 subnormal / normal boundary and the largest finite value
    for target_bits in (0x007fffff, 0x00800000, 0x00000001, 0x7f7fffff):
        t = Fraction(int(np.array([target_bits], np.uint32).view(np.float32)[0].item() * 2 ** 160)) / 2 ** 160
        for K in (1, 3, 2560):
            E = 200 if target_bits == 0x7f7fffff else 60
            v = int(t * K / Fraction(2) ** (2 * E - 364))
            for dv in (-1, 0, 1):
                if 0 < v + dv < 2 ** 128:
                    cases.append(((v + dv) >> 64, (v + dv) & (2 ** 64 - 1), E, K, EPS_BITS, 3))
    check(prog, cases)


# ---------------------------------------------------------------- float-float fast path
FAST_SRC = os.path.join(ROOT, "tests", "host_progs", "rms_fast_check.cu")


@pytest.fixture(scope="module")
def fast_prog(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("rfc") / "rms_fast_check")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a", FAST_SRC, "-o", out],
                   check=True, capture_output=True)
    return out


def exact_ms_bits(x):
    """fl32(fl64(fl64(sum x^2) / K)) from exact rationals."""
    S = sum(Fraction(float(v)) ** 2 for v in x)
    R = float(S)
    with np.errstate(over="ignore", under="ignore"):
        return int(np.float32(R / len(x)).view(np.uint32))


def run_fast(prog, rows, C=0):
    text = "".join(f"{len(r)} {C} " + " ".join(str(int(b)) for b in np.asarray(r, np.float32).view(np.uint32)) + "\n"
                   for r in rows)
    out = subprocess.run([prog], input=text, capture_output=True, text=True, check=True).stdout.split("\n")
    return [tuple(int(v) for v in line.split()) for line in out if line.strip()]


def near_midpoint_row(rng, K, scale, big):
    """K values whose mean square lands within about an fp32 ulp * 2^-11 of a rounding midpoint."""
    x = (rng.standard_normal(K) * scale).astype(np.float32)
    if big:
        x[-1] = np.float32(scale * 30.0)  # the last element carries most of the sum
    rest = sum(Fraction(float(v)) ** 2 for v in x[:-1])
    total = Fraction(float(np.float32(float(sum(Fraction(float(v)) ** 2 for v in x)) / K))) * K
    ms = np.float32(total / K)
    ulp = Fraction(float(np.spacing(ms)))
    mid = Fraction(float(ms)) + ulp / 2
    need = mid * K - rest
    if need <= 0:
        return x
    x[-1] = np.float32(float(need) ** 0.5)
    return x


def test_fast_path_never_disagrees_with_exact(fast_prog):
    rng = np.random.default_rng(11)
    rows = []
    for K in (2560, 6912, 4096, 64, 1536):
        for s in (1e-3, 1.0, 37.0):
            rows.append((rng.standard_normal(K) * s).astype(np.float32))
            rows.append(near_midpoint_row(rng, K, s, big=False))
            rows.append(near_midpoint_row(rng, K, s, big=True))
    for _ in range(40):  # spread exponents, a few huge or tiny outliers
        K = int(rng.choice([2560, 6912, 128]))
        x = (rng.standard_normal(K) * np.exp2(rng.integers(-20, 20, K))).astype(np.float32)
        rows.append(x)
    got = run_fast(fast_prog, rows)
    assert len(got) == len(rows)
    n_ok = 0
    for x, (ok, bits) in zip(rows, got):
        if ok:
            n_ok += 1
            assert bits == exact_ms_bits(x), (len(x), hex(bits), hex(exact_ms_bits(x)))
    assert n_ok >= len(rows) // 2  # the fast path decides most rows, even these adversarial ones


def test_fast_path_refuses_out_of_range_sums(fast_prog):
    rows = [np.full(256, 1e-30, np.float32), np.full(256, 1e25, np.float32), np.zeros(256, np.float32)]
    got = run_fast(fast_prog, rows)
    assert [ok for ok, _ in got] == [0, 0, 0]


@pytest.mark.parametrize("C", [2, 4, 8])
def test_fast_path_in_cluster_order(fast_prog, C):
    """The order of the cluster-shared prologue (each rank a chunk of 16-element groups, four
    component accumulators per thread, warp butterflies, then sequential sums over warps and
    ranks): whenever the decision is taken, its mean square is the exact one."""
    rng = np.random.default_rng(100 + C)
    rows = []
    for K in (8192, 12288, 16448, 28672):
        for s in (1e-3, 1.0, 37.0):
            rows.append((rng.standard_normal(K) * s).astype(np.float32))
            rows.append(near_midpoint_row(rng, K, s, big=False))
            rows.append(near_midpoint_row(rng, K, s, big=True))
    for _ in range(6):
        K = int(rng.choice([8192, 14336]))
        rows.append((rng.standard_normal(K) * np.exp2(rng.integers(-20, 20, K))).astype(np.float32))
    got = run_fast(fast_prog, rows, C)
    assert len(got) == len(rows)
    n_ok = 0
    for x, (ok, bits) in zip(rows, got):
        if ok:
            n_ok += 1
            assert bits == exact_ms_bits(x), (len(x), C, hex(bits), hex(exact_ms_bits(x)))
    assert n_ok >= len(rows) // 2
