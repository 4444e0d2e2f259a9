"""Pins for the oracle's five-trits-per-byte functions (CPU only).

The layout is a reading of "BitNet 1 位 LLM 独立推理引擎：位串行 GEMM 内核与 LUT 优化工程实践",
正文 paragraph 3 (TL2: several weights share one small index, so fewer bytes are loaded): byte
i of a row holds weights 4i..4i+3 as base-3 digits 0..3 and weight 4 RB + i as digit 4, each
digit t + 1, with RB = 16 ceil(K / 80) bytes per row.  Each test below would fail for a
plausible slip: a swapped digit order or region (hand-worked bytes), a lost or doubled code
(the 243-value bijection), wrong padding (size and rejection), or a decode that disagrees with
the 2-bit path (identical int32 products on the same weights).
"""
import itertools
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "trits5_bytes.txt")


def _golden_rows():
    rows, name, spec = [], None, None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, rest = line.split(" ", 1)
        if head == "row":
            name, spec = rest.split(" ", 1)
        elif head == "bytes":
            rows.append((name, spec, [int(v) for v in rest.split()]))
    return rows


def _row_from_spec(spec, K):
    if spec == "all+1":
        return np.ones(K, np.int8)
    if spec == "all-1":
        return -np.ones(K, np.int8)
    t = np.zeros(K, np.int8)
    for item in spec.split(","):
        k, v = item.split(":")
        t[int(k)] = int(v)
    return t


@pytest.mark.parametrize("name,spec,expect", _golden_rows())
def test_hand_worked_bytes(name, spec, expect):
    K = 68
    t = _row_from_spec(spec, K)[None, :]
    got = oracle.pack_trits5(t)
    assert got.shape == (1, 16)
    assert got[0].tolist() == expect, name
    assert (oracle.unpack_trits5(got, K) == t).all()


def test_row_bytes():
    # 16 * ceil(K / 80): hand values, never below ceil(K / 5), equal to K / 5 when 80 | K
    for K, rb in [(4, 16), (68, 16), (80, 16), (84, 32), (2560, 512), (4096, 832), (6912, 1392),
                  (8192, 1648), (14336, 2880), (28672, 5744)]:
        assert oracle.t5_row_bytes(K) == rb, K
        assert rb >= -(-K // 5)
        assert (rb == K // 5) == (K % 80 == 0)


def test_all_243_codes_round_trip():
    """Every 5-tuple of trits, placed in byte 0 of a K = 80 row (weights 0..3 and 64),
    gives a distinct byte; together they are exactly 0..242, and each decodes back."""
    K = 80
    tuples = list(itertools.product((-1, 0, 1), repeat=5))
    t = np.zeros((len(tuples), K), np.int8)
    for r, tup in enumerate(tuples):
        t[r, 0:4] = tup[:4]
        t[r, 64] = tup[4]
    p = oracle.pack_trits5(t)
    assert sorted(p[:, 0].tolist()) == list(range(243))
    assert (p[:, 1:] == 121).all()
    assert (oracle.unpack_trits5(p, K) == t).all()


def test_invalid_bytes_and_padding_rejected():
    K = 68
    p = oracle.pack_trits5(np.zeros((1, K), np.int8))
    for v in range(243, 256):
        bad = p.copy()
        bad[0, 7] = v
        with pytest.raises(oracle.OracleError):
            oracle.unpack_trits5(bad, K)
    bad = p.copy()
    bad[0, 4] = 121 + 81  # weight 68 (past K) set to +1
    with pytest.raises(oracle.OracleError):
        oracle.unpack_trits5(bad, K)
    with pytest.raises(oracle.OracleError):
        oracle.pack_trits5(np.full((1, K), 2, np.int8))


@pytest.mark.parametrize("K", [4, 64, 68, 80, 84, 160, 2560, 6912])
def test_random_round_trip(K):
    rng = np.random.default_rng(K)
    t = rng.integers(-1, 2, size=(7, K)).astype(np.int8)
    p = oracle.pack_trits5(t)
    assert p.shape == (7, oracle.t5_row_bytes(K))
    assert (oracle.unpack_trits5(p, K) == t).all()
    assert p.max() <= 242


@pytest.mark.parametrize("M,N,K", [(1, 9, 68), (3, 17, 2560), (2, 5, 6912), (4, 33, 84)])
def test_product_equals_two_bit_product_and_dense(M, N, K):
    """The same weights give the same int32 results through both layouts, and both equal a
    dense int64 product of the decoded weights."""
    rng = np.random.default_rng(M * 1000 + K)
    t = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    xq = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    xq[0, :] = -128  # extreme token
    sx = rng.uniform(0.1, 4.0, size=M).astype(np.float32)
    gamma = np.float32(0.37)
    p2 = oracle.pack_rows_with_scale(t.astype(np.float32), np.float32(1.0))
    y2, a2 = oracle.ternary_matmul(p2, gamma, xq, sx)
    y5, a5 = oracle.ternary_matmul5(oracle.pack_trits5(t), gamma, xq, sx)
    assert (a5 == a2).all()
    assert (y5.view(np.uint32) == y2.view(np.uint32)).all()
    assert (a5 == xq.astype(np.int64) @ t.T.astype(np.int64)).all()
    y5o, a5o = oracle.ternary_matmul5(oracle.pack_trits5(t), gamma, xq, sx, openmp=True)
    assert (a5o == a5).all() and (y5o.view(np.uint32) == y5.view(np.uint32)).all()


def test_pack_ternary5_matches_two_bit_pack():
    rng = np.random.default_rng(5)
    W = rng.standard_normal((13, 6912)).astype(np.float32)
    p2, g2 = oracle.pack_ternary(W)
    p5, g5 = oracle.pack_ternary5(W)
    assert g5 == g2
    assert (oracle.unpack_trits5(p5, 6912) == oracle.unpack_ternary(p2, 6912)).all()
