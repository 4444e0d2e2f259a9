"""Pins for the oracle functions of the fused epilogue (CPU only): the fp32 residual add
(hand-worked roundings, tests/golden/residual_add.txt) and the RMSNorm scale on its own (it
must be the scale two_rmsnorm applies, itself pinned by hand-worked rows in
test_oracle_pins.py)."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "residual_add.txt")


def _bits(s):
    return np.array([int(s, 16)], np.uint32).view(np.float32)[0]


def test_residual_add_hand_worked():
    rows = [line.split() for line in open(GOLDEN) if line.strip() and not line.startswith("#")]
    assert len(rows) >= 8
    h = np.array([_bits(r[0]) for r in rows], np.float32)
    y = np.array([_bits(r[1]) for r in rows], np.float32)
    want = np.array([int(r[2], 16) for r in rows], np.uint32)
    got = oracle.residual_add(h, y).view(np.uint32)
    assert (got == want).all(), [hex(v) for v in got]


def test_residual_add_rejects_non_finite():
    with pytest.raises(oracle.OracleError):
        oracle.residual_add(np.array([1.0, np.inf], np.float32), np.zeros(2, np.float32))


@pytest.mark.parametrize("K,seed", [(4, 0), (64, 1), (2560, 2), (6912, 3)])
def test_rms_inv_is_the_scale_rmsnorm_applies(K, seed):
    """With g = 1 and x[0] = 1, two_rmsnorm's u[0] = fl(1 * inv) * 1 = inv exactly."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((3, K)).astype(np.float32)
    x[2] *= 1e-20  # a tiny row (its first element is set to 1 below like the others)
    x[:, 0] = 1.0
    inv = oracle.rms_inv(x, 1e-6)
    u, _ = oracle.rmsnorm(x, np.ones(K, np.float32), 1e-6)
    assert (inv.view(np.uint32) == u[:, 0].view(np.uint32)).all()
