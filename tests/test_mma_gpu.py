"""GPU parity of the mma.sync (f16 tensor-core) product for 5 .. 16 tokens against the CPU oracle.

The kernel feeds the 2-bit codes to the tensor cores as raw f16 bit patterns (mostly
subnormals) and the activations scaled by powers of 4; these tests check, through the C ABI,
that every accumulator is the oracle's integer and every output within 1e-6 relative:
every token count from 5 to 16 (and the dispatch of tw_ternary_matmul up to 64), ragged row counts (not multiples of the 16-row tile), K from
one 64-step to the largest allowed, the row-tile and K-slice splits of the launch plan, and
the largest accumulator magnitudes the int8 range allows (|sum c x| up to 256 K, just below
2^24 at K = 65472), which would expose a flushed subnormal or any rounding.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

REL = 1e-6


@pytest.fixture(scope="module")
def tw():
    import ternary_weight_quant_b300 as tw
    return tw


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def run(tw, fn, packed, gamma, xq, sx):
    M, N = xq.shape[0], packed.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    acc = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    getattr(tw, fn)(dev(packed), dev(np.array([gamma], np.float32)), dev(xq), dev(sx), y, None, acc)
    out = host(y), host(acc)
    assert tw.tw_device_status() == 0
    return out


def check(y, acc, y_ref, acc_ref):
    bad = acc != acc_ref
    assert not bad.any(), f"{bad.sum()} accumulators differ, first at {np.argwhere(bad)[0]}"
    y64, r64 = y.astype(np.float64), y_ref.astype(np.float64)
    far = np.abs(y64 - r64) > REL * np.abs(r64)
    assert not far.any(), f"{far.sum()} outputs beyond 1e-6 relative"


@pytest.mark.parametrize("N,K", [(37, 64), (100, 2560), (640, 6912), (3840, 2560)])
def test_mma_every_token_count(tw, N, K):
    """1 .. 16 tokens through tw_ternary_gemv (the mma.sync kernel from 5, and from 3 on the
    shorter rows), 1 .. 64 through tw_ternary_matmul (17 tokens and more: the tcgen05 GEMM)."""
    W, x = si.gemv_case(64, N, K, seed=N + K, outliers=True)
    packed, gamma = oracle.pack_ternary(W)
    xq_all, sx_all, _ = oracle.quant_act(x)  # per token: the first M tokens are the M-token case
    y_all, acc_all = oracle.ternary_matmul(packed, gamma, xq_all, sx_all, openmp=True)
    for M in range(1, 65):
        xq, sx, y_ref, acc_ref = xq_all[:M], sx_all[:M], y_all[:M], acc_all[:M]
        if M <= 16:
            check(*run(tw, "tw_ternary_gemv", packed, gamma, xq, sx), y_ref, acc_ref)
        check(*run(tw, "tw_ternary_matmul", packed, gamma, xq, sx), y_ref, acc_ref)


@pytest.mark.parametrize("M,N,K", [(8, 13824, 2560), (16, 2560, 6912), (16, 6912, 2560), (13, 5000, 1024),
                                   (9, 17, 12800), (16, 1, 64), (5, 3000, 40000), (3, 10240, 8192),
                                   (4, 6144, 4096)])
def test_mma_layer_shapes_and_plans(tw, M, N, K):
    """Shapes that take every launch plan: many tiles per CTA (groups of tiles), few tiles
    (K slices), a single row, tiles that end past N."""
    W, x = si.gemv_case(M, N, K, seed=M * 7 + N, outliers=True)
    packed, gamma = oracle.pack_ternary(W)
    xq, sx, _ = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx, openmp=True)
    check(*run(tw, "tw_ternary_gemv", packed, gamma, xq, sx), y_ref, acc_ref)


@pytest.mark.parametrize("M,N,K", [(8, 30000, 4096), (16, 30000, 4096), (5, 6000, 14336), (12, 6000, 14336),
                                   (7, 20011, 1024)])
def test_mma_persistent_double_buffered(tw, M, N, K):
    """Matrices with more row blocks than one wave of CTAs: the persistent plan, each CTA
    loading its next block into one buffer while it computes from the other (two CTAs per
    SM at K = 4096; one CTA with a larger budget at K = 14336, where two buffers of one tile
    do not fit twice; a ragged last block at N = 20011)."""
    W, x = si.gemv_case(M, N, K, seed=M + N + K, outliers=True)
    packed, gamma = oracle.pack_ternary(W)
    xq, sx, _ = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx, openmp=True)
    check(*run(tw, "tw_ternary_gemv", packed, gamma, xq, sx), y_ref, acc_ref)


@pytest.mark.parametrize("wcode,xval", [(2, 127), (2, -128), (0, -128), (0, 127)])
def test_mma_extreme_accumulators(tw, wcode, xval):
    """All weights +1 (code 2) or -1 (code 0) against all activations 127 or -128 at
    K = 65472: |acc| = 128 K and |sum c x| = 256 K, the largest the int8 range allows."""
    M, N, K = 12, 48, 65472
    packed = np.full((N, K // 4), {2: 0xAA, 0: 0x00}[wcode], np.uint8)
    packed[5] = 0x55  # one row of zero weights
    packed[7, ::3] = 0x99  # mixed codes 1, 2, 1, 2
    xq = np.full((M, K), xval, np.int8)
    xq[3, ::2] = -xval if xval != -128 else 127
    sx = np.linspace(0.5, 3.0, M).astype(np.float32)
    gamma = np.float32(0.7)
    y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
    check(*run(tw, "tw_ternary_matmul", packed, gamma, xq, sx), y_ref, acc_ref)
    check(*run(tw, "tw_ternary_gemv", packed, gamma, xq, sx), y_ref, acc_ref)


def test_mma_each_code_position(tw):
    """One nonzero weight per row at every position of its 16-weight word (the code sits in
    a different mask, shift and f16 exponent or subnormal range for each), against random
    activations: the product must pick exactly that activation."""
    M, K = 16, 1024
    N = 16 * 16
    t = np.zeros((N, K), np.int8)
    for r in range(N):
        pos = (r % 16) + 16 * ((r // 16) % (K // 16))
        t[r, pos] = 1 if r % 3 else -1
    W = t.astype(np.float32)
    packed, gamma = oracle.pack_ternary(W)
    x = si.activations(M, K, seed=3)
    xq, sx, _ = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
    y, acc = run(tw, "tw_ternary_gemv", packed, gamma, xq, sx)
    check(y, acc, y_ref, acc_ref)
    assert (acc_ref == (xq.astype(np.int64) @ t.T.astype(np.int64))).all()
