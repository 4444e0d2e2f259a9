"""GPU parity of the tensor-core GEMM (tw_ternary_gemm) against the CPU oracle.

Same seeded inputs into both sides; int32 accumulators bit-exact, fp32 outputs within
1e-6 relative.  Shapes span several 128-row weight tiles, token tiles of 16..256
(and more than one token tile), K split over clusters of CTAs, ragged tails in all
three dimensions, and the largest accumulator magnitudes the int8 range allows
(which would expose any rounding in the fp32 tensor-core accumulation).
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


def run_gemm(tw, packed, gamma, xq, sx, fn="tw_ternary_gemm", ws=True):
    """ws=True passes the optional workspace (activations widened once per call, TMA-loaded
    with hardware swizzle); ws=False makes every CTA widen its own activation tiles."""
    M, N = xq.shape[0], packed.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    acc = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    work = None
    if ws:
        work = torch.full((tw.tw_gemm_workspace_bytes(M, xq.shape[1]) + 256,), 0x5A, dtype=torch.uint8,
                          device="cuda")
    getattr(tw, fn)(dev(packed), dev(np.array([gamma], np.float32)), dev(xq), dev(sx), y, None, acc, workspace=work)
    out = host(y), host(acc)
    assert tw.tw_device_status() == 0
    return out


def check(y, acc, y_ref, acc_ref):
    bad = acc != acc_ref
    assert not bad.any(), f"{bad.sum()} accumulators differ, first at {np.argwhere(bad)[0]}"
    y64, r64 = y.astype(np.float64), y_ref.astype(np.float64)
    far = np.abs(y64 - r64) > REL * np.abs(r64)
    assert not far.any(), f"{far.sum()} outputs beyond 1e-6 relative"


def case(M, N, K, seed, outliers=True):
    W, x = si.gemv_case(M, N, K, seed=seed, outliers=outliers)
    packed, gamma = oracle.pack_ternary(W)
    xq, sx, _ = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
    return packed, gamma, xq, sx, y_ref, acc_ref


@pytest.mark.parametrize("ws", [True, False])
@pytest.mark.parametrize("M", [1, 15, 16, 17, 64, 65, 200, 256, 257])
@pytest.mark.parametrize("N,K", [(128, 64), (7, 80), (200, 2560), (640, 2560), (300, 6912)])
def test_gemm_parity(tw, M, N, K, ws):
    packed, gamma, xq, sx, y_ref, acc_ref = case(M, N, K, seed=M * 7 + N + K)
    y, acc = run_gemm(tw, packed, gamma, xq, sx, ws=ws)
    check(y, acc, y_ref, acc_ref)


@pytest.mark.parametrize("M,N,K", [(64, 3840, 2560), (256, 2560, 2560), (8, 2560, 6912), (64, 13824, 2560)])
def test_gemm_layer_shapes(tw, M, N, K):
    """2B-layer shapes (the fused q|k|v, o, gate|up and down matrices) at batched-decode sizes."""
    packed, gamma, xq, sx, y_ref, acc_ref = case(M, N, K, seed=N + M)
    y, acc = run_gemm(tw, packed, gamma, xq, sx)
    check(y, acc, y_ref, acc_ref)


@pytest.mark.parametrize("ws", [True, False])
@pytest.mark.parametrize("K", [16, 4096, 28672, 65472, 65520])
def test_gemm_extreme_accumulators(tw, K, ws):
    """Tokens chosen as +-127/-128 times a weight row's signs give |acc| = 127..128 * nnz,
    up to 8.4e6 (< 2^24): every partial sum must stay exact in the fp32 accumulation."""
    N, M = 160, 48
    W = si.weights(N, K, seed=K)
    W[3] = 0.0
    W[4] = np.abs(W[4]) + 1.0       # all +1
    packed, gamma = oracle.pack_ternary(W)
    t = oracle.unpack_ternary(packed, K).astype(np.int32)
    xq = np.empty((M, K), np.int8)
    for m in range(M):
        row = t[m % N]
        if m % 3 == 0:
            xq[m] = np.where(row > 0, 127, np.where(row < 0, -128, 0))
        elif m % 3 == 1:
            xq[m] = np.where(row > 0, -128, 127)
        else:
            xq[m] = np.full(K, -128 if m % 2 else 127, np.int8)
    sx = np.linspace(0.5, 40.0, M).astype(np.float32)
    y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
    assert np.abs(acc_ref).max() > 100 * K // 4
    y, acc = run_gemm(tw, packed, gamma, xq, sx, ws=ws)
    check(y, acc, y_ref, acc_ref)


def test_gemm_repeatable(tw):
    packed, gamma, xq, sx, y_ref, acc_ref = case(96, 1000, 2560, seed=5)
    outs = [run_gemm(tw, packed, gamma, xq, sx, ws=w) for w in (True, True, False)]
    for y, acc in outs:
        check(y, acc, y_ref, acc_ref)
        assert (y == outs[0][0]).all()


def test_gemm_zero_and_negated_weights(tw):
    M, N, K = 80, 256, 1024
    W, x = si.gemv_case(M, N, K, seed=31)
    W[:7] = 0.0
    xq, sx, _ = oracle.quant_act(x)
    ys = []
    for Wv in (W, -W):
        packed, gamma = oracle.pack_ternary(Wv)
        y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
        y, acc = run_gemm(tw, packed, gamma, xq, sx)
        check(y, acc, y_ref, acc_ref)
        assert (acc[:, :7] == 0).all() and (y[:, :7] == 0).all()
        ys.append(y)
    assert (ys[0] == -ys[1]).all()


@pytest.mark.parametrize("M", [17, 48, 64, 100, 256])
def test_matmul_dispatch_parity(tw, M):
    """tw_ternary_matmul picks the GEMV or the GEMM by M; both must give the oracle's result."""
    packed, gamma, xq, sx, y_ref, acc_ref = case(M, 384, 2560, seed=M)
    y, acc = run_gemm(tw, packed, gamma, xq, sx, fn="tw_ternary_matmul")
    check(y, acc, y_ref, acc_ref)


@pytest.mark.parametrize("ws", [True, False])
@pytest.mark.parametrize("M", [11, 12, 16])
def test_matmul_large_matrix_crossover(tw, M, ws):
    """For matrices of 2^24 weights or more (here 2560 x 6912) the dispatch hands 12..16 tokens
    to the GEMM when a workspace is given, and keeps the GEMV otherwise: the same exact result."""
    packed, gamma, xq, sx, y_ref, acc_ref = case(M, 2560, 6912, seed=300 + M)
    y, acc = run_gemm(tw, packed, gamma, xq, sx, fn="tw_ternary_matmul", ws=ws)
    check(y, acc, y_ref, acc_ref)
