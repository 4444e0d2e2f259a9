"""GPU parity of the five-trits-per-byte layout against the CPU oracle.

tw_pack_ternary_t5 must write the oracle's bytes and scale bit for bit; tw_ternary_gemv_t5
must return the oracle's int32 accumulators exactly and y within 1e-6 relative, at every
2B layer shape, at shapes with ragged tails (K not a multiple of 80, chunks past K, rows not
a multiple of the CTA's share), at the largest K the kernel takes (16 slices), with extreme
accumulators, and chained behind the quantisation kernel under programmatic dependent
launch.  The same weights through the 2-bit GEMV must give the same accumulators.
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


def gemv_t5(tw, p5, gamma, xq, sx):
    M, N = xq.shape[0], p5.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    acc = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    tw.tw_ternary_gemv_t5(dev(p5), dev(np.array([gamma], np.float32)), dev(xq), dev(sx), y, acc)
    return host(y), host(acc)


def check(y, acc, y_ref, acc_ref):
    bad = acc != acc_ref
    assert not bad.any(), f"{bad.sum()} accumulators differ, first at {np.argwhere(bad)[0]}"
    far = np.abs(y.astype(np.float64) - y_ref.astype(np.float64)) > REL * np.abs(y_ref.astype(np.float64))
    assert not far.any(), f"{far.sum()} outputs beyond 1e-6 relative"


@pytest.mark.parametrize("N,K", [(5, 4), (37, 68), (256, 256), (40, 84), (3840, 2560), (2560, 6912),
                                 (640, 4096), (9, 28672)])
def test_pack_t5_bit_exact(tw, N, K):
    W = si.weights(N, K, seed=N + K)
    p_ref, g_ref = oracle.pack_ternary5(W)
    p5, g = tw.pack_t5(dev(W))
    assert host(g)[0].view(np.uint32) == np.float32(g_ref).view(np.uint32)
    got = host(p5)
    assert got.shape == p_ref.shape
    assert (got == p_ref).all(), f"{(got != p_ref).sum()} bytes differ"


SHAPES_2B = [(v[0], v[1]) for v in si.layer_shapes("2B").values()] + \
            [(v[0], v[1]) for v in si.fused_layer_shapes("2B").values()]


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", sorted(set(SHAPES_2B)))
def test_gemv_t5_every_2b_shape(tw, N, K, M):
    W, x = si.gemv_case(M, N, K, seed=N * 3 + K + M, outliers=True)
    p5, gamma = oracle.pack_ternary5(W)
    xq, sx, _ = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul5(p5, gamma, xq, sx, openmp=True)
    check(*gemv_t5(tw, p5, gamma, xq, sx), y_ref, acc_ref)


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (2, 37, 64), (1, 100, 80), (2, 33, 96), (1, 9, 4096),
                                   (2, 300, 8192), (1, 7, 14336), (2, 3, 28672), (1, 17, 40960),
                                   (1, 1000, 2560), (2, 4099, 1024)])
def test_gemv_t5_ragged_and_wide(tw, M, N, K):
    """Tails past K inside a chunk, partial last slice, 1..16 slices, uneven CTA row shares."""
    W, x = si.gemv_case(M, N, K, seed=M + 7 * N + K, outliers=True)
    p5, gamma = oracle.pack_ternary5(W)
    xq, sx, _ = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul5(p5, gamma, xq, sx, openmp=True)
    check(*gemv_t5(tw, p5, gamma, xq, sx), y_ref, acc_ref)


@pytest.mark.parametrize("sign,xval", [(1, -128), (-1, -128), (1, 127), (-1, 127)])
def test_gemv_t5_extreme_accumulators(tw, sign, xval):
    """All weights +1 or -1 against all activations 127 or -128 at the largest K: |acc| up
    to 128 * 40960; one row of zeros, one of alternating signs."""
    M, N, K = 2, 24, 40960
    t = np.full((N, K), sign, np.int8)
    t[5] = 0
    t[7, ::2] = -sign
    p5 = oracle.pack_trits5(t)
    xq = np.full((M, K), xval, np.int8)
    xq[1, ::3] = 0
    sx = np.array([1.5, 0.25], np.float32)
    gamma = np.float32(0.8)
    y_ref, acc_ref = oracle.ternary_matmul5(p5, gamma, xq, sx)
    check(*gemv_t5(tw, p5, gamma, xq, sx), y_ref, acc_ref)


def test_gemv_t5_every_byte_value(tw):
    """All 243 byte values in every byte position of a 16-byte chunk, against random
    activations: the table and the digit-4 gather are exercised for every code."""
    M, K = 2, 2560
    RB = oracle.t5_row_bytes(K)
    N = 243
    p5 = np.empty((N, RB), np.uint8)
    for r in range(N):
        p5[r] = (np.arange(RB) * 7 + r) % 243
    t = oracle.unpack_trits5(p5, K)
    xq = np.random.default_rng(1).integers(-128, 128, size=(M, K)).astype(np.int8)
    sx = np.array([0.9, 2.0], np.float32)
    y_ref, acc_ref = oracle.ternary_matmul5(p5, np.float32(1.0), xq, sx)
    assert (acc_ref == xq.astype(np.int64) @ t.T.astype(np.int64)).all()
    check(*gemv_t5(tw, p5, np.float32(1.0), xq, sx), y_ref, acc_ref)


@pytest.mark.parametrize("N,K", [(3840, 2560), (2560, 6912)])
def test_gemv_t5_equals_2bit_gemv_on_device(tw, N, K):
    """Pack the same device tensor both ways and run both products: identical int32."""
    W = si.device_normal((N, K), seed=9)
    p2, g2 = tw.pack(W)
    p5, g5 = tw.pack_t5(W)
    x = si.device_normal((1, K), seed=10)
    xq, sx, xs = tw.quantize(x)
    y2 = torch.empty((1, N), dtype=torch.float32, device="cuda")
    a2 = torch.empty((1, N), dtype=torch.int32, device="cuda")
    y5, a5 = torch.empty_like(y2), torch.empty_like(a2)
    tw.tw_ternary_gemv(p2, g2, xq, sx, y2, xs, a2)
    tw.tw_ternary_gemv_t5(p5, g5, xq, sx, y5, a5)
    assert (host(a5) == host(a2)).all()
    assert (host(y5).view(np.uint32) == host(y2).view(np.uint32)).all()


def test_gemv_t5_chained_behind_quantisation(tw):
    """RMSNorm + quantisation, then the product, back to back on one stream and repeated
    with fresh activations: under programmatic dependent launch the product must read the
    x_q of its own step."""
    N, K = 3840, 2560
    W = si.weights(N, K, seed=21)
    p5_np, gamma = oracle.pack_ternary5(W)
    p5, gd = dev(p5_np), dev(np.array([gamma], np.float32))
    g = si.rms_gain(K, seed=22)
    gdev = dev(g)
    xq = torch.empty((1, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(1, dtype=torch.float32, device="cuda")
    xs = torch.empty(1, dtype=torch.int32, device="cuda")
    ys = []
    xs_host = []
    for step in range(4):
        x = si.activations(1, K, seed=30 + step)
        xs_host.append(x)
        y = torch.empty((1, N), dtype=torch.float32, device="cuda")
        tw.tw_rmsnorm_quant_act(dev(x), gdev, si.RMS_EPS, xq, sx, xs)
        tw.tw_ternary_gemv_t5(p5, gd, xq, sx, y)
        ys.append(y)
    torch.cuda.synchronize()
    for x, y in zip(xs_host, ys):
        q_ref, s_ref, _ = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
        y_ref, _ = oracle.ternary_matmul5(p5_np, gamma, q_ref, s_ref)
        far = np.abs(host(y).astype(np.float64) - y_ref) > REL * np.abs(y_ref)
        assert not far.any()
