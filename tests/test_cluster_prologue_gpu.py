"""GPU parity of the fused quantisation + GEMV when its CTAs share the quantisation in a
thread-block cluster (the streaming kernel from K = 12288, and from K = 8192 with RMSNorm).

Each CTA of a cluster quantises one chunk of K and pushes the chunk's statistics and its
quantised groups to the other CTAs through distributed shared memory.  The launcher takes
clusters of 4 CTAs and shrinks the grid to the clusters that can be resident (284 of 296 CTAs
on 148 SMs at two CTAs per SM), or falls back to clusters of 2.  Covered: grids of 148 and 296
CTAs (kept, and shrunk to 284), odd and small grids (37 and 146 CTAs, shrunk to a multiple
of 4), 1 to 4 tokens (padding tokens included), chunks of 192 to 448 groups, rows that take the
exact mean-square path (all-zero, wide exponent range, subnormal, one-hot, exact ties), tokens
whose quotients sit next to the rounding ties, and launches chained under programmatic
dependent launch.  x_q, s_x and x_sum bit for bit, the accumulators exactly and y within 1e-6,
against the oracle.
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


def assert_y_close(y_gpu, y_ref):
    y_gpu = y_gpu.astype(np.float64)
    y_ref = y_ref.astype(np.float64)
    bad = np.abs(y_gpu - y_ref) > REL * np.abs(y_ref)
    assert not bad.any(), f"{bad.sum()} outputs beyond 1e-6 relative, first at {np.argwhere(bad)[0]}"


def fused(tw, x, p_ref, g_ref, g):
    M, K = x.shape
    N = p_ref.shape[0]
    packed, gamma = dev(p_ref), dev(np.array([g_ref], np.float32))
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    acc = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    xq = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sx = torch.zeros(M, dtype=torch.float32, device="cuda")
    xs = torch.zeros(M, dtype=torch.int32, device="cuda")
    gd = None if g is None else dev(g)
    tw.tw_quant_gemv(dev(x), packed, gamma, y, g=gd, eps=si.RMS_EPS, x_q=xq, s_x=sx, x_sum=xs, acc_out=acc)
    y2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tw.tw_quant_gemv(dev(x), packed, gamma, y2, g=gd, eps=si.RMS_EPS)
    return host(y), host(acc), host(xq), host(sx), host(xs), host(y2)


def check(tw, x, W, g, rows=None):
    p_ref, g_ref = oracle.pack_ternary(W)
    if g is None:
        q_ref, s_ref, sum_ref = oracle.quant_act(x)
    else:
        q_ref, s_ref, sum_ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
    rows = np.arange(W.shape[0]) if rows is None else rows
    y_ref, acc_ref = oracle.ternary_matmul(p_ref[rows], g_ref, q_ref, s_ref, openmp=True)
    y, acc, xq, sx, xs, y2 = fused(tw, x, p_ref, g_ref, g)
    assert (xq == q_ref).all(), f"{(xq != q_ref).sum()} x_q bytes differ"
    assert (sx.view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (xs == sum_ref).all()
    assert (acc[:, rows] == acc_ref).all()
    assert_y_close(y[:, rows], y_ref)
    assert (y2 == y).all()
    assert tw.tw_device_status() == 0


# (N, K, M): 146 rows at K = 12288 (grid 146 -> 144), 3000 (296 -> 284), 28672 with 2500 rows
# (296 -> 284) and 1000 (148), 16448 (257 groups per rank), 2 tokens (148), 3 tokens (296 ->
# 284), 4 tokens (148), 37 rows (grid 36), and K = 8192 (clusters with RMSNorm only)
CASES = [(146, 12288, 1), (3000, 12288, 1), (2500, 28672, 1), (1000, 28672, 1), (2000, 16448, 1),
         (1000, 12288, 2), (700, 12288, 3), (300, 12288, 4), (37, 12288, 1), (640, 8192, 4)]


@pytest.mark.parametrize("N,K,M", CASES)
@pytest.mark.parametrize("rms", [False, True])
def test_cluster_prologue_parity(tw, N, K, M, rms):
    W, x = si.gemv_case(M, N, K, seed=3 * N + K + M + rms, outliers=(M % 2 == 1))
    g = si.rms_gain(K, seed=K + 5) if rms else None
    rows = None
    if N * K > 20_000_000:
        rows = np.sort(np.random.default_rng(N + K).choice(N, min(N, 1024), replace=False))
    check(tw, x, W, g, rows)


def special_tokens(K):
    """All-zero, exponents spread from 2^-140 to 2^60 (mean square outside the float-float
    range: the exact path), subnormal only (likewise), one-hot, exact ties."""
    rng = np.random.default_rng(K)
    x = si.activations(6, K, seed=11)
    x[1] = 0.0
    x[2] = (rng.standard_normal(K) * np.ldexp(1.0, rng.integers(-140, 60, size=K))).astype(np.float32)
    x[3] = np.float32(1e-40) * np.sign(x[3])
    x[4, :] = 0.0
    x[4, K - 7] = -3.0  # in the last chunk
    x[5] = np.array([127, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5] * (K // 8), np.float32)
    return x


@pytest.mark.parametrize("K,N", [(12288, 300), (28672, 1300)])
def test_cluster_prologue_special_tokens(tw, K, N):
    x = special_tokens(K)
    W = si.weights(N, K, seed=70)
    g = si.rms_gain(K, seed=71)
    M = 3 if K <= 12288 else 1  # several tokens of K = 28672 exceed the fused kernel
    for m0 in range(0, 6, M):
        for gg in (None, g):
            check(tw, x[m0:m0 + M], W, gg)


def near_ties(K, M, seed):
    """Quotients x 127 / max|x| on, or a few ulps either side of, the half-integers."""
    rng = np.random.default_rng(seed)
    x = np.empty((M, K), np.float32)
    for m in range(M):
        a = np.float32(rng.uniform(0.5, 4.0))
        k = rng.integers(-127, 127, size=K).astype(np.float32) + np.float32(0.5)
        v = (k * a / np.float32(127.0)).astype(np.float32)
        steps = rng.integers(-3, 4, size=K)
        for s in range(1, 4):  # s ulps up or down
            up, dn = steps == s, steps == -s
            for _ in range(s):
                v[up] = np.nextafter(v[up], np.float32(np.inf))
                v[dn] = np.nextafter(v[dn], np.float32(-np.inf))
        v[K // 2] = a if m % 2 == 0 else -a
        x[m] = v
    return x


def test_cluster_prologue_near_ties(tw):
    K, N, M = 12288, 640, 4
    check(tw, near_ties(K, M, seed=5), si.weights(N, K, seed=72), None)


def test_cluster_prologue_chain_pdl(tw):
    """Back-to-back fused launches of clustered kernels (each reads the previous output) in a
    graph replayed three times: every launch must quantise its own input."""
    N = K = 12288
    packs = [oracle.pack_ternary(si.weights(N, K, seed=80 + i)) for i in range(2)]
    x0 = si.activations(1, K, seed=90)
    g = si.rms_gain(K, seed=91)
    ref = [x0]
    for p, gm in packs:
        q, s, _ = oracle.rmsnorm_quant_act(ref[-1], g, si.RMS_EPS)
        y, _ = oracle.ternary_matmul(p, gm, q, s, openmp=True)
        ref.append(y)
    bufs = [dev(x0)] + [torch.empty((1, N), dtype=torch.float32, device="cuda") for _ in packs]
    dp = [(dev(p), dev(np.array([gm], np.float32))) for p, gm in packs]
    gd = dev(g)

    def chain():
        for i, (p, gm) in enumerate(dp):
            tw.tw_quant_gemv(bufs[i], p, gm, bufs[i + 1], g=gd, eps=si.RMS_EPS)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain()
    torch.cuda.current_stream().wait_stream(s)
    for i in range(len(packs)):
        assert_y_close(host(bufs[i + 1]), ref[i + 1])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    for b in bufs[1:]:
        b.zero_()
    for _ in range(3):
        graph.replay()
    for i in range(len(packs)):
        assert_y_close(host(bufs[i + 1]), ref[i + 1])
    assert tw.tw_device_status() == 0
