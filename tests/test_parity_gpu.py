"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Same seeded inputs into both sides.  Bar: packed bytes, gamma bits, int8 activations,
activation scales, activation sums and int32 accumulators bit-exact; fp32 outputs
within 1e-6 relative (the tolerance stated for the method; the kernels' epilogue
is 3 fp32 roundings from the exact value, <= 1.8e-7 relative).
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


def gpu_pack(tw, W_np):
    packed, ws = tw.pack(dev(W_np))
    return host(packed), host(ws)[0]


def assert_y_close(y_gpu, y_ref):
    y_gpu = y_gpu.astype(np.float64)
    y_ref = y_ref.astype(np.float64)
    bad = np.abs(y_gpu - y_ref) > REL * np.abs(y_ref)
    assert not bad.any(), f"{bad.sum()} outputs beyond 1e-6 relative, first at {np.argwhere(bad)[0]}"


def wide_range(N, K, seed):
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((N, K)) * np.ldexp(1.0, rng.integers(-140, 60, size=(N, K)))
    return W.astype(np.float32)


# ----------------------------------------------------------------------------- pack
PACK_CASES = [(256, 256, 0), (1, 4, 1), (7, 68, 2), (7, 64, 3), (33, 640, 4), (5, 12, 5),
              (3, 4, 6), (1000, 1000, 7), (6912, 2560, 8)]


@pytest.mark.parametrize("N,K,seed", PACK_CASES)
def test_pack_parity(tw, N, K, seed):
    W = si.weights(N, K, seed=seed)
    p_ref, g_ref = oracle.pack_ternary(W)
    p_gpu, g_gpu = gpu_pack(tw, W)
    assert np.float32(g_gpu).view(np.uint32) == np.float32(g_ref).view(np.uint32)
    assert (p_gpu == p_ref).all()


@pytest.mark.parametrize("kind", ["zeros", "constant", "outliers", "wide", "ties"])
def test_pack_special(tw, kind):
    N, K = 37, 96
    if kind == "zeros":
        W = np.zeros((N, K), np.float32)
    elif kind == "constant":
        W = np.full((N, K), -0.3, np.float32)
    elif kind == "outliers":
        W = si.activations(N, K, seed=3, outliers=True)
    elif kind == "wide":
        W = wide_range(N, K, 4)
    else:  # many exact half-way quotients: W in multiples of gamma/2
        W = (np.random.default_rng(5).integers(-3, 4, size=(N, K)) * 0.5).astype(np.float32)
    p_ref, g_ref = oracle.pack_ternary(W)
    p_gpu, g_gpu = gpu_pack(tw, W)
    assert np.float32(g_gpu).view(np.uint32) == np.float32(g_ref).view(np.uint32)
    assert (p_gpu == p_ref).all()


def test_pack_repeatable_with_dirty_workspace(tw):
    W = si.weights(64, 256, seed=9)
    Wd = dev(W)
    ws = torch.full((tw.tw_pack_workspace_bytes(64, 256),), 0xAB, dtype=torch.uint8, device="cuda")
    packed = torch.empty((64, 64), dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(2):
        tw.tw_pack_ternary(Wd, packed, g, ws)
        outs.append((host(packed).copy(), host(g).copy()))
    p_ref, g_ref = oracle.pack_ternary(W)
    for p, gg in outs:
        assert (p == p_ref).all() and gg[0] == g_ref


# ----------------------------------------------------------------------------- activation quant
# 2 to 16 tokens with K >= 6144 take the cluster-shared kernel: 2 CTAs per token below 8192, 4
# below 16384, 8 above (K = 6148 and 16388: chunks that do not divide the row evenly)
ACT_CASES = [(1, 256, 0), (3, 68, 1), (16, 2560, 2), (17, 64, 3), (64, 4, 4), (65, 6912, 5),
             (1, 28672, 6), (2, 12, 7), (4, 4096, 8), (7, 6912, 9), (3, 6148, 10), (5, 8192, 11),
             (16, 12288, 12), (2, 16388, 13), (2, 65472, 14), (17, 8192, 15)]


@pytest.mark.parametrize("M,K,seed", ACT_CASES)
@pytest.mark.parametrize("outliers", [False, True])
def test_quant_act_parity(tw, M, K, seed, outliers):
    x = si.activations(M, K, seed=seed, outliers=outliers)
    q_ref, s_ref, sum_ref = oracle.quant_act(x)
    q, s, sm = tw.quantize(dev(x))
    assert (host(q) == q_ref).all()
    assert (host(s).view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (host(sm) == sum_ref).all()


@pytest.mark.parametrize("M,K,seed", ACT_CASES)
def test_rmsnorm_quant_act_parity(tw, M, K, seed):
    x = si.activations(M, K, seed=seed, outliers=(seed % 2 == 0))
    g = si.rms_gain(K, seed=seed)
    q_ref, s_ref, sum_ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
    q, s, sm = tw.quantize(dev(x), dev(g), si.RMS_EPS)
    assert (host(q) == q_ref).all()
    assert (host(s).view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (host(sm) == sum_ref).all()


def special_rows(K=64):
    x = si.activations(6, K, seed=11)
    x[1] = 0.0                                          # all-zero token
    x[2] = wide_range(1, K, 12)[0]                      # exponents from 2^-140 to 2^60
    x[3] = np.float32(1e-40) * np.sign(x[3])            # subnormal values only
    x[4, :] = 0.0
    x[4, 5] = -3.0                                      # one-hot
    x[5] = np.array([127, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5] * (K // 8), np.float32)  # exact ties
    return x


def test_act_special_rows(tw):
    K = 64
    x = special_rows(K)
    g = si.rms_gain(K, seed=13)
    for use_rms in (False, True):
        if use_rms:
            ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
            got = tw.quantize(dev(x), dev(g), si.RMS_EPS)
        else:
            ref = oracle.quant_act(x)
            got = tw.quantize(dev(x))
        for a, b in zip(got, ref):
            assert (host(a).view(np.uint8) == b.view(np.uint8)).all(), use_rms


@pytest.mark.parametrize("K", [6912, 8192, 28672])
def test_act_special_rows_cluster(tw, K):
    """The special rows (six tokens) at row lengths the cluster-shared kernel takes (2, 4 and 8
    CTAs per token): all-zero, exponents 2^-140..2^60 and subnormal rows take the exact
    mean-square path in every CTA of the cluster; one-hot and exact ties."""
    x = special_rows(K)
    x[4, :] = 0.0
    x[4, K - 3] = -3.0  # in the last CTA's chunk
    g = si.rms_gain(K, seed=13)
    for use_rms in (False, True):
        if use_rms:
            ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
            got = tw.quantize(dev(x), dev(g), si.RMS_EPS)
        else:
            ref = oracle.quant_act(x)
            got = tw.quantize(dev(x))
        for a, b in zip(got, ref):
            assert (host(a).view(np.uint8) == b.view(np.uint8)).all(), (K, use_rms)
    assert tw.tw_device_status() == 0


def near_tie_tokens(K=256, M=8, seed=0):
    """Tokens whose quotients x*127/max|x| sit on, or a few ulps either side of, the
    half-integers where round-half-even decides (the kernels take a fast reciprocal
    path away from them and the IEEE divide near them)."""
    rng = np.random.default_rng(seed)
    x = np.empty((M, K), np.float32)
    for m in range(M):
        a = np.float32(rng.uniform(0.5, 4.0))
        k = rng.integers(-127, 127, size=K).astype(np.float32) + np.float32(0.5)
        v = (k * a / np.float32(127.0)).astype(np.float32)
        steps = rng.integers(-3, 4, size=K)
        for i in range(K):
            for _ in range(abs(int(steps[i]))):
                v[i] = np.nextafter(v[i], np.float32(np.inf) if steps[i] > 0 else np.float32(-np.inf))
        v[0] = a if m % 2 == 0 else -a
        x[m] = v
    return x


def test_quant_near_rounding_ties(tw):
    x = near_tie_tokens()
    ref = oracle.quant_act(x)
    got = tw.quantize(dev(x))
    for a_, b_ in zip(got, ref):
        assert (host(a_).view(np.uint8) == b_.view(np.uint8)).all()
    W = si.weights(64, x.shape[1], seed=3)
    p_ref, g_ref = oracle.pack_ternary(W)
    for m0 in (0, 4):
        xs_ = x[m0:m0 + 4]
        q_ref, s_ref, _ = oracle.quant_act(xs_)
        y_ref, acc_ref = oracle.ternary_matmul(p_ref, g_ref, q_ref, s_ref)
        y, acc, xq, sx, _, _ = fused_run(tw, xs_, p_ref, g_ref, None)
        assert (xq == q_ref).all() and (acc == acc_ref).all()


@pytest.mark.parametrize("spread", [30, 32, 33, 40])
def test_rmsnorm_exponent_spread_edges(tw, spread):
    """Rows whose smallest nonzero element is 2^-spread below the largest: up to 2^-32 the
    kernels sum the squares in 128-bit fixed point, beyond it they take the exponent-bucket
    path; both must give the oracle's x_q and s_x bit for bit (standalone and fused)."""
    K, N = 256, 64
    x = si.activations(3, K, seed=spread)
    x[:, 0] = 1024.0
    x[:, 1] = np.float32(1024.0 * 2.0 ** -spread)
    x[1, 2] = np.float32(1024.0 * 2.0 ** -spread * 1.5)
    x[2] *= np.float32(2.0 ** -120)          # the same spread near the bottom of the range
    g = si.rms_gain(K, seed=spread)
    ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
    got = tw.quantize(dev(x), dev(g), si.RMS_EPS)
    for a_, b_ in zip(got, ref):
        assert (host(a_).view(np.uint8) == b_.view(np.uint8)).all()
    W = si.weights(N, K, seed=spread + 1)
    p_ref, g_ref = oracle.pack_ternary(W)
    y_ref, acc_ref = oracle.ternary_matmul(p_ref, g_ref, ref[0], ref[1])
    y, acc, xq, sx, xs, _ = fused_run(tw, x, p_ref, g_ref, g)
    assert (xq == ref[0]).all() and (sx.view(np.uint32) == ref[1].view(np.uint32)).all()
    assert (acc == acc_ref).all()
    assert_y_close(y, y_ref)


# ----------------------------------------------------------------------------- GEMV / matmul
def product_case(M, N, K, seed, outliers=False):
    W, x = si.gemv_case(M, N, K, seed=seed, outliers=outliers)
    packed, gamma = oracle.pack_ternary(W)
    xq, sx, xs = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
    return packed, gamma, xq, sx, xs, y_ref, acc_ref


def run_product(tw, fn, packed, gamma, xq, sx, xs=None):
    M, N = xq.shape[0], packed.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    g = dev(np.array([gamma], np.float32))
    getattr(tw, fn)(dev(packed), g, dev(xq), dev(sx), y, None if xs is None else dev(xs), acc)
    return host(y), host(acc)


GEMV_SHAPES = [(256, 256), (7, 68), (1, 4), (33, 64), (100, 80), (640, 2560), (37, 6912)]


@pytest.mark.parametrize("N,K", GEMV_SHAPES)
@pytest.mark.parametrize("M", list(range(1, 17)))
def test_gemv_parity(tw, M, N, K):
    case = product_case(M, N, K, seed=M * 100 + N % 97, outliers=(M % 3 == 0))
    packed, gamma, xq, sx, xs, y_ref, acc_ref = case
    y, acc = run_product(tw, "tw_ternary_gemv", packed, gamma, xq, sx)
    assert (acc == acc_ref).all()
    assert_y_close(y, y_ref)
    # with the activation sums supplied by the caller
    y2, acc2 = run_product(tw, "tw_ternary_gemv", packed, gamma, xq, sx, xs)
    assert (acc2 == acc_ref).all() and (y2 == y).all()


@pytest.mark.parametrize("M", [17, 31, 63, 64, 65, 128, 256])
@pytest.mark.parametrize("N,K", [(256, 256), (7, 68), (130, 64), (200, 2560)])
def test_matmul_parity(tw, M, N, K):
    packed, gamma, xq, sx, xs, y_ref, acc_ref = product_case(M, N, K, seed=M + N, outliers=True)
    y, acc = run_product(tw, "tw_ternary_matmul", packed, gamma, xq, sx)
    assert (acc == acc_ref).all()
    assert_y_close(y, y_ref)


def test_gemv_zero_rows_and_negation(tw):
    M, N, K = 4, 48, 256
    W, x = si.gemv_case(M, N, K, seed=17)
    W[5] = 0.0
    for Wv in (W, -W):
        packed, gamma = oracle.pack_ternary(Wv)
        xq, sx, _ = oracle.quant_act(x)
        y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
        y, acc = run_product(tw, "tw_ternary_gemv", packed, gamma, xq, sx)
        assert (acc == acc_ref).all() and (acc[:, 5] == 0).all() and (y[:, 5] == 0).all()
        assert_y_close(y, y_ref)


def test_gemv_extreme_activations(tw):
    # x_q = -128 and +127 everywhere: the largest |acc| the int8 range allows
    N, K = 64, 4096
    W = si.weights(N, K, seed=19)
    packed, gamma = oracle.pack_ternary(W)
    for val in (-128, 127):
        xq = np.full((2, K), val, np.int8)
        sx = np.array([1.0, 3.0], np.float32)
        y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
        y, acc = run_product(tw, "tw_ternary_gemv", packed, gamma, xq, sx)
        assert (acc == acc_ref).all()
        assert_y_close(y, y_ref)


# ----------------------------------------------------------------------------- fused quant + GEMV
FUSED_SHAPES = [(256, 256), (37, 6912), (640, 2560), (1, 64), (149, 128), (300, 28672), (13824, 2560)]


def fused_run(tw, x, p_ref, g_ref, g=None):
    M, K = x.shape
    N = p_ref.shape[0]
    packed, gamma = dev(p_ref), dev(np.array([g_ref], np.float32))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    xs = torch.empty(M, dtype=torch.int32, device="cuda")
    tw.tw_quant_gemv(dev(x), packed, gamma, y, g=None if g is None else dev(g), eps=si.RMS_EPS,
                     x_q=xq, s_x=sx, x_sum=xs, acc_out=acc)
    y2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tw.tw_quant_gemv(dev(x), packed, gamma, y2, g=None if g is None else dev(g), eps=si.RMS_EPS)
    return host(y), host(acc), host(xq), host(sx), host(xs), host(y2)


@pytest.mark.parametrize("N,K", FUSED_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("rms", [False, True])
def test_quant_gemv_parity(tw, M, N, K, rms):
    """Every shape at 1..4 tokens, with and without RMSNorm.  Above 4 M weights with more
    than one token the oracle computes 512 sampled rows (the GPU computes all of them)."""
    W, x = si.gemv_case(M, N, K, seed=N + K + M, outliers=(M % 2 == 0))
    g = si.rms_gain(K, seed=K) if rms else None
    p_ref, g_ref = oracle.pack_ternary(W)
    if rms:
        q_ref, s_ref, sum_ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
    else:
        q_ref, s_ref, sum_ref = oracle.quant_act(x)
    rows = np.arange(N)
    if N * K > 4_000_000 and M > 1:
        rows = np.sort(np.random.default_rng(N + M).choice(N, min(N, 512), replace=False))
    y_ref, acc_ref = oracle.ternary_matmul(p_ref[rows], g_ref, q_ref, s_ref)
    try:
        y, acc, xq, sx, xs, y2 = fused_run(tw, x, p_ref, g_ref, g)
    except tw.TWError as err:
        # the documented refusal: several tokens of very long rows do not fit the fused
        # kernel's shared memory (the separate quantisation + GEMV calls take them)
        assert err.status == tw.TW_ERR_UNSUPPORTED and M > 1 and K >= 28672, err
        return
    assert (xq == q_ref).all()
    assert (sx.view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (xs == sum_ref).all()
    assert (acc[:, rows] == acc_ref).all()
    assert_y_close(y[:, rows], y_ref)
    assert (y2 == y).all()
    assert tw.tw_device_status() == 0


@pytest.mark.parametrize("N,K,rms", [(30000, 2560, True), (30000, 2560, False), (8000, 8192, True),
                                     (9001, 8192, False), (2500, 14336, False), (30000, 4096, True)])
def test_quant_gemv_one_token_large_blocks(tw, N, K, rms):
    """One token, quantisation fused, on matrices whose CTA block exceeds the one-token
    kernel's shared memory (the streaming kernel takes them): K = 2560 to 14336, with and
    without RMSNorm, row counts that do not divide evenly over the CTAs.  Every output against
    the oracle."""
    W, x = si.gemv_case(1, N, K, seed=N + K, outliers=True)
    g = si.rms_gain(K, seed=K + 1) if rms else None
    p_ref, g_ref = oracle.pack_ternary(W)
    if rms:
        q_ref, s_ref, sum_ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
    else:
        q_ref, s_ref, sum_ref = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(p_ref, g_ref, q_ref, s_ref, openmp=True)
    y, acc, xq, sx, xs, y2 = fused_run(tw, x, p_ref, g_ref, g)
    assert (xq == q_ref).all() and (xs == sum_ref).all()
    assert (sx.view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (acc == acc_ref).all()
    assert_y_close(y, y_ref)
    assert (y2 == y).all()
    assert tw.tw_device_status() == 0


@pytest.mark.parametrize("N,K", [(9500, 6144), (6500, 8192), (5000, 12288), (3500, 16384)])
def test_stream_one_token_several_batches(tw, N, K):
    """One token on the streaming kernel with six words per lane and row and several batches
    of rows per warp group (two CTAs per SM; with RMSNorm at K >= 8192 in clusters).  The
    product on a given x_q and the fused launch with and without RMSNorm, every output
    against the oracle (the 70B gate|up takes this path in tests/test_fullsize_gpu.py)."""
    W, x = si.gemv_case(1, N, K, seed=N + 3 * K, outliers=True)
    p_ref, g_ref = oracle.pack_ternary(W)
    rows = np.arange(N)
    packed, gamma = dev(p_ref), dev(np.array([g_ref], np.float32))
    q_ref, s_ref, sum_ref = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(p_ref[rows], g_ref, q_ref, s_ref, openmp=True)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    acc = torch.empty((1, N), dtype=torch.int32, device="cuda")
    tw.tw_ternary_gemv(packed, gamma, dev(q_ref), dev(s_ref), y, dev(sum_ref), acc)
    assert (host(acc)[:, rows] == acc_ref).all()
    assert_y_close(host(y)[:, rows], y_ref)
    for g in (None, si.rms_gain(K, seed=K + 9)):
        if g is not None:
            q_ref, s_ref, _ = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
            y_ref, acc_ref = oracle.ternary_matmul(p_ref[rows], g_ref, q_ref, s_ref, openmp=True)
        yf, accf, xq, sx, _, y2 = fused_run(tw, x, p_ref, g_ref, g)
        assert (xq == q_ref).all() and (sx.view(np.uint32) == s_ref.view(np.uint32)).all()
        assert (accf[:, rows] == acc_ref).all()
        assert_y_close(yf[:, rows], y_ref)
        assert (y2 == yf).all()
    assert tw.tw_device_status() == 0


def test_quant_gemv_special_rows(tw):
    K, N = 64, 40
    x = special_rows(K)
    W = si.weights(N, K, seed=70)
    p_ref, g_ref = oracle.pack_ternary(W)
    g = si.rms_gain(K, seed=71)
    for m0 in range(0, 6, 3):
        xs_ = x[m0:m0 + 3]
        for gg in (None, g):
            if gg is None:
                q_ref, s_ref, _ = oracle.quant_act(xs_)
            else:
                q_ref, s_ref, _ = oracle.rmsnorm_quant_act(xs_, gg, si.RMS_EPS)
            y_ref, acc_ref = oracle.ternary_matmul(p_ref, g_ref, q_ref, s_ref)
            y, acc, xq, sx, _, _ = fused_run(tw, xs_, p_ref, g_ref, gg)
            assert (xq == q_ref).all() and (sx.view(np.uint32) == s_ref.view(np.uint32)).all()
            assert (acc == acc_ref).all()
            assert_y_close(y, y_ref)


def test_quant_gemv_chain_pdl(tw):
    """Back-to-back fused launches (programmatic dependent launch) in a graph: each launch
    reads the previous launch's output as its input, so a missing wait would show up."""
    N = K = 2560
    Ws = [si.weights(N, K, seed=50 + i) for i in range(6)]
    packs = [oracle.pack_ternary(W) for W in Ws]
    x0 = si.activations(1, K, seed=60)
    g = si.rms_gain(K, seed=61)
    ref = [x0]
    for p, gm in packs:
        q, s, _ = oracle.rmsnorm_quant_act(ref[-1], g, si.RMS_EPS)
        y, _ = oracle.ternary_matmul(p, gm, q, s)
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


def _decode_case_check(tw, x, g, N=640, seed=0):
    """One-token fused launch (RMSNorm) on x [1][K] with gain g, against the oracle."""
    K = x.shape[1]
    W = si.weights(N, K, seed=seed)
    p_ref, g_ref = oracle.pack_ternary(W)
    q_ref, s_ref, sum_ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
    y_ref, acc_ref = oracle.ternary_matmul(p_ref, g_ref, q_ref, s_ref)
    y, acc, xq, sx, xs, y2 = fused_run(tw, x, p_ref, g_ref, g)
    assert (xq == q_ref).all()
    assert (sx.view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (xs == sum_ref).all() and (acc == acc_ref).all()
    assert_y_close(y, y_ref)
    assert (y2 == y).all()


def _inv_rms_f32(x_row, eps):
    """fl32 RMSNorm scale of one row, for building test inputs (not a check): exact sum of
    squares (math.fsum of exact double squares), one rounding to fp32 of the mean, IEEE
    fp32 square root and divide."""
    import math
    f32 = np.float32
    ms = f32(math.fsum(float(v) * float(v) for v in x_row) / len(x_row))
    return f32(1.0) / np.sqrt(f32(ms + f32(eps)))


def test_decode_scale_candidate_not_the_maximum(tw):
    """One token with RMSNorm: the element with the largest fl(|x g|) is not the one with the
    largest |u| = fl(fl(x inv) g) (two products a fraction of an ulp apart whose roundings
    cross).  The one-token kernel takes the first as its candidate scale and must notice
    that another |u| exceeds it."""
    f32 = np.float32
    K = 2560
    rng = np.random.default_rng(11)
    x = si.activations(1, K, seed=901)
    g = si.rms_gain(K, seed=902)
    i, j = 100, 1700
    for _ in range(200000):
        xi, gi = f32(rng.uniform(7, 9)), f32(rng.uniform(1.1, 1.3))
        xj = f32(xi * (1 + rng.uniform(-3, 3) * 2.0 ** -23))
        gj = f32(gi * (1 + rng.uniform(-3, 3) * 2.0 ** -23))
        x[0, i], g[i], x[0, j], g[j] = xi, gi, xj, gj
        inv = _inv_rms_f32(x[0], si.RMS_EPS)
        p_i, p_j = abs(f32(xi * gi)), abs(f32(xj * gj))
        u_i, u_j = abs(f32(f32(xi * inv) * gi)), abs(f32(f32(xj * inv) * gj))
        if p_i > p_j and u_j > u_i:
            break
    else:
        pytest.fail("no crossing pair found")
    assert np.abs(x[0] * g).argmax() == i  # the candidate is element i ...
    _decode_case_check(tw, x, g)
    _, s_ref, _ = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
    assert s_ref[0] == u_j  # ... and the scale is element j's


@pytest.mark.parametrize("kind", ["underflow", "ties", "zero_gain"])
def test_decode_scale_edge_rows(tw, kind):
    """One token with RMSNorm where the products |x g| tell nothing about max |u|: they
    underflow to zero while u does not; many exactly equal products; an all-zero gain."""
    K = 2560
    x = si.activations(1, K, seed=903)
    g = si.rms_gain(K, seed=904)
    if kind == "underflow":  # |x g| < 2^-150 but x inv g is a nonzero subnormal or small normal
        x = (x * np.float32(5e-21)).astype(np.float32)
        g = (g * np.float32(1e-26)).astype(np.float32)
        assert (np.float32(np.abs(x) * np.abs(g)) == 0).all()
    elif kind == "ties":  # every |x| equal: all products tie in exact arithmetic on 1/g
        x = np.where(x >= 0, np.float32(3.0), np.float32(-3.0)).astype(np.float32)
        g = np.float32(0.75) * np.ones(K, np.float32)
        g[::7] = np.float32(0.7500001)
    else:
        g = np.zeros(K, np.float32)
    _decode_case_check(tw, x, g)


@pytest.mark.parametrize("M", [1, 2, 4])
def test_long_stream_two_ctas_per_sm(tw, M):
    """A matrix with more rows than one register batch of every warp (the kernel then runs
    two CTAs per SM and loads later batches inside the loop): full comparison."""
    N, K = 20000, 2560
    W, x = si.gemv_case(M, N, K, seed=123 + M)
    p_ref, g_ref = oracle.pack_ternary(W)
    q_ref, s_ref, sum_ref = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(p_ref, g_ref, q_ref, s_ref)
    y, acc = run_product(tw, "tw_ternary_gemv", p_ref, g_ref, q_ref, s_ref)
    assert (acc == acc_ref).all()
    assert_y_close(y, y_ref)
    yf, accf, xq, _, _, _ = fused_run(tw, x, p_ref, g_ref, None)
    assert (xq == q_ref).all() and (accf == acc_ref).all()
    assert_y_close(yf, y_ref)


# ----------------------------------------------------------------------------- full decode layer (2B)
def test_2b_layer_full_parity(tw):
    """Every GEMV of a 2B-shaped decoder layer at M = 1, fully compared (fused q|k|v and gate|up)."""
    shapes = si.fused_layer_shapes("2B")
    g = si.cpu_generator(2024)
    for name, (N, K) in shapes.items():
        W = si.weights(N, K, gen=g)
        x = si.activations(1, K, gen=g)
        p_ref, g_ref = oracle.pack_ternary(W)
        p_gpu, g_gpu = gpu_pack(tw, W)
        assert g_gpu == g_ref and (p_gpu == p_ref).all(), name
        if name in ("qkv", "gateup"):
            gain = si.rms_gain(K, seed=5)
            xq_ref, sx_ref, xs_ref = oracle.rmsnorm_quant_act(x, gain, si.RMS_EPS)
            xq, sx, xs = tw.quantize(dev(x), dev(gain), si.RMS_EPS)
        else:
            gain = None
            xq_ref, sx_ref, xs_ref = oracle.quant_act(x)
            xq, sx, xs = tw.quantize(dev(x))
        assert (host(xq) == xq_ref).all() and (host(sx) == sx_ref).all() and (host(xs) == xs_ref).all()
        y_ref, acc_ref = oracle.ternary_matmul(p_ref, g_ref, xq_ref, sx_ref)
        y, acc = run_product(tw, "tw_ternary_gemv", p_ref, g_ref, xq_ref, sx_ref, xs_ref)
        assert (acc == acc_ref).all(), name
        assert_y_close(y, y_ref)
        yf, accf, _, _, _, _ = fused_run(tw, x, p_ref, g_ref, gain)
        assert (accf == acc_ref).all(), name
        assert_y_close(yf, y_ref)


# ----------------------------------------------------------------------------- graph capture
def test_graph_capture_replay(tw):
    M, N, K = 1, 512, 2560
    W, x = si.gemv_case(M, N, K, seed=23)
    packed, gamma = tw.pack(dev(W))
    xd = dev(x)
    gain = dev(si.rms_gain(K, seed=23))
    x_q = torch.empty((M, K), dtype=torch.int8, device="cuda")
    s_x = torch.empty(M, dtype=torch.float32, device="cuda")
    x_sum = torch.empty(M, dtype=torch.int32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        tw.tw_rmsnorm_quant_act(xd, gain, si.RMS_EPS, x_q, s_x, x_sum)
        tw.tw_ternary_gemv(packed, gamma, x_q, s_x, y, x_sum)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        tw.tw_rmsnorm_quant_act(xd, gain, si.RMS_EPS, x_q, s_x, x_sum)
        tw.tw_ternary_gemv(packed, gamma, x_q, s_x, y, x_sum)
    y.zero_()
    graph.replay()
    p_ref, g_ref = oracle.pack_ternary(W)
    xq_ref, sx_ref, _ = oracle.rmsnorm_quant_act(x, si.rms_gain(K, seed=23), si.RMS_EPS)
    y_ref, _ = oracle.ternary_matmul(p_ref, g_ref, xq_ref, sx_ref)
    assert_y_close(host(y), y_ref)


# ----------------------------------------------------------------------------- error paths on a GPU
def test_host_pointers_rejected(tw):
    lib = tw.lib()
    K, N = 64, 8
    xq_host = np.zeros((1, K), np.int8)
    pinned = torch.zeros((1, K), dtype=torch.int8).pin_memory()
    packed = torch.zeros((N, K // 4), dtype=torch.uint8, device="cuda")
    g = torch.ones(1, device="cuda")
    sx = torch.ones(1, device="cuda")
    y = torch.empty((1, N), device="cuda")
    for bad in (xq_host.ctypes.data, pinned.data_ptr()):
        st = lib.tw_ternary_gemv(packed.data_ptr(), g.data_ptr(), bad, sx.data_ptr(), None, 1, N, K,
                                 y.data_ptr(), None, None)
        assert st == tw.TW_ERR_NOT_DEVICE_PTR
    torch.cuda.synchronize()


def _near_mean_square_midpoint(rng, K, scale, big):
    """A row whose mean square lies within about 2^-35 (relative) of an fp32 rounding
    midpoint: the fused prologue's float-float path must either decide it correctly or
    hand it to the exact path."""
    from fractions import Fraction
    x = (rng.standard_normal(K) * scale).astype(np.float32)
    if big:
        x[-1] = np.float32(scale * 30.0)
    rest = sum(Fraction(float(v)) ** 2 for v in x[:-1])
    ms = np.float32(float((rest + Fraction(float(x[-1])) ** 2) / K))
    mid = Fraction(float(ms)) + Fraction(float(np.spacing(ms))) / 2
    need = mid * K - rest
    if need > 0:
        x[-1] = np.float32(float(need) ** 0.5)
    return x


def test_rmsnorm_mean_square_near_midpoints(tw):
    rng = np.random.default_rng(2026)
    K, N = 2560, 256
    rows = [_near_mean_square_midpoint(rng, K, s, b) for s in (0.01, 1.0, 50.0) for b in (False, True)]
    W = si.weights(N, K, seed=99)
    p_ref, g_ref = oracle.pack_ternary(W)
    g = si.rms_gain(K, seed=98)
    for i in range(0, len(rows), 3):
        x = np.stack(rows[i:i + 3])
        ref = oracle.rmsnorm_quant_act(x, g, si.RMS_EPS)
        got = tw.quantize(dev(x), dev(g), si.RMS_EPS)
        for a_, b_ in zip(got, ref):
            assert (host(a_).view(np.uint8) == b_.view(np.uint8)).all()
        y_ref, acc_ref = oracle.ternary_matmul(p_ref, g_ref, ref[0], ref[1])
        y, acc, xq, sx, xs, _ = fused_run(tw, x, p_ref, g_ref, g)
        assert (xq == ref[0]).all() and (sx.view(np.uint32) == ref[1].view(np.uint32)).all()
        assert (acc == acc_ref).all()
        assert_y_close(y, y_ref)
