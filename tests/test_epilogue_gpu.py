"""GPU parity of the fused epilogue against the CPU oracle (one decode token).

tw_quant_gemv_residual: the int32 accumulators, y (bit for bit: the epilogue forms y as the
definition states it) and h_out = fl32(h + y) (bit for bit).  tw_quant_gemv_stats, from the
partial statistics that call left: the next layer's x_q, s_x and sum x_q bit for bit and y
within 1e-6, against the oracle's RMSNorm + quantisation of the oracle's h_out.  Also: a
scale candidate below the true largest |u| (the quantisation must notice and redo), and two
decoder layers chained back to back under programmatic dependent launch.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

REL = 1e-6
EPS = si.RMS_EPS


@pytest.fixture(scope="module")
def tw():
    import ternary_weight_quant_b300 as tw
    return tw


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def residual_case(N, K, seed):
    """Weights [N][K], the token x [K], the residual stream h [N] (larger than y, as a
    decoder's residual stream is) and the next RMSNorm's gain [N]."""
    W, x = si.gemv_case(1, N, K, seed=seed, outliers=True)
    h = (4.0 * si.activations(1, N, seed=seed + 1)).ravel()
    g_next = si.rms_gain(N, seed=seed + 2)
    return W, x, h, g_next


def run_residual(tw, x, g, packed, gamma, h, g_next, ws):
    N = packed.shape[0]
    h_out = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    y = torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda")
    acc = torch.full((1, N), -7, dtype=torch.int32, device="cuda")
    tw.tw_quant_gemv_residual(dev(x), dev(packed), dev(np.array([gamma], np.float32)), dev(h), h_out, dev(g_next),
                              ws, g=None if g is None else dev(g), eps=EPS, y=y, acc_out=acc)
    return host(y), host(acc), h_out


def oracle_residual(x, g, packed, gamma, h):
    xq, sx, _ = oracle.quant_act(x) if g is None else oracle.rmsnorm_quant_act(x, g, EPS)
    y, acc = oracle.ternary_matmul(packed, gamma, xq, sx)
    return y, acc, oracle.residual_add(h, y.ravel())


@pytest.mark.parametrize("N,K,rms", [(2560, 2560, False), (2560, 6912, False), (2560, 2560, True),
                                     (640, 2560, True), (4096, 4096, False), (64, 64, True), (192, 1024, False)])
def test_residual_then_stats(tw, N, K, rms):
    """The residual call, then the next RMSNorm + quantisation + GEMV (N2 = 3 rows of length
    N) from the statistics it left."""
    W, x, h, g_next = residual_case(N, K, seed=N + K + rms)
    g = si.rms_gain(K, seed=9) if rms else None
    packed, gamma = oracle.pack_ternary(W)
    ws = tw.epilogue_workspace()
    y, acc, h_out = run_residual(tw, x, g, packed, gamma, h, g_next, ws)
    y_ref, acc_ref, h_ref = oracle_residual(x, g, packed, gamma, h)
    assert (acc == acc_ref).all()
    assert (bits(y) == bits(y_ref)).all(), "y is not the defined value"
    assert (bits(host(h_out)) == bits(h_ref)).all(), "h_out differs"
    N2 = 3
    p2, g2 = oracle.pack_ternary(si.weights(N2, N, seed=N + 1))
    y2 = torch.empty((1, N2), dtype=torch.float32, device="cuda")
    xq2 = torch.empty((1, N), dtype=torch.int8, device="cuda")
    sx2 = torch.empty(1, dtype=torch.float32, device="cuda")
    tw.tw_quant_gemv_stats(h_out, dev(g_next), ws, dev(p2), dev(np.array([g2], np.float32)), y2, eps=EPS, x_q=xq2,
                           s_x=sx2)
    q_ref, s_ref, _ = oracle.rmsnorm_quant_act(h_ref, g_next, EPS)
    assert (host(xq2) == q_ref).all() and bits(host(sx2)) == bits(s_ref)
    y2_ref, _ = oracle.ternary_matmul(p2, g2, q_ref, s_ref)
    assert (np.abs(host(y2).astype(np.float64) - y2_ref) <= REL * np.abs(y2_ref)).all()
    assert tw.tw_device_status() == 0


@pytest.mark.parametrize("N2", [3840, 13824, 2560, 7])
def test_stats_consumer_matches_oracle(tw, N2):
    """The residual call's h_out and statistics feed the next RMSNorm + GEMV (layer shapes)."""
    N, K = 2560, 2560
    W, x, h, g_next = residual_case(N, K, seed=N2)
    packed, gamma = oracle.pack_ternary(W)
    W2 = si.weights(N2, N, seed=N2 + 5)
    p2, g2 = oracle.pack_ternary(W2)
    ws = tw.epilogue_workspace()
    xd, hd, gnd = dev(x), dev(h), dev(g_next)
    h_out = torch.empty(N, dtype=torch.float32, device="cuda")
    tw.tw_quant_gemv_residual(xd, dev(packed), dev(np.array([gamma], np.float32)), hd, h_out, gnd, ws, eps=EPS)
    y2 = torch.empty((1, N2), dtype=torch.float32, device="cuda")
    acc2 = torch.empty((1, N2), dtype=torch.int32, device="cuda")
    xq2 = torch.empty((1, N), dtype=torch.int8, device="cuda")
    sx2 = torch.empty(1, dtype=torch.float32, device="cuda")
    xs2 = torch.empty(1, dtype=torch.int32, device="cuda")
    tw.tw_quant_gemv_stats(h_out, gnd, ws, dev(p2), dev(np.array([g2], np.float32)), y2, eps=EPS, x_q=xq2, s_x=sx2,
                           x_sum=xs2, acc_out=acc2)
    _, _, h_ref = oracle_residual(x, None, packed, gamma, h)
    q_ref, s_ref, sum_ref = oracle.rmsnorm_quant_act(h_ref, g_next, EPS)
    y2_ref, acc2_ref = oracle.ternary_matmul(p2, g2, q_ref, s_ref)
    assert (host(xq2) == q_ref).all()
    assert bits(host(sx2)) == bits(s_ref) and (host(xs2) == sum_ref).all()
    assert (host(acc2) == acc2_ref).all()
    yv = host(y2).astype(np.float64)
    assert (np.abs(yv - y2_ref) <= REL * np.abs(y2_ref)).all()
    assert tw.tw_device_status() == 0


def test_stats_consumer_redoes_a_low_candidate(tw):
    """Partials whose scale candidate is a small element (not the largest |u|): the
    quantisation finds elements above it and takes the true largest.  The partials are laid
    out as the residual epilogue writes them, one float4 per CTA of a launch over K outputs
    (min(K, SMs) of them): (sum of squares as hi + lo, candidate h, its gain g).  x holds
    multiples of 1/4 so that the sum of squares is exact in fp32 (hi = the sum, lo = 0)."""
    N, K = 3840, 2560
    rng = np.random.default_rng(44)
    h = (rng.integers(-40, 41, size=K) / 4.0).astype(np.float32)
    g = si.rms_gain(K, seed=42)
    W = si.weights(N, K, seed=43)
    p, gamma = oracle.pack_ternary(W)
    S = float(np.sum(h.astype(np.float64) ** 2))
    assert np.float32(S) == S
    k_small = int(np.argmin(np.abs(h) + (h == 0) * 100.0))  # a small nonzero element
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nparts = min(K, sms)
    parts = np.zeros((tw.tw_epilogue_workspace_bytes() // 16, 4), np.float32)
    parts[0] = [S, 0.0, h[k_small], g[k_small]]
    assert nparts <= parts.shape[0]
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    xq = torch.empty((1, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(1, dtype=torch.float32, device="cuda")
    tw.tw_quant_gemv_stats(dev(h), dev(g), dev(parts.view(np.uint8).ravel()), dev(p),
                           dev(np.array([gamma], np.float32)), y, eps=EPS, x_q=xq, s_x=sx)
    q_ref, s_ref, _ = oracle.rmsnorm_quant_act(h, g, EPS)
    y_ref, _ = oracle.ternary_matmul(p, gamma, q_ref, s_ref)
    u, _ = oracle.rmsnorm(h, g, EPS)
    assert abs(u.ravel()[k_small]) < np.abs(u).max()  # the candidate really is too small
    assert (host(xq) == q_ref).all() and bits(host(sx)) == bits(s_ref)
    assert (np.abs(host(y).astype(np.float64) - y_ref) <= REL * np.abs(y_ref)).all()


def test_two_layers_chained(tw):
    """o (residual) -> gate|up (statistics) -> down (residual) -> q|k|v (statistics) -> ...
    for two 2B-shaped layers, enqueued back to back in place on one residual buffer."""
    shapes = si.fused_layer_shapes("2B")
    hid = shapes["o"][0]
    rng_seed = 500
    h0 = (4.0 * si.activations(1, hid, seed=rng_seed)).ravel()
    hd = dev(h0)
    ws = tw.epilogue_workspace()
    ref_h = h0.copy()
    checks = []
    for layer in range(2):
        for name in ("o", "gateup", "down", "qkv"):
            N, K = shapes[name]
            seed = rng_seed + 10 * layer + len(checks)
            W = si.weights(N, K, seed=seed)
            p, gamma = oracle.pack_ternary(W)
            pd, gd = dev(p), dev(np.array([gamma], np.float32))
            if name in ("o", "down"):  # their input comes from outside the path: synthetic
                x = si.activations(1, K, seed=seed + 1)
                g_next = si.rms_gain(hid, seed=seed + 2)
                y = torch.empty((1, N), dtype=torch.float32, device="cuda")
                tw.tw_quant_gemv_residual(dev(x), pd, gd, hd, hd, dev(g_next), ws, eps=EPS, y=y)
                y_ref, _, ref_h = oracle_residual(x, None, p, gamma, ref_h)
                checks.append(("y_" + name, y, y_ref, True))
                checks.append(("h_" + name, hd.clone(), ref_h.copy(), True))
                last_g = g_next
            else:
                y = torch.empty((1, N), dtype=torch.float32, device="cuda")
                xq = torch.empty((1, K), dtype=torch.int8, device="cuda")
                tw.tw_quant_gemv_stats(hd, dev(last_g), ws, pd, gd, y, eps=EPS, x_q=xq)
                q_ref, s_ref, _ = oracle.rmsnorm_quant_act(ref_h, last_g, EPS)
                y_ref, _ = oracle.ternary_matmul(p, gamma, q_ref, s_ref)
                checks.append(("xq_" + name, xq, q_ref, True))
                checks.append(("y_" + name, y, y_ref, False))
    torch.cuda.synchronize()
    for what, got, ref, exact in checks:
        g_ = host(got).reshape(ref.shape)
        if exact:
            assert (g_.view(np.uint32 if g_.dtype == np.float32 else g_.dtype) ==
                    ref.view(np.uint32 if ref.dtype == np.float32 else ref.dtype)).all(), what
        else:
            assert (np.abs(g_.astype(np.float64) - ref) <= REL * np.abs(ref)).all(), what
    assert tw.tw_device_status() == 0
