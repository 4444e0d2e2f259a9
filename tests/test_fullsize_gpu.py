"""Parity at the benchmark's full 8B and 70B sizes, in the configuration bench.py times.

The weights are drawn on the device with the benchmark's seeded generator and packed
there; the oracle packs the same fp32 tensor on the host and every packed byte and the
scale's bits must match.  The fused decode launch (RMSNorm + quantisation + GEMV for the
q|k|v and gate|up shapes, quantisation + GEMV for o and down, M = 1) then runs over the
full matrix; x_q, s_x and Σx_q are compared whole and the outputs on 1 024 rows drawn at
random, which the oracle computes one by one.  These shapes reach the kernel paths the
small cases do not: more rows than one register batch per warp (two CTAs per SM, later
batches loaded inside the loop) and, for K = 14 336 and 28 672, activations too large to
stage in shared memory (every prologue pass reads them from global memory).
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

CASES = [("8B", "down"), ("8B", "gateup"), ("70B", "down"), ("70B", "gateup")]


@pytest.fixture(scope="module")
def tw():
    import ternary_weight_quant_b300 as m
    return m


@pytest.mark.parametrize("model,name", CASES)
def test_fullsize_sampled_rows(tw, model, name):
    N, K = si.fused_layer_shapes(model)[name]
    rms = name in ("qkv", "gateup")
    seed = 4100 + 10 * len(model) + len(name)
    W = si.device_normal((N, K), seed=seed)
    packed, gamma = tw.pack(W)
    W_h = W.cpu().numpy()
    del W
    p_ref, g_ref = oracle.pack_ternary(W_h)
    del W_h
    assert gamma.cpu().numpy().view(np.uint32)[0] == np.array([g_ref], np.float32).view(np.uint32)[0]
    assert np.array_equal(packed.cpu().numpy(), p_ref)

    x = si.activations(1, K, seed=seed + 1)
    gain = si.rms_gain(K, seed=seed + 2) if rms else None
    if rms:
        xq_ref, sx_ref, xs_ref = oracle.rmsnorm_quant_act(x, gain, si.RMS_EPS)
    else:
        xq_ref, sx_ref, xs_ref = oracle.quant_act(x)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    acc = torch.empty((1, N), dtype=torch.int32, device="cuda")
    xq = torch.empty((1, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(1, dtype=torch.float32, device="cuda")
    xs = torch.empty(1, dtype=torch.int32, device="cuda")
    tw.tw_quant_gemv(torch.from_numpy(x).cuda(), packed, gamma, y,
                     g=None if gain is None else torch.from_numpy(gain).cuda(), eps=si.RMS_EPS,
                     x_q=xq, s_x=sx, x_sum=xs, acc_out=acc)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert sx.cpu().numpy().view(np.uint32)[0] == sx_ref.view(np.uint32)[0]
    assert xs.cpu().numpy()[0] == xs_ref[0]

    rows = np.sort(np.random.default_rng(seed).choice(N, 1024, replace=False))
    y_ref, acc_ref = oracle.ternary_matmul(np.ascontiguousarray(p_ref[rows]), g_ref, xq_ref, sx_ref)
    acc_g = acc.cpu().numpy()[:, rows]
    y_g = y.cpu().numpy()[:, rows].astype(np.float64)
    assert np.array_equal(acc_g, acc_ref)
    assert not (np.abs(y_g - y_ref) > 1e-6 * np.abs(y_ref.astype(np.float64))).any()
    assert tw.tw_device_status() == 0
