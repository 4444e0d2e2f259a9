"""The tensor-core GEMM's failure handling, driven without a GPU fault.

tw_debug_gemm_abort(1) makes each GEMM launch start with its abort flag raised, the state a
bounded mbarrier wait leaves when it gives up: every role must stop before issuing work, the
copies already in flight must land, tensor memory must be released, no output may be
written, and tw_device_status must report TW_ERR_TIMEOUT.  Each of the three GEMM kernels is
driven (the tokens-on-M kernel with split-K clusters, the TMA kernel, the kernel for K not a
multiple of 64), and the next normal GEMM on the same context must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tw():
    import ternary_weight_quant_b300 as tw
    yield tw
    tw.lib().tw_debug_gemm_abort(0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("M,N,K,with_ws", [(64, 3840, 2560, True), (200, 2560, 2560, False), (40, 300, 80, False)])
def test_gemm_abort_path_then_normal(tw, M, N, K, with_ws):
    W, x = si.gemv_case(M, N, K, seed=M + N + K)
    packed, gamma = oracle.pack_ternary(W)
    xq, sx, _ = oracle.quant_act(x)
    y_ref, acc_ref = oracle.ternary_matmul(packed, gamma, xq, sx)
    pd, gd, xd, sd = dev(packed), dev(np.array([gamma], np.float32)), dev(xq), dev(sx)
    ws = tw.gemm_workspace(M, K) if with_ws else None
    assert tw.tw_device_status() == 0

    assert tw.lib().tw_debug_gemm_abort(1) == tw.TW_OK
    try:
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        acc = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
        tw.tw_ternary_gemm(pd, gd, xd, sd, y, acc_out=acc, workspace=ws)
        torch.cuda.synchronize()
        assert tw.tw_device_status() == tw.TW_ERR_TIMEOUT
        assert torch.isnan(y).all() and (acc == -7).all(), "an aborted launch wrote outputs"
    finally:
        assert tw.lib().tw_debug_gemm_abort(0) == tw.TW_OK

    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    tw.tw_ternary_gemm(pd, gd, xd, sd, y, acc_out=acc, workspace=ws)
    torch.cuda.synchronize()
    assert tw.tw_device_status() == 0
    assert (acc.cpu().numpy() == acc_ref).all()
    yv = y.cpu().numpy().astype(np.float64)
    assert (np.abs(yv - y_ref) <= 1e-6 * np.abs(y_ref)).all()
