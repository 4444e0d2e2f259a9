"""tw_pack_ternary_noalloc: packing for callers that cannot allocate device memory.

Some callers (a plug-in inside a framework that owns every device allocation, a
service with memory pools fixed at start-up) cannot hand the packer a workspace.
This entry point keeps its scratch in the library's own device memory.  Its results
must equal those of tw_pack_ternary (bit-exact: packed bytes and the scale's bits),
on two calls in a row, since the scratch keeps the previous call's contents.

Collected last on purpose (file name), so that a run stopping at the first failure
has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu


def _lib():
    import ternary_weight_quant_b300 as tw
    return tw, tw.lib()


def _pack_with_workspace(tw, W):
    N, K = W.shape
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(tw.tw_pack_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    tw.tw_pack_ternary(W, packed, scale, ws)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scale.cpu().numpy().view(np.uint32)[0]


def _pack_noalloc_raw(lib, W):
    N, K = W.shape
    packed = torch.full((N, K // 4), 0xEE, dtype=torch.uint8, device="cuda")
    scale = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.tw_pack_ternary_noalloc(ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_void_p(packed.data_ptr()),
                                     ctypes.c_void_p(scale.data_ptr()), ctypes.c_void_p(stream))
    torch.cuda.synchronize()
    return st, packed.cpu().numpy(), scale.cpu().numpy().view(np.uint32)[0]


@pytest.mark.parametrize("N,K,seed", [(256, 256, 0), (6912, 2560, 1), (7, 68, 2)])
def test_noalloc_matches_workspace_entry_point_twice(N, K, seed):
    tw, lib = _lib()
    W = si.device_normal((N, K), seed=seed)
    ref_packed, ref_scale = _pack_with_workspace(tw, W)
    for _ in range(2):  # the second call starts from the first call's scratch contents
        st, packed, scale = _pack_noalloc_raw(lib, W)
        assert st == tw.TW_OK, lib.tw_status_string(st).decode()
        assert scale == ref_scale
        assert (packed == ref_packed).all()


def test_noalloc_after_a_different_tensor():
    tw, lib = _lib()
    Wa = si.device_normal((512, 1024), seed=11)
    Wb = 3.0 * si.device_normal((300, 640), seed=12)
    st_a, packed_a, scale_a = _pack_noalloc_raw(lib, Wa)  # leaves Wa's histogram in the scratch
    ref_packed_a, ref_scale_a = _pack_with_workspace(tw, Wa)
    assert st_a == tw.TW_OK and scale_a == ref_scale_a and (packed_a == ref_packed_a).all()
    st, packed, scale = _pack_noalloc_raw(lib, Wb)
    ref_packed, ref_scale = _pack_with_workspace(tw, Wb)
    assert st == tw.TW_OK and scale == ref_scale and (packed == ref_packed).all()


def test_noalloc_rejects_bad_sizes():
    tw, lib = _lib()
    W = torch.zeros((4, 16), dtype=torch.float32, device="cuda")
    out = torch.empty(16, dtype=torch.uint8, device="cuda")
    sc = torch.empty(1, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert lib.tw_pack_ternary_noalloc(p(W), 1 << 30, 1 << 12, p(out), p(sc), None) == tw.TW_ERR_SHAPE
    assert lib.tw_pack_ternary_noalloc(p(W), 4, 18, p(out), p(sc), None) == tw.TW_ERR_SHAPE
    assert lib.tw_pack_ternary_noalloc(None, 4, 16, p(out), p(sc), None) == tw.TW_ERR_NULL
