"""Python binding of libtw.so: the W1.58A8 ternary-weight product on one B300.

Thin ctypes marshalling only: every function takes torch CUDA tensors (or raw
device addresses), passes their pointers and sizes to the C entry point of the
same name, and raises TWError on a non-zero status.  All arithmetic runs in the
CUDA kernels of libtw.so; there is no CPU path.  If libtw.so is missing or cannot
be loaded, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtw.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "ternary_w158a8.h")

TW_OK, TW_ERR_NULL, TW_ERR_SHAPE, TW_ERR_ALIGN, TW_ERR_NOT_DEVICE_PTR = 0, 1, 2, 3, 4
TW_ERR_CUDA, TW_ERR_UNSUPPORTED, TW_ERR_TIMEOUT, TW_ERR_WORKSPACE = 5, 6, 7, 8
GEMV_MAX_M = 16
QUANT_GEMV_MAX_M = 4
MAX_K = 65532


class TWError(RuntimeError):
    def __init__(self, status: int, fn: str):
        super().__init__(f"{fn}: {_lib.tw_status_string(status).decode()}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtw.so not built at {LIB_PATH}; run __graft_entry__.build() "
                          "or python ternary_weight_quant_b300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    p, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    sigs = {
        "tw_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "tw_version": ([], ctypes.c_int),
        "tw_pack_workspace_bytes": ([i64, i64], sz),
        "tw_pack_ternary": ([p, i64, i64, p, p, p, sz, p], ctypes.c_int),
        "tw_pack_ternary_noalloc": ([p, i64, i64, p, p, p], ctypes.c_int),
        "tw_quant_act": ([p, i64, i64, p, p, p, p], ctypes.c_int),
        "tw_rmsnorm_quant_act": ([p, p, ctypes.c_float, i64, i64, p, p, p, p], ctypes.c_int),
        "tw_ternary_gemv": ([p, p, p, p, p, i64, i64, i64, p, p, p], ctypes.c_int),
        "tw_ternary_gemm": ([p, p, p, p, p, i64, i64, i64, p, p, p, sz, p], ctypes.c_int),
        "tw_ternary_matmul": ([p, p, p, p, p, i64, i64, i64, p, p, p, sz, p], ctypes.c_int),
        "tw_gemm_workspace_bytes": ([i64, i64], sz),
        "tw_quant_gemv": ([p, p, ctypes.c_float, p, p, i64, i64, i64, p, p, p, p, p, p], ctypes.c_int),
        "tw_device_status": ([p], ctypes.c_int),
        "tw_epilogue_workspace_bytes": ([], sz),
        "tw_quant_gemv_residual": ([p, p, ctypes.c_float, p, p, i64, i64, p, p, p, p, p, p, sz, p], ctypes.c_int),
        "tw_quant_gemv_stats": ([p, p, ctypes.c_float, p, p, p, i64, i64, p, p, p, p, p, p], ctypes.c_int),
        "tw_debug_gemm_abort": ([ctypes.c_int], ctypes.c_int),
        "tw_t5_row_bytes": ([i64], sz),
        "tw_pack_ternary_t5": ([p, i64, i64, p, p, p, sz, p], ctypes.c_int),
        "tw_ternary_gemv_t5": ([p, p, p, p, i64, i64, i64, p, p, p], ctypes.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def lib():
    """The loaded ctypes library (raw entry points, raw pointers)."""
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name, *args):
    st = getattr(_lib, name)(*args)
    if st != TW_OK:
        raise TWError(st, name)


def tw_pack_workspace_bytes(N: int, K: int) -> int:
    return int(_lib.tw_pack_workspace_bytes(N, K))


def tw_pack_ternary(W, packed, w_scale, workspace, N=None, K=None, stream=None):
    """W fp32 [N][K] -> packed uint8 [N][K/4], w_scale fp32 [1] (all device tensors)."""
    N = W.shape[0] if N is None else N
    K = W.shape[1] if K is None else K
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    _call("tw_pack_ternary", _ptr(W), N, K, _ptr(packed), _ptr(w_scale), _ptr(workspace), ws_bytes,
          _stream(stream))


def tw_pack_ternary_noalloc(W, packed, w_scale, N=None, K=None, stream=None):
    """tw_pack_ternary with the library's own device scratch (no workspace argument).

    For callers that cannot allocate device memory when they pack; calls that overlap
    on the GPU share one scratch array and must be serialised."""
    N = W.shape[0] if N is None else N
    K = W.shape[1] if K is None else K
    _call("tw_pack_ternary_noalloc", _ptr(W), N, K, _ptr(packed), _ptr(w_scale), _stream(stream))


def tw_quant_act(x, x_q, s_x, x_sum=None, M=None, K=None, stream=None):
    M = x.shape[0] if M is None else M
    K = x.shape[-1] if K is None else K
    _call("tw_quant_act", _ptr(x), M, K, _ptr(x_q), _ptr(s_x), _ptr(x_sum), _stream(stream))


def tw_rmsnorm_quant_act(x, g, eps, x_q, s_x, x_sum=None, M=None, K=None, stream=None):
    M = x.shape[0] if M is None else M
    K = x.shape[-1] if K is None else K
    _call("tw_rmsnorm_quant_act", _ptr(x), _ptr(g), float(eps), M, K, _ptr(x_q), _ptr(s_x), _ptr(x_sum),
          _stream(stream))


def _product(name, packed, w_scale, x_q, s_x, y, x_sum=None, acc_out=None, M=None, N=None, K=None,
             stream=None):
    M = x_q.shape[0] if M is None else M
    K = x_q.shape[-1] if K is None else K
    N = packed.shape[0] if N is None else N
    _call(name, _ptr(packed), _ptr(w_scale), _ptr(x_q), _ptr(s_x), _ptr(x_sum), M, N, K, _ptr(y),
          _ptr(acc_out), _stream(stream))


def tw_ternary_gemv(packed, w_scale, x_q, s_x, y, x_sum=None, acc_out=None, **kw):
    _product("tw_ternary_gemv", packed, w_scale, x_q, s_x, y, x_sum, acc_out, **kw)


def tw_gemm_workspace_bytes(M: int, K: int) -> int:
    return int(_lib.tw_gemm_workspace_bytes(M, K))


def _product_ws(name, packed, w_scale, x_q, s_x, y, x_sum=None, acc_out=None, workspace=None, M=None, N=None,
                K=None, stream=None):
    M = x_q.shape[0] if M is None else M
    K = x_q.shape[-1] if K is None else K
    N = packed.shape[0] if N is None else N
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    _call(name, _ptr(packed), _ptr(w_scale), _ptr(x_q), _ptr(s_x), _ptr(x_sum), M, N, K, _ptr(y),
          _ptr(acc_out), _ptr(workspace), ws_bytes, _stream(stream))


def tw_ternary_gemm(packed, w_scale, x_q, s_x, y, x_sum=None, acc_out=None, workspace=None, **kw):
    """Tensor-core product; workspace (optional, tw_gemm_workspace_bytes(M, K) bytes) speeds it up."""
    _product_ws("tw_ternary_gemm", packed, w_scale, x_q, s_x, y, x_sum, acc_out, workspace, **kw)


def tw_ternary_matmul(packed, w_scale, x_q, s_x, y, x_sum=None, acc_out=None, workspace=None, **kw):
    _product_ws("tw_ternary_matmul", packed, w_scale, x_q, s_x, y, x_sum, acc_out, workspace, **kw)


def tw_quant_gemv(x, packed, w_scale, y, g=None, eps=1e-6, x_q=None, s_x=None, x_sum=None, acc_out=None,
                  M=None, N=None, K=None, stream=None):
    """Fused (RMSNorm +) activation quantisation + ternary GEMV: x fp32 [M][K] -> y [M][N]."""
    M = x.shape[0] if M is None else M
    K = x.shape[-1] if K is None else K
    N = packed.shape[0] if N is None else N
    _call("tw_quant_gemv", _ptr(x), _ptr(g), float(eps), _ptr(packed), _ptr(w_scale), M, N, K, _ptr(y),
          _ptr(x_q), _ptr(s_x), _ptr(x_sum), _ptr(acc_out), _stream(stream))


def tw_epilogue_workspace_bytes() -> int:
    return int(_lib.tw_epilogue_workspace_bytes())


def epilogue_workspace(device="cuda"):
    """Allocate the workspace that carries the statistics from tw_quant_gemv_residual to
    tw_quant_gemv_stats."""
    return torch.empty(tw_epilogue_workspace_bytes(), dtype=torch.uint8, device=device)


def tw_quant_gemv_residual(x, packed, w_scale, h, h_out, g_next, workspace, g=None, eps=1e-6, y=None,
                           acc_out=None, N=None, K=None, stream=None):
    """One token: (RMSNorm +) quantisation + GEMV, then h_out = h + y and the partial
    statistics of the next RMSNorm (gain g_next) into workspace."""
    K = x.shape[-1] if K is None else K
    N = packed.shape[0] if N is None else N
    ws_bytes = workspace.numel() * workspace.element_size()
    _call("tw_quant_gemv_residual", _ptr(x), _ptr(g), float(eps), _ptr(packed), _ptr(w_scale), N, K, _ptr(h),
          _ptr(h_out), _ptr(g_next), _ptr(y), _ptr(acc_out), _ptr(workspace), ws_bytes, _stream(stream))


def tw_quant_gemv_stats(x, g, workspace, packed, w_scale, y, eps=1e-6, x_q=None, s_x=None, x_sum=None,
                        acc_out=None, N=None, K=None, stream=None):
    """One token: RMSNorm from the statistics a residual epilogue left + quantisation + GEMV."""
    K = x.shape[-1] if K is None else K
    N = packed.shape[0] if N is None else N
    _call("tw_quant_gemv_stats", _ptr(x), _ptr(g), float(eps), _ptr(workspace), _ptr(packed), _ptr(w_scale), N, K,
          _ptr(y), _ptr(x_q), _ptr(s_x), _ptr(x_sum), _ptr(acc_out), _stream(stream))


def tw_t5_row_bytes(K: int) -> int:
    """Bytes per row of the five-trits-per-byte layout (0 for a K the calls reject)."""
    return int(_lib.tw_t5_row_bytes(K))


def tw_pack_ternary_t5(W, packed5, w_scale, workspace, N=None, K=None, stream=None):
    """W fp32 [N][K] -> packed5 uint8 [N][tw_t5_row_bytes(K)] (five trits per byte), w_scale [1]."""
    N = W.shape[0] if N is None else N
    K = W.shape[1] if K is None else K
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    _call("tw_pack_ternary_t5", _ptr(W), N, K, _ptr(packed5), _ptr(w_scale), _ptr(workspace), ws_bytes,
          _stream(stream))


def tw_ternary_gemv_t5(packed5, w_scale, x_q, s_x, y, acc_out=None, M=None, N=None, K=None, stream=None):
    """The GEMV over five-trits-per-byte rows (1 or 2 tokens)."""
    M = x_q.shape[0] if M is None else M
    K = x_q.shape[-1] if K is None else K
    N = packed5.shape[0] if N is None else N
    _call("tw_ternary_gemv_t5", _ptr(packed5), _ptr(w_scale), _ptr(x_q), _ptr(s_x), M, N, K, _ptr(y),
          _ptr(acc_out), _stream(stream))


def tw_device_status() -> int:
    """Read and clear the device status word (0 or a TW_ERR_* code); synchronises the device."""
    out = ctypes.c_int32(0)
    _call("tw_device_status", ctypes.addressof(out))
    return int(out.value)


# ------------------------------------------------------------------ conveniences
def pack(W: torch.Tensor, stream=None):
    """Allocate outputs and pack a device fp32 [N][K] tensor. Returns (packed, w_scale)."""
    N, K = W.shape
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=W.device)
    w_scale = torch.empty(1, dtype=torch.float32, device=W.device)
    ws = torch.empty(max(tw_pack_workspace_bytes(N, K), 8), dtype=torch.uint8, device=W.device)
    tw_pack_ternary(W, packed, w_scale, ws, stream=stream)
    return packed, w_scale


def pack_t5(W: torch.Tensor, stream=None):
    """Allocate outputs and pack a device fp32 [N][K] tensor five trits per byte.
    Returns (packed5, w_scale)."""
    N, K = W.shape
    packed5 = torch.empty((N, tw_t5_row_bytes(K)), dtype=torch.uint8, device=W.device)
    w_scale = torch.empty(1, dtype=torch.float32, device=W.device)
    ws = torch.empty(max(tw_pack_workspace_bytes(N, K), 8), dtype=torch.uint8, device=W.device)
    tw_pack_ternary_t5(W, packed5, w_scale, ws, stream=stream)
    return packed5, w_scale


def quantize(x: torch.Tensor, g: torch.Tensor | None = None, eps: float = 1e-6, stream=None):
    """Allocate outputs and quantise a device fp32 [M][K] tensor (RMSNorm first if g is given)."""
    M, K = x.shape
    x_q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    s_x = torch.empty(M, dtype=torch.float32, device=x.device)
    x_sum = torch.empty(M, dtype=torch.int32, device=x.device)
    if g is None:
        tw_quant_act(x, x_q, s_x, x_sum, stream=stream)
    else:
        tw_rmsnorm_quant_act(x, g, eps, x_q, s_x, x_sum, stream=stream)
    return x_q, s_x, x_sum


def gemm_workspace(M: int, K: int, device="cuda"):
    """Allocate the optional tensor-core workspace for an M x K activation block."""
    return torch.empty(max(tw_gemm_workspace_bytes(M, K), 256), dtype=torch.uint8, device=device)


def matmul(packed, w_scale, x_q, s_x, x_sum=None, acc=False, workspace=None, stream=None):
    """Allocate y (and optionally acc) and run tw_ternary_matmul."""
    M, N = x_q.shape[0], packed.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x_q.device)
    a = torch.empty((M, N), dtype=torch.int32, device=x_q.device) if acc else None
    tw_ternary_matmul(packed, w_scale, x_q, s_x, y, x_sum, a, workspace=workspace, stream=stream)
    return (y, a) if acc else y
