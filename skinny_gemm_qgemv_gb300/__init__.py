"""Python binding of libqgemv, the GB300 (sm_103a) quantized GEMV library.

Thin ctypes marshalling over the C ABI in ``include/qgemv.h``: every function
takes CUDA tensors, passes their device pointers and the current torch stream,
and raises on a non-OK status. All arithmetic runs in the library's kernels;
there is no fallback path. PyTorch only supplies device memory and streams.

Entry points (same names as the C ABI):
  qgemv_w4a16, qgemm_w4a16_skinny, moe_mxfp4_expert_forward,
  hadamard32_quant_i8, gemm_w8a8_i32; GemvGroup wraps qgemv_w4a16_group_* and
  SkinnyGroup qgemm_w4a16_skinny_group_*
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemv.so")

QG_OK = 0
_STATUS = {0: "QG_OK", 1: "QG_ERR_INVALID_ARG", 2: "QG_ERR_MISALIGNED", 3: "QG_ERR_UNSUPPORTED",
           4: "QG_ERR_WORKSPACE", 5: "QG_ERR_CUDA", 6: "QG_ERR_DEVICE_TIMEOUT"}

EXPORTS = [
    "qg_status_string", "qg_version", "qgemv_w4a16", "qg_gemv_workspace_size", "qgemm_w4a16_skinny",
    "qg_skinny_workspace_size", "moe_mxfp4_expert_forward", "qg_moe_workspace_size",
    "qg_moe_workspace_h_offset", "hadamard32_quant_i8", "gemm_w8a8_i32", "qg_set_pdl", "qg_device_error",
    "moe_mxfp4_expert_forward_noalloc", "qg_moe_noalloc_max_bytes",
    "qgemv_w4a16_group_create", "qgemv_w4a16_group_run", "qgemv_w4a16_group_destroy",
    "qgemm_w4a16_skinny_group_create", "qgemm_w4a16_skinny_group_run", "qgemm_w4a16_skinny_group_destroy",
    "qgemv_w8a16", "qgemm_affine",
    "qgemv_w4a16_chain_create", "qgemv_w4a16_chain_run", "qgemv_w4a16_chain_destroy", "qgemv_w4a16_chain_bytes",
    "qg_last_cuda_error", "qg_last_cuda_error_string", "qg_selftest_wait_timeout",
    "qgemv_w4a16_chain_trace_enable", "qgemv_w4a16_chain_trace_read", "qgemv_w4a16_chain_trace_shape",
    "gemm_w8a8_hadamard", "qg_w8a8_hadamard_workspace_size", "qg_workspace_size",
]

OP_GEMV_W4A16, OP_SKINNY_W4A16, OP_MOE_MXFP4, OP_HADAMARD_I8, OP_W8A8_I32, OP_W8A8_HADAMARD = range(6)

X_BF16, X_COPY, X_SWIGLU = 0, 1, 2


class _GemvDesc(ctypes.Structure):
    _fields_ = [("wq", ctypes.c_void_p), ("scales_f16", ctypes.c_void_p), ("biases_f16", ctypes.c_void_p),
                ("x_bf16", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int), ("K", ctypes.c_int)]


class _GemmDesc(ctypes.Structure):
    _fields_ = [("wq", ctypes.c_void_p), ("scales_f16", ctypes.c_void_p), ("biases_f16", ctypes.c_void_p),
                ("x_bf16", ctypes.c_void_p), ("y", ctypes.c_void_p), ("M", ctypes.c_int), ("N", ctypes.c_int),
                ("K", ctypes.c_int)]


class _ChainDesc(ctypes.Structure):
    _fields_ = [("wq", ctypes.c_void_p), ("scales_f16", ctypes.c_void_p), ("biases_f16", ctypes.c_void_p),
                ("N", ctypes.c_int), ("K", ctypes.c_int), ("level", ctypes.c_int), ("x_op", ctypes.c_int),
                ("x_src", ctypes.c_void_p), ("x_alpha", ctypes.c_float), ("y", ctypes.c_void_p)]


class QGError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)}")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libqgemv.so (built by build.py). Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libqgemv.so is not built ({LIB_PATH}); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.qg_status_string.restype = ctypes.c_char_p
        L.qg_status_string.argtypes = [I]
        L.qg_version.restype = I
        L.qgemv_w4a16.restype = I
        L.qgemv_w4a16.argtypes = [P, P, P, P, P, I, I, I, P, Z, P]
        L.qgemm_affine.restype = I
        L.qgemm_affine.argtypes = [P, I, P, P, P, P, I, I, I, I, P]
        L.qgemv_w8a16.restype = I
        L.qgemv_w8a16.argtypes = [P, P, P, P, I, I, P]
        L.qg_gemv_workspace_size.restype = Z
        L.qg_gemv_workspace_size.argtypes = [I, I, I]
        L.qgemm_w4a16_skinny.restype = I
        L.qgemm_w4a16_skinny.argtypes = [P, P, P, P, P, I, I, I, I, P, Z, P]
        L.qg_skinny_workspace_size.restype = Z
        L.qg_skinny_workspace_size.argtypes = [I, I, I, I]
        L.moe_mxfp4_expert_forward.restype = I
        L.moe_mxfp4_expert_forward.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, Z, P]
        L.qg_moe_workspace_size.restype = Z
        L.qg_moe_workspace_size.argtypes = [I, I, I, I, I]
        L.qg_moe_workspace_h_offset.restype = Z
        L.qg_moe_workspace_h_offset.argtypes = [I, I, I, I, I]
        L.qg_workspace_size.restype = Z
        L.qg_workspace_size.argtypes = [I, I, I, I, I, I, I]
        L.hadamard32_quant_i8.restype = I
        L.hadamard32_quant_i8.argtypes = [P, P, P, P, I, I, P]
        L.gemm_w8a8_i32.restype = I
        L.gemm_w8a8_i32.argtypes = [P, P, P, I, I, I, P]
        L.qg_set_pdl.restype = None
        L.qg_set_pdl.argtypes = [I]
        L.qg_device_error.restype = I
        L.qg_device_error.argtypes = [P, I]
        L.moe_mxfp4_expert_forward_noalloc.restype = I
        L.moe_mxfp4_expert_forward_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, P, P]
        L.qg_moe_noalloc_max_bytes.restype = Z
        L.qg_moe_noalloc_max_bytes.argtypes = []
        L.qgemv_w4a16_group_create.restype = I
        L.qgemv_w4a16_group_create.argtypes = [ctypes.POINTER(_GemvDesc), I, I, ctypes.POINTER(P)]
        L.qgemv_w4a16_group_run.restype = I
        L.qgemv_w4a16_group_run.argtypes = [P, P]
        L.qgemv_w4a16_group_destroy.restype = None
        L.qgemv_w4a16_group_destroy.argtypes = [P]
        L.qgemm_w4a16_skinny_group_create.restype = I
        L.qgemm_w4a16_skinny_group_create.argtypes = [ctypes.POINTER(_GemmDesc), I, I, ctypes.POINTER(P)]
        L.qgemm_w4a16_skinny_group_run.restype = I
        L.qgemm_w4a16_skinny_group_run.argtypes = [P, P]
        L.qgemm_w4a16_skinny_group_destroy.restype = None
        L.qgemm_w4a16_skinny_group_destroy.argtypes = [P]
        L.qgemv_w4a16_chain_create.restype = I
        L.qgemv_w4a16_chain_create.argtypes = [ctypes.POINTER(_ChainDesc), I, I, ctypes.POINTER(P)]
        L.qgemv_w4a16_chain_run.restype = I
        L.qgemv_w4a16_chain_run.argtypes = [P, P]
        L.qgemv_w4a16_chain_destroy.restype = None
        L.qgemv_w4a16_chain_destroy.argtypes = [P]
        L.gemm_w8a8_hadamard.restype = I
        L.gemm_w8a8_hadamard.argtypes = [P, P, P, P, P, I, I, I, P, Z, P]
        L.qg_w8a8_hadamard_workspace_size.restype = Z
        L.qg_w8a8_hadamard_workspace_size.argtypes = [I, I]
        L.qg_selftest_wait_timeout.restype = I
        L.qg_selftest_wait_timeout.argtypes = [I, ctypes.c_uint32, P]
        L.qg_last_cuda_error.restype = I
        L.qg_last_cuda_error.argtypes = []
        L.qg_last_cuda_error_string.restype = ctypes.c_char_p
        L.qg_last_cuda_error_string.argtypes = []
        L.qgemv_w4a16_chain_trace_enable.restype = I
        L.qgemv_w4a16_chain_trace_enable.argtypes = [P, I]
        L.qgemv_w4a16_chain_trace_read.restype = I
        L.qgemv_w4a16_chain_trace_read.argtypes = [P, P, Z]
        L.qgemv_w4a16_chain_trace_shape.restype = None
        L.qgemv_w4a16_chain_trace_shape.argtypes = [P, ctypes.POINTER(I), ctypes.POINTER(I)]
        L.qgemv_w4a16_chain_bytes.restype = Z
        L.qgemv_w4a16_chain_bytes.argtypes = [P]
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != QG_OK:
        if status == 5:  # QG_ERR_CUDA: name the runtime error behind it
            where = f"{where} ({lib().qg_last_cuda_error_string().decode()})"
        raise QGError(status, where)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype_bytes, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.element_size() != dtype_bytes:
        raise ValueError(f"{name} must have {dtype_bytes}-byte elements")


def set_pdl(enable: bool):
    lib().qg_set_pdl(1 if enable else 0)


def device_error(clear: bool = True) -> int:
    code = ctypes.c_uint32(0)
    lib().qg_device_error(ctypes.byref(code), 1 if clear else 0)
    return code.value


def qgemv_w4a16(wq, scales, biases, x, y=None, workspace=None, stream=None):
    """y[n] = sum_k (s q + b) x[k]; wq int32 [N][K/8], scales/biases fp16
    [N][K/64], x bf16 [K] -> y fp32 [N]."""
    N, K8 = wq.shape
    K = K8 * 8
    for t, b, n in ((wq, 4, "wq"), (scales, 2, "scales"), (biases, 2, "biases"), (x, 2, "x")):
        _need(t, b, n)
    if y is None:
        y = torch.empty(N, device=wq.device, dtype=torch.float32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().qgemv_w4a16(_p(wq), _p(scales), _p(biases), _p(x), _p(y), N, K, K // scales.shape[1],
                             _p(workspace), ws_bytes, _stream(stream)), "qgemv_w4a16")
    return y


def qgemm_affine(wq, bits, scales, biases, x, y=None, stream=None):
    """Y[m][n] = sum_k (s q + b) X[m][k] with `bits`-bit codes (2, 3, 4, 5, 6
    or 8) packed as one little-endian bit stream per row: wq int32
    [N][K*bits/32], scales/biases fp16 [N][K/group], X bf16 [M][K] or [K] ->
    Y fp32 [M][N] (or [N])."""
    N, W = wq.shape
    K = W * 32 // bits
    vec = x.dim() == 1
    xx = x[None, :] if vec else x
    M = xx.shape[0]
    for t, b, n in ((wq, 4, "wq"), (scales, 2, "scales"), (biases, 2, "biases"), (xx, 2, "x")):
        _need(t, b, n)
    if y is None:
        y = torch.empty(M, N, device=wq.device, dtype=torch.float32)
    _check(lib().qgemm_affine(_p(wq), int(bits), _p(scales), _p(biases), _p(xx), _p(y), M, N, K,
                              K // scales.shape[1], _stream(stream)), "qgemm_affine")
    return y[0] if vec and y.dim() == 2 else y


def qgemv_w8a16(wq, scales, x, y=None, stream=None):
    """y[n] = s[n] sum_k q[n][k] x[k]; wq int8 [N][K], scales fp32 [N],
    x bf16 [K] -> y fp32 [N] (the row-int8 output head)."""
    N, K = wq.shape
    for t, b, n in ((wq, 1, "wq"), (scales, 4, "scales"), (x, 2, "x")):
        _need(t, b, n)
    if y is None:
        y = torch.empty(N, device=wq.device, dtype=torch.float32)
    _check(lib().qgemv_w8a16(_p(wq), _p(scales), _p(x), _p(y), N, K, _stream(stream)), "qgemv_w8a16")
    return y


_WS = {}


def skinny_workspace(nbytes, device, stream=None):
    """A zero-filled workspace for qgemm_w4a16_skinny, cached per (device,
    stream) and reused (every call leaves it zero-filled): calls on one stream
    are ordered, so they may share it, and calls on different streams get
    different ones. Inside a stream capture a fresh one is made (the zero fill
    is captured too) and not cached."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    key = (str(device), stream.cuda_stream)
    ws = _WS.get(key)
    if ws is not None and ws.numel() >= nbytes:
        return ws
    if torch.cuda.is_current_stream_capturing():
        return torch.zeros(nbytes, device=device, dtype=torch.uint8)
    ws = torch.zeros(max(nbytes, 1 << 20), device=device, dtype=torch.uint8)
    _WS[key] = ws
    return ws


def qgemm_w4a16_skinny(wq, scales, biases, x, y=None, workspace=None, stream=None):
    """Y[m][n] = sum_k (s q + b) X[m][k]; X bf16 [M][K] -> Y fp32 [M][N]."""
    N, K8 = wq.shape
    K = K8 * 8
    M = x.shape[0]
    for t, b, n in ((wq, 4, "wq"), (scales, 2, "scales"), (biases, 2, "biases"), (x, 2, "x")):
        _need(t, b, n)
    if y is None:
        y = torch.empty(M, N, device=wq.device, dtype=torch.float32)
    need = lib().qg_skinny_workspace_size(M, N, K, K // scales.shape[1])
    if workspace is None and need:
        workspace = skinny_workspace(need, wq.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().qgemm_w4a16_skinny(_p(wq), _p(scales), _p(biases), _p(x), _p(y), M, N, K,
                                    K // scales.shape[1], _p(workspace), ws_bytes, _stream(stream)),
           "qgemm_w4a16_skinny")
    return y


class GemvGroup:
    """Many independent M = 1 projections run as one persistent launch.

    `items` is a list of (wq, scales, biases, x, y) CUDA tensors with the
    layouts of qgemv_w4a16 (y preallocated, fp32 [N]). The tensors are held
    by the group: every run reads the x's and writes the y's in place."""

    def __init__(self, items):
        descs = (_GemvDesc * len(items))()
        for d, (wq, s, b, x, y) in zip(descs, items):
            for t, nb, n in ((wq, 4, "wq"), (s, 2, "scales"), (b, 2, "biases"), (x, 2, "x"), (y, 4, "y")):
                _need(t, nb, n)
            d.wq, d.scales_f16, d.biases_f16 = wq.data_ptr(), s.data_ptr(), b.data_ptr()
            d.x_bf16, d.y = x.data_ptr(), y.data_ptr()
            d.N, d.K = wq.shape[0], wq.shape[1] * 8
        self._items = list(items)
        self._h = ctypes.c_void_p()
        _check(lib().qgemv_w4a16_group_create(descs, len(items), 64, ctypes.byref(self._h)),
               "qgemv_w4a16_group_create")

    def run(self, stream=None):
        _check(lib().qgemv_w4a16_group_run(self._h, _stream(stream)), "qgemv_w4a16_group_run")

    def close(self):
        if self._h:
            lib().qgemv_w4a16_group_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class GemvChain:
    """M = 1 projections in dependency order as one persistent launch.

    `items` is a list of dicts with keys wq, scales, biases (the layouts of
    qgemv_w4a16), level (non-decreasing), op (X_BF16, X_COPY or X_SWIGLU), x
    (bf16 [K] for X_BF16, fp32 [K] / [2K] for X_COPY / X_SWIGLU, typically an
    earlier level's y), alpha (float, default 1) and y (fp32 [N], written).
    The weights are copied into the kernel's layout at construction; the x
    and y tensors are held and used by every run."""

    def __init__(self, items):
        descs = (_ChainDesc * len(items))()
        for d, it in zip(descs, items):
            wq, s, b, x, y = it["wq"], it["scales"], it["biases"], it["x"], it["y"]
            for t, nb, n in ((wq, 4, "wq"), (s, 2, "scales"), (b, 2, "biases"), (y, 4, "y")):
                _need(t, nb, n)
            op = it.get("op", X_BF16)
            _need(x, 2 if op == X_BF16 else 4, "x")
            d.wq, d.scales_f16, d.biases_f16 = wq.data_ptr(), s.data_ptr(), b.data_ptr()
            d.N, d.K = wq.shape[0], wq.shape[1] * 8
            d.level, d.x_op, d.x_alpha = int(it["level"]), int(op), float(it.get("alpha", 1.0))
            d.x_src, d.y = x.data_ptr(), y.data_ptr()
        self._items = [dict(x=it["x"], y=it["y"]) for it in items]
        self._h = ctypes.c_void_p()
        _check(lib().qgemv_w4a16_chain_create(descs, len(items), 64, ctypes.byref(self._h)),
               "qgemv_w4a16_chain_create")

    def run(self, stream=None):
        _check(lib().qgemv_w4a16_chain_run(self._h, _stream(stream)), "qgemv_w4a16_chain_run")

    def device_bytes(self):
        return lib().qgemv_w4a16_chain_bytes(self._h)

    def trace(self, enable=True):
        """Switch per-(CTA, level) timestamps on or off (see the header)."""
        _check(lib().qgemv_w4a16_chain_trace_enable(self._h, 1 if enable else 0), "qgemv_w4a16_chain_trace_enable")

    def trace_read(self):
        """The stamps of the last runs as a uint64 numpy array [grid][levels][4] (ns)."""
        import numpy as np
        g, lv = ctypes.c_int(0), ctypes.c_int(0)
        lib().qgemv_w4a16_chain_trace_shape(self._h, ctypes.byref(g), ctypes.byref(lv))
        out = np.zeros((g.value, lv.value, 4), dtype=np.uint64)
        _check(lib().qgemv_w4a16_chain_trace_read(self._h, out.ctypes.data_as(ctypes.c_void_p), out.size),
               "qgemv_w4a16_chain_trace_read")
        return out

    def close(self):
        if self._h:
            lib().qgemv_w4a16_chain_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class SkinnyGroup:
    """Many independent skinny projections (2 <= M <= 32) as one persistent
    tensor-core launch.

    `items` is a list of (wq, scales, biases, x, y) CUDA tensors with the
    layouts of qgemm_w4a16_skinny (x bf16 [M][K], y preallocated fp32 [M][N]).
    The tensors are held by the group: every run reads the x's and writes the
    y's in place."""

    def __init__(self, items):
        descs = (_GemmDesc * len(items))()
        for d, (wq, s, b, x, y) in zip(descs, items):
            for t, nb, n in ((wq, 4, "wq"), (s, 2, "scales"), (b, 2, "biases"), (x, 2, "x"), (y, 4, "y")):
                _need(t, nb, n)
            d.wq, d.scales_f16, d.biases_f16 = wq.data_ptr(), s.data_ptr(), b.data_ptr()
            d.x_bf16, d.y = x.data_ptr(), y.data_ptr()
            d.M, d.N, d.K = x.shape[0], wq.shape[0], wq.shape[1] * 8
        self._items = list(items)
        self._h = ctypes.c_void_p()
        _check(lib().qgemm_w4a16_skinny_group_create(descs, len(items), 64, ctypes.byref(self._h)),
               "qgemm_w4a16_skinny_group_create")

    def run(self, stream=None):
        _check(lib().qgemm_w4a16_skinny_group_run(self._h, _stream(stream)), "qgemm_w4a16_skinny_group_run")

    def close(self):
        if self._h:
            lib().qgemm_w4a16_skinny_group_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_workspace_size(T, H, I, E, top_k):
    return lib().qg_moe_workspace_size(T, H, I, E, top_k)


def workspace_size(op, M=0, N=0, K=0, T=0, E=0, top_k=0):
    """Device bytes operation `op` (one of the OP_* constants) needs; the
    single query of the boundary (group size 64 where it applies)."""
    return lib().qg_workspace_size(op, M, N, K, T, E, top_k)


def moe_workspace_h_offset(T, H, I, E, top_k):
    return lib().qg_moe_workspace_h_offset(T, H, I, E, top_k)


def moe_mxfp4_expert_forward(x, logits, gate_q, gate_s, up_q, up_s, down_q, down_s, top_k,
                             y=None, topk_idx=None, topk_w=None, workspace=None, stream=None):
    """Routed MXFP4 expert MoE. x bf16 [T][H], logits fp32 [T][E], gate/up codes
    uint8 [E][I][H/2] + scales [E][I][H/32], down codes [E][H][I/2] + scales
    [E][H][I/32]. Returns (y fp32 [T][H], topk_idx int32 [T][k], topk_w fp32)."""
    T, H = x.shape
    E = logits.shape[1]
    I = gate_q.shape[1]
    dev = x.device
    if y is None:
        y = torch.empty(T, H, device=dev, dtype=torch.float32)
    if topk_idx is None:
        topk_idx = torch.empty(T, top_k, device=dev, dtype=torch.int32)
    if topk_w is None:
        topk_w = torch.empty(T, top_k, device=dev, dtype=torch.float32)
    need = moe_workspace_size(T, H, I, E, top_k)
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().moe_mxfp4_expert_forward(_p(x), _p(logits), _p(gate_q), _p(gate_s), _p(up_q), _p(up_s),
                                          _p(down_q), _p(down_s), T, H, I, E, top_k, _p(y), _p(topk_idx),
                                          _p(topk_w), _p(workspace), ws_bytes, _stream(stream)),
           "moe_mxfp4_expert_forward")
    return y, topk_idx, topk_w


def hadamard32_quant_i8(x, sign_bits, q=None, scale=None, stream=None):
    """x bf16 [M][K], sign_bits int32 [K/32] -> (q int8 [M][K], scale fp32 [M])."""
    M, K = x.shape
    _need(x, 2, "x")
    _need(sign_bits, 4, "sign_bits")
    if q is None:
        q = torch.empty(M, K, device=x.device, dtype=torch.int8)
    if scale is None:
        scale = torch.empty(M, device=x.device, dtype=torch.float32)
    _check(lib().hadamard32_quant_i8(_p(x), _p(sign_bits), _p(q), _p(scale), M, K, _stream(stream)),
           "hadamard32_quant_i8")
    return q, scale


_W8WS = {}


def gemm_w8a8_hadamard(x, sign_bits, w, sw, y=None, workspace=None, stream=None):
    """y[m][n] = C[m][n] s_a[m] s_w[n] / 32 in one launch: x bf16 [M][K] is
    transformed and quantized like hadamard32_quant_i8 (bit-exact), C = q_a w^T
    exactly; w int8 [N][K] and sw fp32 [N] are the weights quantized the same
    way. The zero-filled workspace is cached per (device, stream) (every call
    leaves it zeroed)."""
    M, K = x.shape
    N = w.shape[0]
    for t, b, n in ((x, 2, "x"), (sign_bits, 4, "sign_bits"), (w, 1, "w"), (sw, 4, "sw")):
        _need(t, b, n)
    if y is None:
        y = torch.empty(M, N, device=x.device, dtype=torch.float32)
    need = lib().qg_w8a8_hadamard_workspace_size(M, K)
    if workspace is None:
        st = stream if stream is not None else torch.cuda.current_stream(x.device)
        key = (str(x.device), st.cuda_stream)
        workspace = _W8WS.get(key)
        if workspace is None or workspace.numel() < need:
            if torch.cuda.is_current_stream_capturing():
                workspace = torch.zeros(need, device=x.device, dtype=torch.uint8)
            else:
                workspace = torch.zeros(max(need, 1 << 16), device=x.device, dtype=torch.uint8)
                _W8WS[key] = workspace
    _check(lib().gemm_w8a8_hadamard(_p(x), _p(sign_bits), _p(w), _p(sw), _p(y), M, N, K, _p(workspace),
                                    workspace.numel(), _stream(stream)), "gemm_w8a8_hadamard")
    return y


def gemm_w8a8_i32(a, w, c=None, stream=None):
    """a int8 [M][K], w int8 [N][K] -> c int32 [M][N] = a @ w^T (exact)."""
    M, K = a.shape
    N = w.shape[0]
    _need(a, 1, "a")
    _need(w, 1, "w")
    if c is None:
        c = torch.empty(M, N, device=a.device, dtype=torch.int32)
    _check(lib().gemm_w8a8_i32(_p(a), _p(w), _p(c), M, N, K, _stream(stream)), "gemm_w8a8_i32")
    return c
