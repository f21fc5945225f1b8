"""Oracle: plain CPU reference of the quantized GEMV / skinny GEMM path.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The product library
(``skinny_gemm_qgemv_gb300``) never imports it and shares no code with it.

Floating-point results are float64 from the exact input values; the integer
codes of the Hadamard + int8 path are decided in fp32 (see oracle.c). The C
loops live in ``oracle.c`` (built into ``liboracle.so`` by :func:`build`); this
module marshals numpy arrays and composes the MoE forward from those loops.

Sources (page title, section):
  * "MLX Runner: An Inference Engine You Can Read", "Architecture: one command
    buffer per token" -- affine W4 groups (weight = scale x code + bias).
  * "Krill Teardown", "Core mechanisms" -- several rows share one weight read.
  * "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin), "How it
    works" and "Technical approach / compute" -- top-16 routed experts per
    layer, fused MXFP4 expert GEMV.
  * Uzu article, "How Uzu optimizes bytes and tokens per pass" -- block-32
    randomized Hadamard, 8-bit activations, int8 matrix products.

Readings taken where the pages are silent (each listed in the design notes):
router = softmax of the fp32 logits, top-k by logit value descending with ties
to the lower expert index, routing weights = the un-renormalized softmax
probabilities; expert FFN = down(silu(gate x) * up x); unnormalized Hadamard
with fixed butterfly order; symmetric int8 in [-127, 127] with RNE.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

TOL_REL = 2e-3   # |y - y_ref| <= TOL_REL * sum|x*w| + TOL_ABS
TOL_ABS = 1e-5


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no fast-math, no FP contraction, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_max_threads.restype = I
            lib.oracle_f16_to_double.restype = ctypes.c_double
            lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_e2m1.restype = ctypes.c_double
            lib.oracle_e2m1.argtypes = [I]
            lib.oracle_e8m0.restype = ctypes.c_double
            lib.oracle_e8m0.argtypes = [I]
            lib.oracle_w4a16.argtypes = [P, P, P, P, I, I, I, I, P, P, I]
            lib.oracle_w4a16_rows.argtypes = [P, P, P, P, I, I, I, P, I, ctypes.c_int64,
                                              P, P, I]
            lib.oracle_mxfp4_gemv.argtypes = [P, P, I, I, P, P, P, P, P, I]
            lib.oracle_hadamard32.argtypes = [P, P, I, P]
            lib.oracle_hadamard32_quant_i8.argtypes = [P, P, I, I, P, P, P, I]
            lib.oracle_quant_i8_row.argtypes = [P, I, P, P]
            lib.oracle_w8a8.argtypes = [P, P, I, I, I, P, I]
            lib.oracle_w8a16.argtypes = [P, P, P, I, I, I, P, P, I]
            lib.oracle_affine.argtypes = [P, I, P, P, P, I, I, I, I, P, P, I]
            lib.oracle_w8a8.restype = I
            _lib = lib
    return _lib


def _np(a, dtype):
    """torch tensor or array -> C-contiguous numpy array of `dtype` (bit view)."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().contiguous()
        import torch
        bits = {np.uint16: torch.int16, np.uint32: torch.int32, np.uint8: torch.uint8,
                np.int8: torch.int8, np.int32: torch.int32, np.float32: torch.float32,
                np.float64: torch.float64}[dtype]
        if a.dtype != bits and a.element_size() == np.dtype(dtype).itemsize:
            a = a.view(bits)
        a = a.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" \
                and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return _L().oracle_max_threads()


def f16_to_double(h: int) -> float:
    return _L().oracle_f16_to_double(int(h) & 0xFFFF)


def bf16_to_double(b: int) -> float:
    return _L().oracle_bf16_to_double(int(b) & 0xFFFF)


def e2m1_value(code: int) -> float:
    return _L().oracle_e2m1(int(code))


def e8m0_value(e: int) -> float:
    return _L().oracle_e8m0(int(e))


# --------------------------------------------------------------------------
# W4A16 GEMV / skinny GEMM
# --------------------------------------------------------------------------

def w4a16(wq, scales, biases, x, group=64, threads=0):
    """y[m][n] = sum_k (s*q + b) * x[m][k] in float64, plus sum_k |w*x|.

    wq uint32 [N][K/8], scales/biases fp16 bits [N][K/group], x bf16 bits
    [M][K] (or [K]). Returns (y [M][N], absdot [M][N]) as float64.
    """
    wq = _np(wq, np.uint32)
    s = _np(scales, np.uint16)
    b = _np(biases, np.uint16)
    x = _np(x, np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    N = wq.shape[0]
    assert wq.shape == (N, K // 8) and s.shape == (N, K // group) and b.shape == s.shape
    y = np.zeros((M, N), np.float64)
    ad = np.zeros((M, N), np.float64)
    _L().oracle_w4a16(_ptr(wq), _ptr(s), _ptr(b), _ptr(x), M, N, K, group,
                      _ptr(y), _ptr(ad), threads)
    return y, ad


def w4a16_rows(wq, scales, biases, x, rows, group=64, threads=0, row_base=0):
    """The same definition for selected output rows only; returns [M][len(rows)]."""
    wq = _np(wq, np.uint32)
    s = _np(scales, np.uint16)
    b = _np(biases, np.uint16)
    x = _np(x, np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    M, K = x.shape
    y = np.zeros((M, len(rows)), np.float64)
    ad = np.zeros((M, len(rows)), np.float64)
    _L().oracle_w4a16_rows(_ptr(wq), _ptr(s), _ptr(b), _ptr(x), M, K, group,
                           _ptr(rows), len(rows), int(row_base), _ptr(y), _ptr(ad), threads)
    return y, ad


def affine(wq, bits, scales, biases, x, group=64, threads=0):
    """Affine quantized matvec at 2, 3, 4, 5, 6 or 8 bits: y[m][n] = sum_k
    (s q + b) x[m][k] in float64 plus sum_k |w x|. wq uint32 [N][K*bits/32]
    (each row one little-endian bit stream of K codes), scales/biases fp16
    bits [N][K/group], x bf16 bits [M][K] (or [K])."""
    assert bits in (2, 3, 4, 5, 6, 8) and group in (32, 64, 128)
    wq = _np(wq, np.uint32)
    s = _np(scales, np.uint16)
    b = _np(biases, np.uint16)
    x = _np(x, np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    N = wq.shape[0]
    assert K % 32 == 0 and K % group == 0
    assert wq.shape == (N, K * bits // 32) and s.shape == (N, K // group) and b.shape == s.shape
    y = np.zeros((M, N), np.float64)
    ad = np.zeros((M, N), np.float64)
    _L().oracle_affine(_ptr(wq), bits, _ptr(s), _ptr(b), _ptr(x), M, N, K, group, _ptr(y), _ptr(ad), threads)
    return y, ad


def tolerance(absdot):
    return TOL_REL * np.asarray(absdot) + TOL_ABS


# --------------------------------------------------------------------------
# Inputs of the dependent projections of a decode step
# --------------------------------------------------------------------------
# "MLX Runner: An Inference Engine You Can Read", "Architecture: one command
# buffer per token": a token runs the layer's projections one after another,
# each consuming the previous one's output. Between the fp32 output of one
# projection and the bf16 activation of the next the chain applies either a
# scaled copy or the SwiGLU of a fused gate/up output (the expert FFN form
# down(silu(gate x) * up x) used for the MoE below); both end in one rounding
# to bf16, nearest even.

X_BF16, X_COPY, X_SWIGLU = 0, 1, 2


def bf16_bits(v):
    """Round real values (float64 or float32 arrays) to bf16 in ONE step,
    nearest with ties to even; returns the uint16 bit patterns.

    Normal range: the float64 significand is rounded at bit 45 (bf16 keeps 7
    of float64's 52 fraction bits); magnitudes below 2^-126 are bf16
    subnormals, multiples of 2^-133 rounded with ties to even. Results beyond
    the largest bf16 become infinities."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    b = v.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    normal = r.view(np.float64)
    sub = np.round(v / 2.0 ** -133) * 2.0 ** -133  # np.round: ties to even
    out = np.where(np.abs(v) < 2.0 ** -126, sub, normal)
    with np.errstate(over="ignore"):
        f = out.astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def chain_x(src, op, alpha, K):
    """The bf16 activation (uint16 bits [K]) a projection reads from an earlier
    projection's fp32 output `src`:
      X_COPY:   bf16(alpha * src[k]), the product taken in fp32 (one IEEE
                rounding, as the kernel does), then rounded to bf16;
      X_SWIGLU: bf16(silu(g) * u * alpha) with g = src[k], u = src[K + k], the
                value computed in float64 and rounded once (the kernel
                evaluates it in fp32, so a value within a few fp32 ulps of a
                bf16 rounding boundary may land one bf16 ulp apart)."""
    src = _np(src, np.float32).reshape(-1)
    if op == X_COPY:
        assert src.size >= K
        return bf16_bits((np.float32(alpha) * src[:K]).astype(np.float64))
    if op == X_SWIGLU:
        assert src.size >= 2 * K
        g = src[:K].astype(np.float64)
        u = src[K:2 * K].astype(np.float64)
        return bf16_bits(silu(g) * u * float(alpha))
    raise ValueError(f"unknown op {op}")


# --------------------------------------------------------------------------
# MXFP4 routed-expert MoE
# --------------------------------------------------------------------------

def mxfp4_gemv(codes, scales, v, wv=None, threads=0):
    """out[r] = sum_c W[r][c] v[c] (float64) with W decoded from MXFP4.
    Returns (out, sum_c |W v|, sum_c |W| wv  or None)."""
    codes = _np(codes, np.uint8)
    scales = _np(scales, np.uint8)
    R, C2 = codes.shape
    C = 2 * C2
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    out = np.zeros(R, np.float64)
    ab = np.zeros(R, np.float64)
    aw = None
    wvp = None
    if wv is not None:
        wv = np.ascontiguousarray(np.asarray(wv, dtype=np.float64))
        aw = np.zeros(R, np.float64)
        wvp = _ptr(wv)
    _L().oracle_mxfp4_gemv(_ptr(codes), _ptr(scales), R, C, _ptr(v), wvp, _ptr(out),
                           _ptr(ab), _ptr(aw) if aw is not None else None, threads)
    return out, ab, aw


def mxfp4_dequant(codes, scales):
    """Dense float64 [R][C] of an MXFP4 matrix, decoded through the oracle's
    per-element definition (one-hot GEMV per column is too slow; this walks
    the same table). Small matrices only."""
    codes = _np(codes, np.uint8)
    scales = _np(scales, np.uint8)
    R, C2 = codes.shape
    lo = codes & 15
    hi = codes >> 4
    cod = np.empty((R, 2 * C2), np.int64)
    cod[:, 0::2] = lo
    cod[:, 1::2] = hi
    table = np.array([e2m1_value(c) for c in range(16)])
    sc = np.array([e8m0_value(e) if e != 255 else np.nan for e in range(256)])
    return table[cod] * np.repeat(sc[scales.astype(np.int64)], 32, axis=1)


def router(logits, top_k):
    """Softmax over experts (float64 from the fp32 logits) and top-k by logit
    value, descending, ties to the lower expert index. Returns
    (idx int32 [T][k], weight float64 [T][k], p float64 [T][E])."""
    lg = _np(logits, np.float32).astype(np.float64)
    T, E = lg.shape
    mx = lg.max(axis=1, keepdims=True)
    ex = np.exp(lg - mx)
    p = ex / ex.sum(axis=1, keepdims=True)
    idx = np.zeros((T, top_k), np.int32)
    wts = np.zeros((T, top_k), np.float64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-lg[t, e], e))[:top_k]
        idx[t] = order
        wts[t] = p[t, order]
    return idx, wts, p


def silu(g):
    return g / (1.0 + np.exp(-g))


def dsilu(g):
    sg = 1.0 / (1.0 + np.exp(-g))
    return sg * (1.0 + g * (1.0 - sg))


def moe_forward(x, logits, gate_q, gate_s, up_q, up_s, down_q, down_s, top_k,
                tokens=None, threads=0, h_override=None, get_expert=None):
    """Routed-expert MoE forward for the selected tokens, float64.

    x bf16 bits [T][H]; logits fp32 [T][E]; gate/up codes [E][I][H/2] with
    scales [E][I][H/32]; down codes [E][H][I/2] with scales [E][H][I/32].
    For token t and slot j with expert e = idx[t][j], weight p = w[t][j]:
        g = W_g[e] x_t,  u = W_u[e] x_t,  h = silu(g) * u,  o = W_d[e] h,
        y_t = sum_j p * o.
    The result also carries a per-element error bound: the per-stage
    tolerance 2e-3*sum|x w| + 1e-5 on g and u, propagated to first order
    through SwiGLU and the down product (see tolerance notes in the tests).
    If h_override[(t, j)] is given, that h replaces the oracle's own h for the
    down product (stage-wise check of the down GEMV on the kernel's h).
    get_expert(e) -> (gq, gs, uq, us, dq, ds) of expert e may replace the six
    arrays (then pass None for them), so large expert sets stay off the host.
    """
    xs = _np(x, np.uint16)
    T, H = xs.shape
    idx, wts, _ = router(logits, top_k)
    if get_expert is None:
        arrs = [_np(a, np.uint8) for a in (gate_q, gate_s, up_q, up_s, down_q, down_s)]
        get_expert = lambda e: tuple(a[e] for a in arrs)  # noqa: E731
    if tokens is None:
        tokens = range(T)
    xf = (xs.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = {"idx": idx, "w": wts, "y": {}, "ybound": {}, "h": {}, "hbound": {},
           "g": {}, "u": {}, "gtol": {}, "utol": {}, "o": {}}
    for t in tokens:
        y = np.zeros(H, np.float64)
        yb = np.zeros(H, np.float64)
        for j in range(top_k):
            e = int(idx[t, j])
            p = float(wts[t, j])
            gq, gs, uq, us, dq, ds = get_expert(e)
            g, ag, _ = mxfp4_gemv(gq, gs, xf[t], threads=threads)
            u, au, _ = mxfp4_gemv(uq, us, xf[t], threads=threads)
            tg = TOL_REL * ag + TOL_ABS
            tu = TOL_REL * au + TOL_ABS
            h = silu(g) * u
            # first-order propagation of the g/u tolerance through SwiGLU,
            # with the second-order term of the product kept as well
            dh = (np.abs(dsilu(g) * u) * tg + np.abs(silu(g)) * tu
                  + 1.1 * tg * tu + 0.25 * tg * tg * np.abs(u))
            hin = h if h_override is None else np.asarray(h_override[(t, j)], np.float64)
            o, ao, aw = mxfp4_gemv(dq, ds, hin, wv=dh, threads=threads)
            y += p * o
            yb += p * (TOL_REL * ao + TOL_ABS + aw) + 1e-6 * p * np.abs(o)
            out["g"][(t, j)] = g
            out["u"][(t, j)] = u
            out["gtol"][(t, j)] = tg
            out["utol"][(t, j)] = tu
            out["h"][(t, j)] = h
            out["hbound"][(t, j)] = dh
            out["o"][(t, j)] = o
        out["y"][t] = y
        out["ybound"][t] = yb + TOL_ABS
    return out


# --------------------------------------------------------------------------
# Hadamard + int8, W8A8
# --------------------------------------------------------------------------

def hadamard32(v, sign_bits):
    """fp32 block-32 randomized Walsh-Hadamard of a fp32 vector [K]."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    sb = _np(sign_bits, np.uint32)
    K = v.shape[0]
    z = np.zeros(K, np.float32)
    _L().oracle_hadamard32(_ptr(v), _ptr(sb), K, _ptr(z))
    return z


def quant_i8_row(z):
    """Per-token symmetric int8 of one fp32 row: (q int8 [K], scale fp32)."""
    z = np.ascontiguousarray(np.asarray(z, dtype=np.float32))
    q = np.zeros(z.shape[0], np.int8)
    s = np.zeros(1, np.float32)
    _L().oracle_quant_i8_row(_ptr(z), z.shape[0], _ptr(q), _ptr(s))
    return q, s[0]


def hadamard32_quant_i8(x, sign_bits, threads=0):
    """x bf16 bits [M][K] -> (q int8 [M][K], scale fp32 [M], z fp32 [M][K])."""
    xs = _np(x, np.uint16)
    if xs.ndim == 1:
        xs = xs[None, :]
    sb = _np(sign_bits, np.uint32)
    M, K = xs.shape
    q = np.zeros((M, K), np.int8)
    s = np.zeros(M, np.float32)
    z = np.zeros((M, K), np.float32)
    _L().oracle_hadamard32_quant_i8(_ptr(xs), _ptr(sb), M, K, _ptr(q), _ptr(s), _ptr(z),
                                    threads)
    return q, s, z


def w8a8_dequant(x, w, sign_bits, threads=0):
    """The whole int8 matrix path in float64 (Uzu article, "How Uzu optimizes
    bytes and tokens per pass"): both operands take the same sign flip and
    block-32 Walsh-Hadamard transform and are quantized per row to int8
    (hadamard32_quant_i8), multiplied exactly (w8a8), and dequantized. The
    transform is invertible, (H D a) . (H D w) = 32 a . w (D^2 = I, H H^T =
    32 I), so y[m][n] = C[m][n] s_a[m] s_w[n] / 32 approximates x . w.
    x, w bf16 bits [M][K], [N][K]. Returns (y [M][N] float64, parts) with the
    quantized operands and scales in `parts`."""
    qa, sa, za = hadamard32_quant_i8(x, sign_bits, threads)
    qw, sw, zw = hadamard32_quant_i8(w, sign_bits, threads)
    c = w8a8(qa, qw, threads)
    y = c.astype(np.float64) * sa.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :] / 32.0
    return y, {"qa": qa, "sa": sa, "za": za, "qw": qw, "sw": sw, "zw": zw, "c": c}


def w8a16(wq, scales, x, threads=0):
    """Row-int8 GEMV: y[m][n] = sum_k s[n] q[n][k] x[m][k] in float64, plus
    sum_k |w x| (the tolerance's scale). wq int8 [N][K], scales fp32 [N],
    x bf16 bits [M][K] (or [K]). Returns (y [M][N], absdot [M][N])."""
    wq = _np(wq, np.int8)
    s = _np(scales, np.float32)
    x = _np(x, np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    N = wq.shape[0]
    assert wq.shape == (N, K) and s.shape == (N,)
    y = np.zeros((M, N), np.float64)
    ad = np.zeros((M, N), np.float64)
    _L().oracle_w8a16(_ptr(wq), _ptr(s), _ptr(x), M, N, K, _ptr(y), _ptr(ad), threads)
    return y, ad


def w8a8(a, w, threads=0):
    """C[m][n] = sum_k a[m][k] w[n][k] (exact, int64 accumulate) as int32."""
    a = _np(a, np.int8)
    w = _np(w, np.int8)
    M, K = a.shape
    N = w.shape[0]
    c = np.zeros((M, N), np.int32)
    ovf = _L().oracle_w8a8(_ptr(a), _ptr(w), M, N, K, _ptr(c), threads)
    if ovf:
        raise OverflowError("W8A8 result does not fit in int32")
    return c
