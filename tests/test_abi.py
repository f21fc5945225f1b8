"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the header declares, and rejects malformed requests before any
launch (validation returns a status without touching the device)."""
import ctypes
import os
import re

import pytest

import skinny_gemm_qgemv_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")


@pytest.fixture(scope="module")
def L():
    from skinny_gemm_qgemv_gb300 import build
    build.build()
    return q.lib()


def header_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^QG_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    fns = header_functions()
    for name in ["qgemv_w4a16", "qgemm_w4a16_skinny", "moe_mxfp4_expert_forward",
                 "hadamard32_quant_i8", "gemm_w8a8_i32"]:
        assert name in fns


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name
    assert set(header_functions()) == set(q.EXPORTS)


def test_status_strings(L):
    for s in range(7):
        assert L.qg_status_string(s)
    assert L.qg_status_string(0) == b"QG_OK"
    assert L.qg_version() >= 100


A = 0x10000   # fake, 16-byte-aligned "device" addresses: never dereferenced,
B = 0x20010   # because every call below fails validation first
P = ctypes.c_void_p


def test_single_workspace_query(L):
    # the one query of the boundary gives what the per-operation queries give
    assert L.qg_workspace_size(q.OP_GEMV_W4A16, 1, 4096, 4096, 0, 0, 0) == L.qg_gemv_workspace_size(4096, 4096, 64)
    for M, N, K in ((16, 129, 12288), (32, 4096, 4096), (3, 64, 512)):
        assert L.qg_workspace_size(q.OP_SKINNY_W4A16, M, N, K, 0, 0, 0) == L.qg_skinny_workspace_size(M, N, K, 64)
    for T, H, I, E, k in ((1, 7168, 2048, 384, 16), (16, 512, 256, 8, 2)):
        assert L.qg_workspace_size(q.OP_MOE_MXFP4, 0, H, I, T, E, k) == L.qg_moe_workspace_size(T, H, I, E, k) > 0
    assert L.qg_workspace_size(q.OP_W8A8_HADAMARD, 16, 0, 4096, 0, 0, 0) == \
        L.qg_w8a8_hadamard_workspace_size(16, 4096) > 0
    assert L.qg_workspace_size(q.OP_HADAMARD_I8, 16, 0, 4096, 0, 0, 0) == 0
    assert L.qg_workspace_size(q.OP_W8A8_I32, 16, 4096, 4096, 0, 0, 0) == 0
    assert L.qg_workspace_size(99, 16, 4096, 4096, 1, 8, 2) == 0


def test_w4a16_validation(L):
    f = L.qgemv_w4a16
    assert f(None, P(A), P(A), P(A), P(A), 16, 128, 64, None, 0, None) == 1
    assert f(P(A), P(A), P(A), P(A), P(A), 0, 128, 64, None, 0, None) == 1
    assert f(P(A), P(A), P(A), P(A), P(A), 16, 100, 64, None, 0, None) == 1     # K % 64
    assert f(P(A), P(A), P(A), P(A), P(A), 16, 112, 32, None, 0, None) == 1     # K % 32
    assert f(P(A), P(A), P(A), P(A), P(A), 16, 192, 128, None, 0, None) == 1    # K % 128
    assert f(P(A), P(A), P(A), P(A), P(A), 16, 256, 256, None, 0, None) == 1    # group 256
    assert f(P(A), P(A), P(A), P(A), P(A), 16, 128, 48, None, 0, None) == 1
    assert f(P(A + 4), P(A), P(A), P(A), P(A), 16, 128, 64, None, 0, None) == 2
    g = L.qgemm_w4a16_skinny
    assert g(P(A), P(A), P(A), P(A), P(A), 33, 16, 128, 64, None, 0, None) == 1  # M > 32
    assert g(P(A), P(A), P(A), P(A), P(A), 0, 16, 128, 64, None, 0, None) == 1
    assert g(P(A), P(A), P(A), P(B + 2), P(A), 4, 16, 128, 64, None, 0, None) == 2


def test_affine_validation(L):
    f = L.qgemm_affine
    assert f(None, 3, P(A), P(A), P(A), P(A), 1, 16, 128, 64, None) == 1
    for bits in (0, 1, 7, 16):
        assert f(P(A), bits, P(A), P(A), P(A), P(A), 1, 16, 128, 64, None) == 1
    assert f(P(A), 3, P(A), P(A), P(A), P(A), 1, 16, 128, 48, None) == 1     # group 48
    assert f(P(A), 3, P(A), P(A), P(A), P(A), 1, 16, 80, 32, None) == 1      # K % 32
    assert f(P(A), 3, P(A), P(A), P(A), P(A), 1, 16, 96, 64, None) == 1      # K % group
    assert f(P(A), 3, P(A), P(A), P(A), P(A), 0, 16, 128, 64, None) == 1     # M < 1
    assert f(P(A), 3, P(A), P(A), P(A), P(A), 33, 16, 128, 64, None) == 1    # M > 32
    assert f(P(A + 4), 3, P(A), P(A), P(A), P(A), 1, 16, 128, 64, None) == 2  # misaligned


def test_w8a16_validation(L):
    f = L.qgemv_w8a16
    assert f(None, P(A), P(A), P(A), 16, 128, None) == 1
    assert f(P(A), P(A), P(A), P(A), 0, 128, None) == 1
    assert f(P(A), P(A), P(A), P(A), 16, 100, None) == 1      # K % 16
    assert f(P(A), P(A), P(A), P(A), 16, 8, None) == 1        # K < 16
    assert f(P(A), P(A), P(A), P(A), 16, 65552, None) == 1    # K > 65536
    assert f(P(A + 4), P(A), P(A), P(A), 16, 128, None) == 2  # weights misaligned
    assert f(P(A), P(A), P(A + 2), P(A), 16, 128, None) == 2  # x misaligned


def test_moe_validation(L):
    f = L.moe_mxfp4_expert_forward
    ptrs = [P(A)] * 8
    outs = [P(A)] * 3
    ws = L.qg_moe_workspace_size(1, 128, 128, 8, 2)
    assert ws > 0
    assert L.qg_moe_workspace_h_offset(1, 128, 128, 8, 2) < ws
    assert f(*ptrs, 1, 128, 128, 8, 9, *outs, P(A), ws, None) == 1        # top_k > E
    assert f(*ptrs, 1, 100, 128, 8, 2, *outs, P(A), ws, None) == 1        # H % 64
    assert f(*ptrs, 1, 128, 128, 8, 2, *outs, P(A), ws - 1, None) == 4    # workspace
    assert f(*ptrs, 1, 128, 128, 8, 2, *outs, None, ws, None) == 4
    assert f(*ptrs, 1, 128, 128, 2048, 2, *outs, P(A), 1 << 30, None) == 3  # E > 1024
    assert f(*([P(A)] * 7 + [P(A + 8)]), 1, 128, 128, 8, 2, *outs, P(A), ws, None) == 2
    assert f(*([None] + [P(A)] * 7), 1, 128, 128, 8, 2, *outs, P(A), ws, None) == 1


def test_hadamard_and_w8a8_validation(L):
    h = L.hadamard32_quant_i8
    assert h(P(A), P(A), P(A), P(A), 4, 100, None) == 1     # K % 32
    assert h(P(A), P(A), P(A), P(A), 0, 128, None) == 1
    assert h(P(A), P(A + 4), P(A), P(A), 4, 128, None) == 2
    g = L.gemm_w8a8_i32
    assert g(P(A), P(A), P(A), 16, 64, 96, None) == 1        # K % 64
    assert g(P(A), P(A), P(A), 33, 64, 128, None) == 1       # M > 32
    assert g(P(A), P(A), P(A), 16, 64, 1 << 20, None) == 1   # K too large for int32
    assert g(P(A + 1), P(A), P(A), 16, 64, 128, None) == 2


def test_gemv_group_validation(L):
    Desc = q._GemvDesc
    out = P()

    def make(*shapes, ptr=A):
        ds = (Desc * len(shapes))()
        for d, (N, K) in zip(ds, shapes):
            d.wq = d.scales_f16 = d.biases_f16 = d.x_bf16 = d.y = ptr
            d.N, d.K = N, K
        return ds

    f = L.qgemv_w4a16_group_create
    assert f(make((16, 4096)), 0, 64, ctypes.byref(out)) == 1               # empty group
    assert f(None, 1, 64, ctypes.byref(out)) == 1
    assert f(make((16, 4096)), 1, 64, None) == 1
    assert f(make((16, 4096), (0, 4096)), 2, 64, ctypes.byref(out)) == 1    # N < 1
    assert f(make((16, 4096), (8, 1024)), 2, 64, ctypes.byref(out)) == 3    # K % 2048
    assert f(make((16, 32768)), 1, 64, ctypes.byref(out)) == 3              # K > 16384
    assert f(make((16, 4096)), 1, 32, ctypes.byref(out)) == 3               # group 32
    assert f(make((16, 4096), ptr=A + 4), 1, 64, ctypes.byref(out)) == 2   # misaligned
    assert L.qgemv_w4a16_group_run(None, None) == 1
    L.qgemv_w4a16_group_destroy(None)


def test_skinny_group_validation(L):
    Desc = q._GemmDesc
    out = P()

    def make(*shapes, ptr=A):
        ds = (Desc * len(shapes))()
        for d, (M, N, K) in zip(ds, shapes):
            d.wq = d.scales_f16 = d.biases_f16 = d.x_bf16 = d.y = ptr
            d.M, d.N, d.K = M, N, K
        return ds

    f = L.qgemm_w4a16_skinny_group_create
    assert f(make((16, 128, 4096)), 0, 64, ctypes.byref(out)) == 1                   # empty group
    assert f(None, 1, 64, ctypes.byref(out)) == 1
    assert f(make((16, 128, 4096)), 1, 64, None) == 1
    assert f(make((16, 128, 4096), (16, 0, 4096)), 2, 64, ctypes.byref(out)) == 1    # N < 1
    assert f(make((33, 128, 4096)), 1, 64, ctypes.byref(out)) == 1                   # M > 32
    assert f(make((1, 128, 4096)), 1, 64, ctypes.byref(out)) == 3                    # M < 2
    assert f(make((16, 128, 4096), (16, 128, 448)), 2, 64, ctypes.byref(out)) == 3   # K % 512
    assert f(make((16, 128, 65536)), 1, 64, ctypes.byref(out)) == 3                  # K > 32768
    assert f(make((16, 128, 4096), (17, 128, 4096)), 2, 64, ctypes.byref(out)) == 3  # mixed classes
    assert f(make((16, 128, 4096)), 1, 128, ctypes.byref(out)) == 3                  # group 128
    assert f(make((16, 128, 4096), ptr=A + 4), 1, 64, ctypes.byref(out)) == 2       # misaligned
    assert L.qgemm_w4a16_skinny_group_run(None, None) == 1
    L.qgemm_w4a16_skinny_group_destroy(None)
