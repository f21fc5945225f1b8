"""GPU parity of gemm_w8a8_hadamard: the int8 matrix path of the Uzu article
("How Uzu optimizes bytes and tokens per pass") in one launch.

The weights are transformed and quantized by the oracle; the kernel's y must
equal C s_a s_w / 32 of the oracle (C exact, s_a bit-exact), so the only
difference is the fp32 rounding of the three products (a few ulps), and it must
be bit-identical to the same products formed from the two-launch path
(hadamard32_quant_i8 + gemm_w8a8_i32). Repeated calls on one workspace give the
same bits (the workspace is left zeroed).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def q():
    from skinny_gemm_qgemv_gb300 import build
    build.build()
    import skinny_gemm_qgemv_gb300 as qq
    qq.lib()
    qq.device_error(clear=True)
    yield qq
    assert qq.device_error(clear=True) == 0


@pytest.mark.parametrize("M,N,K", [(16, 4096, 4096), (16, 12288, 4096), (1, 100, 1024), (5, 1000, 2048),
                                   (16, 33, 3072), (13, 4097, 4096), (16, 1, 1024)])
def test_w8a8_hadamard_fused_vs_oracle(q, M, N, K):
    seed = 90 + M + N % 7
    x = synth.outlier_activations(M, K, seed, 0)
    wb = synth.bf16_normal((N, K), seed, 1)
    sb = synth.sign_bits(K, seed, 2)
    qw, sw, _ = oracle.hadamard32_quant_i8(wb, sb)
    yref, parts = oracle.w8a8_dequant(x, wb, sb)
    xd, sbd = x.to(DEV), sb.to(DEV)
    qwd, swd = torch.from_numpy(qw).to(DEV), torch.from_numpy(sw).to(DEV)
    y = q.gemm_w8a8_hadamard(xd, sbd, qwd, swd)
    torch.cuda.synchronize()
    yy = y.cpu().double().numpy()
    assert np.isfinite(yy).all()
    # C exact and s_a bit-exact: only the fp32 products round (3 roundings)
    tol = 4 * 2.0 ** -24 * np.abs(yref) + 1e-30
    bad = np.abs(yy - yref) > tol
    assert not bad.any(), f"{bad.sum()} outside fp32 rounding; worst {np.max(np.abs(yy - yref) / tol):.3g}x"
    # the same products from the two-launch path, bit for bit
    qa, sa = q.hadamard32_quant_i8(xd, sbd)
    c = q.gemm_w8a8_i32(qa, qwd)
    y2 = (c.float() * sa[:, None]) * (swd[None, :] * 0.03125)
    torch.cuda.synchronize()
    assert np.array_equal(sa.cpu().numpy(), parts["sa"])
    assert torch.equal(y, y2)
    # again on the same (cached) workspace, with other activations, then the first ones
    x2 = synth.outlier_activations(M, K, seed + 1, 0).to(DEV)
    y3 = q.gemm_w8a8_hadamard(x2, sbd, qwd, swd)
    y4 = q.gemm_w8a8_hadamard(xd, sbd, qwd, swd)
    torch.cuda.synchronize()
    assert torch.equal(y4, y)
    yref3, _ = oracle.w8a8_dequant(x2.cpu(), wb, sb)
    assert np.all(np.abs(y3.cpu().double().numpy() - yref3) <= 4 * 2.0 ** -24 * np.abs(yref3) + 1e-30)
    assert q.device_error() == 0


def test_w8a8_hadamard_zero_rows_and_refusals(q):
    import ctypes
    M, N, K = 4, 64, 1024
    x = synth.outlier_activations(M, K, 5, 0)
    x[2] = 0  # an all-zero row: s_a = 0, y = 0
    wb = synth.bf16_normal((N, K), 5, 1)
    sb = synth.sign_bits(K, 5, 2)
    qw, sw, _ = oracle.hadamard32_quant_i8(wb, sb)
    y = q.gemm_w8a8_hadamard(x.to(DEV), sb.to(DEV), torch.from_numpy(qw).to(DEV), torch.from_numpy(sw).to(DEV))
    torch.cuda.synchronize()
    assert torch.all(y[2] == 0)
    L = q.lib()
    p = ctypes.c_void_p(y.data_ptr())
    ws = torch.zeros(L.qg_w8a8_hadamard_workspace_size(16, 4096), dtype=torch.uint8, device=DEV)
    w = ctypes.c_void_p(ws.data_ptr())
    assert L.gemm_w8a8_hadamard(p, p, p, p, p, 17, 64, 1024, w, ws.numel(), None) == 3   # M > 16
    assert L.gemm_w8a8_hadamard(p, p, p, p, p, 4, 64, 8192, w, ws.numel(), None) == 3   # K > 4096
    assert L.gemm_w8a8_hadamard(p, p, p, p, p, 4, 64, 1536, w, ws.numel(), None) == 3   # K % 1024
    assert L.gemm_w8a8_hadamard(p, p, p, p, p, 4, 64, 1024, w, 16, None) == 4           # workspace
    assert L.gemm_w8a8_hadamard(p, p, p, p, p, 4, 64, 1000, w, ws.numel(), None) == 1   # K % 32
    assert q.device_error() == 0
