"""Guard bands around every output buffer (the stand-in for a memory checker,
which is closed on this machine): each entry point writes into the middle of a
larger allocation whose two guard bands hold a fixed byte pattern; after the
call the bands must be unchanged and the outputs must still match the oracle.
Shapes are ragged (N not a multiple of the kernels' tiles) so every kernel's
last tile is partial."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 4096          # bytes on each side (keeps the inner slice 16-byte aligned)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def q():
    from skinny_gemm_qgemv_gb300 import build
    build.build()
    import skinny_gemm_qgemv_gb300 as qq
    qq.lib()
    qq.device_error(clear=True)
    yield qq
    assert qq.device_error(clear=True) == 0


class Guarded:
    """A device tensor of `shape`/`dtype` inside guard bands of PATTERN bytes."""

    def __init__(self, shape, dtype):
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=DEV)
        self.nbytes = nbytes
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        lo = self.raw[:GUARD].cpu().numpy()
        hi = self.raw[GUARD + self.nbytes:].cpu().numpy()
        return bool((lo == PATTERN).all() and (hi == PATTERN).all())


def test_canaries_w4a16_gemv_skinny_and_groups(q):
    N, K = 1000, 2048
    wq, s, b = synth.w4_weights(N, K, seed=800, slot=0)
    x = synth.bf16_normal((5, K), seed=800, slot=1)
    d = [t.to(DEV) for t in (wq, s, b)]
    y1 = Guarded((N,), torch.float32)
    q.qgemv_w4a16(*d, x[0].contiguous().to(DEV), y1.t)
    y5 = Guarded((5, N), torch.float32)
    q.qgemm_w4a16_skinny(*d, x.to(DEV), y5.t)
    g1 = Guarded((N,), torch.float32)
    grp = q.GemvGroup([(d[0], d[1], d[2], x[1].contiguous().to(DEV), g1.t)])
    grp.run()
    g5 = Guarded((5, N), torch.float32)
    sgrp = q.SkinnyGroup([(d[0], d[1], d[2], x.to(DEV), g5.t)])
    sgrp.run()
    for gb in (y1, y5, g1, g5):
        assert gb.intact()
    ref, ad = oracle.w4a16(wq, s, b, x)
    for y, r, a in ((y1.t, ref[0], ad[0]), (y5.t, ref, ad), (g1.t, ref[1], ad[1]), (g5.t, ref, ad)):
        assert np.all(np.abs(y.cpu().double().numpy() - r) <= oracle.tolerance(a))
    grp.close()
    sgrp.close()


def test_canaries_hadamard_w8a8_w8a16_affine(q):
    M, K, N = 16, 1024, 1300
    xa = synth.outlier_activations(M, K, seed=801, slot=0)
    sb = synth.sign_bits(K, seed=801, slot=1)
    qa = Guarded((M, K), torch.int8)
    sa = Guarded((M,), torch.float32)
    q.hadamard32_quant_i8(xa.to(DEV), sb.to(DEV), qa.t, sa.t)
    w8 = torch.randint(-128, 128, (N, K), generator=synth.gen(801, 2), dtype=torch.int16).to(torch.int8)
    c = Guarded((M, N), torch.int32)
    q.gemm_w8a8_i32(qa.t, w8.to(DEV), c.t)
    wq16, s16 = synth.w8_row_weights(N, K, seed=801, slot=3)
    y16 = Guarded((N,), torch.float32)
    q.qgemv_w8a16(wq16.to(DEV), s16.to(DEV), xa[0].contiguous().to(DEV), y16.t)
    wqa, sca, bia = synth.affine_weights(N, K, 3, seed=801, slot=4)
    ya = Guarded((3, N), torch.float32)
    q.qgemm_affine(wqa.to(DEV), 3, sca.to(DEV), bia.to(DEV), xa[:3].contiguous().to(DEV), ya.t)
    for gb in (qa, sa, c, y16, ya):
        assert gb.intact()
    qr, sr, _ = oracle.hadamard32_quant_i8(xa, sb)
    assert np.array_equal(qa.t.cpu().numpy(), qr) and np.array_equal(sa.t.cpu().numpy(), sr)
    assert np.array_equal(c.t.cpu().numpy(), oracle.w8a8(qr, w8))
    r16, a16 = oracle.w8a16(wq16, s16, xa[0])
    assert np.all(np.abs(y16.t.cpu().double().numpy() - r16[0]) <= oracle.tolerance(a16[0]))
    ra, aa = oracle.affine(wqa, 3, sca, bia, xa[:3])
    assert np.all(np.abs(ya.t.cpu().double().numpy() - ra) <= oracle.tolerance(aa))


@pytest.mark.parametrize("T", [1, 5])
def test_canaries_moe(q, T):
    E, H, I, k = 16, 1536, 1024, 4
    x = synth.bf16_normal((T, H), 802, 0)
    lg = synth.router_logits(T, E, 802, 1)
    gq, gs = synth.mxfp4_weights(E * I, H, 802, 2)
    uq, us = synth.mxfp4_weights(E * I, H, 802, 3)
    dq, ds = synth.mxfp4_weights(E * H, I, 802, 4)
    w = [t.reshape(E, rows, -1).contiguous() for t, rows in ((gq, I), (gs, I), (uq, I), (us, I), (dq, H), (ds, H))]
    y = Guarded((T, H), torch.float32)
    idx = Guarded((T, k), torch.int32)
    wt = Guarded((T, k), torch.float32)
    ws = Guarded((q.moe_workspace_size(T, H, I, E, k),), torch.uint8)
    q.moe_mxfp4_expert_forward(x.to(DEV), lg.to(DEV), *[t.to(DEV) for t in w], top_k=k, y=y.t,
                               topk_idx=idx.t, topk_w=wt.t, workspace=ws.t)
    for gb in (y, idx, wt, ws):
        assert gb.intact()
    ref = oracle.moe_forward(x, lg, *w, top_k=k)
    assert np.array_equal(idx.t.cpu().numpy(), ref["idx"])
    for t in range(T):
        assert np.all(np.abs(y.t[t].cpu().double().numpy() - ref["y"][t]) <= ref["ybound"][t])
