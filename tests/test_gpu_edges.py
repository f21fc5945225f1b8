"""GPU parity at the edges of the stored formats.

* MXFP4 (E2M1 codes, E8M0 block scales): the smallest exponents e = 0 (the
  oracle's 2^-127; the warp-level MMA path reads it as 0, a difference far
  below the absolute tolerance) and e = 1, large ones (e = 200, i.e. 2^73) in
  the down projection, and e = 254 on blocks whose codes are all zero.
  Sources: "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin),
  "Technical approach / compute" (MXFP4 expert weights).
* Affine 4-bit W4A16 groups ("MLX Runner: An Inference Engine You Can Read",
  "Architecture: one command buffer per token") with fp16 scales and biases at
  the ends of fp16's range: subnormals (down to 2^-24) and 65504, on every M =
  1 and skinny path.
Tolerance as everywhere: |y - y_ref| <= 2e-3 sum|x w| + 1e-5.
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


def close(y_gpu, y_ref, absdot, what=""):
    y = y_gpu.detach().cpu().double().numpy().reshape(y_ref.shape)
    tol = oracle.tolerance(absdot)
    bad = np.abs(y - y_ref) > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst "
                           f"{np.max(np.abs(y - y_ref) / tol):.3g}x tol")
    assert np.isfinite(y).all()


def _moe_edge_inputs(E, H, I, T, seed):
    x = synth.bf16_normal((T, H), seed, 0)
    lg = synth.router_logits(T, E, seed, 1)
    gq, gs = synth.mxfp4_weights(E * I, H, seed, 2)
    uq, us = synth.mxfp4_weights(E * I, H, seed, 3)
    dq, ds = synth.mxfp4_weights(E * H, I, seed, 4)
    r = np.random.default_rng(seed)
    gs, us, ds = gs.numpy().copy(), us.numpy().copy(), ds.numpy().copy()
    gq, uq, dq = gq.numpy().copy(), uq.numpy().copy(), dq.numpy().copy()
    # gate/up: a fifth of the blocks at the smallest exponents
    for s in (gs, us):
        m = r.random(s.shape) < 0.2
        s[m] = r.choice(np.array([0, 1], np.uint8), size=int(m.sum()))
    # down: large exponents on some blocks, 254 on blocks whose codes are zero
    m = r.random(ds.shape) < 0.1
    ds[m] = 200
    z = r.random(ds.shape) < 0.05
    ds[z] = 254
    rows, blks = np.nonzero(z)
    for rr, bb in zip(rows, blks):
        dq[rr, 16 * bb:16 * bb + 16] = 0  # the block's 32 codes (two per byte)
    w = [torch.from_numpy(t).reshape(E, n, -1).contiguous() for t, n in
         ((gq, I), (gs, I), (uq, I), (us, I), (dq, H), (ds, H))]
    return x, lg, w


@pytest.mark.parametrize("E,H,I,T,k", [(8, 512, 512, 4, 2), (16, 1024, 512, 16, 4), (8, 256, 128, 3, 2),
                                       (16, 512, 512, 40, 4)])
def test_moe_e8m0_extreme_exponents(q, E, H, I, T, k):
    # (8, 512, 512): warp-level MMA path; (8, 256, 128): one warp per row;
    # T = 40: block-scaled tcgen05 path
    x, lg, w = _moe_edge_inputs(E, H, I, T, seed=60 + T)
    assert (w[5] == 254).any() and (w[5] == 200).any() and (w[1] == 0).any()
    dev = [t.to(DEV) for t in w]
    y, idx, wt = q.moe_mxfp4_expert_forward(x.to(DEV), lg.to(DEV), *dev, top_k=k)
    torch.cuda.synchronize()
    cache = {}

    def get_expert(e):
        if e not in cache:
            cache[e] = tuple(t[e].numpy() for t in w)
        return cache[e]

    ref = oracle.moe_forward(x, lg, None, None, None, None, None, None, k, get_expert=get_expert)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    yy = y.cpu().double().numpy()
    assert np.isfinite(yy).all()
    for t, yr in ref["y"].items():
        d = np.abs(yy[t] - yr)
        assert np.all(d <= ref["ybound"][t]), f"token {t}: worst {np.max(d / ref['ybound'][t]):.3g}x"
    assert np.abs(yy).max() > 1e15  # the 2^73 blocks did contribute


def _extreme_affine(N, K, seed):
    wq, s, b = synth.w4_weights(N, K, seed=seed, slot=0)
    r = np.random.default_rng(seed)
    sh = s.numpy().view(np.uint16).copy()
    bh = b.numpy().view(np.uint16).copy()
    pick = r.random(sh.shape)
    # fp16 subnormals (2^-24 .. 1023 * 2^-24), the largest finite value, and
    # the smallest normal, with random signs for the biases
    sh[pick < 0.15] = r.integers(1, 1024, int((pick < 0.15).sum()), dtype=np.uint16)
    sh[(pick >= 0.15) & (pick < 0.25)] = 0x7BFF
    sh[(pick >= 0.25) & (pick < 0.3)] = 0x0400
    pick = r.random(bh.shape)
    bh[pick < 0.15] = r.integers(1, 1024, int((pick < 0.15).sum()), dtype=np.uint16) | \
        (r.integers(0, 2, int((pick < 0.15).sum()), dtype=np.uint16) << 15)
    bh[(pick >= 0.15) & (pick < 0.25)] = 0xFBFF  # -65504
    s = torch.from_numpy(sh.view(np.int16)).view(torch.float16)
    b = torch.from_numpy(bh.view(np.int16)).view(torch.float16)
    return wq, s, b


@pytest.mark.parametrize("N,K", [(300, 4096), (77, 12288), (1000, 2048)])
def test_w4a16_gemv_extreme_fp16_scales(q, N, K):
    wq, s, b = _extreme_affine(N, K, seed=70 + N)
    x = synth.bf16_normal((K,), 71, 1)
    yr, ad = oracle.w4a16(wq, s, b, x)
    y = q.qgemv_w4a16(wq.to(DEV), s.to(DEV), b.to(DEV), x.to(DEV))
    close(y, yr[0], ad[0], f"gemv {N}x{K}")
    # the same projection through the chain (one level)
    yc = torch.empty(N, device=DEV)
    ch = q.GemvChain([dict(wq=wq.to(DEV), scales=s.to(DEV), biases=b.to(DEV), level=0, op=q.X_BF16,
                           x=x.to(DEV), y=yc)])
    ch.run()
    torch.cuda.synchronize()
    close(yc, yr[0], ad[0], f"chain {N}x{K}")
    ch.close()


@pytest.mark.parametrize("M", [2, 4, 16, 24])
def test_w4a16_skinny_extreme_fp16_scales(q, M):
    N, K = 520, 4096
    wq, s, b = _extreme_affine(N, K, seed=80 + M)
    x = synth.bf16_normal((M, K), 81, 1)
    yr, ad = oracle.w4a16(wq, s, b, x)
    y = q.qgemm_w4a16_skinny(wq.to(DEV), s.to(DEV), b.to(DEV), x.to(DEV))
    close(y, yr, ad, f"skinny M={M}")
    ys = torch.full((M, N), float("nan"), device=DEV)
    grp = q.SkinnyGroup([(wq.to(DEV), s.to(DEV), b.to(DEV), x.to(DEV), ys)])
    grp.run()
    torch.cuda.synchronize()
    close(ys, yr, ad, f"skinny group M={M}")
    grp.close()
