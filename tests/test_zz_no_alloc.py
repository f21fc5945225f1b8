"""The allocation-free MoE entry point, called through the C ABI.

moe_mxfp4_expert_forward_noalloc serves callers that cannot allocate device
memory when they run the layer (a plugin handed only its input and output
buffers, a runtime with one pre-reserved pool, code recorded during CUDA graph
capture): its scratch is a fixed-size array inside the library. This test runs
it twice in a row and compares each result with the workspace entry point on
the same inputs, within the accuracy bound the other MoE tests use (computed
by the CPU oracle). It lives in its own file, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice():
    from skinny_gemm_qgemv_gb300 import build
    build.build()
    import skinny_gemm_qgemv_gb300 as q
    L = q.lib()
    dev = "cuda"
    E, H, I, T, k = 16, 512, 256, 4, 4
    x = synth.bf16_normal((T, H), 51, 0)
    lg = synth.router_logits(T, E, 51, 1)
    gq, gs = synth.mxfp4_weights(E * I, H, 51, 2)
    uq, us = synth.mxfp4_weights(E * I, H, 51, 3)
    dq, ds = synth.mxfp4_weights(E * H, I, 51, 4)
    w = [t.reshape(E, rows, -1).contiguous() for t, rows in
         ((gq, I), (gs, I), (uq, I), (us, I), (dq, H), (ds, H))]
    wd = [t.to(dev) for t in w]
    xd, lgd = x.to(dev), lg.to(dev)

    # reference: the workspace entry point (through the same C ABI)
    y_ref, idx_ref, w_ref = q.moe_mxfp4_expert_forward(xd, lgd, *wd, top_k=k)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(x, lg, *w, top_k=k)

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        y = torch.full((T, H), float("nan"), device=dev)
        idx = torch.full((T, k), -1, dtype=torch.int32, device=dev)
        wt = torch.full((T, k), float("nan"), device=dev)
        st = L.moe_mxfp4_expert_forward_noalloc(_ptr(xd), _ptr(lgd), *[_ptr(t) for t in wd], T, H, I, E, k,
                                                _ptr(y), _ptr(idx), _ptr(wt), stream)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref)
        assert np.array_equal(idx.cpu().numpy(), ref["idx"])
        assert np.allclose(wt.cpu().double().numpy(), w_ref.cpu().double().numpy(), rtol=1e-6, atol=0)
        for t in range(T):
            d = np.abs(y[t].cpu().double().numpy() - y_ref[t].cpu().double().numpy())
            assert np.all(d <= ref["ybound"][t]), f"call {call} token {t}"
            assert np.all(np.abs(y[t].cpu().double().numpy() - ref["y"][t]) <= ref["ybound"][t])
    assert q.device_error(clear=True) == 0


def test_noalloc_refuses_problems_beyond_its_scratch():
    import skinny_gemm_qgemv_gb300 as q
    L = q.lib()
    cap = L.qg_moe_noalloc_max_bytes()
    assert cap == 8 << 20
    # 384 experts of 7168 x 2048, top-16: 40 tokens need more than the scratch
    assert L.qg_moe_workspace_size(40, 7168, 2048, 384, 16) > cap
    dummy = torch.empty(1024, dtype=torch.uint8, device="cuda")
    p = _ptr(dummy)
    st = L.moe_mxfp4_expert_forward_noalloc(p, p, p, p, p, p, p, p, 40, 7168, 2048, 384, 16, p, p, p, None)
    assert st == 4  # QG_ERR_WORKSPACE, nothing launched
