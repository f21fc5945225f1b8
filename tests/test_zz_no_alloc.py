"""The allocation-free MoE entry point, called through the C ABI.

moe_mxfp4_expert_forward_noalloc serves callers that cannot allocate device
memory when they run the layer (a plugin handed only its input and output
buffers, a runtime with one pre-reserved pool, code recorded during CUDA graph
capture): its scratch is a fixed-size array inside the library. The test runs
it on four shapes -- the one-warp-per-row path at 4 and at 36 tokens, and the
warp-level MMA path that serves the real expert shapes at 4 tokens and at its
largest batch of 32 (larger batches of the real shapes need more scratch than
the array holds) -- twice in a row with
different inputs (so that anything a call read from the scratch without
writing it first would show), and requires each result to be bit-identical to
the workspace entry point's on the same inputs (the same kernels run on the
same data) and within the oracle's accuracy bound. It lives in its own file,
collected last.
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


def _inputs(E, H, I, T, seed):
    x = synth.bf16_normal((T, H), seed, 0)
    lg = synth.router_logits(T, E, seed, 1)
    gq, gs = synth.mxfp4_weights(E * I, H, seed, 2)
    uq, us = synth.mxfp4_weights(E * I, H, seed, 3)
    dq, ds = synth.mxfp4_weights(E * H, I, seed, 4)
    w = [t.reshape(E, rows, -1).contiguous() for t, rows in
         ((gq, I), (gs, I), (uq, I), (us, I), (dq, H), (ds, H))]
    return x, lg, w


# (E, H, I, T, top_k): one-warp-per-row path (I not a multiple of 512), warp-level
# MMA path at 4 and at 32 tokens, and a batch above 32 tokens on the
# one-warp-per-row path
@pytest.mark.parametrize("E,H,I,T,k", [(16, 512, 256, 4, 4), (64, 512, 512, 4, 8), (32, 1024, 512, 32, 8),
                                       (8, 256, 128, 36, 2)])
def test_noalloc_matches_workspace_entry_point_twice(E, H, I, T, k):
    from skinny_gemm_qgemv_gb300 import build
    build.build()
    import skinny_gemm_qgemv_gb300 as q
    L = q.lib()
    dev = "cuda"
    assert L.qg_moe_workspace_size(T, H, I, E, k) <= L.qg_moe_noalloc_max_bytes()
    x, lg, w = _inputs(E, H, I, T, 51)
    wd = [t.to(dev) for t in w]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        # the second call routes differently (other logits and activations)
        if call == 1:
            x = synth.bf16_normal((T, H), 52, 0)
            lg = synth.router_logits(T, E, 52, 1)
        xd, lgd = x.to(dev), lg.to(dev)
        y_ref, idx_ref, w_ref = q.moe_mxfp4_expert_forward(xd, lgd, *wd, top_k=k)
        torch.cuda.synchronize()
        ref = oracle.moe_forward(x, lg, *w, top_k=k)
        y = torch.full((T, H), float("nan"), device=dev)
        idx = torch.full((T, k), -1, dtype=torch.int32, device=dev)
        wt = torch.full((T, k), float("nan"), device=dev)
        st = L.moe_mxfp4_expert_forward_noalloc(_ptr(xd), _ptr(lgd), *[_ptr(t) for t in wd], T, H, I, E, k,
                                                _ptr(y), _ptr(idx), _ptr(wt), stream)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref), f"call {call}"
        assert torch.equal(wt, w_ref), f"call {call}"
        assert torch.equal(y, y_ref), f"call {call}"
        assert np.array_equal(idx.cpu().numpy(), ref["idx"])
        for t in range(T):
            assert np.all(np.abs(y[t].cpu().double().numpy() - ref["y"][t]) <= ref["ybound"][t]), \
                f"call {call} token {t}"
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
