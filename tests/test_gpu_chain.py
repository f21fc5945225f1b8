"""GPU parity of the W4A16 projection chain (qgemv_w4a16_chain_*): M = 1
projections with dependency levels in one persistent launch ("MLX Runner: An
Inference Engine You Can Read", "Architecture: one command buffer per token").

Each projection's y is checked against the oracle's W4A16 definition applied
to the input that projection read: given bf16, or derived by the oracle's
chain_x from the GPU's own output of the earlier level (so errors of one
level do not compound into the next). Tolerance as everywhere:
|y - y_ref| <= 2e-3 sum|x w| + 1e-5.
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


def _x_of(item, ys_by_id):
    """bf16 bits of the input a chain item read (host numpy)."""
    if item["op"] == oracle.X_BF16:
        return item["x"].cpu()
    src = ys_by_id[id(item["x"])].cpu().numpy()
    return oracle.chain_x(src, item["op"], item.get("alpha", 1.0), item["wq"].shape[1] * 8)


def _check(items, what):
    ys = {id(it["y"]): it["y"] for it in items}
    for i, it in enumerate(items):
        x = _x_of(it, ys)
        yr, ad = oracle.w4a16(it["wq"].cpu(), it["scales"].cpu(), it["biases"].cpu(), x)
        close(it["y"], yr[0], ad[0], f"{what} item {i}")


def _w(N, K, seed, slot):
    return [t.to(DEV) for t in synth.w4_weights(N, K, seed=seed, slot=slot)]


def test_chain_levels_ops_and_ragged_shapes(q):
    # level 0: two projections reading one bf16 x; level 1: a scaled copy of
    # one and the SwiGLU of the other; level 2: a three-group K; level 3: a
    # two-chunk K (4096 + 192) and a single-row output.
    x0 = synth.bf16_normal((512,), 21, 0).to(DEV)
    f32 = lambda n: torch.full((n,), float("nan"), device=DEV)  # noqa: E731
    A = dict(zip(("wq", "scales", "biases"), _w(256, 512, 21, 1)), level=0, op=q.X_BF16, x=x0, y=f32(256))
    B = dict(zip(("wq", "scales", "biases"), _w(1024, 512, 21, 2)), level=0, op=q.X_BF16, x=x0, y=f32(1024))
    C = dict(zip(("wq", "scales", "biases"), _w(4288, 256, 21, 3)), level=1, op=q.X_COPY, x=A["y"], alpha=0.5,
             y=f32(4288))
    D = dict(zip(("wq", "scales", "biases"), _w(200, 512, 21, 4)), level=1, op=q.X_SWIGLU, x=B["y"], alpha=1.0,
             y=f32(200))
    E = dict(zip(("wq", "scales", "biases"), _w(77, 192, 21, 5)), level=2, op=q.X_COPY, x=D["y"], alpha=0.7,
             y=f32(77))
    F = dict(zip(("wq", "scales", "biases"), _w(33, 4288, 21, 6)), level=3, op=q.X_COPY, x=C["y"], alpha=0.25,
             y=f32(33))
    G = dict(zip(("wq", "scales", "biases"), _w(1, 64, 21, 7)), level=3, op=q.X_COPY, x=E["y"], alpha=1.0,
             y=f32(1))
    items = [A, B, C, D, E, F, G]
    ch = q.GemvChain(items)
    ch.run()
    torch.cuda.synchronize()
    _check(items, "small chain")
    assert q.device_error() == 0
    ch.close()


def test_chain_repeated_runs_are_bit_identical(q):
    # the level counters return to zero after every run; results are deterministic
    x0 = synth.bf16_normal((4096,), 22, 0).to(DEV)
    items = []
    prev = None
    for lvl, (N, K) in enumerate([(4096, 4096), (24576, 4096), (4096, 12288), (1000, 4096)]):
        it = dict(zip(("wq", "scales", "biases"), _w(N, K, 22, 1 + lvl)), level=lvl,
                  y=torch.empty(N, device=DEV))
        if prev is None:
            it.update(op=q.X_BF16, x=x0)
        elif K == 12288:
            it.update(op=q.X_SWIGLU, x=prev["y"], alpha=1.0)
        else:
            it.update(op=q.X_COPY, x=prev["y"], alpha=0.4)
        items.append(it)
        prev = it
    ch = q.GemvChain(items)
    ch.run()
    torch.cuda.synchronize()
    first = [it["y"].clone() for it in items]
    _check(items, "four-level chain")
    for _ in range(3):
        ch.run()
    torch.cuda.synchronize()
    for a, it in zip(first, items):
        assert torch.equal(a, it["y"])
    assert q.device_error() == 0
    ch.close()


def test_chain_one_level_matches_group_results_within_tolerance(q):
    # all projections independent (one level): the same step as the grouped launch
    specs = [(4096, 4096), (1024, 4096), (1024, 4096), (24576, 4096), (4096, 12288)]
    items = []
    for i, (N, K) in enumerate(specs):
        x = synth.bf16_normal((K,), 23, 10 + i).to(DEV)
        items.append(dict(zip(("wq", "scales", "biases"), _w(N, K, 23, i)), level=0, op=q.X_BF16, x=x,
                          y=torch.empty(N, device=DEV)))
    ch = q.GemvChain(items)
    ch.run()
    torch.cuda.synchronize()
    _check(items, "one-level chain")
    ch.close()


def decoder_items(q, mats, x0, dev):
    """The decode step of the dense stack in dependency order: per layer
    {q, k, v} (level 4l, reading the layer input), o (reading q's output: the
    stand-in for attention), gate_up (reading o's output), down (reading the
    gate half of gate_up's output); the next layer and the lm_head read down's
    output. Every input is a copy scaled by 1 / (0.02 sqrt(K_src)) -- the
    weights' std is 0.02, so each level keeps the activations O(1), in place
    of the norm layers; a fixed-scale SwiGLU would square them every layer
    (the small chain tests cover it)."""
    items, level, layer_in = [], 0, (q.X_BF16, x0, 1.0)
    by = {}
    for name, N, K, wq, s, b in mats:
        kind = name.split(".")[-1]
        y = torch.empty(N, device=dev)
        if kind in ("q", "k", "v") or kind == "lm_head":
            op, x, alpha = layer_in
            lvl = level
        elif kind == "o":
            op, x, alpha, lvl = q.X_COPY, by["q"], 1.0 / (0.02 * 64.0), level + 1
        elif kind == "gate_up":
            op, x, alpha, lvl = q.X_COPY, by["o"], 1.0 / (0.02 * 64.0), level + 2
        else:  # down
            op, x, alpha, lvl = q.X_COPY, by["gate_up"], 1.0 / (0.02 * 64.0), level + 3
        items.append(dict(wq=wq, scales=s, biases=b, level=lvl, op=op, x=x, alpha=alpha, y=y))
        by[kind] = y
        if kind == "down":
            level += 4
            layer_in = (q.X_COPY, y, 1.0 / (0.02 * 12288 ** 0.5))
    return items


def test_chain_full_decoder_stack_sampled_rows(q):
    # the bench's dependent-order step: 36 layers + lm_head, 145 levels, one launch
    shapes = synth.stack_layer_shapes()
    mats = []
    for i, (name, N, K) in enumerate(shapes):
        wq, s, b = synth.w4_weights(N, K, seed=1, slot=10 + i, device=DEV)
        mats.append((name, N, K, wq, s, b))
    x0 = synth.bf16_normal((4096,), 1, 4999, device=DEV)
    items = decoder_items(q, mats, x0, DEV)
    assert items[-1]["level"] == 144
    ch = q.GemvChain(items)
    ch.run()
    torch.cuda.synchronize()
    ys = {id(it["y"]): it["y"] for it in items}
    rng = np.random.default_rng(24)
    for i, it in enumerate(items):
        N = it["y"].numel()
        rows = np.unique(np.concatenate([rng.integers(0, N, 6), [0, N - 1]]))
        x = _x_of(it, ys)
        ridx = torch.from_numpy(rows).to(DEV)
        yr, ad = oracle.w4a16_rows(it["wq"][ridx].cpu(), it["scales"][ridx].cpu(), it["biases"][ridx].cpu(),
                                   x, np.arange(len(rows)))
        close(it["y"][ridx], yr[0], ad[0], f"{shapes[i][0]} rows {rows.tolist()}")
        assert torch.isfinite(it["y"]).all()
    assert q.device_error() == 0
    ch.close()


def test_chain_rejects_bad_descriptors(q):
    import ctypes
    wq, s, b = _w(64, 128, 25, 0)
    x = synth.bf16_normal((128,), 25, 1).to(DEV)
    y = torch.empty(64, device=DEV)
    ok = dict(wq=wq, scales=s, biases=b, level=0, op=q.X_BF16, x=x, y=y)
    with pytest.raises(q.QGError) as e:  # levels must not decrease
        q.GemvChain([dict(ok, level=1), dict(ok, level=0, y=torch.empty(64, device=DEV))])
    assert e.value.status == 1
    # K = 96 is not a multiple of 64
    wq2 = torch.zeros((64, 12), dtype=torch.int32, device=DEV)
    s2 = torch.zeros((64, 8), dtype=torch.float16, device=DEV)
    with pytest.raises(q.QGError) as e:
        q.GemvChain([dict(ok, wq=wq2, scales=s2, biases=s2)])
    assert e.value.status == 1
    wq3, s3, b3 = _w(8, 16384 + 64, 25, 3)  # K above 16384
    with pytest.raises(q.QGError) as e:
        q.GemvChain([dict(ok, wq=wq3, scales=s3, biases=b3, x=synth.bf16_normal((16448,), 25, 4).to(DEV),
                          y=torch.empty(8, device=DEV))])
    assert e.value.status == 3
    L = q.lib()
    h = ctypes.c_void_p()
    assert L.qgemv_w4a16_chain_create(None, 1, 64, ctypes.byref(h)) == 1
    assert L.qgemv_w4a16_chain_run(None, None) == 1
    L.qgemv_w4a16_chain_destroy(None)
