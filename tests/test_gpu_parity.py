"""GPU parity: every entry point of the C ABI against the CPU oracle.

Float outputs must satisfy |y - y_ref| <= 2e-3 * sum|x w| + 1e-5 per element
(the oracle computes y_ref and sum|x w| in float64); integer outputs (int8
codes and scales of the Hadamard path, int32 W8A8, MoE expert indices) must
match bit for bit. Inputs come from the seeded generators in `synth`.
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


def w4_case(N, K, M, seed, device="cpu"):
    wq, s, b = synth.w4_weights(N, K, seed=seed, slot=0, device=device)
    x = synth.bf16_normal((M, K), seed=seed, slot=1, device=device)
    return wq, s, b, x


# ---------------------------------------------------------------- W4A16 GEMV, M = 1

@pytest.mark.parametrize("N,K", [
    (1024, 1024),     # the single-GEMV workload (N = K = 1024)
    (300, 4096),      # ragged last tile
    (77, 2048),
    (1, 4096),        # one row
    (2050, 12288),    # down-projection K, ragged N
    (513, 3072),      # K % 2048 != 0 -> 32 codes per lane
])
def test_gemv_fast_path(q, N, K):
    wq, s, b, x = w4_case(N, K, 1, seed=100 + N)
    y = q.qgemv_w4a16(wq.to(DEV), s.to(DEV), b.to(DEV), x[0].to(DEV))
    yr, ad = oracle.w4a16(wq, s, b, x)
    close(y, yr[0], ad[0], f"gemv {N}x{K}")


@pytest.mark.parametrize("N,K", [(33, 64), (64, 960), (17, 192), (128, 1600)])
def test_gemv_generic_shapes(q, N, K):
    wq, s, b, x = w4_case(N, K, 1, seed=200 + K)
    y = q.qgemv_w4a16(wq.to(DEV), s.to(DEV), b.to(DEV), x[0].to(DEV))
    yr, ad = oracle.w4a16(wq, s, b, x)
    close(y, yr[0], ad[0], f"generic {N}x{K}")


def test_gemv_deterministic(q):
    wq, s, b, x = w4_case(4096, 4096, 1, seed=7, device=DEV)
    y1 = q.qgemv_w4a16(wq, s, b, x[0])
    y2 = q.qgemv_w4a16(wq, s, b, x[0])
    assert torch.equal(y1, y2)


def test_gemv_special_values(q):
    # all-zero codes: y = sum_g b_g * sum_{k in g} x_k ; zero activations: y = 0
    N, K = 64, 2048
    wq = torch.zeros(N, K // 8, dtype=torch.int32)
    s = (torch.rand(N, K // 64, generator=synth.gen(5, 0)) * 0.01).half()
    b = (torch.randn(N, K // 64, generator=synth.gen(5, 1)) * 0.05).half()
    x = synth.bf16_normal((1, K), 5, 2)
    y = q.qgemv_w4a16(wq.to(DEV), s.to(DEV), b.to(DEV), x[0].to(DEV))
    yr, ad = oracle.w4a16(wq, s, b, x)
    close(y, yr[0], ad[0], "zero codes")
    y0 = q.qgemv_w4a16(wq.to(DEV), s.to(DEV), b.to(DEV), torch.zeros(K, dtype=torch.bfloat16, device=DEV))
    assert torch.count_nonzero(y0) == 0


# ---------------------------------------------------------------- skinny GEMM

@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16, 32])
def test_skinny_vs_oracle(q, M):
    N, K = 320, 4096
    wq, s, b, x = w4_case(N, K, M, seed=300 + M)
    y = q.qgemm_w4a16_skinny(wq.to(DEV), s.to(DEV), b.to(DEV), x.to(DEV))
    yr, ad = oracle.w4a16(wq, s, b, x)
    close(y, yr, ad, f"skinny M={M}")


@pytest.mark.parametrize("M,N,K", [(16, 129, 12288), (5, 1000, 1024), (32, 64, 64), (2, 4097, 2048)])
def test_skinny_shapes(q, M, N, K):
    wq, s, b, x = w4_case(N, K, M, seed=400 + M)
    y = q.qgemm_w4a16_skinny(wq.to(DEV), s.to(DEV), b.to(DEV), x.to(DEV))
    yr, ad = oracle.w4a16(wq, s, b, x)
    close(y, yr, ad, f"skinny {M}x{N}x{K}")


def test_skinny_rows_match_gemv(q):
    N, K, M = 512, 4096, 8
    wq, s, b, x = w4_case(N, K, M, seed=9, device=DEV)
    Y = q.qgemm_w4a16_skinny(wq, s, b, x)
    yr, ad = oracle.w4a16(wq, s, b, x)
    for m in range(M):
        ym = q.qgemv_w4a16(wq, s, b, x[m].contiguous())
        # both within tolerance of the same exact value: within 2x of each other
        d = (Y[m] - ym).abs().cpu().double().numpy()
        assert np.all(d <= 2 * oracle.tolerance(ad[m]))


# ------------------------------------------- full-size shapes, sampled rows

STACK = [("q", 4096, 4096), ("k", 1024, 4096), ("gate_up", 24576, 4096), ("down", 4096, 12288),
         ("lm_head", 151936, 4096)]


@pytest.mark.parametrize("name,N,K", STACK)
@pytest.mark.parametrize("M", [1, 16])
def test_full_size_sampled_rows(q, name, N, K, M):
    wq, s, b, x = w4_case(N, K, M, seed=1, device=DEV)
    if M == 1:
        y = q.qgemv_w4a16(wq, s, b, x[0]).unsqueeze(0)
    else:
        y = q.qgemm_w4a16_skinny(wq, s, b, x)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(N + M)
    rows = sorted(set(torch.randint(0, N, (48,), generator=g).tolist()) | {0, N - 1})
    ridx = torch.tensor(rows, device=DEV)
    yr, ad = oracle.w4a16(wq[ridx].cpu(), s[ridx].cpu(), b[ridx].cpu(), x.cpu())
    close(y[:, ridx], yr, ad, f"{name} M={M} sampled")


# ---------------------------------------------------------------- Hadamard + int8

@pytest.mark.parametrize("M,K", [(16, 4096), (16, 12288), (3, 32), (1, 96), (33, 1024)])
def test_hadamard_quant_bit_exact(q, M, K):
    x = synth.outlier_activations(M, K, seed=4, slot=0)
    sb = synth.sign_bits(K, seed=4, slot=5)
    qg, sg = q.hadamard32_quant_i8(x.to(DEV), sb.to(DEV))
    qr, sr, _ = oracle.hadamard32_quant_i8(x, sb)
    assert np.array_equal(sg.cpu().numpy().view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(qg.cpu().numpy(), qr)


def test_hadamard_zero_row_and_plain_normals(q):
    x = synth.bf16_normal((4, 256), 6, 0)
    x[2] = 0
    sb = synth.sign_bits(256, 6, 1)
    qg, sg = q.hadamard32_quant_i8(x.to(DEV), sb.to(DEV))
    qr, sr, _ = oracle.hadamard32_quant_i8(x, sb)
    assert sg[2].item() == 0.0 and torch.count_nonzero(qg[2]) == 0
    assert np.array_equal(qg.cpu().numpy(), qr)
    assert np.array_equal(sg.cpu().numpy().view(np.uint32), sr.view(np.uint32))


# ---------------------------------------------------------------- W8A8

@pytest.mark.parametrize("M,N,K", [(16, 4096, 4096), (16, 12288, 4096), (1, 64, 64), (5, 100, 320),
                                   (32, 256, 1024), (5, 2000, 1088), (32, 1300, 2048), (16, 1217, 64),
                                   (7, 1000, 1024), (16, 130, 3072)])
def test_w8a8_exact(q, M, N, K):
    x = synth.outlier_activations(M, K, seed=4, slot=0)
    sb = synth.sign_bits(K, seed=4, slot=5)
    qa, _, _ = oracle.hadamard32_quant_i8(x, sb)
    w = torch.randint(-127, 128, (N, K), generator=synth.gen(4, 7), dtype=torch.int8)
    c = q.gemm_w8a8_i32(torch.from_numpy(qa).to(DEV), w.to(DEV))
    assert np.array_equal(c.cpu().numpy(), oracle.w8a8(qa, w))


@pytest.mark.parametrize("N", [64, 384])
def test_w8a8_extremes(q, N):
    K = 4096
    a = torch.full((16, K), 127, dtype=torch.int8)
    a[1::2] = -127
    a[3::8, ::2] = -128
    w = torch.full((N, K), -127, dtype=torch.int8)
    w[:, ::3] = 127
    w[1::5, 1::7] = -128  # the full int8 range on the weight side
    c = q.gemm_w8a8_i32(a.to(DEV), w.to(DEV))
    assert np.array_equal(c.cpu().numpy(), oracle.w8a8(a, w))


# ---------------------------------------------------------------- other affine group sizes

@pytest.mark.parametrize("group", [32, 128])
@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (1, 77, 4096), (5, 130, 2048), (32, 64, 512)])
def test_w4a16_group_sizes_32_128(q, group, M, N, K):
    wq, s, b = synth.w4_weights(N, K, seed=600 + M, slot=group, group=group)
    x = synth.bf16_normal((M, K), seed=600 + M, slot=1)
    if M == 1:
        y = q.qgemv_w4a16(wq.to(DEV), s.to(DEV), b.to(DEV), x[0].to(DEV))[None, :]
    else:
        y = q.qgemm_w4a16_skinny(wq.to(DEV), s.to(DEV), b.to(DEV), x.to(DEV))
    torch.cuda.synchronize()
    ref, ad = oracle.w4a16(wq, s, b, x, group=group)
    d = np.abs(y.cpu().double().numpy() - ref)
    assert np.all(d <= oracle.tolerance(ad)), f"worst {np.max(d / oracle.tolerance(ad)):.3g}x"


# ---------------------------------------------------------------- W8A16 row-int8 GEMV

@pytest.mark.parametrize("N,K", [(1, 16), (3, 48), (1000, 4096), (4099, 1024), (257, 12288), (33, 65536)])
def test_w8a16_vs_oracle(q, N, K):
    wq, s = synth.w8_row_weights(N, K, seed=500 + N, slot=1)
    x = synth.bf16_normal((K,), seed=500 + N, slot=2)
    y = q.qgemv_w8a16(wq.to(DEV), s.to(DEV), x.to(DEV))
    torch.cuda.synchronize()
    ref, ad = oracle.w8a16(wq, s, x)
    d = np.abs(y.cpu().double().numpy() - ref[0])
    assert np.all(d <= oracle.tolerance(ad[0])), f"worst {np.max(d / oracle.tolerance(ad[0])):.3g}x"


def test_w8a16_extremes_and_scales(q):
    # full int8 range, tiny and large activations (the fp16 prescale), zero x
    N, K = 96, 2048
    g = torch.Generator().manual_seed(7)
    wq = torch.randint(-128, 128, (N, K), generator=g, dtype=torch.int16).to(torch.int8)
    wq[0] = -128
    wq[1] = 127
    s = torch.rand(N, generator=g) * 4 + 1e-3
    for xscale in (1e-6, 1.0, 3e4):
        x = (torch.randn(K, generator=g) * xscale).to(torch.bfloat16)
        y = q.qgemv_w8a16(wq.to(DEV), s.to(DEV), x.view(torch.int16).to(DEV).view(torch.bfloat16))
        torch.cuda.synchronize()
        ref, ad = oracle.w8a16(wq, s, x)
        d = np.abs(y.cpu().double().numpy() - ref[0])
        assert np.all(d <= oracle.tolerance(ad[0]))
    y = q.qgemv_w8a16(wq.to(DEV), s.to(DEV), torch.zeros(K, dtype=torch.bfloat16, device=DEV))
    assert torch.count_nonzero(y).item() == 0


def test_w8a16_full_size_lm_head(q):
    # the int8 output head of the 9B-class decoder: 151936 x 4096
    N, K = 151936, 4096
    wq, s = synth.w8_row_weights(N, K, seed=3, slot=1, device=DEV)
    x = synth.bf16_normal((K,), seed=3, slot=2, device=DEV)
    y = q.qgemv_w8a16(wq, s, x)
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(0, 64), np.arange(N - 64, N), np.arange(1000, N, 4999)])
    ref, ad = oracle.w8a16(wq[rows].cpu(), s[rows].cpu(), x.cpu())
    d = np.abs(y.cpu().double().numpy()[rows] - ref[0])
    assert np.all(d <= oracle.tolerance(ad[0]))


# ---------------------------------------------------------------- MXFP4 MoE

def moe_inputs(E, H, I, T, seed, device="cpu"):
    x = synth.bf16_normal((T, H), seed, 0, device)
    lg = synth.router_logits(T, E, seed, 1, device)
    gq, gs = synth.mxfp4_weights(E * I, H, seed, 2, device)
    uq, us = synth.mxfp4_weights(E * I, H, seed, 3, device)
    dq, ds = synth.mxfp4_weights(E * H, I, seed, 4, device)
    w = [t.reshape(E, rows, -1).contiguous() for t, rows in
         ((gq, I), (gs, I), (uq, I), (us, I), (dq, H), (ds, H))]
    return x, lg, w


def check_moe(q, x, lg, w, top_k, tokens=None):
    T, H = x.shape
    E = lg.shape[1]
    I = w[0].shape[1]
    dev = [t.to(DEV) for t in w]
    ws = torch.empty(q.moe_workspace_size(T, H, I, E, top_k), dtype=torch.uint8, device=DEV)
    y, idx, wt = q.moe_mxfp4_expert_forward(x.to(DEV), lg.to(DEV), *dev, top_k=top_k, workspace=ws)
    torch.cuda.synchronize()
    cache = {}

    def get_expert(e):
        if e not in cache:
            cache[e] = tuple(t[e].cpu().numpy() for t in w)
        return cache[e]

    ref = oracle.moe_forward(x.cpu(), lg.cpu(), None, None, None, None, None, None, top_k,
                             tokens=tokens, get_expert=get_expert)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.allclose(wt.cpu().double().numpy(), ref["w"], rtol=1e-6, atol=0)
    # stage-wise: the kernel's fp32 h against g, u of the oracle
    off = q.moe_workspace_h_offset(T, H, I, E, top_k)
    hk = ws[off:off + 4 * T * top_k * I].view(torch.float32).reshape(T * top_k, I).cpu().double().numpy()
    for (t, j), h in ref["h"].items():
        assert np.all(np.abs(hk[t * top_k + j] - h) <= ref["hbound"][(t, j)]), f"h of pair {(t, j)}"
    for t, yr in ref["y"].items():
        d = np.abs(y[t].cpu().double().numpy() - yr)
        assert np.all(d <= ref["ybound"][t]), f"token {t}: worst {np.max(d / ref['ybound'][t]):.3g}x"
    return y, idx


@pytest.mark.parametrize("E,H,I,T,k", [(8, 256, 128, 3, 2), (16, 512, 256, 5, 4), (4, 64, 64, 1, 4),
                                       (32, 1024, 512, 16, 8), (24, 1536, 1024, 7, 6), (8, 512, 512, 32, 4),
                                       (40, 2048, 512, 12, 8), (300, 7168, 512, 2, 16),
                                       (16, 4096, 1024, 3, 4), (8, 8192, 512, 2, 2), (700, 512, 512, 2, 8)])
def test_moe_small(q, E, H, I, T, k):
    x, lg, w = moe_inputs(E, H, I, T, seed=30 + E)
    check_moe(q, x, lg, w, k)


def test_moe_tied_logits_pick_lower_index(q):
    E, H, I, T, k = 16, 128, 64, 2, 5
    x, lg, w = moe_inputs(E, H, I, T, seed=41)
    lg = torch.zeros_like(lg)
    lg[1, [3, 9, 12]] = 0.5
    y, idx = check_moe(q, x, lg, w, k)
    assert idx[0].tolist() == [0, 1, 2, 3, 4]
    assert idx[1].tolist() == [3, 9, 12, 0, 1]


def test_moe_ties_at_the_threshold_main_path(q):
    # H, I multiples of 512: the warp radix-select router. Equal logits
    # straddle the k-th place; -0.0 and +0.0 compare equal.
    E, H, I, T, k = 64, 512, 512, 4, 8
    x, lg, w = moe_inputs(E, H, I, T, seed=43)
    lg[0] = 0.0
    lg[1] = 0.0
    lg[1, [3, 9, 12, 40, 41]] = 1.0
    lg[2] = -1.0
    lg[2, 5] = -0.0
    lg[2, 6] = 0.0
    lg[2, [20, 21, 30]] = 2.0
    y, idx = check_moe(q, x, lg, w, k)
    assert idx[0].tolist() == list(range(8))
    assert idx[1].tolist() == [3, 9, 12, 40, 41, 0, 1, 2]
    assert idx[2].tolist()[:5] == [20, 21, 30, 5, 6]
    assert idx[2].tolist()[5:] == [0, 1, 2]


def test_moe_shared_experts_split_into_virtual_experts(q):
    # every token picks experts 0..k-1 (zero logits, ties to the lower index):
    # 20 pairs per expert, more than one MMA's 8 columns
    E, H, I, T, k = 12, 1024, 512, 20, 3
    x, lg, w = moe_inputs(E, H, I, T, seed=47)
    lg = torch.zeros_like(lg)
    y, idx = check_moe(q, x, lg, w, k)
    assert (idx == torch.tensor([0, 1, 2], dtype=idx.dtype, device=idx.device)).all()


@pytest.mark.parametrize("T", [1, 16, 24])
def test_moe_full_size(q, T):
    # hidden 7168, intermediate 2048, 384 experts, top-16; tokens sampled
    E, H, I, k = 384, 7168, 2048, 16
    x, lg, w = moe_inputs(E, H, I, T, seed=3, device=DEV)
    check_moe(q, x, lg, w, k, tokens=[0] if T == 1 else [0, 7, T - 1])


# Batches of 33..64 tokens run on the block-scaled tensor-core path (one
# accumulator buffer once a batch's columns no longer fit two; B spans that
# start past the first 16-column block; ranges that start mid-window).
@pytest.mark.parametrize("E,H,I,T,k", [(24, 1024, 512, 33, 6), (64, 512, 512, 40, 8), (48, 1536, 1024, 64, 4),
                                       (16, 2048, 512, 48, 2)])
def test_moe_tc_batches(q, E, H, I, T, k):
    x, lg, w = moe_inputs(E, H, I, T, seed=60 + T, device=DEV)
    check_moe(q, x, lg, w, k)


def test_moe_tc_full_size(q):
    # the full layer (384 experts of 7168 x 2048, top-16) at a 48-token batch; tokens sampled
    E, H, I, T, k = 384, 7168, 2048, 48, 16
    x, lg, w = moe_inputs(E, H, I, T, seed=3, device=DEV)
    check_moe(q, x, lg, w, k, tokens=[0, 17, 33, T - 1])


# ---------------------------------------------------------------- grouped M = 1 GEMV

def test_gemv_group_vs_oracle(q):
    shapes = [(300, 4096), (77, 2048), (1, 4096), (2050, 12288), (513, 6144), (129, 16384), (1024, 4096),
              (1023, 8192)]
    cases = [w4_case(N, K, 1, seed=400 + i) for i, (N, K) in enumerate(shapes)]
    dev = [(wq.to(DEV), s.to(DEV), b.to(DEV), x[0].to(DEV), torch.empty(wq.shape[0], device=DEV))
           for wq, s, b, x in cases]
    grp = q.GemvGroup(dev)
    grp.run()
    torch.cuda.synchronize()
    first = [d[4].clone() for d in dev]
    for (wq, s, b, x), d, (N, K) in zip(cases, dev, shapes):
        yr, ad = oracle.w4a16(wq, s, b, x)
        close(d[4], yr[0], ad[0], f"group {N}x{K}")
    # a second run gives the same bits; a changed activation is picked up
    grp.run()
    torch.cuda.synchronize()
    for d, f in zip(dev, first):
        assert torch.equal(d[4], f)
    wq, s, b, x = cases[0]
    x2 = synth.bf16_normal((1, 4096), seed=999, slot=1)
    dev[0][3].copy_(x2[0].to(DEV))
    grp.run()
    torch.cuda.synchronize()
    yr, ad = oracle.w4a16(wq, s, b, x2)
    close(dev[0][4], yr[0], ad[0], "group rerun with new x")
    grp.close()


def test_gemv_group_full_stack_layer_sampled(q):
    # one decoder layer of the stack plus the lm_head as one group, full size
    shapes = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
              ("gate_up", 24576, 4096), ("down", 4096, 12288), ("lm_head", 151936, 4096)]
    items, host = [], []
    for i, (name, N, K) in enumerate(shapes):
        wq, s, b, x = w4_case(N, K, 1, seed=50 + i, device=DEV)
        items.append((wq, s, b, x[0], torch.empty(N, device=DEV)))
    grp = q.GemvGroup(items)
    grp.run()
    torch.cuda.synchronize()
    for (name, N, K), (wq, s, b, x, y) in zip(shapes, items):
        g = torch.Generator().manual_seed(N)
        rows = sorted(set(torch.randint(0, N, (32,), generator=g).tolist()) | {0, N - 1})
        ridx = torch.tensor(rows, device=DEV)
        yr, ad = oracle.w4a16(wq[ridx].cpu(), s[ridx].cpu(), b[ridx].cpu(), x.unsqueeze(0).cpu())
        close(y[ridx].unsqueeze(0), yr, ad, f"group {name} sampled")
    grp.close()


# ------------------------------------------- grouped skinny GEMM (tcgen05)

@pytest.mark.parametrize("M", [2, 3, 16, 17, 32])
def test_skinny_group_vs_oracle(q, M):
    # several projections of mixed N (ragged last tiles, a one-row matrix) and
    # mixed K in one launch; each against the oracle
    shapes = [(300, 4096), (77, 512), (1, 1024), (2050, 12288), (513, 6144), (129, 1536), (1024, 4096)]
    cases = [w4_case(N, K, M, seed=700 + 13 * M + i) for i, (N, K) in enumerate(shapes)]
    dev = [(wq.to(DEV), s.to(DEV), b.to(DEV), x.to(DEV), torch.full((M, wq.shape[0]), float("nan"), device=DEV))
           for wq, s, b, x in cases]
    grp = q.SkinnyGroup(dev)
    grp.run()
    torch.cuda.synchronize()
    first = [d[4].clone() for d in dev]
    for (wq, s, b, x), d, (N, K) in zip(cases, dev, shapes):
        yr, ad = oracle.w4a16(wq, s, b, x)
        close(d[4], yr, ad, f"skinny group M={M} {N}x{K}")
    # a second run gives the same bits; a changed activation is picked up
    grp.run()
    torch.cuda.synchronize()
    for d, f in zip(dev, first):
        assert torch.equal(d[4], f)
    wq, s, b, x = cases[0]
    x2 = synth.bf16_normal((M, 4096), seed=998, slot=1)
    dev[0][3].copy_(x2.to(DEV))
    grp.run()
    torch.cuda.synchronize()
    yr, ad = oracle.w4a16(wq, s, b, x2)
    close(dev[0][4], yr, ad, "skinny group rerun with new x")
    grp.close()


def test_skinny_group_matches_single_calls(q):
    # the grouped launch and the one-matrix launch compute the same sums for
    # full-K tiles: identical bits when the single call does not split K
    N, K, M = 4096, 4096, 16
    wq, s, b, x = w4_case(N, K, M, seed=31, device=DEV)
    y = torch.empty(M, N, device=DEV)
    grp = q.SkinnyGroup([(wq, s, b, x, y)])
    grp.run()
    torch.cuda.synchronize()
    yr, ad = oracle.w4a16(wq.cpu(), s.cpu(), b.cpu(), x.cpu())
    close(y, yr, ad, "skinny group one matrix")
    grp.close()


def test_skinny_group_full_stack_layer_sampled(q):
    # one decoder layer of the stack plus the lm_head as one group, M = 16, full size
    shapes = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
              ("gate_up", 24576, 4096), ("down", 4096, 12288), ("lm_head", 151936, 4096)]
    M = 16
    items = []
    for i, (name, N, K) in enumerate(shapes):
        wq, s, b, x = w4_case(N, K, M, seed=80 + i, device=DEV)
        items.append((wq, s, b, x, torch.empty(M, N, device=DEV)))
    grp = q.SkinnyGroup(items)
    grp.run()
    torch.cuda.synchronize()
    for (name, N, K), (wq, s, b, x, y) in zip(shapes, items):
        g = torch.Generator().manual_seed(N + 7)
        rows = sorted(set(torch.randint(0, N, (32,), generator=g).tolist()) | {0, N - 1})
        ridx = torch.tensor(rows, device=DEV)
        yr, ad = oracle.w4a16(wq[ridx].cpu(), s[ridx].cpu(), b[ridx].cpu(), x.cpu())
        close(y[:, ridx], yr, ad, f"skinny group {name} sampled")
    grp.close()
