"""Pins of the oracle to facts outside itself (closed forms, hand-derived
golden values, textbook/library special cases, brute force, invariants).

Each group names the page passage the oracle function follows:
  * W4A16 affine: "MLX Runner: An Inference Engine You Can Read",
    "Architecture: one command buffer per token".
  * Skinny rows: "Krill Teardown", "Core mechanisms" (continuous batcher).
  * MXFP4 MoE: "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin),
    "How it works" / "Technical approach / compute".
  * Hadamard + int8, W8A8: Uzu article, "How Uzu optimizes bytes and tokens
    per pass".
  * W8A16 row-int8 GEMV: "Running Kimi K3 (2.8T) on one Apple Silicon Mac"
    (Deltafin), "Technical approach / compute" (packed int8 output head).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def bf16_bits(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f16_bits(vals):
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


def pack_codes(q):
    """codes [N][K] (0..15) -> uint32 words, code k in bits 4(k%8).. of word k/8"""
    q = np.asarray(q, dtype=np.uint64)
    N, K = q.shape
    q = q.reshape(N, K // 8, 8)
    w = np.zeros((N, K // 8), dtype=np.uint64)
    for i in range(8):
        w |= q[:, :, i] << np.uint64(4 * i)
    return w.astype(np.uint32)


# ---------------------------------------------------------------- scalar decoders

def test_f16_decode_matches_numpy_for_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(p)) for p in pats[::7]])
    r = ref[::7]
    finite = np.isfinite(r)
    assert np.array_equal(got[finite], r[finite])
    assert np.all(np.isnan(got[np.isnan(r)]))
    assert np.all(np.isinf(got[np.isinf(r)]) & (np.sign(got[np.isinf(r)]) == np.sign(r[np.isinf(r)])))


def test_bf16_decode_matches_torch():
    pats = np.arange(0, 65536, 5, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(int(p)) for p in pats])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])


# ---------------------------------------------------------------- W4A16

def test_w4a16_golden_hand_example():
    g = json.load(open(os.path.join(GOLD, "w4a16_hand.json")))
    K, N = g["K"], g["N"]
    words = np.zeros((N, K // 8), np.uint32)
    words[0, :] = 0x33333333
    words[1, 0::2] = 0x76543210
    words[1, 1::2] = 0xFEDCBA98
    words[2, :] = 0x11111111
    sc = np.array([[int(v, 16) for v in r["scale_f16"]] for r in g["rows"]], np.uint16)
    bi = np.array([[int(v, 16) for v in r["bias_f16"]] for r in g["rows"]], np.uint16)
    x = np.zeros((2, K), np.uint16)
    x[0, :64] = 0x3F80
    x[0, 64:] = 0xC000
    x[1, :] = 0x3F00
    y, ad = oracle.w4a16(words, sc, bi, x)
    assert np.array_equal(y, np.array(g["y"]))
    assert np.array_equal(ad, np.array(g["absdot"]))


def test_w4a16_nibble_order_low_first():
    # word 0x76543210 holds codes 0..7 in order; s = 1, b = 0; one-hot x picks code k
    K = 64
    words = np.full((1, K // 8), 0x76543210, np.uint32)
    s = f16_bits([[1.0]])
    b = f16_bits([[0.0]])
    for k in range(K):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y, _ = oracle.w4a16(words, s, b, x)
        assert y[0, 0] == k % 8


def test_w4a16_one_hot_returns_dequantized_column():
    wq, s, b = synth.w4_weights(8, 256, seed=11, slot=0)
    wq_np = wq.numpy().view(np.uint32)
    s_np = s.view(torch.int16).numpy().view(np.uint16)
    b_np = b.view(torch.int16).numpy().view(np.uint16)
    for k in [0, 7, 8, 63, 64, 129, 255]:
        x = np.zeros((1, 256), np.uint16)
        x[0, k] = 0x3F80
        y, _ = oracle.w4a16(wq_np, s_np, b_np, x)
        q = (wq_np[:, k // 8] >> np.uint32(4 * (k % 8))) & np.uint32(15)
        exp = s.float().numpy()[:, k // 64].astype(np.float64) * q + \
            b.float().numpy()[:, k // 64].astype(np.float64)
        assert np.array_equal(y[0], exp)


def test_w4a16_zero_codes_reduce_to_bias_times_group_sums():
    rng = np.random.default_rng(3)
    N, K = 5, 256
    words = np.zeros((N, K // 8), np.uint32)
    s = f16_bits(rng.normal(size=(N, 4)) * 0.01)
    b = f16_bits(rng.normal(size=(N, 4)) * 0.05)
    x = bf16_bits(rng.normal(size=(3, K)))
    y, _ = oracle.w4a16(words, s, b, x)
    xf = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    gs = xf.reshape(3, 4, 64).sum(axis=2)                 # [M][groups]
    exp = gs @ b.view(np.float16).astype(np.float64).T    # sum_g b_g * sum_{k in g} x_k
    assert np.allclose(y, exp, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("group", [32, 128])
def test_w4a16_other_group_sizes_zero_codes_and_one_hot(group):
    # zero codes: y = sum_g b_g * (sum of x over group g); one-hot x: the
    # dequantized column with the scale and bias of group k // group
    rng = np.random.default_rng(4)
    N, K = 5, 512
    G = K // group
    words = np.zeros((N, K // 8), np.uint32)
    s = f16_bits(rng.normal(size=(N, G)) * 0.01)
    b = f16_bits(rng.normal(size=(N, G)) * 0.05)
    x = bf16_bits(rng.normal(size=(2, K)))
    y, _ = oracle.w4a16(words, s, b, x, group=group)
    xf = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    exp = xf.reshape(2, G, group).sum(axis=2) @ b.view(np.float16).astype(np.float64).T
    assert np.allclose(y, exp, rtol=1e-13, atol=1e-13)
    q = rng.integers(0, 16, size=(N, K))
    wq = pack_codes(q)
    for k in (0, group - 1, group, K - 1):
        xh = np.zeros((1, K), np.uint16)
        xh[0, k] = 0x3F80  # 1.0
        y1, _ = oracle.w4a16(wq, s, b, xh, group=group)
        col = s.view(np.float16).astype(np.float64)[:, k // group] * q[:, k] + \
            b.view(np.float16).astype(np.float64)[:, k // group]
        assert np.array_equal(y1[0], col)


def test_w4a16_integer_inputs_exact():
    # s = 1, b = 0 and small integer x: y is an exact integer sum
    rng = np.random.default_rng(5)
    N, K = 4, 192
    q = rng.integers(0, 16, size=(N, K))
    x_int = rng.integers(-8, 9, size=(2, K))
    y, _ = oracle.w4a16(pack_codes(q), f16_bits(np.ones((N, 3))), f16_bits(np.zeros((N, 3))),
                        bf16_bits(x_int.astype(np.float32)))
    exact = [[int(sum(int(q[n, k]) * int(x_int[m, k]) for k in range(K))) for n in range(N)]
             for m in range(2)]
    assert np.array_equal(y, np.array(exact, dtype=np.float64))


def test_w4a16_skinny_rows_equal_per_row_gemv_and_linear():
    wq, s, b = synth.w4_weights(16, 320, seed=2, slot=0)
    X = synth.bf16_normal((4, 320), seed=2, slot=1)
    Y, _ = oracle.w4a16(wq, s, b, X)
    for m in range(4):
        y1, _ = oracle.w4a16(wq, s, b, X[m:m + 1])
        assert np.array_equal(Y[m], y1[0])
    # linearity in x (exact up to double rounding)
    x2 = (X[0].float() * 2).to(torch.bfloat16)           # exact doubling
    y2, _ = oracle.w4a16(wq, s, b, x2[None])
    assert np.allclose(y2[0], 2 * Y[0], rtol=1e-14, atol=1e-15)


def test_w4a16_rows_entry_matches_full():
    wq, s, b = synth.w4_weights(40, 256, seed=4, slot=0)
    X = synth.bf16_normal((3, 256), seed=4, slot=1)
    Y, A = oracle.w4a16(wq, s, b, X)
    rows = [0, 7, 39, 20]
    y, a = oracle.w4a16_rows(wq, s, b, X, rows)
    assert np.array_equal(y, Y[:, rows]) and np.array_equal(a, A[:, rows])
    y, a = oracle.w4a16_rows(wq[8:], s[8:], b[8:], X, [8, 30], row_base=8)
    assert np.array_equal(y, Y[:, [8, 30]])


def test_w4a16_absdot_bounds_result():
    wq, s, b = synth.w4_weights(32, 512, seed=6, slot=0)
    X = synth.bf16_normal((2, 512), seed=6, slot=1)
    Y, A = oracle.w4a16(wq, s, b, X)
    assert np.all(np.abs(Y) <= A + 1e-12)


def test_affine_encoder_reconstructs_within_half_step():
    # the input recipe: dequantized weights lie within scale/2 of the fp32 draw
    w = synth.normal_f32((6, 128), 0.02, seed=0, slot=9)
    wq, s, b = synth.affine_w4_encode(w)
    x = np.zeros((1, 128), np.uint16)
    for k in [0, 5, 64, 127]:
        x[:] = 0
        x[0, k] = 0x3F80
        y, _ = oracle.w4a16(wq, s, b, x)
        err = np.abs(y[0] - w[:, k].double().numpy())
        assert np.all(err <= s.float().double().numpy()[:, k // 64] * 0.5 + 2e-5)


# ---------------------------------------------------------------- MXFP4

def e2m1_from_bits(code):
    """OCP MX v1.0 E2M1: sign bit 3, 2-bit exponent (bias 1), 1-bit mantissa;
    exponent 0 is subnormal (m * 2^-1)."""
    sign = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    mag = m * 0.5 if e == 0 else math.ldexp(1.0 + m / 2.0, e - 1)
    return sign * mag


def test_e2m1_table_matches_bit_field_definition():
    for c in range(16):
        got = oracle.e2m1_value(c)
        exp = e2m1_from_bits(c)
        assert got == exp and math.copysign(1.0, got) == math.copysign(1.0, exp)


def test_e8m0_is_power_of_two():
    for e in [0, 1, 100, 126, 127, 128, 200, 254]:
        assert oracle.e8m0_value(e) == math.ldexp(1.0, e - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_mxfp4_golden_hand_example():
    g = json.load(open(os.path.join(GOLD, "mxfp4_hand.json")))
    codes = np.full((1, 16), 0x9A, np.uint8)
    scales = np.full((1, 1), g["scale_e8m0"], np.uint8)
    out, _, _ = oracle.mxfp4_gemv(codes, scales, np.ones(32))
    assert out[0] == g["cases"][0]["out"]
    out, _, _ = oracle.mxfp4_gemv(codes, scales, np.arange(32, dtype=np.float64))
    assert out[0] == g["cases"][1]["out"]


def test_mxfp4_low_nibble_is_even_element():
    codes = np.zeros((1, 16), np.uint8)
    codes[0, 3] = 0x42     # element 6 -> code 2 (1.0), element 7 -> code 4 (2.0)
    scales = np.full((1, 1), 127, np.uint8)
    for c, exp in [(6, 1.0), (7, 2.0), (5, 0.0), (8, 0.0)]:
        v = np.zeros(32)
        v[c] = 1.0
        out, _, _ = oracle.mxfp4_gemv(codes, scales, v)
        assert out[0] == exp


def test_mxfp4_encoder_roundtrip_and_scale_rule():
    w = synth.normal_f32((4, 64), 0.02, seed=3, slot=7)
    codes, e = synth.mxfp4_encode(w)
    D = oracle.mxfp4_dequant(codes, e)
    # every block's scale puts amax in [4, 8) * 2^X, i.e. within the E2M1 range
    blocks = w.double().numpy().reshape(4, 2, 32)
    amax = np.abs(blocks).max(axis=2)
    sc = np.ldexp(1.0, e.numpy().astype(int) - 127)
    assert np.all(amax >= 4 * sc) and np.all(amax < 8 * sc)
    # rounding error at most half of the largest gap (2 * scale) of the grid
    err = np.abs(D - w.double().numpy()).reshape(4, 2, 32)
    assert np.all(err <= 1.0 * sc[:, :, None] + 1e-12)


def softmax_ref(x):
    from scipy.special import softmax
    return softmax(np.asarray(x, np.float64), axis=-1)


def test_router_softmax_and_topk_order():
    lg = synth.router_logits(5, 384, seed=3, slot=3)
    idx, w, p = oracle.router(lg, 16)
    assert np.allclose(p, softmax_ref(lg.double().numpy()), rtol=1e-13, atol=0)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-13)
    order = np.argsort(-lg.double().numpy(), axis=1, kind="stable")[:, :16]
    assert np.array_equal(idx, order)
    assert np.array_equal(w, np.take_along_axis(p, order, axis=1))


def test_router_ties_go_to_lower_index():
    lg = np.zeros((2, 12), np.float32)
    lg[1, [3, 7, 9]] = 1.0
    idx, w, _ = oracle.router(lg, 5)
    assert list(idx[0]) == [0, 1, 2, 3, 4]
    assert list(idx[1]) == [3, 7, 9, 0, 1]
    assert np.allclose(w[0], 1.0 / 12)


def dense_from_bits(codes, scales):
    """Independent decode (bit-field E2M1 and ldexp E8M0) for the FFN pins."""
    codes = np.asarray(codes)
    R, C2 = codes.shape
    tab = np.array([e2m1_from_bits(c) for c in range(16)])
    cod = np.empty((R, 2 * C2), np.int64)
    cod[:, 0::2] = codes & 15
    cod[:, 1::2] = codes >> 4
    sc = np.ldexp(1.0, np.asarray(scales).astype(np.int64) - 127)
    return tab[cod] * np.repeat(sc, 32, axis=1)


def _tiny_moe(E, H, I, T, seed):
    x = synth.bf16_normal((T, H), seed, 0)
    lg = synth.router_logits(T, E, seed, 1)
    gq, gs = synth.mxfp4_weights(E * I, H, seed, 2)
    uq, us = synth.mxfp4_weights(E * I, H, seed, 3)
    dq, ds = synth.mxfp4_weights(E * H, I, seed, 4)
    r = lambda a, rows: a.reshape(E, rows, -1)
    return x, lg, r(gq, I), r(gs, I), r(uq, I), r(us, I), r(dq, H), r(ds, H)


def test_moe_single_expert_is_plain_swiglu_ffn():
    E, H, I = 1, 64, 96
    x, lg, gq, gs, uq, us, dq, ds = _tiny_moe(E, H, I, 2, seed=21)
    out = oracle.moe_forward(x, lg, gq, gs, uq, us, dq, ds, top_k=1)
    xf = x.double().numpy()
    Wg = dense_from_bits(gq[0].numpy(), gs[0].numpy())
    Wu = dense_from_bits(uq[0].numpy(), us[0].numpy())
    Wd = dense_from_bits(dq[0].numpy(), ds[0].numpy())
    for t in range(2):
        g = Wg @ xf[t]
        u = Wu @ xf[t]
        h = g / (1 + np.exp(-g)) * u
        assert out["w"][t, 0] == 1.0
        assert np.allclose(out["y"][t], Wd @ h, rtol=1e-12, atol=1e-14)


def test_moe_all_experts_equal_logits_is_mean():
    E, H, I = 4, 64, 32
    x, _, gq, gs, uq, us, dq, ds = _tiny_moe(E, H, I, 1, seed=22)
    lg = torch.zeros((1, E))
    out = oracle.moe_forward(x, lg, gq, gs, uq, us, dq, ds, top_k=E)
    xf = x.double().numpy()[0]
    acc = np.zeros(H)
    for e in range(E):
        g = dense_from_bits(gq[e].numpy(), gs[e].numpy()) @ xf
        u = dense_from_bits(uq[e].numpy(), us[e].numpy()) @ xf
        acc += dense_from_bits(dq[e].numpy(), ds[e].numpy()) @ (g / (1 + np.exp(-g)) * u)
    assert list(out["idx"][0]) == [0, 1, 2, 3]
    assert np.allclose(out["y"][0], acc / E, rtol=1e-12, atol=1e-14)


def test_moe_brute_force_tiny():
    E, H, I, T, k = 8, 64, 64, 3, 2
    x, lg, gq, gs, uq, us, dq, ds = _tiny_moe(E, H, I, T, seed=23)
    out = oracle.moe_forward(x, lg, gq, gs, uq, us, dq, ds, top_k=k)
    xf = x.double().numpy()
    lgn = lg.double().numpy()
    for t in range(T):
        p = softmax_ref(lgn[t])
        sel = sorted(range(E), key=lambda e: (-lgn[t, e], e))[:k]
        acc = np.zeros(H)
        for e in sel:
            g = dense_from_bits(gq[e].numpy(), gs[e].numpy()) @ xf[t]
            u = dense_from_bits(uq[e].numpy(), us[e].numpy()) @ xf[t]
            acc += p[e] * (dense_from_bits(dq[e].numpy(), ds[e].numpy()) @ (g / (1 + np.exp(-g)) * u))
        assert np.allclose(out["y"][t], acc, rtol=1e-12, atol=1e-14)
        assert np.all(out["ybound"][t] > 0)


# ---------------------------------------------------------------- Hadamard + int8

def sylvester(n=32):
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1)


def test_hadamard_columns_are_sylvester_and_orthogonal():
    H = np.zeros((32, 32), np.int64)
    zero_signs = np.zeros(1, np.uint32)
    for j in range(32):
        e = np.zeros(32, np.float32)
        e[j] = 1.0
        H[:, j] = oracle.hadamard32(e, zero_signs).astype(np.int64)
    assert np.array_equal(H, sylvester())
    assert np.array_equal(H @ H.T, 32 * np.eye(32, dtype=np.int64))


def test_hadamard_inverse_recovers_input_exactly_for_small_integers():
    rng = np.random.default_rng(1)
    v = rng.integers(-50, 51, size=128).astype(np.float32)
    sb = synth.sign_bits(128, seed=9, slot=0)
    z = oracle.hadamard32(v, sb)
    back = oracle.hadamard32(z, np.zeros(4, np.uint32)) / 32.0   # H z / 32 = D v
    signs = np.array([((int(sb[k // 32]) & 0xFFFFFFFF) >> (k % 32)) & 1 for k in range(128)])
    assert np.array_equal(np.where(signs == 1, -back, back), v)


def test_hadamard_constant_block_energy_in_bin_zero():
    z = oracle.hadamard32(np.full(32, 3.0, np.float32), np.zeros(1, np.uint32))
    assert z[0] == 96.0 and np.all(z[1:] == 0.0)


def test_hadamard_sign_bit_negates_that_input():
    rng = np.random.default_rng(2)
    v = rng.normal(size=32).astype(np.float32)
    for j in [0, 5, 31]:
        w = v.copy()
        w[j] = -w[j]
        a = oracle.hadamard32(v, np.array([1 << j], np.uint32))
        b = oracle.hadamard32(w, np.zeros(1, np.uint32))
        assert np.array_equal(a, b)


def test_quant_row_rounds_half_to_even_and_saturates():
    q, s = oracle.quant_i8_row([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -127.0])
    assert s == np.float32(1.0)
    assert list(q) == [127, 2, 4, -2, -4, 0, 2, -127]
    q, s = oracle.quant_i8_row(np.zeros(8))
    assert s == 0.0 and not q.any()


def test_quant_error_within_half_step_and_amax_maps_to_127():
    x = synth.outlier_activations(16, 1024, seed=4, slot=0)
    sb = synth.sign_bits(1024, seed=4, slot=5)
    q, s, z = oracle.hadamard32_quant_i8(x, sb)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    for m in range(16):
        assert s[m] == np.float32(np.abs(z[m]).max() / np.float32(127.0))
        err = np.abs(z[m].astype(np.float64) - s[m].astype(np.float64) * q[m])
        assert np.all(err <= 0.5 * s[m] * (1 + 1e-5))
        assert np.abs(q[m]).max() == 127


def test_hadamard_quant_uses_the_transform():
    x = synth.outlier_activations(3, 256, seed=4, slot=0)
    sb = synth.sign_bits(256, seed=4, slot=5)
    _, _, z = oracle.hadamard32_quant_i8(x, sb)
    for m in range(3):
        xf = x[m].float().numpy()
        assert np.array_equal(z[m], oracle.hadamard32(xf, sb))


def test_hadamard_spreads_outliers_statistic():
    # reported, loose check: the transform lowers max|.|/rms on outlier inputs
    x = synth.outlier_activations(16, 4096, seed=4, slot=0)
    sb = synth.sign_bits(4096, seed=4, slot=5)
    _, _, z = oracle.hadamard32_quant_i8(x, sb)
    xf = x.float().numpy()
    r_in = np.abs(xf).max(1) / np.sqrt((xf ** 2).mean(1))
    r_out = np.abs(z).max(1) / np.sqrt((z.astype(np.float64) ** 2).mean(1))
    assert np.median(r_out) < np.median(r_in)


# ---------------------------------------------------------------- W8A8

def test_w8a8_matches_integer_matmul():
    rng = np.random.default_rng(8)
    a = rng.integers(-127, 128, size=(16, 512)).astype(np.int8)
    w = rng.integers(-127, 128, size=(40, 512)).astype(np.int8)
    c = oracle.w8a8(a, w)
    assert np.array_equal(c, a.astype(np.int64) @ w.astype(np.int64).T)


def test_w8a8_extremes_and_overflow_detection():
    a = np.full((1, 4096), 127, np.int8)
    w = np.full((2, 4096), -127, np.int8)
    assert np.array_equal(oracle.w8a8(a, w), np.full((1, 2), -127 * 127 * 4096))
    a = np.full((1, 140000), 127, np.int8)
    with pytest.raises(OverflowError):
        oracle.w8a8(a, a)


# ---------------------------------------------------------------- W8A16 row-int8 GEMV

def test_w8a16_one_hot_selects_scaled_column():
    # x = e_k: y[n] = s[n] * q[n][k] (catches a transposed operand or a lost scale)
    rng = np.random.default_rng(5)
    N, K = 7, 48
    q = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    s = np.array([0.5, 2.0, 0.25, 1.0, 3.0, 0.125, 8.0], np.float32)
    for k in (0, 17, 47):
        x = np.zeros(K, np.float32)
        x[k] = 1.0
        y, ad = oracle.w8a16(q, s, bf16_bits(x))
        assert np.array_equal(y[0], s.astype(np.float64) * q[:, k])
        assert np.array_equal(ad[0], np.abs(s.astype(np.float64) * q[:, k]))


def test_w8a16_all_ones_codes_give_scaled_sum():
    rng = np.random.default_rng(6)
    N, K = 5, 64
    x = rng.integers(-8, 9, size=K).astype(np.float32)  # integers: exact in bf16 and double
    s = np.array([1.0, 0.5, -2.0, 4.0, 0.75], np.float32)
    for code in (1, -1, 127, -128):
        q = np.full((N, K), code, np.int8)
        y, _ = oracle.w8a16(q, s, bf16_bits(x))
        assert np.array_equal(y[0], s.astype(np.float64) * code * x.sum())


def test_w8a16_agrees_with_w4a16_on_shared_cases():
    # codes 0..15, scale representable in fp16, zero bias: both definitions coincide
    rng = np.random.default_rng(7)
    N, K = 6, 128
    q = rng.integers(0, 16, size=(N, K))
    s16 = np.array([0.5, 0.25, 1.5, 0.125, 2.0, 0.375], np.float16)
    x = bf16_bits(rng.standard_normal(K))
    y8, _ = oracle.w8a16(q.astype(np.int8), s16.astype(np.float32), x)
    scales = np.repeat(s16[:, None], K // 64, axis=1).view(np.uint16)
    biases = np.zeros_like(scales)
    y4, _ = oracle.w4a16(pack_codes(q), scales, biases, x)
    assert np.allclose(y8, y4, rtol=1e-12, atol=0)


def test_w8a16_rows_of_x_are_independent():
    rng = np.random.default_rng(8)
    N, K, M = 4, 32, 3
    q = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    s = rng.random(N).astype(np.float32)
    x = bf16_bits(rng.standard_normal((M, K)))
    y, _ = oracle.w8a16(q, s, x)
    for m in range(M):
        ym, _ = oracle.w8a16(q, s, x[m])
        assert np.array_equal(y[m], ym[0])


# ---------------------------------------------------------------- affine 2/3/4/5/6/8 bits

def pack_bitstream(q, bits):
    """codes [N][K] -> uint32 [N][K*bits/32]: each row one little-endian bit
    stream (numpy.packbits with little bit order, then little-endian words)."""
    q = np.asarray(q, dtype=np.uint64)
    N, K = q.shape
    bitarr = ((q[:, :, None] >> np.arange(bits, dtype=np.uint64)) & np.uint64(1)).astype(np.uint8)
    by = np.packbits(bitarr.reshape(N, K * bits), axis=1, bitorder="little")
    return np.ascontiguousarray(by).view("<u4").astype(np.uint32)


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
@pytest.mark.parametrize("group", [32, 128])
def test_affine_one_hot_returns_dequantized_column(bits, group):
    rng = np.random.default_rng(bits * 10 + group)
    N, K = 6, 256
    q = rng.integers(0, 1 << bits, size=(N, K))
    wq = pack_bitstream(q, bits)
    s = f16_bits(rng.normal(size=(N, K // group)) * 0.01)
    b = f16_bits(rng.normal(size=(N, K // group)) * 0.05)
    sf = s.view(np.float16).astype(np.float64)
    bf = b.view(np.float16).astype(np.float64)
    for k in (0, 1, 10, 31, 32, 100, 255):  # codes that straddle word boundaries for 3, 5, 6 bits
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y, _ = oracle.affine(wq, bits, s, b, x, group=group)
        assert np.array_equal(y[0], sf[:, k // group] * q[:, k] + bf[:, k // group])


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
def test_affine_constant_codes_closed_form(bits):
    rng = np.random.default_rng(40 + bits)
    N, K, group = 3, 512, 64
    x = bf16_bits(rng.integers(-4, 5, size=(2, K)).astype(np.float32))  # small integers: exact
    xf = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    gsum = xf.reshape(2, K // group, group).sum(axis=2)
    s = f16_bits(np.full((N, K // group), 0.5))
    b = f16_bits(np.full((N, K // group), -0.25))
    for code in (0, (1 << bits) - 1):
        wq = pack_bitstream(np.full((N, K), code), bits)
        y, _ = oracle.affine(wq, bits, s, b, x, group=group)
        exp = (0.5 * code - 0.25) * gsum.sum(axis=1)
        assert np.array_equal(y, np.repeat(exp[:, None], N, axis=1))


@pytest.mark.parametrize("group", [32, 64, 128])
def test_affine_four_bits_is_the_w4a16_definition(group):
    rng = np.random.default_rng(90 + group)
    N, K = 5, 512
    q = rng.integers(0, 16, size=(N, K))
    s = f16_bits(rng.normal(size=(N, K // group)) * 0.01)
    b = f16_bits(rng.normal(size=(N, K // group)) * 0.05)
    x = bf16_bits(rng.normal(size=(3, K)))
    ya, _ = oracle.affine(pack_bitstream(q, 4), 4, s, b, x, group=group)
    y4, _ = oracle.w4a16(pack_codes(q), s, b, x, group=group)
    assert np.array_equal(pack_bitstream(q, 4), pack_codes(q))
    assert np.allclose(ya, y4, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- fused int8 path (Hadamard -> int8 -> W8A8 -> dequant)

def test_w8a8_dequant_within_the_quantization_bound():
    # |y - x.w| is bounded by the int8 rounding of both transformed operands:
    # with z = H D v and |z/s - q| <= 1/2 per element,
    # 32 |y - x.w| <= sum_k (|z_a| s_w + |z_w| s_a) / 2 + K s_a s_w / 4.
    rng = np.random.default_rng(11)
    M, N, K = 3, 5, 256
    x = bf16_bits(rng.normal(size=(M, K)))
    w = bf16_bits(rng.normal(size=(N, K)) * 0.02)
    sb = synth.sign_bits(K, seed=11, slot=0).numpy()
    y, p = oracle.w8a8_dequant(x, w, sb)
    xf = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    wf = torch.from_numpy(w.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    exact = xf @ wf.T
    za, zw = p["za"].astype(np.float64), p["zw"].astype(np.float64)
    sa, sw = p["sa"].astype(np.float64), p["sw"].astype(np.float64)
    bound = (np.abs(za).sum(1)[:, None] * sw[None, :] + np.abs(zw).sum(1)[None, :] * sa[:, None]) / 2 \
        + K * sa[:, None] * sw[None, :] / 4
    assert np.all(np.abs(y - exact) * 32 <= bound * (1 + 1e-9) + 1e-12)
    # and the transform is what makes it work: the same rows without outliers agree closely
    assert np.max(np.abs(y - exact)) < 0.05 * np.max(np.abs(exact))


def test_w8a8_dequant_scales_with_the_activations():
    # per-token symmetric quantization is scale-invariant: x -> 2x gives y -> 2y exactly
    rng = np.random.default_rng(12)
    M, N, K = 2, 4, 128
    xv = rng.normal(size=(M, K)).astype(np.float32)
    x1, x2 = bf16_bits(xv), bf16_bits(2 * xv)
    w = bf16_bits(rng.normal(size=(N, K)) * 0.02)
    sb = synth.sign_bits(K, seed=12, slot=0).numpy()
    y1, _ = oracle.w8a8_dequant(x1, w, sb)
    y2, _ = oracle.w8a8_dequant(x2, w, sb)
    assert np.array_equal(y2, 2 * y1)


# ------------------------------------------------ decode-step chain inputs
# "MLX Runner: An Inference Engine You Can Read", "Architecture: one command
# buffer per token": each projection consumes the previous one's output,
# rounded to bf16 (scaled copy, or the SwiGLU of a fused gate/up output).

def test_bf16_rounding_single_step_ties_even_and_subnormals():
    # 1 + 2^-8 lies halfway between bf16 1 and 1 + 2^-7: ties go to the even 1.0
    assert oracle.bf16_bits([1 + 2 ** -8])[0] == 0x3F80
    # 1 + 3 * 2^-8 is halfway between mantissas 1 and 2: the even one
    assert oracle.bf16_bits([1 + 3 * 2 ** -8])[0] == 0x3F82
    # just above the tie (by far less than an fp32 ulp): rounds up. Rounding
    # to fp32 first would land on the tie and give 0x3F80.
    assert oracle.bf16_bits([1 + 2 ** -8 + 2 ** -40])[0] == 0x3F81
    assert oracle.bf16_bits([-(1 + 2 ** -8 + 2 ** -40)])[0] == 0xBF81
    # bf16 subnormals are multiples of 2^-133
    assert oracle.bf16_bits([2.0 ** -130])[0] == 0x0008
    assert oracle.bf16_bits([2.5 * 2.0 ** -133])[0] == 0x0002   # tie -> even
    assert oracle.bf16_bits([3.5 * 2.0 ** -133])[0] == 0x0004
    # beyond the largest bf16 (0x7F7F): infinity
    assert oracle.bf16_bits([3.5e38])[0] == 0x7F80
    assert oracle.bf16_bits([0.0, -0.0]).tolist() == [0x0000, 0x8000]


def test_bf16_rounding_of_fp32_values_matches_torch():
    # from fp32 there is no second rounding: torch's fp32 -> bf16 conversion
    # (nearest even) must agree on every value
    r = np.random.default_rng(3)
    v = (r.standard_normal(200000) * np.exp(r.uniform(-40, 40, 200000))).astype(np.float32)
    ours = oracle.bf16_bits(v.astype(np.float64))
    assert np.array_equal(ours, bf16_bits(v))


def test_chain_copy_is_scaled_fp32_product_then_bf16():
    r = np.random.default_rng(4)
    src = r.standard_normal(640).astype(np.float32)
    for alpha in (1.0, 0.5, 0.7):
        prod = (torch.from_numpy(src[:512]) * torch.tensor(alpha, dtype=torch.float32))
        want = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(oracle.chain_x(src, oracle.X_COPY, alpha, 512), want)


def test_chain_swiglu_identities():
    K = 256
    r = np.random.default_rng(5)
    g = r.uniform(-6, 6, K).astype(np.float32)
    ones = np.ones(K, np.float32)
    # u = 0: zero activations; g = 0: silu(0) = 0
    assert not (oracle.chain_x(np.concatenate([g, 0 * ones]), oracle.X_SWIGLU, 1.0, K) & 0x7FFF).any()
    assert not (oracle.chain_x(np.concatenate([0 * g, ones]), oracle.X_SWIGLU, 1.0, K) & 0x7FFF).any()
    # silu(g) - silu(-g) = g (sigmoid(g) + sigmoid(-g) = 1): catches a sign or
    # a dropped factor
    def val(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    xp = val(oracle.chain_x(np.concatenate([g, ones]), oracle.X_SWIGLU, 1.0, K))
    xm = val(oracle.chain_x(np.concatenate([-g, ones]), oracle.X_SWIGLU, 1.0, K))
    assert np.all(np.abs((xp - xm) - g) <= 2.0 ** -8 * (np.abs(xp) + np.abs(xm)) + 1e-30)
    # large positive gate: silu(g) -> g, so x -> bf16(g u alpha)
    big = np.full(K, 40.0, np.float32)
    u = r.standard_normal(K).astype(np.float32)
    got = val(oracle.chain_x(np.concatenate([big, u]), oracle.X_SWIGLU, 0.25, K))
    assert np.allclose(got, 10.0 * u, rtol=2 ** -8)


def test_chain_of_two_levels_composes_gemv_and_rounding():
    # level 0: y0 = W0 x; level 1 reads bf16(alpha y0) -- the same as calling the
    # pinned W4A16 definition on an input rounded by torch
    N0, K0, N1 = 96, 128, 40
    w0 = synth.w4_weights(N0, K0, seed=7, slot=1)
    w1 = synth.w4_weights(N1, N0 - 32, seed=7, slot=2)
    x = synth.bf16_normal((K0,), 7, 3)
    y0, _ = oracle.w4a16(*w0, x)
    y0f = y0[0].astype(np.float32)
    x1 = oracle.chain_x(y0f, oracle.X_COPY, 0.5, N0 - 32)
    x1_t = (torch.from_numpy(y0f[:N0 - 32]) * 0.5).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(x1, x1_t)
    y1, _ = oracle.w4a16(*w1, x1)
    W1 = synth_dequant(w1)
    want = W1 @ torch.from_numpy(x1_t.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.allclose(y1[0], want, rtol=1e-12, atol=1e-12)


def synth_dequant(w):
    """Dense float64 weights of an affine W4 g64 matrix, unpacked with numpy."""
    wq, s, b = (t.numpy() for t in w)
    N = wq.shape[0]
    K = wq.shape[1] * 8
    words = wq.view(np.uint32)
    q = np.stack([(words >> np.uint32(4 * i)) & np.uint32(15) for i in range(8)], axis=-1).reshape(N, K)
    sc = s.view(np.float16).astype(np.float64).repeat(64, axis=1)
    bi = b.view(np.float16).astype(np.float64).repeat(64, axis=1)
    return sc * q + bi
