"""Seeded synthetic inputs shared by the tests, the bench and the oracle's callers.

This module draws random numbers and encodes weights into the stored formats
the kernels and the oracle consume. It holds no step of the hot path itself:
neither the GEMV/GEMM contractions, the router, SwiGLU, the Hadamard transform
nor the per-token activation quantizer live here. The weight encoders below
(affine at 2..8 bits, row-int8 and MXFP4) are the input recipe of the
workloads, i.e. how the stored codes are produced from fp32 weights before any
kernel runs; the hot path only ever decodes them.

Sources of the recipes:
  * "MLX Runner: An Inference Engine You Can Read", section "Architecture: one
    command buffer per token": affine groups, weight = scale x code + bias.
  * "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin), section
    "Technical approach / compute": MXFP4 experts, E2M1 codes with an E8M0
    scale applied to the exponent.
  * Uzu article, section "How Uzu optimizes bytes and tokens per pass": 8-bit
    activations and outliers motivating the block-32 randomized Hadamard.

Every tensor gets its own torch.Generator seeded with ``seed * 1000 + slot`` so
inputs are reproducible on the device they are drawn on. Values drawn on CPU and
on CUDA differ (different generator families); each run draws once and gives the
same tensors to both sides.
"""
from __future__ import annotations

import math

import torch

__all__ = [
    "gen", "normal_f32", "bf16_normal", "affine_w4_encode", "w4_weights", "affine_encode",
    "affine_weights", "row_int8_encode", "w8_row_weights", "mxfp4_encode", "mxfp4_weights",
    "router_logits", "outlier_activations", "sign_bits", "STACK_SHAPES", "stack_layer_shapes",
]


def gen(seed: int, slot: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000 + int(slot))
    return g


def normal_f32(shape, std, seed, slot, device="cpu") -> torch.Tensor:
    return torch.randn(*shape, generator=gen(seed, slot, device), device=device,
                       dtype=torch.float32) * std


def bf16_normal(shape, seed, slot, device="cpu") -> torch.Tensor:
    """x ~ N(0, 1) rounded to bf16 (round to nearest even)."""
    return normal_f32(shape, 1.0, seed, slot, device).to(torch.bfloat16)


# --------------------------------------------------------------------------
# Affine 4-bit, group 64: weight = scale * code + bias (MLX affine format)
# --------------------------------------------------------------------------

def affine_w4_encode(w: torch.Tensor, group: int = 64):
    """Encode fp32 weights [N][K] per K-group by min/max into uint4 codes.

    scale = fp16(max((max - min) / 15, 0)), bias = fp16(min); the codes are
    computed against the fp16-rounded scale and bias, rounded half to even and
    clamped to 0..15; a group with scale 0 gets all-zero codes. Codes are packed
    8 per 32-bit word, code k of a row in bits [4(k%8), 4(k%8)+3] of word k/8.
    Returns (wq int32 [N][K/8] holding the uint32 bit patterns, scales fp16
    [N][K/group], biases fp16 [N][K/group]).
    """
    N, K = w.shape
    assert K % group == 0 and K % 8 == 0
    wg = w.float().reshape(N, K // group, group)
    mn = wg.amin(dim=2)
    mx = wg.amax(dim=2)
    scale = torch.clamp((mx - mn) / 15.0, min=0.0).to(torch.float16)
    bias = mn.to(torch.float16)
    sf = scale.float().unsqueeze(2)
    bf = bias.float().unsqueeze(2)
    safe = torch.where(sf > 0, sf, torch.ones_like(sf))
    q = torch.round((wg - bf) / safe).clamp_(0, 15)
    q = torch.where(sf > 0, q, torch.zeros_like(q)).to(torch.int64).reshape(N, K // 8, 8)
    shifts = torch.arange(0, 32, 4, device=w.device, dtype=torch.int64)
    words = (q << shifts).sum(dim=2)                     # 0 .. 2^32-1
    words = words - ((words >> 31) & 1) * (1 << 32)      # same bits, int32 range
    return words.to(torch.int32).contiguous(), scale.contiguous(), bias.contiguous()


def affine_encode(w: torch.Tensor, bits: int, group: int = 64):
    """Encode fp32 weights [N][K] per K-group by min/max into `bits`-bit codes
    (2, 3, 4, 5, 6 or 8): the recipe of affine_w4_encode with 2^bits - 1
    levels. Each row's codes form one little-endian bit stream: code k in bits
    [bits*k, bits*k + bits), bit j of the stream in bit j % 32 of word j / 32.
    Returns (wq int32 [N][K*bits/32] holding the uint32 bit patterns, scales
    fp16 [N][K/group], biases fp16 [N][K/group])."""
    N, K = w.shape
    assert K % group == 0 and K % 32 == 0 and bits in (2, 3, 4, 5, 6, 8)
    levels = (1 << bits) - 1
    wg = w.float().reshape(N, K // group, group)
    mn = wg.amin(dim=2)
    mx = wg.amax(dim=2)
    scale = torch.clamp((mx - mn) / levels, min=0.0).to(torch.float16)
    bias = mn.to(torch.float16)
    sf = scale.float().unsqueeze(2)
    bf = bias.float().unsqueeze(2)
    safe = torch.where(sf > 0, sf, torch.ones_like(sf))
    q = torch.round((wg - bf) / safe).clamp_(0, levels)
    q = torch.where(sf > 0, q, torch.zeros_like(q)).to(torch.int64).reshape(N, K)
    # bit stream: bit t of code k goes to stream bit bits*k + t
    bitv = (q.unsqueeze(2) >> torch.arange(bits, device=w.device, dtype=torch.int64)) & 1   # [N][K][bits]
    bitv = bitv.reshape(N, K * bits // 32, 32)
    words = (bitv << torch.arange(32, device=w.device, dtype=torch.int64)).sum(dim=2)
    words = words - ((words >> 31) & 1) * (1 << 32)
    return words.to(torch.int32).contiguous(), scale.contiguous(), bias.contiguous()


def affine_weights(N, K, bits, seed, slot, device="cpu", group=64, std=0.02):
    """Weights ~ N(0, std) encoded as `bits`-bit affine codes (see affine_encode)."""
    return _chunked(N, K, std, seed, slot, device, lambda w: affine_encode(w, bits, group))


def _chunked(R, C, std, seed, slot, device, encode, max_elems=1 << 28):
    """Draw [R][C] ~ N(0, std) in row chunks from one generator and encode each
    chunk, so peak memory stays bounded for multi-GB weight sets."""
    g = gen(seed, slot, device)
    rows = max(1, min(R, max_elems // max(C, 1)))
    outs = []
    for r0 in range(0, R, rows):
        r1 = min(R, r0 + rows)
        w = torch.randn(r1 - r0, C, generator=g, device=device, dtype=torch.float32) * std
        outs.append(encode(w))
        del w
    return tuple(torch.cat([o[i] for o in outs], dim=0) if len(outs) > 1 else outs[0][i]
                 for i in range(len(outs[0])))


def w4_weights(N, K, seed, slot, device="cpu", group=64, std=0.02):
    """Weights ~ N(0, std) encoded as affine uint4 (see affine_w4_encode)."""
    return _chunked(N, K, std, seed, slot, device, lambda w: affine_w4_encode(w, group))


def row_int8_encode(w: torch.Tensor):
    """Row-int8 encoding of fp32 weights [N][K] (a row-int8 checkpoint):
    s = max|w| / 127 per row (fp32), q = round-half-even(w / s) clamped to
    [-127, 127]; an all-zero row gets s = 0 and codes 0.
    Returns (q int8 [N][K], s fp32 [N])."""
    w = w.float()
    amax = w.abs().amax(dim=1)
    s = amax / 127.0
    safe = torch.where(s > 0, s, torch.ones_like(s))
    q = torch.clamp(torch.round(w / safe[:, None]), -127, 127).to(torch.int8)
    q = torch.where((s > 0)[:, None], q, torch.zeros_like(q))
    return q, s


def w8_row_weights(N, K, seed, slot, device="cpu", std=0.02):
    """Weights ~ N(0, std) as row-int8 (see row_int8_encode)."""
    return _chunked(N, K, std, seed, slot, device, row_int8_encode)


# --------------------------------------------------------------------------
# MXFP4: E2M1 codes (2 per byte, low nibble = even index), E8M0 per 32
# --------------------------------------------------------------------------

def mxfp4_encode(w: torch.Tensor):
    """Encode fp32 weights [R][C] as MXFP4 following the OCP MX v1.0 recipe.

    Per block of 32 along C: amax = max|w|; X = floor(log2 amax) - 2 (2 is the
    largest E2M1 exponent), clamped to [-127, 127]; the block scale is stored as
    E8M0 e = X + 127 (amax = 0 gives e = 0 and zero codes). Each w / 2^X is
    rounded to the nearest E2M1 magnitude {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to
    the even mantissa, saturating at 6; bit 3 of the code is the sign.
    Returns (codes uint8 [R][C/2], scales uint8 [R][C/32]).
    """
    R, C = w.shape
    assert C % 32 == 0
    wb = w.float().reshape(R, C // 32, 32)
    amax = wb.abs().amax(dim=2)
    pos = amax > 0
    safe = torch.where(pos, amax, torch.ones_like(amax))
    X = torch.floor(torch.log2(safe)) - 2.0
    # log2 of a float can round up across a power of two: fix so 2^X*4 <= amax
    X = torch.where(torch.ldexp(torch.ones_like(X), X + 2.0) > safe, X - 1.0, X)
    X = torch.where(torch.ldexp(torch.ones_like(X), X + 3.0) <= safe, X + 1.0, X)
    X = torch.clamp(X, -127.0, 127.0)
    X = torch.where(pos, X, torch.full_like(X, -127.0))
    e = (X + 127.0).to(torch.uint8)
    a = (wb / torch.ldexp(torch.ones_like(X), X).unsqueeze(2)).abs()
    # ties: towards the neighbour whose mantissa bit is 0 (even code index)
    idx = torch.zeros_like(a, dtype=torch.int64)
    idx = torch.where(a > 0.25, 1, idx)
    idx = torch.where(a >= 0.75, 2, idx)
    idx = torch.where(a > 1.25, 3, idx)
    idx = torch.where(a >= 1.75, 4, idx)
    idx = torch.where(a > 2.5, 5, idx)
    idx = torch.where(a >= 3.5, 6, idx)
    idx = torch.where(a > 5.0, 7, idx)
    code = idx | torch.where(wb < 0, 8, 0)
    code = torch.where(pos.unsqueeze(2), code, torch.zeros_like(code))
    code = code.reshape(R, C // 2, 2)
    packed = (code[:, :, 0] | (code[:, :, 1] << 4)).to(torch.uint8)
    return packed.contiguous(), e.contiguous()


def mxfp4_weights(R, C, seed, slot, device="cpu", std=0.02):
    """Weights ~ N(0, std) encoded as MXFP4 (see mxfp4_encode)."""
    return _chunked(R, C, std, seed, slot, device, mxfp4_encode)


def router_logits(T, E, seed, slot, device="cpu"):
    return normal_f32((T, E), 1.0, seed, slot, device)


# --------------------------------------------------------------------------
# Activations with outliers and the random sign vector
# --------------------------------------------------------------------------

def outlier_activations(M, K, seed, slot, device="cpu", frac=0.01, factor=50.0):
    """x ~ N(0,1) [M][K] with exactly floor(frac*M*K) positions, drawn without
    replacement, multiplied by `factor`; rounded to bf16."""
    x = normal_f32((M, K), 1.0, seed, slot, device)
    n_out = int(math.floor(frac * M * K))
    perm = torch.randperm(M * K, generator=gen(seed, slot + 1, device), device=device)
    idx = perm[:n_out]
    flat = x.reshape(-1)
    flat[idx] = flat[idx] * factor
    return flat.reshape(M, K).to(torch.bfloat16)


def sign_bits(K, seed, slot, device="cpu"):
    """One random sign per K position, packed: word b bit j set = negate
    element 32*b + j. Returned as int32 [K/32] holding uint32 bit patterns."""
    assert K % 32 == 0
    bits = torch.randint(0, 2, (K // 32, 32), generator=gen(seed, slot, device),
                         device=device, dtype=torch.int64)
    shifts = torch.arange(32, device=device, dtype=torch.int64)
    words = (bits << shifts).sum(dim=1)
    words = words - ((words >> 31) & 1) * (1 << 32)
    return words.to(torch.int32).contiguous()


# --------------------------------------------------------------------------
# The dense 9B-class decoder layer stack (one token): W4A16 g64 projections
# --------------------------------------------------------------------------

# (name, N = output features, K = input features)
STACK_SHAPES = [
    ("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
    ("gate_up", 24576, 4096), ("down", 4096, 12288),
]
STACK_LAYERS = 36
LM_HEAD = ("lm_head", 151936, 4096)


def stack_layer_shapes(layers=STACK_LAYERS):
    """All (name, N, K) of one token's layer stack in issue order."""
    out = []
    for l in range(layers):
        for name, n, k in STACK_SHAPES:
            out.append((f"l{l}.{name}", n, k))
    out.append(LM_HEAD)
    return out
