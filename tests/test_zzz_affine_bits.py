"""GPU parity of qgemm_affine (affine codes at 2, 3, 4, 5, 6 or 8 bits, groups
32/64/128, "MLX Runner: An Inference Engine You Can Read", "Architecture: one
command buffer per token") against the float64 oracle: |y - y_ref| <=
2e-3 * sum|x w| + 1e-5 per element. Inputs come from the seeded generators in
`synth` (each row's codes one little-endian bit stream)."""
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


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
# M <= 4: the chunked kernel (M = 2 and 3 below its 4-row instance; K = 96: fewer
# chunks than lanes); M = 7: the one-code-per-lane kernel
@pytest.mark.parametrize("M,N,K,group", [(1, 300, 1024, 64), (4, 77, 2048, 128), (7, 50, 512, 32),
                                         (2, 130, 96, 32), (3, 33, 4096, 64)])
def test_affine_bits_vs_oracle(q, bits, M, N, K, group):
    wq, s, b = synth.affine_weights(N, K, bits, seed=700 + M, slot=bits, group=group)
    x = synth.bf16_normal((M, K), seed=700 + M, slot=1)
    y = q.qgemm_affine(wq.to(DEV), bits, s.to(DEV), b.to(DEV), x.to(DEV))
    torch.cuda.synchronize()
    ref, ad = oracle.affine(wq, bits, s, b, x, group=group)
    d = np.abs(y.cpu().double().numpy() - ref)
    assert np.all(d <= oracle.tolerance(ad)), f"worst {np.max(d / oracle.tolerance(ad)):.3g}x"
