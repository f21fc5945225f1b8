"""Device-side failure reporting, tested without faulting the GPU.

Every wait in the kernels is bounded; a wait that gives up records a code in
the library's sticky error word and its kernel returns, so the context stays
usable. qg_selftest_wait_timeout launches one kernel whose wait can never be
satisfied (an mbarrier nothing arrives at, bounded by a poll count, and a
device counter nothing raises, bounded by time); the test requires the
timeout to be reported through qg_device_error with the kernel's code, the
word to clear, and the next call on the same context to be correct.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from skinny_gemm_qgemv_gb300 import build
    build.build()
    import skinny_gemm_qgemv_gb300 as qq
    qq.lib()
    qq.device_error(clear=True)
    yield qq
    assert qq.device_error(clear=True) == 0


@pytest.mark.parametrize("kind,limit,code", [(0, 4096, 0x501), (1, 2000, 0x502)])
def test_unsatisfiable_wait_times_out_reports_and_context_stays_usable(q, kind, limit, code):
    L = q.lib()
    stream = torch.cuda.current_stream()
    t0 = time.time()
    assert L.qg_selftest_wait_timeout(kind, limit, ctypes.c_void_p(stream.cuda_stream)) == 0
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    c = ctypes.c_uint32(0)
    assert L.qg_device_error(ctypes.byref(c), 1) == 6  # QG_ERR_DEVICE_TIMEOUT, then cleared
    assert c.value == code
    assert L.qg_device_error(ctypes.byref(c), 0) == 0 and c.value == 0
    # the same context serves the next call correctly
    wq, s, b = synth.w4_weights(1000, 4096, seed=31, slot=0)
    x = synth.bf16_normal((4096,), 31, 1)
    y = q.qgemv_w4a16(wq.cuda(), s.cuda(), b.cuda(), x.cuda())
    yr, ad = oracle.w4a16(wq, s, b, x)
    yy = y.cpu().double().numpy()
    assert np.all(np.abs(yy - yr[0]) <= oracle.tolerance(ad[0]))
    assert q.device_error() == 0


def test_selftest_rejects_bad_arguments(q):
    L = q.lib()
    assert L.qg_selftest_wait_timeout(2, 10, None) == 1
    assert L.qg_selftest_wait_timeout(0, 0, None) == 1
    assert L.qg_selftest_wait_timeout(1, 2000000, None) == 1
    assert q.device_error() == 0
