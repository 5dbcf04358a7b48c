"""Failure detection on the GPU without faulting it.

Every wait in the library's kernels is bounded.  The self-test kernel waits on a barrier that nothing ever
completes; the wait must give up (about one second), record LORA_ERR_TIMEOUT in the workspace status word that
the host reads back, and leave the CUDA context usable for the next call.
"""
import time

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import Dev, compare, to_np

pytestmark = pytest.mark.gpu


def test_wait_limit_is_settable():
    """With the limit lowered to 50 ms the never-completed wait gives up in well under the default second; the
    default is restored afterwards."""
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()
    lib = lm.library()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    try:
        lm.set_wait_limit(0.05)
        t0 = time.perf_counter()
        assert lib.lora_selftest_wait_timeout(ws.data_ptr(), ws.numel(), stream) == 0
        rc = lib.lora_workspace_status(ws.data_ptr(), stream)
        spent = time.perf_counter() - t0
    finally:
        lm.set_wait_limit(1.0)
    assert rc == -11, rc                                   # LORA_ERR_TIMEOUT
    assert 0.04 < spent < 0.5, spent


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()
    lib = lm.library()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.lora_selftest_wait_timeout(ws.data_ptr(), ws.numel(), stream) == 0
    rc = lib.lora_workspace_status(ws.data_ptr(), stream)
    assert rc == -11, rc                                   # LORA_ERR_TIMEOUT
    assert "bounded wait" in lib.lora_last_error().decode()
    # the context is still usable: a normal call on a fresh workspace runs and reports no error
    wl = workloads.config5(K=256, N=384, n_adapters=10, n_decode=40, prefill_tokens=120, len_lo=20, len_hi=80,
                           train_len=40)
    d = Dev(wl)
    wsz = lm.workspace_size(wl.T, wl.K, wl.N, 0, d.pool, wl.segs)
    ws2 = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    y = d.forward(workspace=ws2)
    lm.workspace_status(ws2)
    compare(to_np(y), oracle.forward_wl(wl), "y after a timed-out self-test")
