"""LORA_DEBUG_CHECKS on the GPU: with every store index checked in the kernels (and the plan checked on the host
first), valid batches report LORA_OK in the status word and give bit-for-bit the results of the unchecked path.

No test here provokes a failing check on the device: a kernel that skipped a store would leave its outputs
incomplete, and the cases that would trigger it are planner bugs; the host half of the checker is exercised
against planted planner mistakes in test_plan_check.py.
"""
import numpy as np
import pytest

import workloads
from gpu_util import Dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()


def bits(t):
    import torch
    return t.detach().contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


CASES = {
    "decode_cuda_core_shrink": lambda: workloads.config2(T=300, K=384, N=640, n_adapters=40),
    "cosrv_split_main": lambda: workloads.config5(K=384, N=640, n_adapters=30, n_decode=200, prefill_tokens=600,
                                                  len_lo=40, len_hi=300, train_len=120),
    "cosrv_full_table": lambda: workloads.config5(K=256, N=1024),
    "mixed_saved": lambda: workloads.config3(K=256, N=512, prefill_tokens=600, train_len=150, len_lo=64, len_hi=300),
}


@pytest.mark.parametrize("case", list(CASES))
def test_debug_checks_clean_and_identical(case):
    import torch
    wl = CASES[case]()
    d = Dev(wl)
    save = wl.xa_mode == "save"
    ref = d.forward(save_xa=save)
    got = d.forward(save_xa=save, debug=True, check_status=True)
    ref, got = (ref, got) if save else ((ref,), (got,))
    for a, b in zip(ref, got):
        assert np.array_equal(bits(a), bits(b))
    if any(q[3] for q in wl.segs.tolist()):
        xs = ref[1] if save else None
        g0 = d.backward(xa_saved=xs)
        g1 = d.backward(xa_saved=xs, debug=True, check_status=True)
        torch.cuda.synchronize()
        for a, b in zip(g0, g1):
            assert np.array_equal(bits(a), bits(b))
