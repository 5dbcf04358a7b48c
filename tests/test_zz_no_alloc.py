"""lora_mixed_forward_static: the forward pass for callers that cannot allocate device memory.

Serving engines that own every byte of the GPU through their own memory pool (or code that runs while the
allocator must not be touched) cannot hand the layer a freshly allocated workspace.  This entry point keeps
the forward pass's scratch in a fixed device array owned by the library.  These tests call it through the
C ABI and check it against the regular entry point (which uses a caller workspace) and against the float64
oracle on two different batches in a row, so the second call starts from whatever the first one left in the
shared array; check that the second call leaves the device's free memory unchanged (it allocates nothing) and
that its status word reads clean; and check that a batch too large for the array is refused before anything
runs.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import lora_co_serving_gb300 as lm
import oracle
import workloads
from gpu_util import Dev, compare, to_np


@pytest.fixture(scope="module")
def lib():
    lm.build()
    return lm.library()


def _static(lib, d, y, stream):
    s = lm.segments(d.segs)
    wl = d.wl
    return lib.lora_mixed_forward_static(wl.T, wl.K, wl.N, 0, d.x.data_ptr(), d.Wt.data_ptr(), d.pool.cptr(),
                                         s.ctypes.data, s.shape[0], y.data_ptr(), None, 0, stream)


@pytest.mark.gpu
def test_static_scratch_forward_matches_workspace_forward_twice(lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    batches = [
        workloads.config5(K=512, N=768, n_adapters=24, n_decode=150, prefill_tokens=500, len_lo=30, len_hi=250,
                          train_len=100),
        workloads.config2(seed=77, T=300, K=384, N=640, n_adapters=40),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    for i, wl in enumerate(batches):
        d = Dev(wl)
        ref = d.forward()                                  # regular entry point, caller workspace
        y = torch.full_like(ref, float("nan"))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        rc = _static(lib, d, y, stream)
        assert rc == 0, lib.lora_last_error().decode()
        torch.cuda.synchronize()
        if i > 0:
            # the first call on a device may load the library's array; later calls allocate nothing
            assert torch.cuda.mem_get_info()[0] == free0, "the static-scratch forward changed free device memory"
        assert lib.lora_static_status(stream) == 0, lib.lora_last_error().decode()
        compare(to_np(y), to_np(ref), "static-scratch forward vs workspace forward, call %d" % (i + 1))
        compare(to_np(y), oracle.forward_wl(wl), "static-scratch forward vs oracle, call %d" % (i + 1))


def test_static_scratch_rejects_oversized_batch(lib):
    # the full co-serving batch (8192 x 28672 layer) needs more scratch than the fixed array: refused on the
    # host, before any device call
    wl = workloads.config5(K=64, N=64)
    K, N = 8192, 28672
    rank = np.asarray(wl.rank, np.int32)
    a_off = np.concatenate([[0], np.cumsum(rank[:-1].astype(np.int64) * K)]).astype(np.int64)
    b_off = np.concatenate([[0], np.cumsum(rank[:-1].astype(np.int64) * N)]).astype(np.int64)
    scale = np.full(rank.shape[0], 2.0, np.float32)
    pool = lm._Pool(0x10000000, 0x20000000, a_off.ctypes.data, b_off.ctypes.data, rank.ctypes.data,
                    scale.ctypes.data, rank.shape[0])
    s = lm.segments(wl.segs)
    rc = lib.lora_mixed_forward_static(wl.T, K, N, 0, 0x30000000, 0x40000000, ctypes.addressof(pool),
                                       s.ctypes.data, s.shape[0], 0x50000000, None, 0, None)
    assert rc == -10
    assert "scratch" in lib.lora_last_error().decode()
