"""The layer captured into a CUDA graph and replayed.

Serving engines replay decode (and inference prefill) steps from captured graphs to drop per-launch host cost
("DeltaServe: Host-Agnostic Co-Serving of Inference and Fine-Tuning for LLMs", section 2.5 and section 3.3,
execution modes).  A captured forward + backward must replay to exactly the results of the same calls made
eagerly, after other calls have reused the library's plan staging buffers, and again after new input values are
written into the captured buffers.
"""
import numpy as np
import pytest

import workloads
from gpu_util import Dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()
    lm.library()


def eager(lm, d, ws, stream, sliced=None):
    if sliced is None:
        y = lm.forward(d.x, d.Wt, d.pool, d.segs, workspace=ws, stream=stream)
        g = lm.backward(d.x, d.Wt, d.pool, d.segs, d.dY, recompute=True, workspace=ws, stream=stream)
    else:
        y = lm.sliced_forward(d.x, d.Wt, d.pool, sliced, d.segs, workspace=ws, stream=stream)
        g = lm.sliced_backward(d.x, d.Wt, d.pool, sliced, d.segs, d.dY, recompute=True, workspace=ws, stream=stream)
    return [y] + list(g)


@pytest.mark.parametrize("kind", ["decode", "mixed", "sliced"])
def test_capture_and_replay_bitwise(kind):
    import torch
    import lora_co_serving_gb300 as lm
    if kind == "decode":
        wl = workloads.config2(T=200, K=512, N=768, n_adapters=40)
        wl.dY = workloads.bf16_round(np.random.default_rng(0).standard_normal((wl.T, wl.N)).astype(np.float32))
        # fine-tuning rows so that the backward has work: a 24-token segment on adapter 3 at the end
        segs = wl.segs.tolist()[:176] + [(176, 24, 3, 1)]
        wl.segs = np.asarray(segs, np.int32)
        sliced = None
    elif kind == "mixed":
        wl = workloads.config5(K=512, N=768, n_adapters=24, n_decode=150, prefill_tokens=500, len_lo=30,
                               len_hi=250, train_len=100)
        sliced = None
    else:
        base = workloads.config5(K=64, N=64, n_adapters=24, n_decode=150, prefill_tokens=500, len_lo=30, len_hi=250,
                                 train_len=100)
        wl = workloads.sliced(41, base.T, 512, [0, 512, 768, 1024], base.segs, base.rank)
        sliced = lm.Slices(wl.bounds)
    d = Dev(wl)
    size = (lm.sliced_workspace_size(wl.T, wl.K, wl.N, lm.BF16, d.pool, sliced, d.segs) if sliced is not None
            else lm.workspace_size(wl.T, wl.K, wl.N, lm.BF16, d.pool, d.segs))
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ref = [t.clone() for t in eager(lm, d, ws, s, sliced)]          # eager results (and one-time setup)
        y = torch.empty_like(ref[0])
        dX, dA, dB = [torch.zeros_like(t) for t in ref[1:]]
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        if sliced is None:
            lm.forward(d.x, d.Wt, d.pool, d.segs, y=y, workspace=ws, stream=s)
            lm.backward(d.x, d.Wt, d.pool, d.segs, d.dY, dX=dX, dA=dA, dB=dB, recompute=True, workspace=ws, stream=s)
        else:
            lm.sliced_forward(d.x, d.Wt, d.pool, sliced, d.segs, y=y, workspace=ws, stream=s)
            lm.sliced_backward(d.x, d.Wt, d.pool, sliced, d.segs, d.dY, dX=dX, dA=dA, dB=dB, recompute=True,
                               workspace=ws, stream=s)

    # other calls in between reuse the library's staging buffers and overwrite the shared workspace
    other = workloads.config2(T=64, K=wl.K, N=wl.N, n_adapters=8, seed=77)
    od = Dev(other)
    ows = torch.empty(lm.workspace_size(other.T, other.K, other.N, lm.BF16, od.pool, od.segs), dtype=torch.uint8,
                      device="cuda")
    for _ in range(20):
        od.forward(workspace=ows)
    if sliced is None:
        lm.forward(d.x, d.Wt, d.pool, d.segs, workspace=ws)          # and an eager call on the same workspace
    torch.cuda.synchronize()

    g.replay()
    torch.cuda.synchronize()
    for name, a, b in zip(("y", "dX", "dA", "dB"), (y, dX, dA, dB), ref):
        assert torch.equal(a, b), "replayed %s differs from the eager call" % name

    # new values in the captured input buffers: the replay computes on them
    rng = np.random.default_rng(5)
    x2 = workloads.bf16_round(rng.standard_normal((wl.T, wl.K)).astype(np.float32))
    d.x.copy_(to_dev(x2, "bf16"))
    with torch.cuda.stream(s):
        ref2 = [t.clone() for t in eager(lm, d, ws, s, sliced)]
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for name, a, b in zip(("y", "dX", "dA", "dB"), (y, dX, dA, dB), ref2):
        assert torch.equal(a, b), "replay on new inputs: %s differs from the eager call" % name
    assert not torch.equal(ref2[0], ref[0])
