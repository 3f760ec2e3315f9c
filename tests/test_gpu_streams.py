"""The forward under concurrency and graph capture, through the C-ABI.

The persistent d = 128 forward hands out its tiles through one of 64
per-device queues taken in turn per call, and zeroes it when it completes.
These tests run forwards concurrently on several streams (each call must
still see only its own queue) and inside a captured CUDA graph replayed
several times (the captured call reuses its queue on every replay, which is
clean again when the previous replay completed), and check every result
bit for bit against the same call made alone."""
import pytest
import torch

import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300.inputs import Workload, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


SHAPES = [
    Workload("st-a", T=2000, Hq=16, Hk=4, d=128, L=24, seed=1),
    Workload("st-b", T=777, Hq=8, Hk=1, d=128, L=7, seed=2),
    Workload("st-c", T=1500, Hq=4, Hk=4, d=128, L=0, seed=3),
    Workload("st-d", T=1200, Hq=16, Hk=2, d=64, L=40, seed=4),
    Workload("st-e", T=3000, Hq=16, Hk=4, d=128, L=48, seed=5),
]


def _inputs(w):
    x = {n: t.cuda() for n, t in make_inputs(w).items()}
    if w.L == 0:
        x["kd"] = x["vd"] = None
    return x


def _alone(w, x):
    o, lse = moda.moda_fwd_layer_major(x["q"], x["k"], x["v"], x["kd"], x["vd"], w.scale)
    torch.cuda.synchronize()
    return o.clone(), lse.clone()


def test_concurrent_forwards_on_streams():
    xs = [_inputs(w) for w in SHAPES]
    ref = [_alone(w, x) for w, x in zip(SHAPES, xs)]
    streams = [torch.cuda.Stream() for _ in SHAPES]
    outs = [[(torch.empty_like(x["q"]), torch.empty((w.T, w.Hq), device="cuda")) for _ in range(3)]
            for w, x in zip(SHAPES, xs)]
    torch.cuda.synchronize()
    # every stream launches three forwards without waiting; the launches
    # interleave on the device
    for rep in range(3):
        for i, (w, x, s) in enumerate(zip(SHAPES, xs, streams)):
            o, lse = outs[i][rep]
            moda.moda_fwd_layer_major(x["q"], x["k"], x["v"], x["kd"], x["vd"], w.scale, o=o,
                                      lse=lse, stream=s)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    for i in range(len(SHAPES)):
        for o, lse in outs[i]:
            assert torch.equal(o.view(torch.int16), ref[i][0].view(torch.int16))
            assert torch.equal(lse, ref[i][1])


def test_forward_replayed_from_a_cuda_graph():
    w = SHAPES[0]
    x = _inputs(w)
    o = torch.empty_like(x["q"])
    lse = torch.empty((w.T, w.Hq), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first call outside the capture: library set-up
        moda.moda_fwd_layer_major(x["q"], x["k"], x["v"], x["kd"], x["vd"], w.scale, o=o, lse=lse,
                                  stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moda.moda_fwd_layer_major(x["q"], x["k"], x["v"], x["kd"], x["vd"], w.scale, o=o, lse=lse,
                                  stream=s)
    for seed in (11, 12, 13):
        # new contents in the captured input buffers, then one replay
        gen = torch.Generator(device="cuda").manual_seed(seed)
        x["q"].copy_(torch.randn(x["q"].shape, generator=gen, device="cuda").to(torch.bfloat16))
        x["kd"].copy_(torch.randn(x["kd"].shape, generator=gen, device="cuda").to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert moda.moda_get_device_error() == 0
        o_ref, l_ref = _alone(w, x)
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, l_ref)
