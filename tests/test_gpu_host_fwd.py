"""moda_fwd_layer_major_host: the forward from and to host memory. The
library copies the host inputs into a device workspace, runs the same kernel
as moda_fwd_layer_major and copies o and lse back, so the results must be
bit-identical to the device call on the same inputs (and match the oracle)."""
import numpy as np
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


def _device_call(x, scale):
    q, k, v, kd, vd = (x[n].cuda() for n in ("q", "k", "v", "kd", "vd"))
    L = kd.shape[0]
    o, lse = moda.moda_fwd_layer_major(q, k, v, kd if L else None, vd if L else None, scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def _host(x, pinned):
    return {n: (t.pin_memory() if pinned else t.clone()) for n, t in x.items()}


CASES = [
    Workload("host-T300-G4", T=300, Hq=8, Hk=2, d=128, L=12, seed=61),
    Workload("host-T129-G1-d64", T=129, Hq=3, Hk=3, d=64, L=33, seed=62),
    Workload("host-T64-G16-L0", T=64, Hq=16, Hk=1, d=128, L=0, seed=63),
    Workload("host-T1000-G8-d64", T=1000, Hq=16, Hk=2, d=64, L=64, seed=64),
]


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_host_call_equals_device_call(w, pinned):
    x = make_inputs(w)
    h = _host(x, pinned)
    L = w.L
    o, lse = moda.moda_fwd_layer_major_host(h["q"], h["k"], h["v"], h["kd"] if L else None,
                                            h["vd"] if L else None, w.scale)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    assert not o.is_cuda and not lse.is_cuda
    od, ld = _device_call(x, w.scale)
    assert torch.equal(o.view(torch.int16), od.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ld.view(torch.int32))
    eo, el = gc.compare(x, w.scale, o.float().numpy(), lse.numpy())
    assert eo <= gc.TOL_O and el <= gc.TOL_LSE, (eo, el)


def test_host_call_without_lse():
    w = CASES[0]
    x = make_inputs(w)
    h = _host(x, True)
    o, lse = moda.moda_fwd_layer_major_host(h["q"], h["k"], h["v"], h["kd"], h["vd"], w.scale,
                                            want_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    od, _ = _device_call(x, w.scale)
    assert torch.equal(o.view(torch.int16), od.view(torch.int16))


def test_two_streams_two_workspaces_alternating():
    """Calls alternate between two streams, each with its own workspace and
    host outputs, so one call's copies overlap the other's forward; every
    call's result equals the device call on its own inputs."""
    w = Workload("host-alt", T=700, Hq=16, Hk=4, d=128, L=20, seed=65)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    need = moda.moda_fwd_host_workspace_bytes(w.T, w.Hq, w.Hk, w.d, w.L)
    wss = [torch.empty((need,), dtype=torch.uint8, device="cuda") for _ in range(2)]
    inputs = [make_inputs(w, seed=100 + i) for i in range(6)]
    hosts = [_host(x, True) for x in inputs]
    outs = []
    for i, h in enumerate(hosts):
        s = streams[i % 2]
        o = torch.empty((w.T, w.Hq, w.d), dtype=torch.bfloat16, pin_memory=True)
        lse = torch.empty((w.T, w.Hq), dtype=torch.float32, pin_memory=True)
        moda.moda_fwd_layer_major_host(h["q"], h["k"], h["v"], h["kd"], h["vd"], w.scale, o=o,
                                       lse=lse, workspace=wss[i % 2], stream=s)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    for x, (o, lse) in zip(inputs, outs):
        od, ld = _device_call(x, w.scale)
        assert torch.equal(o.view(torch.int16), od.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ld.view(torch.int32))


def test_workspace_too_small_is_rejected():
    w = CASES[0]
    x = _host(make_inputs(w), True)
    need = moda.moda_fwd_host_workspace_bytes(w.T, w.Hq, w.Hk, w.d, w.L)
    ws = torch.empty((need - 256,), dtype=torch.uint8, device="cuda")
    with pytest.raises(moda.ModaError):
        moda.moda_fwd_layer_major_host(x["q"], x["k"], x["v"], x["kd"], x["vd"], w.scale,
                                       workspace=ws)
    assert moda.moda_get_device_error() == 0
