"""moda_bwd_noalloc -- the backward for callers that cannot give the library
device memory for scratch -- must agree with moda_bwd (caller workspace) on
the same inputs, on two calls in a row. Before the checked calls, one call
with a different upstream gradient fills the shared scratch with other
values, so a row the delta kernel failed to write would show up as wrong
gradients. Both entry points run the same deterministic kernels (no atomics),
so the gradients must agree bit for bit, and a fortiori within the backward
tests' tolerance. Collected last so that a failure here does not hide the
other tests in a run that stops at the first failure."""
import numpy as np
import pytest
import torch

import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import build as mbuild
from sequence_depth_attention_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu
REL = 1e-2  # the backward tests' tolerance: 1 % of each gradient's scale


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    moda.load()


def _grads(w):
    f32 = dict(dtype=torch.float32, device="cuda")
    return (torch.empty((w.T, w.Hq, w.d), **f32), torch.empty((w.T, w.Hk, w.d), **f32),
            torch.empty((w.T, w.Hk, w.d), **f32),
            torch.empty((w.Hk, w.T, w.L, w.d), **f32) if w.L else None,
            torch.empty((w.Hk, w.T, w.L, w.d), **f32) if w.L else None)


@pytest.mark.parametrize("w", [Workload("noalloc-a", T=700, Hq=16, Hk=4, d=128, L=24, seed=21),
                               Workload("noalloc-b", T=300, Hq=8, Hk=2, d=64, L=0, seed=22)],
                         ids=lambda w: w.name)
def test_noalloc_backward_matches_workspace_backward(w):
    x = {n: t.cuda() for n, t in make_inputs(w).items()}
    kd = moda.moda_pack_depth(x["kd"]) if w.L else None
    vd = moda.moda_pack_depth(x["vd"]) if w.L else None
    o, lse = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale)
    g = torch.Generator(device="cuda").manual_seed(5)
    dO = torch.randn((w.T, w.Hq, w.d), generator=g, device="cuda").to(torch.bfloat16)
    dO_other = torch.randn((w.T, w.Hq, w.d), generator=g, device="cuda").to(torch.bfloat16)
    args = (x["q"], x["k"], x["v"], kd, vd, o, lse, dO, w.scale)
    ref = moda.moda_bwd(*args)
    # leaves the scratch holding the deltas of another dO
    moda.moda_bwd_noalloc(x["q"], x["k"], x["v"], kd, vd, o, lse, dO_other, w.scale,
                          grads=_grads(w))
    for _ in range(2):
        got = moda.moda_bwd_noalloc(*args, grads=_grads(w))
        torch.cuda.synchronize()
        assert moda.moda_get_device_error() == 0
        for r, a in zip(ref, got):
            if r is None:
                continue
            r, a = r.cpu().numpy(), a.cpu().numpy()
            assert np.isfinite(a).all()
            assert np.max(np.abs(a - r)) <= REL * max(np.max(np.abs(r)), 1e-30)
            assert np.array_equal(a, r)


def test_noalloc_rejects_oversize():
    w = Workload("noalloc-big", T=(1 << 20) // 16 + 1, Hq=16, Hk=4, d=128, L=0)
    lib = moda.load()
    fake = 0x10000000
    rc = lib.moda_bwd_noalloc(*([fake] * 8), w.T, w.Hq, w.Hk, w.d, w.L, 0.1, *([fake + (1 << 40)] * 5),
                              None)
    assert rc == 2  # MODA_ERR_UNSUPPORTED, nothing launched
