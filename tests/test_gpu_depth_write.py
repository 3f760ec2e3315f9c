"""moda_depth_write: bit-exact slot writes into the packed stream, the
layer-by-layer write path agreeing with moda_pack_depth, and the
sliding-window bounded cache (ring of S slots) matching the oracle on the
last S layers."""
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


@pytest.mark.parametrize("T,Hk,d,L", [(1, 1, 64, 1), (257, 4, 128, 46), (1000, 3, 64, 5)])
def test_layerwise_writes_equal_pack(T, Hk, d, L):
    g = torch.Generator(device="cuda").manual_seed(T + L)
    layers = torch.randn((L, T, Hk, d), generator=g, device="cuda").to(torch.bfloat16)
    dst = torch.full((Hk, T, L, d), float("nan"), device="cuda", dtype=torch.bfloat16)
    for l in range(L):
        moda.moda_depth_write(layers[l].contiguous(), dst, l)
    packed = moda.moda_pack_depth(layers)
    torch.cuda.synchronize()
    assert torch.equal(dst.view(torch.int16), packed.view(torch.int16))


def test_sliding_window_cache_is_the_last_S_layers():
    """Ring of S slots, layer l written to slot l % S: after n > S layers the
    forward over the ring equals the oracle on the last S layers' slots."""
    w = Workload("ring", T=300, Hq=8, Hk=2, d=128, L=11, seed=17)  # 11 layers written
    S = 4
    x = make_inputs(w)
    ring_k = torch.zeros((w.Hk, w.T, S, w.d), device="cuda", dtype=torch.bfloat16)
    ring_v = torch.zeros_like(ring_k)
    for l in range(w.L):
        moda.moda_depth_write(x["kd"][l].cuda().contiguous(), ring_k, l % S)
        moda.moda_depth_write(x["vd"][l].cuda().contiguous(), ring_v, l % S)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = moda.moda_fwd(q, k, v, ring_k, ring_v, w.scale)
    torch.cuda.synchronize()
    last = dict(x, kd=x["kd"][w.L - S:].contiguous(), vd=x["vd"][w.L - S:].contiguous())
    eo, el = gc.compare(last, w.scale, o.float().cpu().numpy(), lse.cpu().numpy())
    assert eo <= gc.TOL_O and el <= gc.TOL_LSE
