"""Seeded random shapes through every forward path and the backward, each
checked against the fp64 oracle in full: T from 1 to 700 (ragged tails, tiles
shorter than one softmax warp's positions), every supported G, one to four
KV heads, d = 64 and 128, L from 0 to 130 (below, at and above one depth
word, and not a multiple of G). Shapes are drawn once from a fixed seed, so
the set is the same on every run."""
import random

import numpy as np
import pytest
import torch

import oracle
import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu


def _shapes(n, seed):
    rnd = random.Random(seed)
    out = []
    for i in range(n):
        G = rnd.choice([1, 2, 4, 8, 16])
        Hk = rnd.choice([1, 2, 3, 4]) if G <= 4 else rnd.choice([1, 2])
        T = rnd.choice([1, 3, rnd.randint(4, 130), rnd.randint(131, 700), rnd.randint(131, 700)])
        L = rnd.choice([0, rnd.randint(1, 33), rnd.randint(1, 33), rnd.randint(34, 130)])
        d = rnd.choice([64, 128])
        out.append(Workload(f"rs{seed}-{i}-T{T}-G{G}-Hk{Hk}-d{d}-L{L}", T=T, Hq=G * Hk, Hk=Hk, d=d,
                            L=L, seed=1000 + i))
    return out


FWD = _shapes(24, seed=5)
BWD = _shapes(8, seed=6)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


@pytest.mark.parametrize("w", FWD, ids=lambda w: w.name)
@pytest.mark.parametrize("layer_major", [False, True], ids=["packed", "layer-major"])
def test_random_shape_forward(w, layer_major):
    gc.check_workload(w, layer_major=layer_major)


@pytest.mark.parametrize("w", BWD, ids=lambda w: w.name)
def test_random_shape_backward(w):
    x = make_inputs(w)
    g = torch.Generator().manual_seed(w.seed)
    dO = torch.randn((w.T, w.Hq, w.d), generator=g).to(torch.bfloat16)
    q, k, v, dOg = (t.cuda() for t in (x["q"], x["k"], x["v"], dO))
    kd = x["kd"].cuda() if w.L else None
    vd = x["vd"].cuda() if w.L else None
    o, lse = moda.moda_fwd_layer_major(q, k, v, kd, vd, w.scale)
    grads = moda.moda_bwd(q, k, v, kd, vd, o, lse, dOg, w.scale, layer_major=True)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    b = {n: bf16_bits(t) for n, t in x.items()}
    ref = oracle.backward(b["q"], b["k"], b["v"], b["kd"] if w.L else None,
                          b["vd"] if w.L else None, bf16_bits(dO), w.scale, nthreads=gc.NTHREADS)
    for name, gg, r in zip(("dq", "dk", "dv", "dkd", "dvd"), grads, ref):
        if r.size == 0:
            continue
        got = gg.cpu().numpy()
        scale = max(float(np.max(np.abs(r))), 1e-30)
        err = float(np.max(np.abs(got - r)))
        assert np.isfinite(got).all(), f"{w.name}.{name}: non-finite"
        assert err <= 1e-2 * scale, f"{w.name}.{name}: {err:.3e} > 1e-2 * {scale:.3e}"
