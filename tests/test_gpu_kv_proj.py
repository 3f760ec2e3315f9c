"""moda_kv_proj_write (an FFN layer's depth K/V, projected from the FFN's input
and written into its slot of the packed streams) against the fp64 oracle.

Tolerance, derived from the arithmetic: bf16 products are exact in fp32, the
fp32 sum over Dm terms errs by at most Dm * 2^-24 * sum|x_c w_c| (taken twice
as a margin), and the final rounding to bf16 adds at most 2^-8 of the value.
Every slot other than `slot` must come back bit-identical."""
import numpy as np
import pytest
import torch

import oracle
from sequence_depth_attention_gb300 import binding as moda
from sequence_depth_attention_gb300.inputs import (PROJ_LONG, ProjWorkload, bf16_bits,
                                                   make_proj_inputs)

pytestmark = pytest.mark.gpu

CASES = [
    ProjWorkload("proj-T200-d64", T=200, Dm=256, Hk=2, d=64, L=5, slot=3),
    ProjWorkload("proj-T300-Hk3", T=300, Dm=512, Hk=3, d=128, L=2, slot=0, seed=4),
    ProjWorkload("proj-T1", T=1, Dm=64, Hk=1, d=128, L=1, slot=0),
    ProjWorkload("proj-T129-last-slot", T=129, Dm=192, Hk=5, d=64, L=7, slot=6, seed=2),
]


def _check(w, x, wk, wv, out_k, out_v, rows):
    """Compare out_k/out_v [n_rows, Hk*d] (GPU, fp32 view of bf16) with the oracle."""
    xb = bf16_bits(x.cpu())
    xv = x.cpu().double().numpy()[rows]
    for wt, got, name in ((wk, out_k, "K"), (wv, out_v, "V")):
        ref = oracle.kv_proj(xb, bf16_bits(wt.cpu()), rows)
        absum = np.abs(xv) @ np.abs(wt.cpu().double().numpy()).T
        tol = 2.0 ** -8 * np.abs(ref) + 2 * w.Dm * 2.0 ** -24 * absum + 1e-30
        err = np.abs(got - ref)
        bad = err > tol
        assert not bad.any(), (f"{w.name} {name}: {bad.sum()} elements out of tolerance, "
                               f"worst {err.max():.3e} (tol there {tol[np.unravel_index(err.argmax(), err.shape)]:.3e})")


def _run(w, dev="cuda"):
    inp = make_proj_inputs(w, device="cpu")
    g = {k: v.to(dev) for k, v in inp.items()}
    kd0, vd0 = g["kd"].clone(), g["vd"].clone()
    moda.moda_kv_proj_write(g["x"], g["wk"], g["wv"], g["kd"], g["vd"], w.slot)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    return inp, g, kd0, vd0


def _slot_rows(t, Hk, d, rows):
    # [Hk, T, d] slot view -> [n_rows, Hk*d] in feature order hk*d + j
    return t[:, rows, :].permute(1, 0, 2).reshape(len(rows), Hk * d).double().cpu().numpy()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_kv_proj_full(w):
    inp, g, kd0, vd0 = _run(w)
    rows = np.arange(w.T)
    _check(w, inp["x"], inp["wk"], inp["wv"], _slot_rows(g["kd"][:, :, w.slot], w.Hk, w.d, rows),
           _slot_rows(g["vd"][:, :, w.slot], w.Hk, w.d, rows), rows)
    others = [l for l in range(w.L) if l != w.slot]
    if others:
        assert torch.equal(g["kd"][:, :, others], kd0[:, :, others])
        assert torch.equal(g["vd"][:, :, others], vd0[:, :, others])


def test_kv_proj_long_sampled():
    w = PROJ_LONG
    g = make_proj_inputs(w, device="cuda")
    kd0_prev = g["kd"][:, :, w.slot - 1].clone()
    vd0_first = g["vd"][:, :, 0].clone()
    moda.moda_kv_proj_write(g["x"], g["wk"], g["wv"], g["kd"], g["vd"], w.slot)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 129, w.T // 2, w.T - 2, w.T - 1],
                                     rng.integers(0, w.T, 56)]))
    _check(w, g["x"], g["wk"], g["wv"], _slot_rows(g["kd"][:, :, w.slot], w.Hk, w.d, rows),
           _slot_rows(g["vd"][:, :, w.slot], w.Hk, w.d, rows), rows)
    assert torch.equal(g["kd"][:, :, w.slot - 1], kd0_prev)
    assert torch.equal(g["vd"][:, :, 0], vd0_first)


def test_kv_proj_two_layers_keep_each_others_slots():
    """Two FFN layers write slots 0 and 1 of the same streams; the second call
    leaves the first one's slot intact."""
    w = ProjWorkload("proj-two", T=256, Dm=128, Hk=2, d=64, L=2, slot=0, seed=7)
    inp, g, kd0, vd0 = _run(w)
    first_k = g["kd"][:, :, 0].clone()
    w2 = ProjWorkload("proj-two", T=256, Dm=128, Hk=2, d=64, L=2, slot=1, seed=8)
    inp2 = make_proj_inputs(w2, device="cpu")
    moda.moda_kv_proj_write(inp2["x"].cuda(), inp2["wk"].cuda(), inp2["wv"].cuda(), g["kd"], g["vd"], 1)
    torch.cuda.synchronize()
    assert torch.equal(g["kd"][:, :, 0], first_k)
    rows = np.arange(w.T)
    _check(w2, inp2["x"], inp2["wk"], inp2["wv"], _slot_rows(g["kd"][:, :, 1], w.Hk, w.d, rows),
           _slot_rows(g["vd"][:, :, 1], w.Hk, w.d, rows), rows)
