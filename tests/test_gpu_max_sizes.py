"""The largest sizes the entry points accept, against the fp64 oracle:
L = 1024 depth slots (every depth schedule at its longest: at G = 1 a tile
runs 1024 depth blocks, a softmax warp's word one slot of its 32 positions)
through the forward in both depth layouts, the backward and the decode, and a
sequence of about 2^20 positions (TMA coordinates and tile queues far past
the other tests' sizes).

Random N(0, 1) scores over thousands of keys give nearly uniform rows, where
a wrong or missing key moves o and lse very little; q is scaled by a power of
two in most cases here so that each row is dominated by a few keys and any
wrong one shows."""
import numpy as np
import pytest
import torch

import oracle
import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs, sample_rows

import gpu_common as gc

pytestmark = pytest.mark.gpu

L_MAX = 1024


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


def _sharpen(x, mul):
    x = dict(x)
    x["q"] = (x["q"].float() * mul).to(torch.bfloat16)  # a power of two: exact
    return x


FWD = [
    (Workload("Lmax-T70-G1", T=70, Hq=2, Hk=2, d=128, L=L_MAX, seed=21), 4.0),
    (Workload("Lmax-T45-G16", T=45, Hq=16, Hk=1, d=128, L=L_MAX, seed=22), 1.0),
    (Workload("Lmax-T130-G2-d64", T=130, Hq=4, Hk=2, d=64, L=L_MAX, seed=23), 4.0),
    (Workload("Lmax-T33-G8-d64", T=33, Hq=8, Hk=1, d=64, L=L_MAX, seed=24), 2.0),
]


@pytest.mark.parametrize("layer_major", [False, True], ids=["packed", "layer-major"])
@pytest.mark.parametrize("w,mul", FWD, ids=lambda c: c.name if isinstance(c, Workload) else None)
def test_max_depth_forward_full(w, mul, layer_major):
    gc.check_workload(w, q_mul=mul, layer_major=layer_major)


BWD_REL = 1e-2  # as the other backward tests: 1 % of each gradient's scale


@pytest.mark.parametrize("layer_major", [False, True], ids=["packed", "layer-major"])
@pytest.mark.parametrize("w", [Workload("Lmax-bwd-T40-G4", T=40, Hq=8, Hk=2, d=128, L=L_MAX, seed=31),
                               Workload("Lmax-bwd-T70-G1-d64", T=70, Hq=2, Hk=2, d=64, L=L_MAX, seed=32)],
                         ids=lambda w: w.name)
def test_max_depth_backward(w, layer_major):
    x = _sharpen(make_inputs(w), 2.0)
    g = torch.Generator().manual_seed(78)
    dO = torch.randn((w.T, w.Hq, w.d), generator=g).to(torch.bfloat16)
    q, k, v, dOg = (t.cuda() for t in (x["q"], x["k"], x["v"], dO))
    if layer_major:
        kd, vd = x["kd"].cuda(), x["vd"].cuda()
        o, lse = moda.moda_fwd_layer_major(q, k, v, kd, vd, w.scale)
    else:
        kd, vd = moda.moda_pack_depth(x["kd"].cuda()), moda.moda_pack_depth(x["vd"].cuda())
        o, lse = moda.moda_fwd(q, k, v, kd, vd, w.scale)
    grads = moda.moda_bwd(q, k, v, kd, vd, o, lse, dOg, w.scale, layer_major=layer_major)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    b = {n: bf16_bits(t) for n, t in x.items()}
    ref = list(oracle.backward(b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), w.scale,
                               nthreads=gc.NTHREADS))
    got = [t.cpu().numpy() for t in grads]
    if not layer_major:  # packed [Hk, T, L, d] -> the oracle's [L, T, Hk, d]
        got[3] = got[3].transpose(2, 1, 0, 3)
        got[4] = got[4].transpose(2, 1, 0, 3)
    for name, gg, r in zip(("dq", "dk", "dv", "dkd", "dvd"), got, ref):
        scale = max(float(np.max(np.abs(r))), 1e-30)
        err = float(np.max(np.abs(gg - r)))
        assert np.isfinite(gg).all(), f"{w.name}.{name}: non-finite values"
        assert err <= BWD_REL * scale, f"{w.name}.{name}: max err {err:.3e} > {BWD_REL} * {scale:.3e}"


@pytest.mark.parametrize("w", [Workload("dec-Lmax-T300-G4", T=300, Hq=8, Hk=2, d=128, L=L_MAX, seed=41),
                               Workload("dec-Lmax-T77-G1-d64", T=77, Hq=3, Hk=3, d=64, L=L_MAX, seed=42)],
                         ids=lambda w: w.name)
def test_max_depth_decode(w):
    x = _sharpen(make_inputs(w), 4.0)
    t = w.T - 1
    q = x["q"][t].cuda().contiguous()
    kt = x["kd"][:, t].cuda().permute(1, 0, 2).contiguous()  # [Hk, L, d]
    vt = x["vd"][:, t].cuda().permute(1, 0, 2).contiguous()
    o, lse = moda.moda_decode(q, x["k"].cuda(), x["v"].cuda(), kt, vt, w.scale)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    ro, rl = gc.oracle_rows(x, w.scale, np.full(w.Hq, t), np.arange(w.Hq))
    eo = float(np.max(np.abs(o.float().cpu().numpy() - ro)))
    el = float(np.max(np.abs(lse.cpu().numpy() - rl)))
    assert eo <= gc.TOL_O and el <= gc.TOL_LSE, (eo, el)


@pytest.mark.parametrize("w", [Workload("Tbig-G4", T=(1 << 20) + 5, Hq=4, Hk=1, d=128, L=2, seed=51),
                               Workload("Tbig-G2-d64", T=(1 << 20) + 37, Hq=2, Hk=1, d=64, L=3, seed=52)],
                         ids=lambda w: w.name)
def test_long_sequence_sampled(w):
    """About 2^20 positions, inputs drawn on the device, both depth layouts
    compared with one oracle evaluation on the stratified row sample (tile
    edges, both ends, 64 random positions)."""
    x = _sharpen(make_inputs(w, device="cuda"), 4.0)
    ts, hs = sample_rows(w.T, w.Hq, w.G)
    ti, hi = torch.from_numpy(ts).cuda(), torch.from_numpy(hs).cuda()
    outs = {}
    for name in ("packed", "layer-major"):
        if name == "packed":
            kd, vd = moda.moda_pack_depth(x["kd"]), moda.moda_pack_depth(x["vd"])
            o, lse = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale)
            del kd, vd
        else:
            o, lse = moda.moda_fwd_layer_major(x["q"], x["k"], x["v"], x["kd"], x["vd"], w.scale)
        torch.cuda.synchronize()
        assert moda.moda_get_device_error() == 0
        outs[name] = (o[ti, hi].float().cpu().numpy(), lse[ti, hi].cpu().numpy())
        del o, lse
    xc = {n: t.cpu() for n, t in x.items()}
    del x
    ro, rl = gc.oracle_rows(xc, w.scale, ts, hs)
    for name, (o, lse) in outs.items():
        assert np.isfinite(o).all() and np.isfinite(lse).all(), name
        eo = float(np.max(np.abs(o - ro)))
        el = float(np.max(np.abs(lse - rl)))
        assert eo <= gc.TOL_O and el <= gc.TOL_LSE, (name, eo, el)
