"""moda_decode (one new token: row t = Tctx-1 of the forward for all heads)
against the fp64 oracle, through the C-ABI."""
import numpy as np
import pytest
import torch

import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


def decode_and_compare(w, packed_view=False, device_inputs=False, layer_major_view=False):
    x = make_inputs(w, device="cuda" if device_inputs else "cpu")
    t = w.T - 1
    q = x["q"][t].cuda().contiguous()
    kc, vc = x["k"].cuda(), x["v"].cuda()
    if w.L == 0:
        kt = vt = None
    elif layer_major_view:
        # the layer-major tensors in place: slot stride T*Hk*d, KV-head stride d
        kdl, vdl = x["kd"].cuda(), x["vd"].cuda()
        kt, vt = kdl[:, t].transpose(0, 1), vdl[:, t].transpose(0, 1)
    elif packed_view:
        kp = moda.moda_pack_depth(x["kd"].cuda())
        vp = moda.moda_pack_depth(x["vd"].cuda())
        kt, vt = kp[:, t], vp[:, t]  # [Hk, L, d] with KV-head stride T*L*d
    else:
        kt = x["kd"][:, t].cuda().permute(1, 0, 2).contiguous()
        vt = x["vd"][:, t].cuda().permute(1, 0, 2).contiguous()
    o, lse = moda.moda_decode(q, kc, vc, kt, vt, w.scale)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    xc = {n: v.cpu() for n, v in x.items()}
    ts = np.full(w.Hq, t)
    hs = np.arange(w.Hq)
    ro, rl = gc.oracle_rows(xc, w.scale, ts, hs)
    eo = float(np.max(np.abs(o.float().cpu().numpy() - ro)))
    el = float(np.max(np.abs(lse.cpu().numpy() - rl)))
    assert eo <= gc.TOL_O and el <= gc.TOL_LSE, (eo, el)
    return o, lse, x


CASES = [
    Workload("dec-T1", T=1, Hq=4, Hk=2, d=128, L=3),
    Workload("dec-T1-L0", T=1, Hq=16, Hk=1, d=64, L=0),
    Workload("dec-T300-G4", T=300, Hq=16, Hk=4, d=128, L=46),
    Workload("dec-T257-G1", T=257, Hq=3, Hk=3, d=64, L=1),
    Workload("dec-T5000-G8", T=5000, Hq=16, Hk=2, d=128, L=24, seed=3),
    Workload("dec-T4096-G16", T=4096, Hq=16, Hk=1, d=128, L=96, seed=4),
    Workload("dec-T65-G2", T=65, Hq=4, Hk=2, d=64, L=130, seed=9),
    Workload("dec-T64-G2", T=64, Hq=6, Hk=3, d=128, L=64, seed=10),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_decode_vs_oracle(w):
    decode_and_compare(w)


@pytest.mark.parametrize("w", [Workload("dec-lm-T777-G4", T=777, Hq=8, Hk=2, d=128, L=13, seed=6),
                               Workload("dec-lm-T300-G1-d64", T=300, Hq=3, Hk=3, d=64, L=70, seed=7),
                               Workload("dec-lm-T129-G16", T=129, Hq=16, Hk=1, d=128, L=5, seed=8)],
                         ids=lambda w: w.name)
def test_decode_reads_layer_major_tensors_in_place(w):
    """moda_decode_strided on [L,T,Hk,d] depth tensors, the token's slots
    T*Hk*d elements apart (the layout moda_fwd_layer_major reads)."""
    decode_and_compare(w, layer_major_view=True)


def test_decode_reads_packed_stream_in_place():
    decode_and_compare(Workload("dec-packed", T=777, Hq=8, Hk=2, d=128, L=13, seed=6), packed_view=True)


def test_decode_long_context():
    decode_and_compare(Workload("dec-64k", T=65536, Hq=16, Hk=4, d=128, L=48), device_inputs=True)


def test_decode_equals_last_forward_row():
    w = Workload("dec-vs-fwd", T=2000, Hq=16, Hk=4, d=128, L=20, seed=8)
    o, lse, x = decode_and_compare(w)
    kd = moda.moda_pack_depth(x["kd"].cuda())
    vd = moda.moda_pack_depth(x["vd"].cuda())
    of, lf = moda.moda_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), kd, vd, w.scale)
    assert (of[-1].float() - o.float()).abs().max().item() <= 2 * gc.TOL_O
    assert (lf[-1] - lse).abs().max().item() <= 2 * gc.TOL_LSE
