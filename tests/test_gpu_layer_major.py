"""The forward and backward on layer-major depth K/V (moda_fwd_layer_major,
moda_bwd_layer_major): kd/vd [L,T,Hk,d] as the layers wrote them, each depth
block gathered by the forward's tensor-memory-accelerator copies (the
chunk-aware grouping of Mixture-of-Depths Attention, Sec. 3.2, Fig. 4,
without a relayout pass), against the fp64 oracle, which reads the same
layer-major tensors."""
import numpy as np
import pytest
import torch

import oracle
import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import inputs as wl
from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


# A softmax warp's word of a depth block holds its PW = 32/G positions times
# G slots; the shapes below cover every G, L below, equal to and above one
# word's slots, L not a multiple of G, ragged T, and tail tiles shorter than
# one warp's positions.
EDGE = [
    Workload("lm-T1-G2", T=1, Hq=4, Hk=2, d=64, L=3),
    Workload("lm-T2-G16", T=2, Hq=16, Hk=1, d=128, L=5),
    Workload("lm-T3-G4", T=3, Hq=8, Hk=2, d=64, L=1),
    Workload("lm-T127-G8", T=127, Hq=16, Hk=2, d=128, L=7),
    Workload("lm-T129-G1", T=129, Hq=3, Hk=3, d=64, L=2),
    Workload("lm-T200-G2-L96", T=200, Hq=4, Hk=2, d=128, L=96),
    Workload("lm-T300-G16-L48", T=300, Hq=16, Hk=1, d=64, L=48),
    Workload("lm-T1000-G4-L24", T=1000, Hq=8, Hk=2, d=128, L=24, seed=4),
    Workload("lm-T1000-G4-L46", T=1000, Hq=8, Hk=2, d=128, L=46, seed=5),
    Workload("lm-T513-G1-L33", T=513, Hq=2, Hk=2, d=128, L=33, seed=6),
    Workload("lm-T385-G4-L46-d64", T=385, Hq=8, Hk=2, d=64, L=46, seed=11),
    Workload("lm-T700-G2-L90-d64", T=700, Hq=4, Hk=2, d=64, L=90, seed=12),
    Workload("lm-T1000-G8-L64-d64", T=1000, Hq=16, Hk=2, d=64, L=64, seed=13),
    Workload("lm-T100-G1-L200-d64", T=100, Hq=2, Hk=2, d=64, L=200, seed=14),
    Workload("lm-T64-G16-L0", T=64, Hq=16, Hk=1, d=128, L=0),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_layer_major_edge_shapes_full(w):
    gc.check_workload(w, layer_major=True)


def test_layer_major_700m_layer_full():
    gc.check_workload(wl.LAYER_700M, layer_major=True)


@pytest.mark.parametrize("w", wl.GQA_SWEEP, ids=lambda w: w.name)
def test_layer_major_gqa_sweep_sampled(w):
    gc.check_workload(w, sampled=True, layer_major=True)


def test_layer_major_long_64k_sampled():
    gc.check_workload(wl.LONG, sampled=True, device_inputs=True, layer_major=True)


def test_layer_major_table2_sampled():
    w = next(w for w in wl.TABLE2 if w.T == 16384)
    gc.check_workload(w, sampled=True, device_inputs=True, layer_major=True)


@pytest.mark.parametrize("w", [Workload("lm-vs-packed-d128", T=1500, Hq=16, Hk=4, d=128, L=48, seed=7),
                               Workload("lm-vs-packed-d64", T=900, Hq=8, Hk=1, d=64, L=20, seed=8)],
                         ids=lambda w: w.name)
def test_layer_major_matches_packed_path(w):
    """Same inputs through moda_pack_depth + moda_fwd: the depth terms are
    summed in another order, so the results agree to rounding."""
    x = make_inputs(w)
    o1, l1 = gc.run_cuda(x, w.scale)
    o2, l2 = gc.run_cuda(x, w.scale, layer_major=True)
    assert np.max(np.abs(o1 - o2)) <= 4e-3
    assert np.max(np.abs(l1 - l2)) <= 1e-5


def test_layer_major_prefix_of_a_larger_buffer():
    """Layer l of a bigger [Lmax, T, Hk, d] buffer: the first L layers are a
    contiguous prefix, so a slice kd[:L] is itself layer-major and exact."""
    w = Workload("lm-prefix", T=300, Hq=8, Hk=2, d=128, L=12, seed=9)
    x = make_inputs(w)
    big = torch.zeros((20, w.T, w.Hk, w.d), dtype=torch.bfloat16)
    big[:w.L] = x["kd"]
    bigv = torch.zeros_like(big)
    bigv[:w.L] = x["vd"]
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = moda.moda_fwd_layer_major(q, k, v, big.cuda()[:w.L], bigv.cuda()[:w.L], w.scale)
    torch.cuda.synchronize()
    eo, el = gc.compare(x, w.scale, o.float().cpu().numpy(), lse.cpu().numpy())
    assert eo <= gc.TOL_O and el <= gc.TOL_LSE


# ---------------------------------------------------------------- backward
BWD_REL = 1e-2  # as the packed backward's tests: 1 % of each gradient's scale


def _bwd_check(name, got, ref):
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    err = float(np.max(np.abs(got - ref)))
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    assert err <= BWD_REL * scale, f"{name}: max err {err:.3e} > {BWD_REL} * {scale:.3e}"


@pytest.mark.parametrize("w", [Workload("lm-bwd-T300-G4", T=300, Hq=8, Hk=2, d=128, L=24, seed=5),
                               Workload("lm-bwd-T200-G1-d64", T=200, Hq=3, Hk=3, d=64, L=33),
                               Workload("lm-bwd-T127-G8", T=127, Hq=16, Hk=2, d=128, L=7)],
                         ids=lambda w: w.name)
def test_layer_major_backward_matches_oracle(w):
    """moda_fwd_layer_major then moda_bwd_layer_major: every gradient against
    the oracle backward, dkd/dvd compared in their own [L,T,Hk,d] layout."""
    x = make_inputs(w)
    g = torch.Generator().manual_seed(77)
    dO = torch.randn((w.T, w.Hq, w.d), generator=g).to(torch.bfloat16)
    q, k, v, kd, vd, dOg = (t.cuda() for t in (x["q"], x["k"], x["v"], x["kd"], x["vd"], dO))
    o, lse = moda.moda_fwd_layer_major(q, k, v, kd, vd, w.scale)
    grads = moda.moda_bwd(q, k, v, kd, vd, o, lse, dOg, w.scale, layer_major=True)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    b = {n: bf16_bits(t) for n, t in x.items()}
    ref = oracle.backward(b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), w.scale,
                          nthreads=gc.NTHREADS)
    for name, gg, r in zip(("dq", "dk", "dv", "dkd", "dvd"), grads, ref):
        _bwd_check(f"{w.name}.{name}", gg.cpu().numpy(), r)


def test_layer_major_backward_equals_packed_backward():
    """Same o, lse and dO into moda_bwd (packed streams) and
    moda_bwd_layer_major: only the depth rows' addresses differ, so every
    gradient is bit-identical (dkd/dvd after the relayout)."""
    w = Workload("lm-bwd-eq", T=700, Hq=16, Hk=4, d=128, L=20, seed=3)
    x = {n: t.cuda() for n, t in make_inputs(w).items()}
    g = torch.Generator(device="cuda").manual_seed(5)
    dO = torch.randn((w.T, w.Hq, w.d), generator=g, device="cuda").to(torch.bfloat16)
    kd = moda.moda_pack_depth(x["kd"])
    vd = moda.moda_pack_depth(x["vd"])
    o, lse = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale)
    gp = moda.moda_bwd(x["q"], x["k"], x["v"], kd, vd, o, lse, dO, w.scale)
    gl = moda.moda_bwd(x["q"], x["k"], x["v"], x["kd"], x["vd"], o, lse, dO, w.scale,
                       layer_major=True)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    for a, b_ in zip(gp[:3], gl[:3]):
        assert torch.equal(a, b_)
    for a, b_ in zip(gp[3:], gl[3:]):
        assert torch.equal(a.permute(2, 1, 0, 3), b_)
