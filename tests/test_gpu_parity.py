"""CUDA path vs the fp64 oracle, element by element, through the C-ABI."""
import numpy as np
import pytest
import torch

import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import inputs as wl
from sequence_depth_attention_gb300.inputs import Workload, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


# ---------------------------------------------------------------- pack
@pytest.mark.parametrize("L,T,Hk,d", [(1, 1, 1, 64), (4, 128, 2, 64), (46, 257, 4, 128),
                                      (3, 1000, 3, 128), (96, 33, 1, 64)])
def test_pack_depth_bit_exact(L, T, Hk, d):
    g = torch.Generator(device="cuda").manual_seed(L * 1000 + T)
    src = torch.randn((L, T, Hk, d), generator=g, device="cuda").to(torch.bfloat16)
    dst = moda.moda_pack_depth(src)
    torch.cuda.synchronize()
    want = src.permute(2, 1, 0, 3).contiguous()
    assert torch.equal(dst.view(torch.int16), want.view(torch.int16))


# ---------------------------------------------------------------- configs
def test_tiny_full():
    gc.check_workload(wl.TINY)


def test_700m_layer_full():
    gc.check_workload(wl.LAYER_700M)


@pytest.mark.parametrize("w", wl.GQA_SWEEP, ids=lambda w: w.name)
def test_gqa_sweep_sampled(w):
    gc.check_workload(w, sampled=True)


@pytest.mark.parametrize("w", wl.DEPTH_SWEEP, ids=lambda w: w.name)
def test_depth_sweep_sampled(w):
    gc.check_workload(w, sampled=True, device_inputs=True)


def test_long_64k_sampled():
    gc.check_workload(wl.LONG, sampled=True, device_inputs=True)


def test_long_64k_l0_sampled():
    gc.check_workload(wl.LONG_L0, sampled=True, device_inputs=True)


# ---------------------------------------------------------------- edges
EDGE = [
    Workload("T1", T=1, Hq=4, Hk=2, d=64, L=3),
    Workload("T1-L0", T=1, Hq=2, Hk=2, d=128, L=0),
    Workload("T2-G16", T=2, Hq=16, Hk=1, d=128, L=5),
    Workload("T3-G4", T=3, Hq=8, Hk=2, d=64, L=1),
    Workload("T127-G8", T=127, Hq=16, Hk=2, d=128, L=7),
    Workload("T129-G1", T=129, Hq=3, Hk=3, d=64, L=2),
    Workload("T200-G2-L96", T=200, Hq=4, Hk=2, d=128, L=96),
    Workload("T300-G16-L48", T=300, Hq=16, Hk=1, d=64, L=48),
    Workload("T513-G4-L0", T=513, Hq=8, Hk=2, d=128, L=0),
    Workload("T1000-G4-L24", T=1000, Hq=8, Hk=2, d=128, L=24, seed=4),
    # d = 64 runs two tiles per CTA: pairs whose tiles use very different
    # K/V blocks (long depth runs of one tile), odd tile counts, a lone tile
    Workload("T200-G1-L33-d64", T=200, Hq=3, Hk=3, d=64, L=33),
    Workload("T385-G4-L46-d64", T=385, Hq=8, Hk=2, d=64, L=46, seed=11),
    Workload("T700-G2-L90-d64", T=700, Hq=4, Hk=2, d=64, L=90, seed=12),
    Workload("T1000-G8-L64-d64", T=1000, Hq=16, Hk=2, d=64, L=64, seed=13),
    Workload("T100-G1-L200-d64", T=100, Hq=2, Hk=2, d=64, L=200, seed=14),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_edge_shapes_full(w):
    gc.check_workload(w)


def test_peaked_softmax():
    """q x 4: far from uniform, so masking and max tracking matter."""
    gc.check_workload(Workload("peaked", T=700, Hq=8, Hk=2, d=128, L=12, seed=9), q_mul=4.0)


def _key_ramp(x):
    # key magnitudes grow 0.5x -> 4x along the sequence and q is doubled, so
    # every row's running max keeps rising: blocks far above the reference
    # force a rescale of O and l after the first block, and blocks a few log2
    # units above it push the block sum past its bound without one
    T = x["k"].shape[0]
    ramp = torch.linspace(0.5, 4.0, T).view(T, 1, 1)
    x["k"] = (x["k"].float() * ramp).to(torch.bfloat16)
    x["q"] = (x["q"].float() * 2.0).to(torch.bfloat16)
    return x


@pytest.mark.parametrize("w", [Workload("ramp-d128", T=1000, Hq=8, Hk=2, d=128, L=12, seed=21),
                               Workload("ramp-d64", T=700, Hq=8, Hk=2, d=64, L=16, seed=22)],
                         ids=lambda w: w.name)
def test_rising_scores_rescale(w):
    gc.check_workload(w, prep=_key_ramp)


def test_depth_slot_permutation_invariance():
    w = Workload("perm", T=300, Hq=8, Hk=2, d=128, L=10, seed=2)
    x = make_inputs(w)
    o1, l1 = gc.run_cuda(x, w.scale)
    perm = torch.randperm(w.L, generator=torch.Generator().manual_seed(0))
    x2 = dict(x, kd=x["kd"][perm].contiguous(), vd=x["vd"][perm].contiguous())
    o2, l2 = gc.run_cuda(x2, w.scale)
    assert np.max(np.abs(o1 - o2)) <= 1e-2
    assert np.max(np.abs(l1 - l2)) <= 1e-4


def test_zero_depth_with_negative_scores():
    """kd = vd = 0 and sequence logits pushed far negative: depth slots carry
    most of the mass with a zero value, o shrinks toward 0."""
    w = Workload("zero-depth", T=257, Hq=4, Hk=1, d=64, L=8, seed=6)
    x = make_inputs(w)
    x["kd"].zero_()
    x["vd"].zero_()
    x["k"] = (x["k"].float().abs() * 2).to(torch.bfloat16)
    x["q"] = (-x["q"].float().abs() * 2).to(torch.bfloat16)
    o, lse = gc.run_cuda(x, w.scale)
    eo, el = gc.compare(x, w.scale, o, lse)
    assert eo <= gc.TOL_O and el <= gc.TOL_LSE


def test_deterministic_repeat():
    w = Workload("repeat", T=1000, Hq=16, Hk=4, d=128, L=24, seed=8)
    x = make_inputs(w)
    o1, l1 = gc.run_cuda(x, w.scale)
    o2, l2 = gc.run_cuda(x, w.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_l0_equals_sdpa_on_gpu():
    """Plain causal GQA (L = 0) against torch SDPA in fp32 on the same device."""
    w = Workload("sdpa", T=2048, Hq=16, Hk=4, d=128, L=0, seed=10)
    x = {n: t.cuda() for n, t in make_inputs(w).items()}
    o, _ = moda.moda_fwd(x["q"], x["k"], x["v"], None, None, w.scale)
    q = x["q"].float().permute(1, 0, 2)
    k = x["k"].float().repeat_interleave(w.G, 1).permute(1, 0, 2)
    v = x["v"].float().repeat_interleave(w.G, 1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=w.scale)
    assert (o.float() - ref.permute(1, 0, 2)).abs().max().item() <= gc.TOL_O


def test_lse_optional_and_status_clean():
    w = Workload("nolse", T=100, Hq=4, Hk=2, d=64, L=2)
    x = {n: t.cuda() for n, t in make_inputs(w).items()}
    kd = moda.moda_pack_depth(x["kd"])
    vd = moda.moda_pack_depth(x["vd"])
    o, lse = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale, want_lse=False)
    assert lse is None
    assert moda.moda_get_device_error() == 0
    o2, _ = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale)
    assert torch.equal(o, o2)


@pytest.mark.parametrize("d", [64, 128])
def test_output_16_byte_aligned_only(d):
    """o at an address that is 16- but not 32-byte aligned (the ABI asks for
    16): the same values as at a 32-byte aligned o (d = 64 then writes its rows
    in 16-byte stores; d = 128 writes through TMA stores, whose tensor map needs
    only 16-byte alignment)."""
    w = Workload(f"o-align-d{d}", T=300, Hq=8, Hk=2, d=d, L=6, seed=31)
    x = {n: t.cuda() for n, t in make_inputs(w).items()}
    kd = moda.moda_pack_depth(x["kd"])
    vd = moda.moda_pack_depth(x["vd"])
    o_ref, l_ref = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale)
    n = w.T * w.Hq * w.d
    buf = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
    base = buf.data_ptr()
    off = next(e for e in range(0, 16) if (base + 2 * e) % 32 == 16)
    o = buf[off:off + n].view(w.T, w.Hq, w.d)
    assert o.data_ptr() % 32 == 16
    moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale, o=o)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
