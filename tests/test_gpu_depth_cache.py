"""Bounded depth KV cache on the GPU (summary, Sec. 6.2) through the C-ABI:
the depth mass against the fp64 oracle, the slot choice against the oracle's
policy on the same fp32 utilities (floating point decides an integer there,
so both sides take the decision from the kernel's values), the device-indexed
slot write, and a layer loop that runs all of it on the stream, checked
against the oracle on the entries the policy kept."""
import numpy as np
import pytest
import torch

import oracle
from oracle import depth_cache
import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import inputs as wl
from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu

# Mass tolerance: each term exp(z - lse) carries the fp32 error of the logit
# and of lse (~1e-6 relative) and of the exponential (2 ulp); the fp32 sums
# over T*G rows add ~n*2^-24 relative. 1e-4 of the largest slot mass bounds
# both with margin and still fails on a wrong row, head or slot (O(1) errors).
MASS_REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


def _mass_both(w, x, scale=None):
    scale = w.scale if scale is None else scale
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    kd = moda.moda_pack_depth(x["kd"].cuda())
    vd = moda.moda_pack_depth(x["vd"].cuda())
    o, lse = moda.moda_fwd(q, k, v, kd, vd, scale)
    mass = moda.moda_depth_mass(q, kd, lse, scale)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    b = {n: bf16_bits(t.cpu()) for n, t in x.items()}
    ref = oracle.depth_mass(b["q"], b["k"], b["v"], b["kd"], b["vd"], scale, nthreads=gc.NTHREADS)
    return mass.cpu().numpy(), ref


MASS_SHAPES = [
    Workload("mass-tiny", T=128, Hq=4, Hk=2, d=64, L=4),
    Workload("mass-G1-L33", T=300, Hq=3, Hk=3, d=128, L=33, seed=3),
    Workload("mass-G16-T1", T=1, Hq=16, Hk=1, d=128, L=7, seed=4),
    Workload("mass-G8-ragged", T=1000, Hq=16, Hk=2, d=64, L=70, seed=5),
    Workload("mass-G2-L1", T=65, Hq=4, Hk=2, d=128, L=1, seed=6),
]


@pytest.mark.parametrize("w", MASS_SHAPES, ids=lambda w: w.name)
def test_depth_mass_matches_oracle(w):
    got, ref = _mass_both(w, make_inputs(w))
    assert np.isfinite(got).all()
    assert np.max(np.abs(got - ref)) <= MASS_REL * np.max(np.abs(ref))


def test_depth_mass_700m_layer():
    w = wl.LAYER_700M
    got, ref = _mass_both(w, make_inputs(w))
    assert np.max(np.abs(got - ref)) <= MASS_REL * np.max(np.abs(ref))


def test_depth_mass_equal_logits():
    """q = 0: every candidate of row t has p = 1/(t+1+L)."""
    w = Workload("mass-q0", T=500, Hq=8, Hk=2, d=128, L=6, seed=7)
    x = make_inputs(w)
    x["q"].zero_()
    got, _ = _mass_both(w, x)
    want = w.G * sum(1.0 / (t + 1 + w.L) for t in range(w.T))
    assert np.max(np.abs(got - want)) <= MASS_REL * want


def _utility_f32(mass):
    """The admit kernel's utility: fp32 sum over KV heads in head order."""
    u = np.zeros(mass.shape[1], np.float32)
    for h in range(mass.shape[0]):
        u = (u + mass[h].astype(np.float32)).astype(np.float32)
    return u


def test_admit_matches_oracle_policy():
    rng = np.random.default_rng(11)
    slot = torch.empty((1,), dtype=torch.int32, device="cuda")
    for S in (1, 3, 7, 32, 33, 200, 1024):
        for trial in range(6):
            ages = rng.permutation(5000)[:S].astype(np.int32)
            if trial == 0:
                ages[rng.choice(S, size=max(1, S // 3), replace=False)] = -1
            Hk = int(rng.integers(1, 5))
            mass = rng.choice(np.array([0.25, 0.5, 1.0, 3.0], np.float32), size=(Hk, S))
            if trial == 1:  # distinct utilities
                mass = rng.random((Hk, S), dtype=np.float32)
            for R in (0, 1, 2, S // 2, S, S + 3):
                ga = torch.tensor(ages, device="cuda")
                moda.moda_depth_cache_admit(ga, torch.tensor(mass, device="cuda"), R, 9000, slot=slot)
                torch.cuda.synchronize()
                got = int(slot.item())
                want = depth_cache.victim(ages.tolist(), _utility_f32(mass).tolist(), R)
                assert got == want, (S, trial, R)
                after = ages.copy()
                after[want] = 9000
                assert np.array_equal(ga.cpu().numpy(), after)


def test_write_at_device_slot():
    T, Hk, d, L = 257, 3, 128, 6
    g = torch.Generator(device="cuda").manual_seed(2)
    src = torch.randn((T, Hk, d), generator=g, device="cuda").to(torch.bfloat16)
    dst = torch.randn((Hk, T, L, d), generator=g, device="cuda").to(torch.bfloat16)
    want = dst.clone()
    want[:, :, 4, :] = src.permute(1, 0, 2)
    slot = torch.tensor([4], dtype=torch.int32, device="cuda")
    moda.moda_depth_write_at(src, dst, slot)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    assert torch.equal(dst.view(torch.int16), want.view(torch.int16))
    # an out-of-range slot writes nothing and is reported by the device error word
    before = dst.clone()
    moda.moda_depth_write_at(src, dst, torch.tensor([L], dtype=torch.int32, device="cuda"))
    assert moda.moda_get_device_error() == 1  # MODA_ERR_INVALID_ARG
    assert torch.equal(dst.view(torch.int16), before.view(torch.int16))
    assert moda.moda_get_device_error() == 0  # read and cleared


@pytest.mark.parametrize("recent", [0, 2, 4], ids=["top-S", "hybrid", "window"])
def test_layer_loop_on_stream(recent):
    """Eleven layers write depth entries into a 4-slot cache; each layer's
    forward reads the cache, its depth mass scores the slots, the policy picks
    the slot and the layer's K/V go there, all enqueued on the stream. The
    slot choices must follow the oracle's policy on the kernel's utilities,
    the cache must hold exactly the chosen layers' K/V, and every forward must
    match the oracle on the layers the cache held when it ran."""
    S, n_layers = 4, 11
    w = Workload("cache-loop", T=300, Hq=8, Hk=2, d=128, L=n_layers, seed=19)
    x = make_inputs(w)  # kd/vd [n_layers, T, Hk, d]: layer i's depth K/V
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    layers_k = [x["kd"][i].cuda().contiguous() for i in range(n_layers)]
    layers_v = [x["vd"][i].cuda().contiguous() for i in range(n_layers)]
    cache_k = torch.zeros((w.Hk, w.T, S, w.d), dtype=torch.bfloat16, device="cuda")
    cache_v = torch.zeros_like(cache_k)
    ages = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    mass = torch.zeros((w.Hk, S), dtype=torch.float32, device="cuda")
    ws = torch.empty(((moda.moda_depth_mass_workspace_bytes(w.T, w.Hk, S) + 3) // 4,),
                     dtype=torch.float32, device="cuda")
    slot = torch.empty((1,), dtype=torch.int32, device="cuda")
    held = [-1] * S  # host mirror, replayed with the oracle's policy
    outs, masses = [], []
    for i in range(n_layers):
        filled = sum(a >= 0 for a in held)
        if filled:
            o, lse = moda.moda_fwd(q, k, v, cache_k[:, :, :filled].contiguous(),
                                   cache_v[:, :, :filled].contiguous(), w.scale)
            outs.append((i, list(held[:filled]), o.clone(), lse.clone()))
        if filled == S:
            moda.moda_depth_mass(q, cache_k, lse, w.scale, mass=mass, workspace=ws)
        moda.moda_depth_cache_admit(ages, mass, recent, i, slot=slot)
        moda.moda_depth_write_at(layers_k[i], cache_k, slot)
        moda.moda_depth_write_at(layers_v[i], cache_v, slot)
        torch.cuda.synchronize()
        m = mass.cpu().numpy()
        masses.append(m.copy())
        want = depth_cache.victim(held, _utility_f32(m).tolist(), recent)
        assert int(slot.item()) == want, (i, held)
        held[want] = i
        assert ages.cpu().tolist() == held
    assert moda.moda_get_device_error() == 0
    # the cache holds exactly the chosen layers' K/V, bit for bit
    for s, layer in enumerate(held):
        assert torch.equal(cache_k[:, :, s].view(torch.int16),
                           layers_k[layer].permute(1, 0, 2).view(torch.int16))
        assert torch.equal(cache_v[:, :, s].view(torch.int16),
                           layers_v[layer].permute(1, 0, 2).view(torch.int16))
    # each forward against the oracle on the layers it read (slot order)
    for i, layers, o, lse in outs[-3:]:
        sub = dict(x, kd=x["kd"][layers].contiguous(), vd=x["vd"][layers].contiguous())
        eo, el = gc.compare(sub, w.scale, o.float().cpu().numpy(), lse.cpu().numpy())
        assert eo <= gc.TOL_O and el <= gc.TOL_LSE, (i, layers)
    if recent >= S:
        assert sorted(held) == list(range(n_layers - S, n_layers))
