"""CUDA backward vs the fp64 oracle backward, through the C-ABI.

Tolerance: every gradient g must satisfy max|g_gpu - g_oracle| <= 1e-2 *
max|g_oracle| (1 % of the gradient's scale). The kernels take bf16 operands
with fp32 accumulation and round P and dS to bf16 (relative 2^-9 per term)
before the tensor-core products; over sums of hundreds of terms of mixed sign
this leaves errors near 1e-3 of the scale, so 1e-2 holds with margin while
still catching any wrong term, index or sign (those give O(1) errors)."""
import numpy as np
import pytest
import torch

import oracle
import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import inputs as wl
from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs, sample_rows

import gpu_common as gc

pytestmark = pytest.mark.gpu
REL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


def run_gpu(x, dO, scale):
    dev = "cuda"
    q, k, v, dOg = (t.to(dev) for t in (x["q"], x["k"], x["v"], dO))
    L = x["kd"].shape[0]
    kd = moda.moda_pack_depth(x["kd"].to(dev)) if L else None
    vd = moda.moda_pack_depth(x["vd"].to(dev)) if L else None
    o, lse = moda.moda_fwd(q, k, v, kd, vd, scale)
    grads = moda.moda_bwd(q, k, v, kd, vd, o, lse, dOg, scale)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    out = [g.cpu().numpy() if g is not None else None for g in grads]
    if L:  # packed [Hk,T,L,d] -> append layout [L,T,Hk,d]
        out[3] = np.ascontiguousarray(out[3].transpose(2, 1, 0, 3))
        out[4] = np.ascontiguousarray(out[4].transpose(2, 1, 0, 3))
    return out


def upstream(w, seed=77):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((w.T, w.Hq, w.d), generator=g).to(torch.bfloat16)


def check(name, got, ref):
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    err = float(np.max(np.abs(got - ref)))
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    assert err <= REL * scale, f"{name}: max err {err:.3e} > {REL} * {scale:.3e}"


def check_full(w):
    x = make_inputs(w)
    dO = upstream(w)
    got = run_gpu(x, dO, w.scale)
    b = {n: bf16_bits(t) for n, t in x.items()}
    L = w.L
    ref = oracle.backward(b["q"], b["k"], b["v"], b["kd"] if L else None, b["vd"] if L else None,
                          bf16_bits(dO), w.scale, nthreads=gc.NTHREADS)
    for name, g, r in zip(("dq", "dk", "dv", "dkd", "dvd"), got, ref):
        if r.size:
            check(f"{w.name}.{name}", g, r)


EDGE = [
    Workload("bwd-tiny", T=128, Hq=4, Hk=2, d=64, L=4),
    Workload("bwd-T1", T=1, Hq=4, Hk=2, d=128, L=3),
    Workload("bwd-T3-G16", T=3, Hq=16, Hk=1, d=64, L=2),
    Workload("bwd-T65-L0", T=65, Hq=8, Hk=2, d=128, L=0),
    Workload("bwd-T127-G8", T=127, Hq=16, Hk=2, d=128, L=7),
    Workload("bwd-T200-G1", T=200, Hq=3, Hk=3, d=64, L=33),
    Workload("bwd-T300-G4", T=300, Hq=8, Hk=2, d=128, L=24, seed=5),
    # many 64-row sub-tiles per key block (both S^T/dP^T buffers reused over many
    # barrier phases) with a ragged tail, at each head dimension
    Workload("bwd-T1000-G2-d64", T=1000, Hq=4, Hk=2, d=64, L=8, seed=9),
    Workload("bwd-T700-G2-d128", T=700, Hq=4, Hk=2, d=128, L=5, seed=11),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_backward_full(w):
    check_full(w)


def test_backward_700m_layer_full():
    check_full(wl.LAYER_700M)


@pytest.mark.parametrize("w", [wl.GQA_SWEEP[3], wl.DEPTH_SWEEP[3]], ids=lambda w: w.name)
def test_backward_large_sampled(w):
    """Sampled rows (dq, depth gradients of their positions) and the tail keys
    (dk, dv), from the oracle's row-subset backward."""
    x = make_inputs(w, device="cuda")
    dO = upstream(w)
    got = run_gpu(x, dO, w.scale)
    x = {n: t.cpu() for n, t in x.items()}
    b = {n: bf16_bits(t) for n, t in x.items()}
    W = 16
    ts, _ = sample_rows(w.T, w.Hq, w.G, n_random=24)
    ts = sorted(set(ts.tolist()) | set(range(w.T - W, w.T)))
    rows = np.array([t * w.Hq + h for t in ts for h in range(w.Hq)])
    dq, dk, dv, dkd, dvd = oracle.default().backward_rows(
        b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), w.scale, rows, w.T - W,
        nthreads=gc.NTHREADS)
    check(f"{w.name}.dq", got[0].reshape(-1, w.d)[rows], dq)
    check(f"{w.name}.dk_tail", got[1][w.T - W:], dk)
    check(f"{w.name}.dv_tail", got[2][w.T - W:], dv)
    if w.L:
        G = w.G
        for i, t in enumerate(ts):
            for hk in range(w.Hk):
                sel = slice(i * w.Hq + hk * G, i * w.Hq + (hk + 1) * G)
                check(f"{w.name}.dkd[t={t},hk={hk}]", got[3][:, t, hk], dkd[sel].sum(0))
                check(f"{w.name}.dvd[t={t},hk={hk}]", got[4][:, t, hk], dvd[sel].sum(0))


@pytest.mark.parametrize("layer_major", [False, True], ids=["packed", "layer-major"])
def test_backward_long_sequence_tail(layer_major):
    """T >= 32768 at d = 128, where the dK/dV kernel's two elementwise
    warpgroups take alternate sub-tiles: dk and dv of the last 1024 keys (key
    blocks walking up to 32 sub-tiles, the ragged last one included), dq and
    the depth gradients of sampled rows, against the oracle's row-subset
    backward over every row that sees those keys."""
    w = Workload("bwd-T32773-G2", T=32768 + 5, Hq=2, Hk=1, d=128, L=3, seed=15)
    x = make_inputs(w, device="cuda")
    dO = upstream(w)
    q, k, v, dOg = x["q"], x["k"], x["v"], dO.cuda()
    if layer_major:
        kd, vd = x["kd"], x["vd"]
        o, lse = moda.moda_fwd_layer_major(q, k, v, kd, vd, w.scale)
    else:
        kd, vd = moda.moda_pack_depth(x["kd"]), moda.moda_pack_depth(x["vd"])
        o, lse = moda.moda_fwd(q, k, v, kd, vd, w.scale)
    dq, dk, dv, dkd, dvd = moda.moda_bwd(q, k, v, kd, vd, o, lse, dOg, w.scale,
                                         layer_major=layer_major)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    if not layer_major:  # packed [Hk,T,L,d] -> append layout [L,T,Hk,d]
        dkd, dvd = dkd.permute(2, 1, 0, 3), dvd.permute(2, 1, 0, 3)
    W = 1024
    ts, _ = sample_rows(w.T, w.Hq, w.G, n_random=24)
    ts = sorted(set(ts.tolist()) | set(range(w.T - W, w.T)))
    rows = np.array([t * w.Hq + h for t in ts for h in range(w.Hq)])
    tsel = torch.tensor(ts, device="cuda")
    got_dq = dq.reshape(-1, w.d)[torch.from_numpy(rows).cuda()].cpu().numpy()
    got_dk, got_dv = dk[w.T - W:].cpu().numpy(), dv[w.T - W:].cpu().numpy()
    got_dkd, got_dvd = dkd[:, tsel].cpu().numpy(), dvd[:, tsel].cpu().numpy()  # [L, n, Hk, d]
    b = {n: bf16_bits(t) for n, t in x.items()}
    del x, dq, dk, dv, dkd, dvd
    r_dq, r_dk, r_dv, r_dkd, r_dvd = oracle.default().backward_rows(
        b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), w.scale, rows, w.T - W,
        nthreads=gc.NTHREADS)
    check("dq", got_dq, r_dq)
    check("dk_tail", got_dk, r_dk)
    check("dv_tail", got_dv, r_dv)
    G = w.G
    for i in range(len(ts)):
        for hk in range(w.Hk):
            sel = slice(i * w.Hq + hk * G, i * w.Hq + (hk + 1) * G)
            check(f"dkd[t={ts[i]},hk={hk}]", got_dkd[:, i, hk], r_dkd[sel].sum(0))
            check(f"dvd[t={ts[i]},hk={hk}]", got_dvd[:, i, hk], r_dvd[sel].sum(0))


def test_backward_deterministic():
    w = Workload("bwd-det", T=500, Hq=8, Hk=2, d=128, L=12, seed=3)
    x = make_inputs(w)
    dO = upstream(w)
    a = run_gpu(x, dO, w.scale)
    b = run_gpu(x, dO, w.scale)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
