"""The d = 64 path at the shape of the pages' kernel-efficiency table
(Mixture-of-Depths Attention, Table 2: B = 1, d = 64, G = 8, Hq = 64, Hk = 8,
L = 64, T from 4K to 64K), checked against the fp64 oracle at the sizes it is
benchmarked at.

d = 64 runs the two-tiles-per-CTA forward, whose paired K/V stages are
released by one arrival per tile; at T = 16384 a KV head has 1024 tiles and
every pair walks long runs of depth blocks, which the small edge shapes do not
reach. Inputs are drawn on the device (Philox, seed 0) and copied to the host
for the oracle, which recomputes a stratified row sample: every head at the
tile edges and the ends of the sequence, plus 64 seeded random positions."""
import numpy as np
import pytest
import torch

import oracle
import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import inputs as wl
from sequence_depth_attention_gb300.inputs import bf16_bits, make_inputs, sample_rows

import gpu_common as gc

pytestmark = pytest.mark.gpu

T16K = next(w for w in wl.TABLE2 if w.T == 16384)
T64K = next(w for w in wl.TABLE2 if w.T == 65536)
REL = 1e-2  # backward: max error <= 1 % of each gradient's largest magnitude


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


@pytest.mark.parametrize("w", [T16K, T64K], ids=lambda w: w.name)
def test_table2_forward_sampled(w):
    gc.check_workload(w, sampled=True, device_inputs=True)


def _check(name, got, ref):
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    err = float(np.max(np.abs(got - ref)))
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    assert err <= REL * scale, f"{name}: max err {err:.3e} > {REL} * {scale:.3e}"


def test_table2_backward_sampled():
    """Backward at T = 16384: dq and the depth gradients of the sampled
    positions, dk and dv of the last 16 keys (every row that sees them is in
    the sample), against the oracle's row-subset backward."""
    w = T16K
    x = make_inputs(w, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(77)
    dO = torch.randn((w.T, w.Hq, w.d), generator=g, device="cuda").to(torch.bfloat16)
    kd = moda.moda_pack_depth(x["kd"])
    vd = moda.moda_pack_depth(x["vd"])
    o, lse = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale)
    dq, dk, dv, dkd, dvd = moda.moda_bwd(x["q"], x["k"], x["v"], kd, vd, o, lse, dO, w.scale)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    W = 16
    ts, _ = sample_rows(w.T, w.Hq, w.G, n_random=24)
    ts = sorted(set(ts.tolist()) | set(range(w.T - W, w.T)))
    tsel = torch.tensor(ts, device="cuda")
    got_dq = dq[tsel].reshape(-1, w.d).cpu().numpy()
    got_dk = dk[w.T - W:].cpu().numpy()
    got_dv = dv[w.T - W:].cpu().numpy()
    got_dkd = dkd[:, tsel].cpu().numpy()  # [Hk, n, L, d]
    got_dvd = dvd[:, tsel].cpu().numpy()
    del dq, dk, dv, dkd, dvd, kd, vd
    b = {n: bf16_bits(t) for n, t in x.items()}
    del x
    rows = np.array([t * w.Hq + h for t in ts for h in range(w.Hq)])
    r_dq, r_dk, r_dv, r_dkd, r_dvd = oracle.default().backward_rows(
        b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), w.scale, rows, w.T - W,
        nthreads=gc.NTHREADS)
    _check("dq", got_dq, r_dq)
    _check("dk_tail", got_dk, r_dk)
    _check("dv_tail", got_dv, r_dv)
    G = w.G
    for i, t in enumerate(ts):
        for hk in range(w.Hk):
            sel = slice(i * w.Hq + hk * G, i * w.Hq + (hk + 1) * G)
            _check(f"dkd[t={t},hk={hk}]", got_dkd[hk, i], r_dkd[sel].sum(0))
            _check(f"dvd[t={t},hk={hk}]", got_dvd[hk, i], r_dvd[sel].sum(0))
