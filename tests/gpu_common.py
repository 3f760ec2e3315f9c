"""Shared helpers for the GPU parity tests: run the CUDA path through the
C-ABI binding and compare with the fp64 oracle on the same seeded inputs."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import build as mbuild
from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs, sample_rows

# Tolerances of the forward: max-abs 2e-2 on o (bf16 output, bf16 P in the
# P.V product) and 1e-3 on lse (fp32 accumulation).
TOL_O = 2e-2
TOL_LSE = 1e-3

NTHREADS = max(1, (os.cpu_count() or 2))


def ensure_built():
    mbuild.build()
    moda.load()


def run_cuda(x, scale, device="cuda", depth_on_cuda_cores=False, layer_major=False):
    """x: dict of bf16 tensors (kd/vd in [L,T,Hk,d]). Returns o, lse on CPU.
    layer_major=True hands kd/vd to moda_fwd_layer_major as they are, else
    they are packed first and go to moda_fwd."""
    q, k, v = (x[n].to(device) for n in ("q", "k", "v"))
    L = x["kd"].shape[0]
    if layer_major:
        kd = x["kd"].to(device).contiguous() if L else None
        vd = x["vd"].to(device).contiguous() if L else None
        o, lse = moda.moda_fwd_layer_major(q, k, v, kd, vd, scale)
        torch.cuda.synchronize()
        assert moda.moda_get_device_error() == 0
        return o.float().cpu().numpy(), lse.cpu().numpy()
    if L:
        kd = moda.moda_pack_depth(x["kd"].to(device))
        vd = moda.moda_pack_depth(x["vd"].to(device))
    else:
        kd = vd = None
    o, lse = moda.moda_fwd(q, k, v, kd, vd, scale, depth_on_cuda_cores=depth_on_cuda_cores)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def oracle_rows(x, scale, ts, hs):
    b = {n: bf16_bits(t) for n, t in x.items()}
    L = x["kd"].shape[0]
    return oracle.rows(b["q"], b["k"], b["v"], b["kd"] if L else None, b["vd"] if L else None,
                       scale, ts, hs, nthreads=NTHREADS)


def compare(x, scale, o, lse, ts=None, hs=None):
    """Max-abs errors of (o, lse) against the oracle on rows (ts, hs) (all rows if None)."""
    T, Hq, _ = x["q"].shape
    if ts is None:
        tt, hh = np.meshgrid(np.arange(T), np.arange(Hq), indexing="ij")
        ts, hs = tt.ravel(), hh.ravel()
    ro, rl = oracle_rows(x, scale, ts, hs)
    eo = float(np.max(np.abs(o[ts, hs] - ro)))
    el = float(np.max(np.abs(lse[ts, hs] - rl)))
    return eo, el


def check_workload(w: Workload, sampled=False, device_inputs=False, q_mul=1.0,
                   depth_on_cuda_cores=False, prep=None, layer_major=False):
    x = make_inputs(w, device="cuda" if device_inputs else "cpu")
    if q_mul != 1.0:
        x["q"] = (x["q"].float() * q_mul).to(torch.bfloat16)
    if prep is not None:  # reshape the inputs' statistics (same tensors go to the oracle)
        x = prep(x)
    o, lse = run_cuda(x, w.scale, depth_on_cuda_cores=depth_on_cuda_cores, layer_major=layer_major)
    if device_inputs:
        x = {n: t.cpu() for n, t in x.items()}
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    ts = hs = None
    if sampled:
        ts, hs = sample_rows(w.T, w.Hq, w.G)
    eo, el = compare(x, w.scale, o, lse, ts, hs)
    assert eo <= TOL_O, f"{w.name}: max|o - oracle| = {eo:.3e} > {TOL_O}"
    assert el <= TOL_LSE, f"{w.name}: max|lse - oracle| = {el:.3e} > {TOL_LSE}"
    return eo, el
