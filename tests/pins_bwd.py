"""Pins for the oracle's backward (gradients of the MoDA forward).

Each ``pin_*`` takes an ``oracle.Oracle`` and returns ``{name: (error, tol)}``.
P9 and P10 compare with torch autograd (a library's reverse mode) through
formulations that share nothing with the oracle's loops; P11 checks exact
identities of the softmax gradient."""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs

import pins


def case(T, Hq, Hk, d, L, seed):
    w = Workload("pin", T, Hq, Hk, d, L, 1.0, seed)
    x = make_inputs(w)
    g = torch.Generator().manual_seed(seed + 1000)
    dO = torch.randn((T, Hq, d), generator=g).to(torch.bfloat16)
    return x, dO


def _err(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.asarray(a).size else 0.0


def autograd_dense(x, dO, scale):
    """Gradients of the pages' dense masked formulation (Sec. 3.2/3.3 masks,
    expanded rows i_q = tG+g) by torch autograd in fp64."""
    leaves = {n: x[n].to(torch.float64).requires_grad_(True) for n in ("q", "k", "v", "kd", "vd")}
    q, k, v, kd, vd = (leaves[n] for n in ("q", "k", "v", "kd", "vd"))
    T, Hq, d = q.shape
    Hk = k.shape[1]
    L = kd.shape[0]
    G = Hq // Hk
    keep = pins.masks_pages(T, G, L)
    outs = []
    for hk in range(Hk):
        qe = q[:, hk * G:(hk + 1) * G, :].reshape(T * G, d)
        keys = torch.cat([k[:, hk, :], kd[:, :, hk, :].permute(1, 0, 2).reshape(T * L, d)], 0)
        vals = torch.cat([v[:, hk, :], vd[:, :, hk, :].permute(1, 0, 2).reshape(T * L, d)], 0)
        out = F.scaled_dot_product_attention(qe[None], keys[None], vals[None], attn_mask=keep[None],
                                             scale=scale)[0]
        outs.append(out.reshape(T, G, d))
    o = torch.cat(outs, dim=1)
    (o * dO.to(torch.float64)).sum().backward()
    return tuple(leaves[n].grad.numpy() for n in ("q", "k", "v", "kd", "vd"))


def pin_bwd_autograd_dense(orc, T=13, Hq=8, Hk=2, d=8, L=5, scale=0.37, seed=31):
    x, dO = case(T, Hq, Hk, d, L, seed)
    b = {n: bf16_bits(t) for n, t in x.items()}
    got = orc.backward(b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), scale)
    ref = autograd_dense(x, dO, scale)
    return {f"P9.{n}": (_err(g, r), 1e-12) for n, g, r in zip(("dq", "dk", "dv", "dkd", "dvd"), got, ref)}


def pin_bwd_l0_sdpa(orc, T=29, Hq=6, Hk=3, d=16, scale=0.21, seed=37):
    x, dO = case(T, Hq, Hk, d, 0, seed)
    b = {n: bf16_bits(t) for n, t in x.items()}
    dq, dk, dv, _, _ = orc.backward(b["q"], b["k"], b["v"], None, None, bf16_bits(dO), scale)
    G = Hq // Hk
    q = x["q"].to(torch.float64).requires_grad_(True)
    k = x["k"].to(torch.float64).requires_grad_(True)
    v = x["v"].to(torch.float64).requires_grad_(True)
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2), k.repeat_interleave(G, 1).permute(1, 0, 2),
                                       v.repeat_interleave(G, 1).permute(1, 0, 2), is_causal=True,
                                       scale=scale).permute(1, 0, 2)
    (o * dO.to(torch.float64)).sum().backward()
    return {"P10.dq": (_err(dq, q.grad.numpy()), 1e-12), "P10.dk": (_err(dk, k.grad.numpy()), 1e-12),
            "P10.dv": (_err(dv, v.grad.numpy()), 1e-12)}


def pin_bwd_identities(orc, T=23, Hq=8, Hk=2, d=16, L=6, scale=0.3, seed=41):
    """Per KV head: sum of all value gradients = sum of dO over the head's rows
    (each probability row sums to 1); sum of all key gradients = 0 (softmax is
    invariant to adding one vector to every key of a row)."""
    x, dO = case(T, Hq, Hk, d, L, seed)
    b = {n: bf16_bits(t) for n, t in x.items()}
    dq, dk, dv, dkd, dvd = orc.backward(b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), scale)
    G = Hq // Hk
    g = dO.to(torch.float64).numpy()
    ev, ek = 0.0, 0.0
    for hk in range(Hk):
        want = g[:, hk * G:(hk + 1) * G, :].sum(axis=(0, 1))
        got = dv[:, hk, :].sum(axis=0) + dvd[:, :, hk, :].sum(axis=(0, 1))
        ev = max(ev, _err(got, want))
        ek = max(ek, float(np.abs(dk[:, hk, :].sum(axis=0) + dkd[:, :, hk, :].sum(axis=(0, 1))).max()))
    return {"P11.sum_dv": (ev, 1e-11), "P11.sum_dk": (ek, 1e-11)}


ALL_BWD_PINS = [pin_bwd_autograd_dense, pin_bwd_l0_sdpa, pin_bwd_identities]


def run_all(orc):
    out = {}
    for pin in ALL_BWD_PINS:
        out.update(pin(orc))
    return out
