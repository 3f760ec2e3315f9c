"""Pins for the oracle's depth mass (the utility of the bounded depth cache,
summary Sec. 6.2) against what the pages and the mathematics fix, none of
which re-runs the oracle's own loops:

  C1  the pages' dense formulation (expanded rows i_q = tG + g, keys
      [K | flat depth axis j_d = tL + l], the grouped causal and block-diagonal
      masks of Sec. 3.2-3.3) softmaxed by torch; slot l's mass is the sum of
      the probability in the depth columns with j_d mod L = l;
  C2  equal logits (q = 0): every candidate of row t has p = 1/(t+1+L), so
      each slot's mass over KV head hk is G * sum_t 1/(t+1+L), written with
      exact fractions (the reading notes' teaching example, Sec. 二.2, is the
      t = 2, L = 4 term: 4/7 of the mass on the depth slots);
  C3  brute force on the integer case of the forward pins, 50-digit mpmath;
  C4  permuting the depth slots permutes the mass (slots form a set, Sec. 2.2);
  C5  additivity over rows: the mass of a row set is the sum over a partition.

Each ``pin_*`` returns ``{name: (error, tol)}`` so a build of the oracle with
a planted mistake must make at least one of them fail.
"""
from __future__ import annotations

from fractions import Fraction

import mpmath
import numpy as np
import torch

import pins
from sequence_depth_attention_gb300.inputs import bf16_bits


def dense_mass(x, scale):
    q, k, kd = (x[n].to(torch.float64) for n in ("q", "k", "kd"))
    T, Hq, d = q.shape
    Hk = k.shape[1]
    L = kd.shape[0]
    G = Hq // Hk
    keep = pins.masks_pages(T, G, L)
    mass = np.zeros((Hk, L))
    for hk in range(Hk):
        qe = q[:, hk * G:(hk + 1) * G, :].reshape(T * G, d)
        kflat = kd[:, :, hk, :].permute(1, 0, 2).reshape(T * L, d)
        keys = torch.cat([k[:, hk, :], kflat], 0)
        s = (scale * qe @ keys.T).masked_fill(~keep, float("-inf"))
        p = torch.softmax(s, dim=-1)[:, T:]  # depth columns j_d = t*L + l
        mass[hk] = p.reshape(T * G, T, L).sum(dim=(0, 1)).numpy()
    return mass


def pin_mass_dense(orc, T=19, Hq=8, Hk=2, d=8, L=5, scale=0.45, seed=31):
    _, x, b = pins.case(T, Hq, Hk, d, L, seed)
    got = orc.depth_mass(b["q"], b["k"], b["v"], b["kd"], b["vd"], scale)
    return {"C1.mass": (pins._err(got, dense_mass(x, scale)), 1e-12)}


def pin_mass_equal_logits(orc, T=11, Hq=6, Hk=3, d=8, L=4, seed=33):
    _, x, b = pins.case(T, Hq, Hk, d, L, seed)
    b["q"] = np.zeros_like(b["q"])  # bf16 zero bits: every logit is 0
    got = orc.depth_mass(b["q"], b["k"], b["v"], b["kd"], b["vd"], 0.7)
    G = Hq // Hk
    want = float(G * sum(Fraction(1, t + 1 + L) for t in range(T)))
    return {"C2.mass": (float(np.max(np.abs(got - want))), 1e-13)}


def pin_mass_brute_force(orc):
    B = pins.BRUTE
    q, k, kd = B["q"], B["k"], B["kd"]
    T, Hq, d, L, G = 3, 2, 2, 2, 2
    mpmath.mp.dps = 50
    want = [mpmath.mpf(0)] * L
    for t in range(T):
        for h in range(Hq):
            hk = h // G
            z = [sum(q[t][h][c] * k[j][hk][c] for c in range(d)) for j in range(t + 1)]
            zd = [sum(q[t][h][c] * kd[l][t][hk][c] for c in range(d)) for l in range(L)]
            Z = mpmath.fsum(mpmath.e ** v for v in z + zd)
            for l in range(L):
                want[l] += mpmath.e ** zd[l] / Z

    def bits(a):
        return bf16_bits(torch.tensor(a, dtype=torch.float32).to(torch.bfloat16))
    b = {n: bits(a) for n, a in B.items()}
    got = orc.depth_mass(b["q"], b["k"], b["v"], b["kd"], b["vd"], 1.0)
    err = max(abs(got[0, l] - float(want[l])) for l in range(L))
    return {"C3.mass": (err, 1e-14)}


def pin_mass_permutation(orc, T=13, Hq=4, Hk=2, d=8, L=6, scale=0.5, seed=35):
    _, x, b = pins.case(T, Hq, Hk, d, L, seed)
    got = orc.depth_mass(b["q"], b["k"], b["v"], b["kd"], b["vd"], scale)
    perm = np.array([3, 0, 5, 1, 4, 2])
    gotp = orc.depth_mass(b["q"], b["k"], b["v"], np.ascontiguousarray(b["kd"][perm]),
                          np.ascontiguousarray(b["vd"][perm]), scale)
    return {"C4.mass": (pins._err(gotp, got[:, perm]), 1e-14)}


def pin_mass_rows_additive(orc, T=10, Hq=4, Hk=1, d=8, L=3, scale=0.6, seed=37):
    _, x, b = pins.case(T, Hq, Hk, d, L, seed)
    a = (b["q"], b["k"], b["v"], b["kd"], b["vd"], scale)
    tt, hh = np.meshgrid(np.arange(T), np.arange(Hq), indexing="ij")
    tt, hh = tt.reshape(-1), hh.reshape(-1)
    first = tt < T // 2
    whole = orc.depth_mass(*a)
    parts = orc.depth_mass(*a, ts=tt[first], hs=hh[first]) + orc.depth_mass(*a, ts=tt[~first], hs=hh[~first])
    return {"C5.mass": (pins._err(whole, parts), 1e-13)}


ALL_PINS = [pin_mass_dense, pin_mass_equal_logits, pin_mass_brute_force, pin_mass_permutation,
            pin_mass_rows_additive]


def run_all(orc):
    out = {}
    for pin in ALL_PINS:
        out.update(pin(orc))
    return out
