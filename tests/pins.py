"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, none of which re-runs the oracle's own per-row loops.

Each ``pin_*`` takes an ``oracle.Oracle`` and returns ``{name: (error, tol)}``
so the same pins can be run against a build of the oracle with a planted
mistake (``test_oracle_mutants.py``) and must then fail.

Citations are to "Mixture-of-Depths Attention" (arXiv 2603.15619) as the pages
present it: Sec. 2.1 Eq. (1)-(2) (GQA), Sec. 2.2 (MoDA, one softmax), Sec. 3.2
(flash-compatible / chunk-aware / group-aware depth layout, masks), Sec. 3.3
(online softmax over sequence then depth blocks), and the reading notes'
teaching example in Sec. 二.2 (4/7 depth mass).
"""
from __future__ import annotations

import math

import mpmath
import numpy as np
import scipy.special
import torch
import torch.nn.functional as F

from sequence_depth_attention_gb300.inputs import Workload, bf16_bits, make_inputs


def case(T, Hq, Hk, d, L, seed=0, depth_scale=1.0):
    w = Workload("pin", T, Hq, Hk, d, L, depth_scale, seed)
    x = make_inputs(w)
    return w, x, {k: bf16_bits(v) for k, v in x.items()}


def _f64(t):
    return t.to(torch.float64)


def _err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


# ---------------------------------------------------------------------------
# P1: L = 0 is ordinary causal GQA attention (Sec. 2.1 Eq. (2); Table 3's
# "Sequence KV" row is vanilla attention). Library routine: torch SDPA in fp64,
# K/V heads repeated G times so query head h reads KV head floor(h/G).
# ---------------------------------------------------------------------------
def sdpa_causal_gqa(x, scale):
    T, Hq, d = x["q"].shape
    G = Hq // x["k"].shape[1]
    q = _f64(x["q"]).permute(1, 0, 2)
    k = _f64(x["k"]).repeat_interleave(G, dim=1).permute(1, 0, 2)
    v = _f64(x["v"]).repeat_interleave(G, dim=1).permute(1, 0, 2)
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale)
    s = scale * (q @ k.transpose(-1, -2))
    s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


def pin_l0_sdpa(orc, T=37, Hq=6, Hk=2, d=16, scale=0.3, seed=3):
    _, x, b = case(T, Hq, Hk, d, 0, seed)
    o, lse = orc.forward(b["q"], b["k"], b["v"], None, None, scale)
    ro, rl = sdpa_causal_gqa(x, scale)
    return {"P1.o": (_err(o, ro), 1e-12), "P1.lse": (_err(lse, rl), 1e-12)}


# ---------------------------------------------------------------------------
# P2: the pages' own dense formulation. Expanded query rows i_q = t*G + g
# (T_q = G*T_kv), keys = [K (T rows) | flash-compatible depth axis of T*L rows,
# j_d = t*L + l] (Sec. 3.2), grouped causal mask floor(i_q/G) >= i_k and the
# block-diagonal depth mask floor(i_q/G) == floor(j_d/L) (Sec. 3.2, Sec. 3.3
# mask equation). Softmax by torch SDPA with that boolean mask.
# ---------------------------------------------------------------------------
def masks_pages(T, G, L):
    iq = torch.arange(T * G)[:, None]
    keep_seq = (iq // G) >= torch.arange(T)[None, :]
    if L == 0:
        return keep_seq
    jd = torch.arange(T * L)[None, :]
    keep_depth = (iq // G) == (jd // L)
    return torch.cat([keep_seq, keep_depth], dim=1)


def dense_pages(x, scale):
    q, k, v, kd, vd = (_f64(x[n]) for n in ("q", "k", "v", "kd", "vd"))
    T, Hq, d = q.shape
    Hk = k.shape[1]
    L = kd.shape[0]
    G = Hq // Hk
    keep = masks_pages(T, G, L)
    o = np.zeros((T, Hq, d))
    lse = np.zeros((T, Hq))
    for hk in range(Hk):
        qe = q[:, hk * G:(hk + 1) * G, :].reshape(T * G, d)
        kflat = kd[:, :, hk, :].permute(1, 0, 2).reshape(T * L, d)
        vflat = vd[:, :, hk, :].permute(1, 0, 2).reshape(T * L, d)
        keys = torch.cat([k[:, hk, :], kflat], 0)
        vals = torch.cat([v[:, hk, :], vflat], 0)
        out = F.scaled_dot_product_attention(qe[None], keys[None], vals[None],
                                             attn_mask=keep[None], scale=scale)[0]
        s = (scale * qe @ keys.T).masked_fill(~keep, float("-inf"))
        o[:, hk * G:(hk + 1) * G, :] = out.reshape(T, G, d).numpy()
        lse[:, hk * G:(hk + 1) * G] = torch.logsumexp(s, -1).reshape(T, G).numpy()
    return o, lse


def pin_dense_pages(orc, T=21, Hq=8, Hk=2, d=8, L=5, scale=0.41, seed=5):
    _, x, b = case(T, Hq, Hk, d, L, seed)
    o, lse = orc.forward(b["q"], b["k"], b["v"], b["kd"], b["vd"], scale)
    ro, rl = dense_pages(x, scale)
    return {"P2.o": (_err(o, ro), 1e-12), "P2.lse": (_err(lse, rl), 1e-12)}


# ---------------------------------------------------------------------------
# P3: T = 1 closed form: softmax over {self} + the L depth slots of position 0
# (Sec. 2.2: the depth path reads the same position only).
# ---------------------------------------------------------------------------
def pin_t1_closed_form(orc, Hq=4, Hk=2, d=16, L=7, scale=0.25, seed=7):
    _, x, b = case(1, Hq, Hk, d, L, seed)
    o, lse = orc.forward(b["q"], b["k"], b["v"], b["kd"], b["vd"], scale)
    G = Hq // Hk
    eo, el = 0.0, 0.0
    for h in range(Hq):
        hk = h // G
        keys = np.concatenate([_f64(x["k"][0, hk])[None].numpy(), _f64(x["kd"][:, 0, hk]).numpy()])
        vals = np.concatenate([_f64(x["v"][0, hk])[None].numpy(), _f64(x["vd"][:, 0, hk]).numpy()])
        z = scale * keys @ _f64(x["q"][0, h]).numpy()
        p = scipy.special.softmax(z)
        eo = max(eo, _err(o[0, h], p @ vals))
        el = max(el, abs(lse[0, h] - scipy.special.logsumexp(z)))
    return {"P3.o": (eo, 1e-12), "P3.lse": (el, 1e-12)}


# ---------------------------------------------------------------------------
# P4: equal logits (q = 0). Every visible candidate gets 1/(t+1+L); o is the
# plain mean of the visible values; lse = ln(t+1+L). The teaching example:
# 1-based position 3 with 4 depth slots -> depth mass 4/7.
# ---------------------------------------------------------------------------
def pin_equal_logits(orc, T=9, Hq=4, Hk=2, d=8, L=4, seed=11, example=None):
    _, x, b = case(T, Hq, Hk, d, L, seed)
    b = dict(b)
    b["q"] = np.zeros_like(b["q"])
    o, lse = orc.forward(b["q"], b["k"], b["v"], b["kd"], b["vd"], 0.7)
    G = Hq // Hk
    eo, el = 0.0, 0.0
    for t in range(T):
        for h in range(Hq):
            hk = h // G
            vis = np.concatenate([_f64(x["v"][:t + 1, hk]).numpy(), _f64(x["vd"][:, t, hk]).numpy()])
            eo = max(eo, _err(o[t, h], vis.mean(axis=0)))
            el = max(el, abs(lse[t, h] - math.log(t + 1 + L)))
    res = {"P4.o": (eo, 1e-13), "P4.lse": (el, 1e-13)}
    if example is not None:
        t0, Lx = example["t_zero_based"], example["L"]
        _, _, b2 = case(t0 + 1, 2, 1, 4, Lx, seed)
        b2 = dict(b2)
        b2["q"] = np.zeros_like(b2["q"])
        _, _, p = orc.row(b2["q"], b2["k"], b2["v"], b2["kd"], b2["vd"], 1.0, t0, 0)
        want = example["depth_mass_num"] / example["depth_mass_den"]
        res["P4.example_len"] = (abs(len(p) - example["candidates"]), 0)
        res["P4.example_mass"] = (abs(p[t0 + 1:].sum() - want), 1e-15)
    return res


# ---------------------------------------------------------------------------
# P5: invariants. (a) each probability row sums to 1; (b) permuting the depth
# slots changes nothing (the depth history is a set, Sec. 2.2); (c) GQA
# equivalence: repeating each KV head G times and running with G = 1 gives
# the same result (Eq. (2) phi(h)).
# ---------------------------------------------------------------------------
def pin_invariants(orc, T=19, Hq=6, Hk=2, d=16, L=6, scale=0.3, seed=13):
    _, x, b = case(T, Hq, Hk, d, L, seed)
    o, lse = orc.forward(b["q"], b["k"], b["v"], b["kd"], b["vd"], scale)
    worst = 0.0
    for t in (0, 1, T // 2, T - 1):
        for h in (0, Hq - 1):
            _, _, p = orc.row(b["q"], b["k"], b["v"], b["kd"], b["vd"], scale, t, h)
            worst = max(worst, abs(p.sum() - 1.0))
    perm = np.random.default_rng(seed).permutation(L)
    op, lp = orc.forward(b["q"], b["k"], b["v"], b["kd"][perm], b["vd"][perm], scale)
    G = Hq // Hk
    rep = {n: bf16_bits(x[n].repeat_interleave(G, dim=1)) for n in ("k", "v")}
    rep.update({n: bf16_bits(x[n].repeat_interleave(G, dim=2)) for n in ("kd", "vd")})
    og, lg = orc.forward(b["q"], rep["k"], rep["v"], rep["kd"], rep["vd"], scale)
    return {"P5.sum1": (worst, 1e-13),
            "P5.perm.o": (_err(o, op), 1e-13), "P5.perm.lse": (_err(lse, lp), 1e-13),
            "P5.gqa.o": (_err(o, og), 0.0), "P5.gqa.lse": (_err(lse, lg), 0.0)}


# ---------------------------------------------------------------------------
# P6: split-merge identity of a joint softmax over two candidate sets (the
# MiTA notes' merge of compressed and routed branches, applied to the
# sequence and depth sets): lse = logaddexp(lse_s, lse_d),
# o = (e^{lse_s} o_s + e^{lse_d} o_d) / e^{lse}. Sequence half from the
# oracle at L = 0 (itself pinned by P1); depth half by scipy.
# ---------------------------------------------------------------------------
def pin_split_merge(orc, T=17, Hq=4, Hk=1, d=16, L=9, scale=0.35, seed=17):
    _, x, b = case(T, Hq, Hk, d, L, seed)
    o, lse = orc.forward(b["q"], b["k"], b["v"], b["kd"], b["vd"], scale)
    os_, ls_ = orc.forward(b["q"], b["k"], b["v"], None, None, scale)
    G = Hq // Hk
    eo, el = 0.0, 0.0
    for t in range(T):
        for h in range(Hq):
            hk = h // G
            z = scale * _f64(x["kd"][:, t, hk]).numpy() @ _f64(x["q"][t, h]).numpy()
            ld = scipy.special.logsumexp(z)
            od = scipy.special.softmax(z) @ _f64(x["vd"][:, t, hk]).numpy()
            lm = np.logaddexp(ls_[t, h], ld)
            om = math.exp(ls_[t, h] - lm) * os_[t, h] + math.exp(ld - lm) * od
            eo = max(eo, _err(o[t, h], om))
            el = max(el, abs(lse[t, h] - lm))
    return {"P6.o": (eo, 1e-12), "P6.lse": (el, 1e-12)}


# ---------------------------------------------------------------------------
# P7: brute force, exact. T=3, G=2, Hk=1, d=2, L=2, scale=1 with small
# integers (exact in bf16): logits are integers, o is a ratio of sums of
# e^integer * integer, evaluated with 50-digit mpmath.
# ---------------------------------------------------------------------------
BRUTE = {
    "q": [[[1, -1], [2, 0]], [[0, 1], [-1, 2]], [[1, 1], [2, -2]]],
    "k": [[[1, 2]], [[-2, 1]], [[0, -1]]],
    "v": [[[3, -1]], [[1, 2]], [[-2, 0]]],
    "kd": [[[[2, 0]], [[1, -1]], [[-1, 2]]], [[[0, 1]], [[2, 2]], [[1, 0]]]],
    "vd": [[[[1, 1]], [[0, -3]], [[2, 2]]], [[[-1, 2]], [[3, 0]], [[-2, 1]]]],
}


def brute_force_exact():
    q, k, v, kd, vd = (BRUTE[n] for n in ("q", "k", "v", "kd", "vd"))
    T, Hq, d, L, G = 3, 2, 2, 2, 2
    mpmath.mp.dps = 50
    o = [[None] * Hq for _ in range(T)]
    lse = [[None] * Hq for _ in range(T)]
    for t in range(T):
        for h in range(Hq):
            hk = h // G
            cand = [(sum(q[t][h][c] * k[j][hk][c] for c in range(d)), v[j][hk]) for j in range(t + 1)]
            cand += [(sum(q[t][h][c] * kd[l][t][hk][c] for c in range(d)), vd[l][t][hk]) for l in range(L)]
            Z = mpmath.fsum(mpmath.e ** z for z, _ in cand)
            o[t][h] = [mpmath.fsum(mpmath.e ** z * val[c] for z, val in cand) / Z for c in range(d)]
            lse[t][h] = mpmath.log(Z)
    return o, lse


def pin_brute_force(orc):
    def bits(a):
        return bf16_bits(torch.tensor(a, dtype=torch.float32).to(torch.bfloat16))
    b = {n: bits(a) for n, a in BRUTE.items()}
    o, lse = orc.forward(b["q"], b["k"], b["v"], b["kd"], b["vd"], 1.0)
    eo_ref, el_ref = brute_force_exact()
    eo, el = 0.0, 0.0
    for t in range(3):
        for h in range(2):
            for c in range(2):
                ref = float(eo_ref[t][h][c])
                eo = max(eo, abs(o[t, h, c] - ref) / max(1.0, abs(ref)))
            ref = float(el_ref[t][h])
            el = max(el, abs(lse[t, h] - ref) / max(1.0, abs(ref)))
    return {"P7.o": (eo, 1e-14), "P7.lse": (el, 1e-14)}


ALL_PINS = [pin_l0_sdpa, pin_dense_pages, pin_t1_closed_form, pin_equal_logits,
            pin_invariants, pin_split_merge, pin_brute_force]


def run_all(orc, example=None):
    out = {}
    for pin in ALL_PINS:
        if pin is pin_equal_logits:
            out.update(pin(orc, example=example))
        else:
            out.update(pin(orc))
    return out
