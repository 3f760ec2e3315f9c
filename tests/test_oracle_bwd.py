"""The oracle's backward against torch autograd and exact identities (CPU),
and planted mistakes in copies of its source that the pins must catch."""
import os

import numpy as np
import pytest

import oracle
import pins_bwd

SRC = os.path.join(os.path.dirname(oracle.__file__), "moda_oracle.c")


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins_bwd.ALL_BWD_PINS, ids=lambda p: p.__name__)
def test_bwd_pin(orc, pin):
    for name, (err, tol) in pin(orc).items():
        assert err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


@pytest.mark.parametrize("shape", [dict(T=1, Hq=2, Hk=1, d=8, L=3), dict(T=9, Hq=16, Hk=1, d=4, L=2),
                                   dict(T=17, Hq=4, Hk=4, d=8, L=1)])
def test_bwd_autograd_more_shapes(orc, shape):
    res = pins_bwd.pin_bwd_autograd_dense(orc, scale=0.5, seed=43, **shape)
    for name, (err, tol) in res.items():
        assert err <= tol, f"{name}: {err:.3e}"


def test_bwd_threads_deterministic(orc):
    x, dO = pins_bwd.case(30, 4, 2, 8, 4, 47)
    from sequence_depth_attention_gb300.inputs import bf16_bits
    b = {n: bf16_bits(t) for n, t in x.items()}
    r1 = orc.backward(b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), 0.3, nthreads=1)
    r4 = orc.backward(b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), 0.3, nthreads=4)
    for a, c in zip(r1, r4):
        assert np.allclose(a, c, rtol=0, atol=1e-13)


BWD_MUTANTS = {
    "missing_D_term": ("const double ds = p * (dp - D);", "const double ds = p * dp;"),
    "ds_sign": ("const double ds = p * (dp - D);", "const double ds = p * (D - dp);"),
    "dv_uses_ds": ("dval[c] += p * g[c];", "dval[c] += ds * g[c];"),
    "dk_no_scale": ("dkey[c] += scale * ds * qr[c];", "dkey[c] += ds * qr[c];"),
    "dq_uses_values": ("dst->dq_row[c] += scale * ds * bf16_to_double(key[c]);",
                       "dst->dq_row[c] += scale * ds * bf16_to_double(val[c]);"),
    "D_from_dO_squared": ("for (int c = 0; c < d; ++c) D += g[c] * o[c];",
                          "for (int c = 0; c < d; ++c) D += g[c] * g[c];"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_bwd_pins_catch_mutant(tmp_path, name):
    before, after = BWD_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    orc = oracle.Oracle(oracle.build(force=True, src=str(path), out=str(tmp_path / "libm.so")))
    failed = [n for n, (err, tol) in pins_bwd.run_all(orc).items() if not err <= tol]
    assert failed, f"no backward pin catches mutant {name}"


def test_bwd_rows_matches_full(orc):
    """The row-subset backward reproduces the full one: dq rows, depth
    gradients summed over the heads of each position, and the tail keys."""
    from sequence_depth_attention_gb300.inputs import bf16_bits
    T, Hq, Hk, d, L = 40, 8, 2, 8, 5
    x, dO = pins_bwd.case(T, Hq, Hk, d, L, 53)
    b = {n: bf16_bits(t) for n, t in x.items()}
    full = orc.backward(b["q"], b["k"], b["v"], b["kd"], b["vd"], bf16_bits(dO), 0.3, nthreads=3)
    k_lo = 30
    ts = [0, 7, 19] + list(range(k_lo, T))
    rows = np.array([t * Hq + h for t in ts for h in range(Hq)])
    dq, dk, dv, dkd, dvd = orc.backward_rows(b["q"], b["k"], b["v"], b["kd"], b["vd"],
                                             bf16_bits(dO), 0.3, rows, k_lo, nthreads=3)
    assert np.allclose(dq, full[0].reshape(T * Hq, d)[rows], atol=1e-12)
    assert np.allclose(dk, full[1][k_lo:], atol=1e-12) and np.allclose(dv, full[2][k_lo:], atol=1e-12)
    G = Hq // Hk
    for i, t in enumerate(ts):
        for hk in range(Hk):
            sel = slice(i * Hq + hk * G, i * Hq + (hk + 1) * G)
            assert np.allclose(dkd[sel].sum(0), full[3][:, t, hk], atol=1e-12)
            assert np.allclose(dvd[sel].sum(0), full[4][:, t, hk], atol=1e-12)
