"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle
import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    kw = {"example": _load("worked_example.json")} if pin is pins.pin_equal_logits else {}
    for name, (err, tol) in pin(orc, **kw).items():
        assert err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


@pytest.mark.parametrize("shape", [
    dict(T=1, Hq=1, Hk=1, d=8, L=0),      # single row, no depth
    dict(T=5, Hq=2, Hk=2, d=4, L=1),      # G = 1
    dict(T=33, Hq=16, Hk=1, d=8, L=3),    # G = 16 (multi-query)
    dict(T=12, Hq=8, Hk=4, d=8, L=12),    # L = T
])
def test_l0_and_dense_at_more_shapes(orc, shape):
    T, Hq, Hk, d, L = (shape[n] for n in ("T", "Hq", "Hk", "d", "L"))
    res = pins.pin_dense_pages(orc, T=T, Hq=Hq, Hk=Hk, d=d, L=L, scale=0.5, seed=23)
    res.update(pins.pin_l0_sdpa(orc, T=T, Hq=Hq, Hk=Hk, d=d, scale=0.5, seed=23))
    for name, (err, tol) in res.items():
        assert err <= tol, f"{name}: {err:.3e}"


def test_group_indexing_facts_from_pages():
    """The mask helper used by P2 reproduces the pages' indexing example and eta."""
    g = _load("group_indexing.json")
    G = g["G"]
    rows = np.array(g["rows"])
    t_base = rows // G
    assert sorted(set(t_base.tolist())) == g["t_base_set"]
    assert int(t_base.min()) == g["t_start"] and int(t_base.max()) + 1 == g["t_end"]
    # depth columns kept for rows 8..15 are exactly those of positions 2 and 3
    L = 3
    keep = pins.masks_pages(T=4, G=G, L=L)
    depth = keep[:, 4:]
    for r in rows:
        cols = np.nonzero(depth[r].numpy())[0]
        assert cols.tolist() == list(range((r // G) * L, (r // G + 1) * L))
    for gs, pct in g["eta_percent"].items():
        assert abs(100.0 * int(gs) / g["C"] - pct) < 1e-12
        assert abs(pct - g["eta_printed_percent"][gs]) < 0.01


def test_rows_threads_match_single(orc):
    _, x, b = pins.case(40, 4, 2, 16, 6, seed=29)
    tt, hh = np.meshgrid(np.arange(40), np.arange(4), indexing="ij")
    o1, l1 = orc.rows(b["q"], b["k"], b["v"], b["kd"], b["vd"], 0.25, tt.ravel(), hh.ravel(), 1)
    o4, l4 = orc.rows(b["q"], b["k"], b["v"], b["kd"], b["vd"], 0.25, tt.ravel(), hh.ravel(), 4)
    assert np.array_equal(o1, o4) and np.array_equal(l1, l4)


def test_rejects_bad_arguments(orc):
    _, x, b = pins.case(4, 2, 1, 8, 2)
    with pytest.raises(ValueError):
        orc.row(b["q"], b["k"], b["v"], b["kd"], b["vd"], 1.0, 4, 0)   # t out of range
    with pytest.raises(ValueError):
        orc.row(b["q"], b["k"], b["v"], b["kd"], b["vd"], 1.0, 0, 2)   # h out of range
    with pytest.raises(TypeError):
        orc.row(b["q"].astype(np.int32), b["k"], b["v"], b["kd"], b["vd"], 1.0, 0, 0)
