"""The oracle side of the bounded depth cache (summary, Sec. 6.2), CPU only:
the depth mass (slot utility) against its pins, planted mistakes in the C
source caught by them, and the slot choice of the three policies against
hand-worked cases and against the policy's definition (which entries the
cache holds afterwards)."""
import itertools
import os

import numpy as np
import pytest

import oracle
from oracle import depth_cache
import pins_cache

SRC = os.path.join(os.path.dirname(oracle.__file__), "moda_oracle.c")


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins_cache.ALL_PINS, ids=lambda p: p.__name__)
def test_mass_pin(orc, pin):
    for name, (err, tol) in pin(orc).items():
        assert err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


MUTANTS = {
    "mass_reads_previous_candidate": ("for (int l = 0; l < jb->L; ++l) m[l] += p[t + 1 + l];",
                                      "for (int l = 0; l < jb->L; ++l) m[l] += p[t + l];"),
    "mass_head_mod": ("double* m = jb->mass + (int64_t)(h / G) * jb->L;",
                      "double* m = jb->mass + (int64_t)(h % jb->Hk) * jb->L;"),
    "mass_slots_reversed": ("for (int l = 0; l < jb->L; ++l) m[l] += p[t + 1 + l];",
                            "for (int l = 0; l < jb->L; ++l) m[l] += p[t + jb->L - l];"),
    "mass_drops_last_thread": ("for (int i = 0; i < nthreads; ++i)\n    for (size_t e = 0; e < nm; ++e) mass[e] += jobs[i].mass[e];",
                               "for (int i = 0; i + 1 < nthreads; ++i)\n    for (size_t e = 0; e < nm; ++e) mass[e] += jobs[i].mass[e];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mass_pins_catch_mutant(tmp_path, name):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    # the additivity pin runs rows over one thread per call; run the dense pin
    # threaded too so a lost thread copy shows
    res = pins_cache.run_all(orc)
    _, x, b = pins_cache.pins.case(23, 8, 2, 8, 5, 41)
    got = orc.depth_mass(b["q"], b["k"], b["v"], b["kd"], b["vd"], 0.4, nthreads=4)
    res["C1.mass.threads"] = (pins_cache.pins._err(got, pins_cache.dense_mass(x, 0.4)), 1e-12)
    failed = [n for n, (err, tol) in res.items() if not err <= tol]
    assert failed, f"no pin catches mutant {name}"


# ---------------------------------------------------------------- slot choice
def test_victim_hand_cases():
    ages = [0, 1, 2, 3]
    u = [0.5, 0.4, 0.05, 0.3]
    assert depth_cache.victim(ages, u, recent=4) == 0      # sliding window: the oldest
    assert depth_cache.victim(ages, u, recent=9) == 0      # R >= S is the window too
    assert depth_cache.victim(ages, u, recent=0) == 2      # top-S: least utility
    assert depth_cache.victim(ages, u, recent=1) == 2      # R = 1 keeps only the new one
    assert depth_cache.victim(ages, u, recent=2) == 2      # age 3 protected; 0.05 leaves
    assert depth_cache.victim(ages, u, recent=3) == 1      # ages 3, 2 protected; 0.4 < 0.5
    # slots need not hold entries in age order
    assert depth_cache.victim([7, 2, 9, 4], [0.1, 0.1, 0.1, 0.1], recent=0) == 1  # tie: older
    assert depth_cache.victim([5, 5, 5, 5], [0.2, 0.1, 0.1, 0.3], recent=0) == 1  # tie: lower slot
    # empty slots fill first, lowest first, whatever the utility
    assert depth_cache.victim([-1, 0, -1], [9.0, 0.0, 9.0], recent=0) == 0
    assert depth_cache.victim([3, 1, -1], [0.0, 0.0, 0.0], recent=3) == 2


def test_victim_matches_definition():
    """The entries held after the write equal, by the policy's definition,
    the R most recent ones plus the highest-utility ones up to S."""
    rng = np.random.default_rng(3)
    for S in (1, 2, 3, 5, 8):
        for trial in range(60):
            ages = list(rng.permutation(40)[:S])
            if trial % 5 == 0:  # some empty slots
                for s in rng.choice(S, size=rng.integers(1, S + 1), replace=False):
                    ages[s] = -1
            u = list(rng.choice([0.1, 0.2, 0.3, 0.5], size=S))  # ties on purpose
            for R in range(0, S + 2):
                v = depth_cache.victim(ages, u, R)
                after = list(ages)
                after[v] = 100
                held = sorted(a for a in after if a >= 0)
                assert held == depth_cache.kept_after(ages, u, R, 100), (S, ages, u, R, v)


def test_sliding_window_is_last_S():
    """R = S over a long run keeps exactly the last S entries (the ring of
    the sliding-window reading)."""
    S = 4
    ages = [-1] * S
    for new in range(11):
        v = depth_cache.victim(ages, [0.0] * S, recent=S)
        ages[v] = new
    assert sorted(ages) == list(range(7, 11))
    # and the slots are reused in ring order
    assert ages == [8, 9, 10, 7]


@pytest.mark.parametrize("S,R", list(itertools.product([3, 6], [0, 2])))
def test_top_s_keeps_high_utility_entries(S, R):
    """With a fixed utility per entry, the cache converges to the R most
    recent entries plus the highest-utility older ones."""
    util = {a: float((a * 37) % 11) / 11 for a in range(30)}
    ages = [-1] * S
    for new in range(30):
        u = [util[a] if a >= 0 else 0.0 for a in ages]
        v = depth_cache.victim(ages, u, R)
        ages[v] = new
    recent = set(range(30 - max(R, 1), 30))
    older = sorted((a for a in range(30) if a not in recent), key=lambda a: (-util[a], -a))
    assert set(ages) == recent | set(older[:S - len(recent)])
