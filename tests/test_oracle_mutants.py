"""Plants plausible mistakes in copies of the oracle source (CPU only) and
checks that the pins catch every one: a dropped term, a wrong index, a wrong
head mapping, a transposed depth operand, a missing scale, a wrong sign."""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moda_oracle.c")

MUTANTS = {
    "self_key_dropped": ("z[j] = scale * dot_bf16(qrow, krow, d);",
                         "z[j] = (j == t) ? -1e300 : scale * dot_bf16(qrow, krow, d);"),
    "head_mod_not_div": ("const int hk = h / G;", "const int hk = h % Hk;"),
    "depth_index_swapped": ("const uint16_t* kdrow = kd + (((int64_t)l * T + t) * Hk + hk) * d;",
                            "const uint16_t* kdrow = kd + (((int64_t)t * L + l) * Hk + hk) * d;"),
    "depth_scale_dropped": ("z[t + 1 + l] = scale * dot_bf16(qrow, kdrow, d);",
                            "z[t + 1 + l] = dot_bf16(qrow, kdrow, d);"),
    "depth_value_from_keys": ("const uint16_t* vdrow = vd +", "const uint16_t* vdrow = kd +"),
    "exp_sign_flipped": ("z[j] = exp(z[j] - m); /* z now holds", "z[j] = exp(m - z[j]); /* z now holds"),
    "lse_without_max": ("*lse = m + log(Z);", "*lse = log(Z);"),
    "depth_previous_position": ("const uint16_t* kdrow = kd + (((int64_t)l * T + t) * Hk + hk) * d;",
                                "const uint16_t* kdrow = kd + (((int64_t)l * T + (t > 0 ? t - 1 : t)) * Hk + hk) * d;"),
    "causal_exclusive_values": ("for (int64_t j = 0; j <= t; ++j) {\n    const double pj",
                                "for (int64_t j = 0; j < t; ++j) {\n    const double pj"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = [n for n, (err, tol) in pins.run_all(orc).items() if not err <= tol]
    assert failed, f"no pin catches mutant {name}"
