"""The oracle's depth-KV projection against its pins, and planted mistakes in
copies of the oracle source that the pins must catch (CPU only)."""
import os

import pytest

import oracle
import pins_kvproj

SRC = os.path.join(os.path.dirname(oracle.__file__), "moda_oracle.c")


@pytest.mark.parametrize("name", sorted(pins_kvproj.PINS))
def test_kv_proj_pin(name):
    err, tol = pins_kvproj.PINS[name](oracle.default())
    assert err <= tol, f"{name}: error {err} > {tol}"


MUTANTS = {
    "weight_index_transposed": ("const uint16_t* wrow = w + (int64_t)n * Dm;",
                                "const uint16_t* wrow = w + (int64_t)n;"),
    "last_term_dropped": ("for (int c = 0; c < Dm; ++c) s += bf16_to_double(xrow[c]) * bf16_to_double(wrow[c]);",
                          "for (int c = 0; c < Dm - 1; ++c) s += bf16_to_double(xrow[c]) * bf16_to_double(wrow[c]);"),
    "row_list_ignored": ("const int64_t t = rows ? rows[r] : r;", "const int64_t t = r;"),
    "input_row_shifted": ("const uint16_t* xrow = x + t * (int64_t)Dm;",
                          "const uint16_t* xrow = x + (t > 0 ? t - 1 : t) * (int64_t)Dm;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_kv_proj_pins_catch_mutant(tmp_path, name):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    orc = oracle.Oracle(oracle.build(force=True, src=str(path), out=str(tmp_path / "libm.so")))
    failed = [n for n, (err, tol) in pins_kvproj.run_all(orc).items() if not err <= tol]
    assert failed, f"no pin catches mutant {name}"
