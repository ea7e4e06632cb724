"""Plant plausible slips in a copy of the oracle (on the CPU) and check that the
pins of test_oracle_pins.py catch every one of them.  The shipped oracle is
never modified; each mutant is a rewritten copy built into a temporary dir."""
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN, rel_l2, to_bf16_bits
from test_oracle_pins import brute_force, tiny_inputs

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "lin_attn_oracle.c")).read()

MUTANTS = {
    "transposed_kv_in_apply": ("kvh[i * D + j]", "kvh[j * D + i]"),
    "last_token_dropped": ("for (int64_t m = 0; m < N; ++m)", "for (int64_t m = 0; m < N - 1; ++m)"),
    "first_token_dropped": ("for (int64_t m = 0; m < N; ++m)", "for (int64_t m = 1; m < N; ++m)"),
    "wrong_sign_in_kv": ("dst[j] += a *", "dst[j] -= a *"),
    "multiply_by_den": ("out[r * D + j] = s / d;", "out[r * D + j] = s * d;"),
    "bad_bf16_decode": ("(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    "v_index_swapped": ("a * bf16_to_f64(vrow[j])", "a * bf16_to_f64(vrow[i])"),
    "q_from_wrong_row": ("const uint16_t *qrow = q + flat * D;", "const uint16_t *qrow = q + (flat / N) * N * D;"),
    "last_dim_dropped": ("for (int64_t i = 0; i < D; ++i)\n                s +=", "for (int64_t i = 0; i < D - 1; ++i)\n                s +="),
    "den_of_wrong_head": ("const double d = (double)den[flat];", "const double d = (double)den[flat % N];"),
}


def pins_hold(lib) -> bool:
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    qb, kb, vb = (to_bf16_bits(g[x])[None] for x in ("q_rot", "k_rot", "v"))
    den = np.array(g["den"], np.float32)[None]
    if not np.array_equal(oracle.forward(qb, kb, vb, den, lib=lib)[0], np.array(g["out"])):
        return False
    qb, kb, vb, den = tiny_inputs(seed=11, H=2, N=256, D=32)
    if rel_l2(oracle.forward(qb, kb, vb, den, lib=lib), brute_force(qb, kb, vb, den)) > 1e-12:
        return False
    cases = json.load(open(os.path.join(GOLDEN, "bf16_patterns.json")))["cases"]
    bits = np.array([int(c["bits"], 16) for c in cases], np.uint16)
    if not np.array_equal(oracle.bf16_decode(bits, lib=lib), [float(c["value"]) for c in cases]):
        return False
    return True


def test_unmodified_oracle_passes(oracle_lib):
    assert pins_hold(oracle_lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    assert SRC.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(SRC.replace(old, new))
    lib = oracle.load(lib_path=str(tmp_path / f"lib{name}.so"), src=str(src))
    assert not pins_hold(lib), f"pins missed the planted slip {name}"
