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
# Slips in the producer step (ReLU, RoPE, normaliser, BF16 rounding).
PRODUCER_MUTANTS = {
    "rope_sign": ("dst[row + 2 * p] = f32_to_bf16_rne(a0 - b0);", "dst[row + 2 * p] = f32_to_bf16_rne(a0 + b0);"),
    "rope_swapped_tables": ("const float c = cos_t[n * P + p], s = sin_t[n * P + p];",
                            "const float s = cos_t[n * P + p], c = sin_t[n * P + p];"),
    "rope_pair_shift": ("const float c = cos_t[n * P + p], s = sin_t[n * P + p];",
                        "const float c = cos_t[n * P + (p + 1) % P], s = sin_t[n * P + (p + 1) % P];"),
    "no_relu_on_rotated": ("x0 = x0 > 0.0f ? x0 : 0.0f;", "x0 = x0;"),
    "no_relu_in_den": ("ksum[i] += ka > 0.0 ? ka : 0.0;", "ksum[i] += ka;"),
    "rounding_truncates": ("u += 0x7fffu + ((u >> 16) & 1u);", "u += 0u;"),
    "rounding_ties_away": ("u += 0x7fffu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    "eps_dropped": ("den[h * N + n] = dot + eps;", "den[h * N + n] = dot;"),
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


# Slips in the softmax anchor attention.
SOFTMAX_MUTANTS = {
    "no_max_subtraction": ("s[m] = exp(s[m] - smax);", "s[m] = exp(s[m]);"),
    "no_scale": ("s[m] = scale * dot;", "s[m] = dot;"),
    "no_normalisation": ("dst[j] /= wsum;", "dst[j] /= 1.0;"),
    "value_of_wrong_key": ("const uint16_t *vrow = v + (h * N + m) * D;",
                           "const uint16_t *vrow = v + (h * N + (N - 1 - m)) * D;"),
    "keys_of_wrong_head": ("const uint16_t *krow = k + (h * N + m) * D;", "const uint16_t *krow = k + m * D;"),
}


def softmax_pins_hold(lib) -> bool:
    from test_oracle_softmax_pins import bf16_randn, torch_sdpa
    from conftest import to_bf16_bits, bits_to_f64
    for shape, qs in (((2, 37, 16), 1.0), ((3, 64, 32), 3.0)):
        qb, kb, vb = bf16_randn(shape, 1, qs), bf16_randn(shape, 2), bf16_randn(shape, 3)
        got = oracle.softmax_attention_rows(qb, kb, vb, lib=lib).reshape(shape)
        if not (np.all(np.isfinite(got)) and rel_l2(got, torch_sdpa(qb, kb, vb)) <= 1e-12):
            return False
    q = np.zeros((1, 6, 16)); q[..., 0] = 4096.0
    k = np.zeros((1, 6, 16)); k[0, 3, 0] = 1.0
    vb = bf16_randn((1, 6, 16), 9)
    got = oracle.softmax_attention_rows(to_bf16_bits(q), to_bf16_bits(k), vb, lib=lib)
    return bool(np.all(np.isfinite(got)) and np.allclose(got, bits_to_f64(vb)[0, 3], rtol=1e-12))


def producer_pins_hold(lib) -> bool:
    from test_oracle_producer_pins import random_case, torch_producer
    for shape in ((2, 64, 32), (3, 17, 112)):
        q, k, cos, sin = random_case(*shape, seed=sum(shape))
        q_rot, k_rot, den = oracle.producer(q, k, cos, sin, lib=lib)
        tq, tk, tden = torch_producer(q, k, cos, sin)
        if not (np.array_equal(q_rot, tq) and np.array_equal(k_rot, tk) and np.allclose(den, tden, rtol=1e-13)):
            return False
    vals = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1.2345678], np.float32)
    import torch
    from conftest import bf16_bits
    return bool(np.array_equal(oracle.f32_to_bf16(vals, lib=lib), bf16_bits(torch.from_numpy(vals).to(torch.bfloat16))))


# Slips in the second GEMM with FP64 denominators (the fused path's reference).
F64DEN_MUTANTS = {
    "f64den_multiply": ("out[r * D + j] = s / dd;", "out[r * D + j] = s * dd;"),
    "f64den_sample_index": ("const double dd = den64[flat];", "const double dd = den64[r];"),
    "f64den_rounded_to_f32": ("const double dd = den64[flat];", "const double dd = (double)(float)den64[flat];"),
    "f64den_den_of_wrong_head": ("const double dd = den64[flat];", "const double dd = den64[flat % N];"),
    "f64den_last_dim_dropped": ("for (int64_t i = 0; i < D; ++i)\n                s += bf16_to_f64(qrow[i]) * kvh[i * D + j];\n            out[r * D + j] = s / dd;",
                                "for (int64_t i = 0; i < D - 1; ++i)\n                s += bf16_to_f64(qrow[i]) * kvh[i * D + j];\n            out[r * D + j] = s / dd;"),
}


def test_unmodified_oracle_passes(oracle_lib):
    from test_oracle_f64den_pins import f64den_pins_hold
    assert pins_hold(oracle_lib)
    assert f64den_pins_hold(oracle_lib)
    assert producer_pins_hold(oracle_lib)
    assert softmax_pins_hold(oracle_lib)


@pytest.mark.parametrize("name", sorted(SOFTMAX_MUTANTS))
def test_softmax_mutant_is_caught(tmp_path, name):
    old, new = SOFTMAX_MUTANTS[name]
    assert SRC.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(SRC.replace(old, new))
    lib = oracle.load(lib_path=str(tmp_path / f"lib{name}.so"), src=str(src))
    assert not softmax_pins_hold(lib), f"pins missed the planted slip {name}"


@pytest.mark.parametrize("name", sorted(PRODUCER_MUTANTS))
def test_producer_mutant_is_caught(tmp_path, name):
    old, new = PRODUCER_MUTANTS[name]
    assert SRC.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(SRC.replace(old, new))
    lib = oracle.load(lib_path=str(tmp_path / f"lib{name}.so"), src=str(src))
    assert not producer_pins_hold(lib), f"pins missed the planted slip {name}"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    assert SRC.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(SRC.replace(old, new))
    lib = oracle.load(lib_path=str(tmp_path / f"lib{name}.so"), src=str(src))
    assert not pins_hold(lib), f"pins missed the planted slip {name}"


@pytest.mark.parametrize("name", sorted(F64DEN_MUTANTS))
def test_f64den_mutant_is_caught(tmp_path, name):
    from test_oracle_f64den_pins import f64den_pins_hold
    old, new = F64DEN_MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / f"{name}.c"
    src.write_text(SRC.replace(old, new))
    lib = oracle.load(lib_path=str(tmp_path / f"lib{name}.so"), src=str(src))
    assert not f64den_pins_hold(lib), f"pins missed the planted slip {name}"
