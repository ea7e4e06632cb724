"""Pins for the FP64 oracle: it is checked against things other than itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong decode or a multiply in
place of the divide) fails at least one of them; test_oracle_mutants.py plants
such slips in a copy of the oracle and confirms that.

Definition followed (page "PR #35728 完整报告 - [diffusion] Accelerate
SANA-Video linear attention in quality=high", 关键源码片段): per head,
KV = K_rot^T V and out = (Q_rot KV) / den, i.e. ((Q_rot K_rot^T) V) / den.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import GOLDEN, bf16_bits, bits_to_f64, rel_l2, to_bf16_bits
from video_diffusion_dit_gb300 import synth


def brute_force(qb, kb, vb, den):
    """((Q K^T) V) / den in FP64 with numpy matmuls: the other association."""
    q, k, v = bits_to_f64(qb), bits_to_f64(kb), bits_to_f64(vb)
    scores = np.einsum("hnd,hmd->hnm", q, k)
    return np.einsum("hnm,hmd->hnd", scores, v) / den.astype(np.float64)[..., None]


def tiny_inputs(seed=0, H=2, N=256, D=32):
    L = synth.make_layer(H, N, D, seed)
    return oracle.torch_inputs_to_numpy(L)


def test_bf16_decode_known_patterns(oracle_lib):
    cases = json.load(open(os.path.join(GOLDEN, "bf16_patterns.json")))["cases"]
    bits = np.array([int(c["bits"], 16) for c in cases], np.uint16)
    want = np.array([float(c["value"]) for c in cases])
    got = oracle.bf16_decode(bits, lib=oracle_lib)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_worked_example_exact(oracle_lib):
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    qb = to_bf16_bits(g["q_rot"])[None]
    kb = to_bf16_bits(g["k_rot"])[None]
    vb = to_bf16_bits(g["v"])[None]
    den = np.array(g["den"], np.float32)[None]
    kv = oracle.kv(kb, vb, lib=oracle_lib)
    assert np.array_equal(kv[0], np.array(g["kv"]))
    out = oracle.forward(qb, kb, vb, den, lib=oracle_lib)
    assert np.array_equal(out[0], np.array(g["out"]))


@pytest.mark.parametrize("shape", [(2, 256, 32), (3, 64, 16), (1, 37, 48), (2, 1, 8)])
def test_associativity_against_brute_force(oracle_lib, shape):
    H, N, D = shape
    qb, kb, vb, den = tiny_inputs(seed=H * 1000 + N, H=H, N=N, D=D)
    out = oracle.forward(qb, kb, vb, den, lib=oracle_lib)
    ref = brute_force(qb, kb, vb, den)
    assert rel_l2(out, ref) <= 1e-12
    assert np.max(np.abs(out - ref)) <= 1e-11 * np.max(np.abs(ref))


def test_kv_against_library_matmul(oracle_lib):
    qb, kb, vb, den = tiny_inputs(seed=7, H=2, N=200, D=24)
    kv = oracle.kv(kb, vb, lib=oracle_lib)
    k, v = bits_to_f64(kb), bits_to_f64(vb)
    ref = np.stack([k[h].T @ v[h] for h in range(k.shape[0])])
    assert rel_l2(kv, ref) <= 1e-13


def test_linearity_in_v(oracle_lib):
    qb, kb, vb, den = tiny_inputs(seed=3, H=2, N=96, D=16)
    v = bits_to_f64(vb)
    rng = np.random.default_rng(3)
    mask = rng.random(v.shape) < 0.5
    v1 = np.where(mask, v, 0.0)
    v2 = np.where(mask, 0.0, v)
    a, b = 2.0, -0.5  # powers of two keep every BF16 value exact
    f = lambda vv: oracle.forward(qb, kb, to_bf16_bits(vv), den, lib=oracle_lib)
    lhs = f(a * v1 + b * v2)
    rhs = a * f(v1) + b * f(v2)
    assert rel_l2(lhs, rhs) <= 1e-13


def test_zero_v_gives_exact_zero(oracle_lib):
    qb, kb, vb, den = tiny_inputs(seed=4)
    out = oracle.forward(qb, kb, np.zeros_like(vb), den, lib=oracle_lib)
    assert np.array_equal(out, np.zeros_like(out))


def test_token_permutation(oracle_lib):
    qb, kb, vb, den = tiny_inputs(seed=5, H=2, N=128, D=16)
    perm = np.random.default_rng(5).permutation(qb.shape[1])
    kv0 = oracle.kv(kb, vb, lib=oracle_lib)
    kv1 = oracle.kv(kb[:, perm], vb[:, perm], lib=oracle_lib)
    assert rel_l2(kv1, kv0) <= 1e-14
    out0 = oracle.forward(qb, kb, vb, den, lib=oracle_lib)
    out1 = oracle.forward(qb[:, perm], kb, vb, den[:, perm], lib=oracle_lib)
    assert np.array_equal(out1, out0[:, perm])


def test_denominator_scaling_and_head_independence(oracle_lib):
    qb, kb, vb, den = tiny_inputs(seed=6, H=3, N=64, D=16)
    out = oracle.forward(qb, kb, vb, den, lib=oracle_lib)
    out2 = oracle.forward(qb, kb, vb, (den * 2).astype(np.float32), lib=oracle_lib)
    assert np.array_equal(out2, out / 2)
    qb2, kb2, vb2 = qb.copy(), kb.copy(), vb.copy()
    qb2[1], kb2[1], vb2[1] = qb[2], kb[0], vb[2]
    out3 = oracle.forward(qb2, kb2, vb2, den, lib=oracle_lib)
    assert np.array_equal(out3[0], out[0]) and np.array_equal(out3[2], out[2])
    assert not np.array_equal(out3[1], out[1])


def test_closed_form_head_dim_one(oracle_lib):
    rng = np.random.default_rng(8)
    N = 50
    q = rng.integers(-64, 64, N) / 8.0
    k = rng.integers(-64, 64, N) / 16.0
    v = rng.integers(-64, 64, N) / 4.0
    den = (rng.integers(1, 100, N) / 4.0).astype(np.float32)
    s = math.fsum(float(a) * float(b) for a, b in zip(k, v))
    want = np.array([qq * s / float(d) for qq, d in zip(q, den)])
    got = oracle.forward(to_bf16_bits(q).reshape(1, N, 1), to_bf16_bits(k).reshape(1, N, 1),
                         to_bf16_bits(v).reshape(1, N, 1), den.reshape(1, N), lib=oracle_lib)
    assert np.allclose(got.ravel(), want, rtol=1e-15, atol=0)


def test_closed_form_single_token(oracle_lib):
    qb, kb, vb, den = tiny_inputs(seed=9, H=2, N=1, D=32)
    q, k, v = bits_to_f64(qb)[:, 0], bits_to_f64(kb)[:, 0], bits_to_f64(vb)[:, 0]
    want = np.stack([(math.fsum(q[h] * k[h]) * v[h]) / float(den[h, 0]) for h in range(2)])
    got = oracle.forward(qb, kb, vb, den, lib=oracle_lib)[:, 0]
    assert rel_l2(got, want) <= 1e-14


def test_apply_rows_matches_full_forward(oracle_lib):
    qb, kb, vb, den = tiny_inputs(seed=10, H=2, N=64, D=32)
    kv = oracle.kv(kb, vb, lib=oracle_lib)
    rows = np.array([0, 63, 64, 100, 127], np.int64)
    part = oracle.apply_rows(qb, kv, den, rows, lib=oracle_lib)
    full = oracle.forward(qb, kb, vb, den, lib=oracle_lib).reshape(-1, 32)
    assert np.array_equal(part, full[rows])
    with pytest.raises(RuntimeError):
        oracle.apply_rows(qb, kv, den, np.array([128], np.int64), lib=oracle_lib)


def test_synth_recipe_properties():
    """The generator's inputs have the recipe's structure (it holds no attention maths)."""
    L = synth.make_layer(2, 64, 32, seed=0)
    assert L["q_rot"].dtype == torch.bfloat16 and L["den"].dtype == torch.float32
    assert tuple(L["q_rot"].shape) == (1, 2, 64, 32) and tuple(L["den"].shape) == (1, 2, 64, 1)
    assert bool((L["den"] >= 1e-6).all())
    # token 0 sits at position 0: RoPE is the identity there, so q_rot = relu'd draws (>= 0)
    assert bool((L["q_rot"][0, :, 0] >= 0).all())
    L2 = synth.make_layer(2, 64, 32, seed=0)
    assert all(torch.equal(L[k], L2[k]) for k in L)
    g = synth.WORKLOADS["720p_193f"]
    assert g.grid[0] * g.grid[1] * g.grid[2] == g.tokens
    g = synth.WORKLOADS["480p_81f"]
    assert g.grid[0] * g.grid[1] * g.grid[2] == g.tokens


def test_synth_rope_is_a_rotation():
    cos, sin = synth.rope_tables(30, 16, grid=(2, 3, 5))
    assert torch.allclose(cos * cos + sin * sin, torch.ones_like(cos), atol=1e-6)
    cos1, sin1 = synth.rope_tables(8, 16)
    assert torch.equal(cos1[0], torch.ones(8)) and torch.equal(sin1[0], torch.zeros(8))
