"""Pins for the oracle's second GEMM with FP64 denominators (oracle_apply_rows_f64den), the
reference of every fused-producer parity check: the producer step forms the normaliser's
denominator in FP64 and the layer divides the second product by it (page "PR #35728 完整报告
- [diffusion] Accelerate SANA-Video linear attention in quality=high", 关键源码片段, snippet
sana_video.py: the normaliser from the un-rotated ReLU'd Q and K, then `* normalizer`).

Each pin is fixed by something other than the routine itself: the FP32-denominator routine
(pinned in test_oracle_pins.py) on denominators both routines see exactly, numpy brute force,
a hand-worked example, a first-order closed form that tells an FP64 denominator from one
rounded to FP32, exact power-of-two scaling, and row selection against the full result."""
import json
import os

import numpy as np

import oracle
from conftest import GOLDEN, rel_l2, to_bf16_bits
from test_oracle_pins import brute_force, tiny_inputs


def f64_den(H, N, seed):
    """Denominators that FP32 cannot hold: 1 + u with u having bits below 2^-24."""
    rng = np.random.default_rng(seed)
    return 0.5 + rng.random((H, N)) + rng.random((H, N)) * 2.0 ** -30


def sample_rows(H, N, seed):
    """Rows of the second and last heads (both ends) plus random ones, shuffled."""
    rng = np.random.default_rng(seed)
    rows = np.concatenate([[N, 2 * N - 1, (H - 1) * N, H * N - 1], rng.choice(H * N, 24, replace=False)])
    return rng.permutation(np.unique(rows)).astype(np.int64)


def f64den_pins_hold(lib=None) -> bool:
    # 1. Denominators exact in FP32: the same numbers as the FP32-denominator call, bit for bit.
    qb, kb, vb, den32 = tiny_inputs(seed=21, H=3, N=70, D=16)
    kv = oracle.kv(kb, vb, lib=lib)
    full = oracle.apply_rows(qb, kv, den32.astype(np.float64), lib=lib)
    if not np.array_equal(full, oracle.forward(qb, kb, vb, den32, lib=lib).reshape(-1, 16)):
        return False
    # 2. Row selection: sampled rows (second and last heads included) are those rows of the full result.
    H, N = 3, 70
    den64 = f64_den(H, N, 5)
    full = oracle.apply_rows(qb, kv, den64, lib=lib)
    rows = sample_rows(H, N, 6)
    if not np.array_equal(oracle.apply_rows(qb, kv, den64, rows, lib=lib), full[rows]):
        return False
    # 3. Doubling every denominator halves every output exactly.
    if not np.array_equal(oracle.apply_rows(qb, kv, den64 * 2.0, lib=lib), full / 2.0):
        return False
    # 4. Brute force ((Q K^T) V) / den with numpy on FP64 denominators.
    if rel_l2(full.reshape(H, N, 16), brute_force(qb, kb, vb, den64)) > 1e-12:
        return False
    # 5. The hand-worked example (H=1, N=2, D=2) with its denominators given in FP64.
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    q, k, v = (to_bf16_bits(g[x])[None] for x in ("q_rot", "k_rot", "v"))
    got = oracle.apply_rows(q, oracle.kv(k, v, lib=lib), np.array(g["den"], np.float64)[None], lib=lib)
    if not np.array_equal(got, np.array(g["out"])):
        return False
    # 6. den = 1 + 2^-40 (FP32 would round it to 1): Q.KV = [[6, 10], [2, 4]], so
    #    out = num / (1 + e) = num - num e + O(e^2); the FP64 quotient lies within one ulp of that.
    e = 2.0 ** -40
    got = oracle.apply_rows(q, oracle.kv(k, v, lib=lib), np.full((1, 2), 1.0 + e), lib=lib)
    num = np.array([[6.0, 10.0], [2.0, 4.0]])
    return bool(np.all(got < num) and np.all(np.abs(got - (num - num * e)) <= np.spacing(num)))


def test_f64_denominator_apply_pins():
    assert f64den_pins_hold()


def test_fp32_exact_denominators_match_forward_on_every_row():
    qb, kb, vb, den32 = tiny_inputs(seed=3, H=4, N=129, D=32)
    got = oracle.apply_rows(qb, oracle.kv(kb, vb), den32.astype(np.float64)).reshape(4, 129, 32)
    assert np.array_equal(got, oracle.forward(qb, kb, vb, den32))


def test_sampled_rows_of_second_and_last_heads():
    qb, kb, vb, _ = tiny_inputs(seed=4, H=5, N=64, D=16)
    kv = oracle.kv(kb, vb)
    den64 = f64_den(5, 64, 9)
    full = oracle.apply_rows(qb, kv, den64)
    rows = sample_rows(5, 64, 10)
    assert np.array_equal(oracle.apply_rows(qb, kv, den64, rows), full[rows])


def test_producer_denominators_end_to_end():
    """The whole fused-path reference (producer -> kv -> apply with FP64 den) against numpy:
    ReLU'd un-rotated Q and K form den, the rotated copies form the two products."""
    from test_oracle_producer_pins import random_case
    from conftest import bits_to_f64
    q, k, cos, sin = random_case(2, 40, 16, seed=13)
    v = to_bf16_bits(np.round(np.random.default_rng(14).standard_normal((2, 40, 16)) * 8) / 8)
    q_rot, k_rot, den64 = oracle.producer(q, k, cos, sin)
    got = oracle.apply_rows(q_rot, oracle.kv(k_rot, v), den64).reshape(2, 40, 16)
    qa, ka = np.maximum(bits_to_f64(q), 0), np.maximum(bits_to_f64(k), 0)
    den = np.einsum("hnd,hd->hn", qa, ka.sum(axis=1)) + 1e-6
    qr, kr, vv = bits_to_f64(q_rot), bits_to_f64(k_rot), bits_to_f64(v)
    want = np.einsum("hnm,hmd->hnd", np.einsum("hnd,hmd->hnm", qr, kr), vv) / den[..., None]
    assert rel_l2(got, want) <= 1e-12
