"""Pins for the oracle's softmax anchor attention (page "[sglang] SANA-Video 2.0 anchor
attention ..." (PR #49219), 코드 분석 §2: F.scaled_dot_product_attention(q, k, v) with no
mask and the default 1/sqrt(D) scale): torch's own float64 SDPA, closed forms (one key,
identical keys, one dominant key), key-permutation invariance, and large logits (which
need the max subtraction)."""
import numpy as np
import pytest
import torch

import oracle
from conftest import bits_to_f64, rel_l2, to_bf16_bits


def bf16_randn(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def torch_sdpa(qb, kb, vb):
    q, k, v = (torch.from_numpy(bits_to_f64(b))[None] for b in (qb, kb, vb))
    return torch.nn.functional.scaled_dot_product_attention(q, k, v)[0].numpy()


@pytest.mark.parametrize("shape,qscale", [((2, 37, 16), 1.0), ((3, 64, 32), 3.0), ((1, 200, 112), 1.0),
                                          ((2, 5, 8), 10.0)])
def test_matches_torch_float64_sdpa(shape, qscale):
    qb, kb, vb = bf16_randn(shape, 1, qscale), bf16_randn(shape, 2), bf16_randn(shape, 3)
    got = oracle.softmax_attention_rows(qb, kb, vb).reshape(shape)
    assert rel_l2(got, torch_sdpa(qb, kb, vb)) <= 1e-12


def test_single_key_returns_its_value():
    qb, kb, vb = bf16_randn((2, 1, 16), 4), bf16_randn((2, 1, 16), 5), bf16_randn((2, 1, 16), 6)
    assert np.array_equal(oracle.softmax_attention_rows(qb, kb, vb).reshape(2, 1, 16), bits_to_f64(vb))


def test_identical_keys_average_the_values():
    H, N, D = 1, 9, 16
    qb = bf16_randn((H, N, D), 7)
    kb = np.repeat(bf16_randn((H, 1, D), 8), N, axis=1)
    vb = to_bf16_bits(np.arange(H * N * D, dtype=np.float64).reshape(H, N, D) / 8.0)
    got = oracle.softmax_attention_rows(qb, kb, vb).reshape(H, N, D)
    want = np.broadcast_to(bits_to_f64(vb).mean(axis=1, keepdims=True), (H, N, D))
    assert np.allclose(got, want, rtol=1e-14, atol=1e-14)


def test_dominant_key_and_large_logits():
    # q = 64 * e0, key 3 = e0 and the rest 0: logits 64/sqrt(D) vs 0 -> weight ~e^-32 elsewhere;
    # scaled up (q = 512 e0) exp() without the max subtraction would overflow.
    H, N, D = 1, 6, 16
    for big in (64.0, 4096.0):
        q = np.zeros((H, N, D)); q[..., 0] = big
        k = np.zeros((H, N, D)); k[0, 3, 0] = 1.0
        vb = bf16_randn((H, N, D), 9)
        got = oracle.softmax_attention_rows(to_bf16_bits(q), to_bf16_bits(k), vb).reshape(H, N, D)
        lead = np.exp(-big / 4.0)  # weight of the other keys relative to key 3
        want = (bits_to_f64(vb)[0, 3] + lead * (bits_to_f64(vb)[0].sum(0) - bits_to_f64(vb)[0, 3])) / (1 + 5 * lead)
        assert np.all(np.isfinite(got))
        assert np.allclose(got[0], np.broadcast_to(want, (N, D)), rtol=1e-12, atol=1e-12)


def test_key_permutation_invariance():
    shape = (2, 50, 32)
    qb, kb, vb = bf16_randn(shape, 10, 2.0), bf16_randn(shape, 11), bf16_randn(shape, 12)
    perm = np.random.default_rng(0).permutation(50)
    a = oracle.softmax_attention_rows(qb, kb, vb)
    b = oracle.softmax_attention_rows(qb, kb[:, perm], vb[:, perm])
    assert rel_l2(b, a) <= 1e-14


def test_selected_rows_match_all_rows():
    shape = (3, 40, 16)
    qb, kb, vb = bf16_randn(shape, 13), bf16_randn(shape, 14), bf16_randn(shape, 15)
    full = oracle.softmax_attention_rows(qb, kb, vb)
    rows = np.array([0, 39, 40, 119], np.int64)
    assert np.array_equal(oracle.softmax_attention_rows(qb, kb, vb, rows=rows), full[rows])
