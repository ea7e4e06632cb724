"""Pins for the oracle's producer step (ReLU, interleaved RoPE, normaliser): checked
against hand-worked values, torch's own binary32 arithmetic and BF16 rounding, and numpy
FP64 for the normaliser.

Definition (page "PR #35728 完整报告 - [diffusion] Accelerate SANA-Video linear
attention in quality=high", 关键源码片段, snippet sana_video.py): query/key -> ReLU ->
interleaved RoPE (only the rotated copies feed the GEMMs); the normaliser uses the
un-rotated activated copies.  The rotation is fixed to binary32 ops in the order
(x0*c - x1*s, x0*s + x1*c), rounded once to BF16 (nearest-even)."""
import numpy as np
import pytest
import torch

import oracle
from conftest import bf16_bits, bits_to_f64, to_bf16_bits
from video_diffusion_dit_gb300 import synth


def torch_producer(q_bits, k_bits, cos, sin, eps=1e-6):
    """The same definition evaluated with torch CPU ops (separate binary32 products and
    sum, torch's BF16 rounding) - an implementation independent of the oracle's C."""
    def rot(bits):
        x = torch.relu(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float())
        x0, x1 = x[..., 0::2], x[..., 1::2]
        c, s = torch.from_numpy(cos), torch.from_numpy(sin)
        y = torch.empty_like(x)
        y[..., 0::2] = x0 * c - x1 * s
        y[..., 1::2] = x0 * s + x1 * c
        return bf16_bits(y.to(torch.bfloat16))
    qa = np.maximum(bits_to_f64(q_bits), 0.0)
    ka = np.maximum(bits_to_f64(k_bits), 0.0)
    den = np.einsum("hnd,hd->hn", qa, ka.sum(axis=1)) + eps
    return rot(q_bits), rot(k_bits), den


def random_case(H, N, D, seed):
    rng = np.random.default_rng(seed)
    q = to_bf16_bits(torch.randn(H, N, D, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16).double())
    k = to_bf16_bits(torch.randn(H, N, D, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16).double())
    ang = rng.uniform(-50, 50, size=(N, D // 2))
    return q, k, np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),          # subnormals
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -126, 3.3e38, -0.0, np.inf, -np.inf],
                 np.float32),                                             # ties, extremes
    ])
    want = bf16_bits(torch.from_numpy(vals).to(torch.bfloat16))
    assert np.array_equal(oracle.f32_to_bf16(vals), want)


def test_hand_worked_rotation():
    q = to_bf16_bits([[[1.5, 0.5, -2.0, 1.0]]])      # second pair: ReLU turns -2 into 0
    k = to_bf16_bits([[[0.25, 0.75, 1.0, 1.0]]])
    cos = np.array([[0.5, 0.0]], np.float32)
    sin = np.array([[0.25, 1.0]], np.float32)
    q_rot, k_rot, den = oracle.producer(q, k, cos, sin, eps=0.0)
    # pair 0: (1.5*0.5 - 0.5*0.25, 1.5*0.25 + 0.5*0.5) = (0.625, 0.625)
    # pair 1: (0*0 - 1*1, 0*1 + 1*0) = (-1, 0)
    assert np.array_equal(bits_to_f64(q_rot)[0, 0], [0.625, 0.625, -1.0, 0.0])
    # k pair 0: (0.125 - 0.1875, 0.0625 + 0.375) = (-0.0625, 0.4375); pair 1: (-1, 1)
    assert np.array_equal(bits_to_f64(k_rot)[0, 0], [-0.0625, 0.4375, -1.0, 1.0])
    # den = relu(q) . relu(k) = 1.5*0.25 + 0.5*0.75 + 0 + 1*1 = 1.75
    assert den[0, 0] == 1.75


def test_identity_and_quarter_turn():
    q, k, _, _ = random_case(2, 33, 16, 3)
    ones, zeros = np.ones((33, 8), np.float32), np.zeros((33, 8), np.float32)
    q_rot, k_rot, _ = oracle.producer(q, k, ones, zeros)
    assert np.array_equal(bits_to_f64(q_rot), np.maximum(bits_to_f64(q), 0))
    q_rot, _, _ = oracle.producer(q, k, zeros, ones)
    qa = np.maximum(bits_to_f64(q), 0)
    assert np.array_equal(bits_to_f64(q_rot)[..., 0::2], -qa[..., 1::2])
    assert np.array_equal(bits_to_f64(q_rot)[..., 1::2], qa[..., 0::2])


@pytest.mark.parametrize("shape", [(2, 64, 32), (3, 17, 112), (1, 5, 2)])
def test_producer_matches_torch_bit_for_bit(shape):
    q, k, cos, sin = random_case(*shape, seed=sum(shape))
    q_rot, k_rot, den = oracle.producer(q, k, cos, sin)
    tq, tk, tden = torch_producer(q, k, cos, sin)
    assert np.array_equal(q_rot, tq) and np.array_equal(k_rot, tk)
    assert np.allclose(den, tden, rtol=1e-13, atol=0)


def test_producer_reproduces_the_input_generator():
    """The generator forms q_rot/k_rot/den from the same pre-ReLU draws with torch; the
    oracle's producer step must give the same BF16 operands and (to FP32 rounding) den."""
    L = synth.make_layer(2, 300, 48, seed=5, grid=(3, 10, 10), producer_inputs=True)
    q_rot, k_rot, den = oracle.producer(bf16_bits(L["q"][0]), bf16_bits(L["k"][0]),
                                        L["rope_cos"].numpy(), L["rope_sin"].numpy())
    assert np.array_equal(q_rot, bf16_bits(L["q_rot"][0]))
    assert np.array_equal(k_rot, bf16_bits(L["k_rot"][0]))
    assert np.array_equal(den.astype(np.float32), L["den"][0, :, :, 0].numpy())
