"""The softmax anchor layer (lin_attn_anchor_forward) against the FP64 oracle.  The
softmax weights go through BF16 before the second product (as in flash attention), so
both output types are held to rel-L2 <= 4e-3; repeated calls must be bitwise identical."""
import numpy as np
import pytest
import torch

import oracle
from conftest import bf16_bits, rel_l2
from video_diffusion_dit_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 4e-3


@pytest.fixture(scope="module")
def la():
    from video_diffusion_dit_gb300 import lin_attn
    return lin_attn


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def check(la, dev, H, N, D, seed=0, logit_scale=1.0, rows=None, dtypes=(torch.bfloat16, torch.float32)):
    L = synth.make_anchor_layer(H, N, D, seed, logit_scale, device=dev)
    qb, kb, vb = (bf16_bits(L[x][0]) for x in ("q", "k", "v"))
    ref = oracle.softmax_attention_rows(qb, kb, vb, rows=rows)
    with la.LinAttn(H, N, D, dev) as ctx:
        for dt in dtypes:
            out = ctx.anchor_forward(L["q"], L["k"], L["v"], out_dtype=dt)
            assert ctx.device_status() == 0
            got = out.reshape(H * N, D)
            if rows is not None:
                got = got[torch.from_numpy(rows).to(dev)]
            err = rel_l2(got.double().cpu().numpy(), ref)
            assert err <= TOL, f"anchor H={H} N={N} D={D} scale={logit_scale} {dt}: rel-L2 {err:.3e}"
        again = ctx.anchor_forward(L["q"], L["k"], L["v"]).clone()
        assert torch.equal(again, ctx.anchor_forward(L["q"], L["k"], L["v"]))


@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 127, 128, 129, 300, 1000])
def test_anchor_token_counts(la, dev, N):
    check(la, dev, 2, N, 112, seed=N)


@pytest.mark.parametrize("D", [16, 32, 48, 64, 80, 96, 112, 128])
def test_anchor_head_dims(la, dev, D):
    check(la, dev, 3, 257, D, seed=D)


@pytest.mark.parametrize("logit_scale", [4.0, 16.0])
def test_anchor_sharp_softmax_exercises_rescale(la, dev, logit_scale):
    # Large logits: row maxima keep growing across key tiles, forcing O rescales.
    check(la, dev, 2, 2000, 64, seed=3, logit_scale=logit_scale)


def test_anchor_480p_sampled(la, dev):
    w = synth.WORKLOADS["480p_81f"]
    H, N, D = w.heads, w.tokens, w.head_dim
    rows = np.unique(np.concatenate([np.random.default_rng(4).choice(H * N, 512, replace=False),
                                     [0, N - 1, N, H * N - 1]])).astype(np.int64)
    check(la, dev, H, N, D, seed=0, rows=rows, dtypes=(torch.bfloat16,))
