"""The fused producer path (lin_attn_forward_fused): ReLU, interleaved RoPE and the
normaliser computed inside the kernels from the pre-activation q, k and FP32 rotation
tables.  Held to the FP64 oracle (its producer step, then the layer) with the same
tolerances as the plain call; and because the rotation is defined bit for bit, the reduced
KV must equal, bitwise, the KV the plain call forms from the generator's Q_rot/K_rot."""
import pytest
import torch

import oracle
from conftest import bf16_bits, rel_l2, whole_and_head_rel_l2
from video_diffusion_dit_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 2e-5, torch.bfloat16: 4e-3}


@pytest.fixture(scope="module")
def la():
    from video_diffusion_dit_gb300 import lin_attn
    return lin_attn


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def oracle_fused(layer, rows=None):
    """Producer step then the layer, all on the oracle; rows = flat sample or None (all)."""
    q, k = bf16_bits(layer["q"][0]), bf16_bits(layer["k"][0])
    q_rot, k_rot, den = oracle.producer(q, k, layer["rope_cos"].cpu().numpy(), layer["rope_sin"].cpu().numpy())
    kv = oracle.kv(k_rot, bf16_bits(layer["v"][0]))
    out = oracle.apply_rows(q_rot, kv, den, rows)
    return out, kv


def check(la, dev, H, N, D, seed, grid=None, dtypes=(torch.float32, torch.bfloat16)):
    layer = synth.make_layer(H, N, D, seed, grid, producer_inputs=True)
    ref, kv_ref = oracle_fused(layer)
    ref = ref.reshape(H, N, D)
    g = {key: t.to(dev) for key, t in layer.items()}
    with la.LinAttn(H, N, D, dev) as ctx:
        for dt in dtypes:
            out = ctx.forward_fused(g["q"], g["k"], g["v"], g["rope_cos"], g["rope_sin"], out_dtype=dt)
            assert ctx.device_status() == 0
            err = rel_l2(out.double().cpu().numpy()[0], ref)
            assert err <= TOL[dt], f"fused H={H} N={N} D={D} {dt}: rel-L2 {err:.3e}"
        kv_fused = ctx.debug_kv().clone()
        assert rel_l2(kv_fused.double().cpu().numpy(), kv_ref) <= 1e-6
        # The plain call on the generator's rotated operands forms bitwise the same KV.
        plain = ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"])
        assert torch.equal(ctx.debug_kv(), kv_fused)
        fused = ctx.forward_fused(g["q"], g["k"], g["v"], g["rope_cos"], g["rope_sin"])
        # Only the denominators differ (FP32 in the kernel vs FP64 -> FP32 in the generator).
        assert rel_l2(fused.double().cpu().numpy(), plain.double().cpu().numpy()) <= 1e-6


@pytest.mark.parametrize("shape", [(2, 256, 32), (3, 777, 112), (2, 1000, 64), (4, 129, 128), (1, 1, 16),
                                   (2, 65, 48)])
def test_fused_small(la, dev, shape):
    check(la, dev, *shape, seed=shape[1])


@pytest.mark.parametrize("shape", [(3, 777, 112), (2, 1000, 64), (4, 129, 128), (2, 65, 48)])
def test_fused_token_major_is_bitwise_the_head_major_call(la, dev, shape):
    # The model's projection layout [1, N, H, D] in, [1, N, H*D] out: the same plan and the
    # same per-token arithmetic, so the same bits as the head-major fused call.
    H, N, D = shape
    g = {key: t.to(dev) for key, t in synth.make_layer(H, N, D, N + 1, producer_inputs=True).items()}
    nhd = {key: g[key].permute(0, 2, 1, 3).contiguous() for key in ("q", "k", "v")}
    with la.LinAttn(H, N, D, dev) as ctx:
        for dt in (torch.float32, torch.bfloat16):
            ref = ctx.forward_fused(g["q"], g["k"], g["v"], g["rope_cos"], g["rope_sin"], out_dtype=dt).clone()
            kv_ref = ctx.debug_kv().clone()
            out = ctx.forward_fused(nhd["q"], nhd["k"], nhd["v"], g["rope_cos"], g["rope_sin"], out_dtype=dt,
                                    layout="nhd")
            assert ctx.device_status() == 0
            assert tuple(out.shape) == (1, N, H * D)
            assert torch.equal(ctx.debug_kv(), kv_ref)
            assert torch.equal(out.reshape(1, N, H, D).permute(0, 2, 1, 3), ref)


def test_fused_480p(la, dev):
    w = synth.WORKLOADS["480p_81f"]
    check(la, dev, w.heads, w.tokens, w.head_dim, w.seed, w.grid, dtypes=(torch.float32,))


@pytest.mark.parametrize("name", ["720p_193f", "720p_193f_d64"])
def test_fused_720p_whole_tensor(la, dev, name):
    """The full 720p layer (and its D=64, H=32 shape) through the fused call, every output
    element against the oracle, both tiers and output types; the model's token-major layout
    gives the same bits; repeated calls are bitwise identical."""
    w = synth.WORKLOADS[name]
    H, N, D = w.heads, w.tokens, w.head_dim
    layer = synth.make_workload(w, device=dev, producer_inputs=True)
    ref, kv_ref = oracle_fused(layer)
    ref = torch.from_numpy(ref.reshape(H, N, D)).to(dev)
    nhd = {key: layer[key].permute(0, 2, 1, 3).contiguous() for key in ("q", "k", "v")}
    tabs = (layer["rope_cos"], layer["rope_sin"])
    with la.LinAttn(H, N, D, dev) as ctx:
        for mode in ("high", "lossless"):
            for dt in (torch.float32, torch.bfloat16):
                out = ctx.forward_fused(layer["q"], layer["k"], layer["v"], *tabs, out_dtype=dt, mode=mode)
                assert ctx.device_status() == 0
                whole, head = whole_and_head_rel_l2(out, ref)
                assert whole <= TOL[dt] and head <= TOL[dt], f"fused {name} {mode} {dt}: {whole:.3e} / {head:.3e}"
                assert rel_l2(ctx.debug_kv().double().cpu().numpy(), kv_ref) <= 1e-6
                tm = ctx.forward_fused(nhd["q"], nhd["k"], nhd["v"], *tabs, out_dtype=dt, mode=mode, layout="nhd")
                assert ctx.device_status() == 0
                assert torch.equal(tm.reshape(1, N, H, D).permute(0, 2, 1, 3), out), (mode, dt)
                del out, tm
        again = ctx.forward_fused(layer["q"], layer["k"], layer["v"], *tabs).clone()
        third = ctx.forward_fused(layer["q"], layer["k"], layer["v"], *tabs)
        assert torch.equal(again, third)


def test_fused_rejects_bad_arguments(la, dev):
    g = {k: t.to(dev) for k, t in synth.make_layer(2, 64, 32, 0, producer_inputs=True).items()}
    with la.LinAttn(2, 64, 32, dev) as ctx:
        out = torch.empty(1, 2, 64, 32, device=dev)
        s = torch.cuda.current_stream().cuda_stream
        args = [g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), g["rope_cos"].data_ptr(),
                g["rope_sin"].data_ptr(), out.data_ptr(), la.OUT_F32, 64]
        assert la.lib.lin_attn_forward_fused(ctx._h, *args, 7, s) == la.ERR_INVALID_ARG
        assert la.lib.lin_attn_forward_fused_layout(ctx._h, *args, la.MODE_HIGH, 5, s) == la.ERR_INVALID_ARG
        bad = list(args)
        bad[3] = 0
        assert la.lib.lin_attn_forward_fused(ctx._h, *bad, la.MODE_HIGH, s) == la.ERR_INVALID_ARG
        with pytest.raises(ValueError):
            ctx.forward_fused(g["q"], g["k"], g["v"], g["rope_cos"][:32], g["rope_sin"])
        assert ctx.device_status() == 0


@pytest.mark.parametrize("shape", [(3, 777, 112), (2, 1000, 64), (4, 129, 128)])
def test_fused_lossless(la, dev, shape):
    # The 'lossless' tier with the producer step fused in: the oracle's numbers within the
    # same tolerances, and bitwise the KV of the plain lossless call on the generator's
    # rotated operands (the rotation is defined bit for bit).
    H, N, D = shape
    layer = synth.make_layer(H, N, D, 7 * N, producer_inputs=True)
    ref, kv_ref = oracle_fused(layer)
    ref = ref.reshape(H, N, D)
    g = {key: t.to(dev) for key, t in layer.items()}
    with la.LinAttn(H, N, D, dev) as ctx:
        for dt in (torch.float32, torch.bfloat16):
            out = ctx.forward_fused(g["q"], g["k"], g["v"], g["rope_cos"], g["rope_sin"], out_dtype=dt,
                                    mode="lossless")
            assert ctx.device_status() == 0
            err = rel_l2(out.double().cpu().numpy()[0], ref)
            assert err <= TOL[dt], f"fused lossless H={H} N={N} D={D} {dt}: rel-L2 {err:.3e}"
        kv_fused = ctx.debug_kv().clone()
        assert rel_l2(kv_fused.double().cpu().numpy(), kv_ref) <= 1e-6
        ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"], mode="lossless")
        assert torch.equal(ctx.debug_kv(), kv_fused)


@pytest.mark.parametrize("shape", [(5, 3001, 112), (3, 777, 64), (20, 120000, 112)])
def test_fused_host_buffers_are_bitwise_the_device_call(la, dev, shape):
    # The host-buffer form pipelines the copies over chunks of heads; every chunk runs the
    # layer's own split, so its result is the device call's bits.  (20, 120000): the spare
    # CTAs share the tails of all heads, so the chunks' launches reproduce shared segments.
    H, N, D = shape
    layer = synth.make_layer(H, N, D, 11 * N + H, producer_inputs=True)
    keys = ("q", "k", "v", "rope_cos", "rope_sin")
    host = {key: layer[key].contiguous().pin_memory() for key in keys}
    g = {key: layer[key].to(dev) for key in keys}
    with la.LinAttn(H, N, D, dev) as ctx:
        for mode in ("high", "lossless"):
            for dt in (torch.float32, torch.bfloat16):
                want = ctx.forward_fused(g["q"], g["k"], g["v"], g["rope_cos"], g["rope_sin"], out_dtype=dt,
                                         mode=mode).cpu()
                got = ctx.forward_fused_host(host["q"], host["k"], host["v"], host["rope_cos"], host["rope_sin"],
                                             out_dtype=dt, mode=mode)
                assert ctx.device_status() == 0
                assert torch.equal(got, want), (mode, dt)
        bad = [host["q"].data_ptr(), host["k"].data_ptr(), host["v"].data_ptr(), 0, host["rope_sin"].data_ptr(),
               got.data_ptr(), la.OUT_BF16, N, la.MODE_HIGH, torch.cuda.current_stream().cuda_stream]
        assert la.lib.lin_attn_forward_fused_host(ctx._h, *bad) == la.ERR_INVALID_ARG
