"""Parity of the CUDA path (through the C ABI) with the FP64 oracle on the same seeded
inputs.  Tolerances: whole-tensor relative L2 <= 2e-5 for FP32 output and <= 4e-3 for
BF16 output; the reduced KV <= 1e-6; repeated calls bitwise identical.  Both quality
tiers have the same exact target, so both are held to the same bounds."""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_l2, whole_and_head_rel_l2
from video_diffusion_dit_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 2e-5, torch.bfloat16: 4e-3}
KV_TOL = 1e-6
MODES = ("high", "lossless")


@pytest.fixture(scope="module")
def la():
    from video_diffusion_dit_gb300 import lin_attn
    return lin_attn


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def to_dev(layer, dev):
    return {k: t.to(dev) for k, t in layer.items()}


def to_token_major(t):
    """[1, H, N, D] -> contiguous [1, N, H, D]."""
    return t.permute(0, 2, 1, 3).contiguous()


def run(ctx, g, mode, dt):
    out = ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"], mode=mode, out_dtype=dt)
    assert ctx.device_status() == 0
    return out


def check_full(la, dev, H, N, D, seed=0, grid=None, modes=MODES, dtypes=(torch.float32, torch.bfloat16)):
    layer = synth.make_layer(H, N, D, seed, grid)
    qb, kb, vb, den = oracle.torch_inputs_to_numpy(layer)
    kv_ref = oracle.kv(kb, vb)
    ref = oracle.apply_rows(qb, kv_ref, den).reshape(H, N, D)
    g = to_dev(layer, dev)
    with la.LinAttn(H, N, D, dev) as ctx:
        for mode in modes:
            for dt in dtypes:
                out = run(ctx, g, mode, dt)
                err = rel_l2(out.double().cpu().numpy()[0], ref)
                assert err <= TOL[dt], f"H={H} N={N} D={D} {mode} {dt}: rel-L2 {err:.3e}"
                kv_err = rel_l2(ctx.debug_kv().double().cpu().numpy(), kv_ref)
                assert kv_err <= KV_TOL, f"H={H} N={N} D={D} {mode}: KV rel-L2 {kv_err:.3e}"


def test_worked_example_bit_exact(la, dev):
    q = torch.zeros(1, 1, 2, 16, dtype=torch.bfloat16)
    k, v = torch.zeros_like(q), torch.zeros_like(q)
    q[0, 0, :, :2] = torch.tensor([[1.0, 1.0], [2.0, 0.0]])
    k[0, 0, :, :2] = torch.tensor([[1.0, 2.0], [0.0, 1.0]])
    v[0, 0, :, :2] = torch.tensor([[1.0, 2.0], [3.0, 4.0]])
    den = torch.tensor([2.0, 4.0]).reshape(1, 1, 2, 1)
    want = torch.zeros(1, 1, 2, 16, dtype=torch.float64)
    want[0, 0, :, :2] = torch.tensor([[3.0, 5.0], [0.5, 1.0]])
    with la.LinAttn(1, 2, 16, dev) as ctx:
        for mode in MODES:
            for dt in (torch.float32, torch.bfloat16):
                out = ctx.forward(q.to(dev), k.to(dev), v.to(dev), den.to(dev), mode=mode, out_dtype=dt)
                assert torch.equal(out.double().cpu(), want), (mode, dt, out)
                kv = ctx.debug_kv().cpu()
                assert torch.equal(kv[0, :2, :2], torch.tensor([[1.0, 2.0], [5.0, 8.0]]))


def test_tiny_config(la, dev):
    check_full(la, dev, 2, 256, 32)


@pytest.mark.parametrize("D", [16, 32, 48, 64, 80, 96, 112, 128])
def test_head_dims(la, dev, D):
    check_full(la, dev, 3, 777, D, seed=D)


@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 127, 128, 129, 1000, 4097])
def test_ragged_token_counts(la, dev, N):
    check_full(la, dev, 2, N, 112, seed=N)


def test_many_heads_d64(la, dev):
    check_full(la, dev, 32, 3000, 64, seed=5)


def test_480p_full_all_modes(la, dev):
    w = synth.WORKLOADS["480p_81f"]
    check_full(la, dev, w.heads, w.tokens, w.head_dim, w.seed, w.grid)


def check_whole(out, ref, dt, what):
    """Whole-tensor and per-head relative L2 of a full-size result against the oracle."""
    whole, head = whole_and_head_rel_l2(out, ref)
    assert whole <= TOL[dt] and head <= TOL[dt], f"{what}: rel-L2 {whole:.3e}, worst head {head:.3e}"


@pytest.mark.parametrize("name", ["720p_193f", "720p_193f_d64"])
def test_full_size_whole_tensor(la, dev, name):
    """Full-size layer in the bench's launch configuration, every output element against the
    oracle, both tiers and output types; the token-major call on the same data gives the
    same bits as the head-major call."""
    w = synth.WORKLOADS[name]
    H, N, D = w.heads, w.tokens, w.head_dim
    layer = synth.make_workload(w, device=dev)
    qb, kb, vb, den = oracle.torch_inputs_to_numpy(layer)
    kv_ref = oracle.kv(kb, vb)
    ref = torch.from_numpy(oracle.apply_rows(qb, kv_ref, den).reshape(H, N, D)).to(dev)
    tm = {k: to_token_major(layer[k]) for k in ("q_rot", "k_rot", "v")}
    with la.LinAttn(H, N, D, dev) as ctx:
        for mode in MODES:
            for dt in (torch.float32, torch.bfloat16):
                out = run(ctx, layer, mode, dt)
                check_whole(out, ref, dt, f"{name} {mode} {dt}")
                kv_err = rel_l2(ctx.debug_kv().double().cpu().numpy(), kv_ref)
                assert kv_err <= KV_TOL, f"{name} {mode}: KV rel-L2 {kv_err:.3e}"
                nhd = ctx.forward(tm["q_rot"], tm["k_rot"], tm["v"], layer["den"], mode=mode, out_dtype=dt,
                                  layout="nhd")
                assert ctx.device_status() == 0
                assert torch.equal(nhd.view(1, N, H, D), to_token_major(out)), (name, mode, dt)
                del out, nhd


@pytest.mark.parametrize("n", synth.SWEEP_TOKENS)
def test_token_sweep_whole_tensor(la, dev, n):
    """The N sweep at H=20, D=112 and at H=32, D=64: every output element and the KV against
    the oracle (FP32 output in both tiers; BF16 output too at N = 65536)."""
    for name in (f"sweep_n{n}", f"sweep_n{n}_d64"):
        w = synth.WORKLOADS[name]
        H, N, D = w.heads, w.tokens, w.head_dim
        layer = synth.make_workload(w, device=dev)
        qb, kb, vb, den = oracle.torch_inputs_to_numpy(layer)
        kv_ref = oracle.kv(kb, vb)
        ref = torch.from_numpy(oracle.apply_rows(qb, kv_ref, den).reshape(H, N, D)).to(dev)
        dtypes = (torch.float32, torch.bfloat16) if n == 65536 else (torch.float32,)
        with la.LinAttn(H, N, D, dev) as ctx:
            for mode in MODES:
                for dt in dtypes:
                    check_whole(run(ctx, layer, mode, dt), ref, dt, f"{name} {mode} {dt}")
                assert rel_l2(ctx.debug_kv().double().cpu().numpy(), kv_ref) <= KV_TOL, (name, mode)


def test_denoise_step_twenty_layers(la, dev):
    """20 sequential layer calls at the 720p shape with fresh seeded inputs per layer on one
    context (the scratch is reused call after call); the first and last layers are held to
    the oracle on every output element, every call must finish with a clean status."""
    w = synth.WORKLOADS["720p_193f"]
    H, N, D = w.heads, w.tokens, w.head_dim
    out = torch.empty(1, H, N, D, device=dev)
    with la.LinAttn(H, N, D, dev) as ctx:
        for mode in MODES:
            for layer_idx in range(synth.DENOISE_LAYERS):
                layer = synth.make_layer(H, N, D, seed=layer_idx, grid=w.grid, device=dev)
                ctx.forward(layer["q_rot"], layer["k_rot"], layer["v"], layer["den"], out=out, mode=mode)
                if layer_idx in (0, synth.DENOISE_LAYERS - 1):
                    assert ctx.device_status() == 0
                    qb, kb, vb, den = oracle.torch_inputs_to_numpy(layer)
                    ref = oracle.apply_rows(qb, oracle.kv(kb, vb), den).reshape(H, N, D)
                    check_whole(out, ref, torch.float32, f"denoise {mode} layer {layer_idx}")
            assert ctx.device_status() == 0


@pytest.mark.parametrize("mode", MODES)
def test_bitwise_deterministic(la, dev, mode):
    w = synth.WORKLOADS["480p_81f"]
    g = synth.make_workload(w, device=dev)
    with la.LinAttn(w.heads, w.tokens, w.head_dim, dev) as ctx:
        a = run(ctx, g, mode, torch.float32).clone()
        kva = ctx.debug_kv()
        # a different call in between must leave no trace
        run(ctx, to_dev(synth.make_layer(w.heads, 5000, w.head_dim, 3), dev), mode, torch.bfloat16)
        b = run(ctx, g, mode, torch.float32)
        assert torch.equal(a, b)
        assert torch.equal(kva, ctx.debug_kv())


@pytest.mark.parametrize("mode", MODES)
def test_zero_v_gives_zero(la, dev, mode):
    g = to_dev(synth.make_layer(2, 1000, 112, 4), dev)
    g["v"].zero_()
    with la.LinAttn(2, 1000, 112, dev) as ctx:
        out = run(ctx, g, mode, torch.float32)
        assert torch.count_nonzero(out).item() == 0


def test_modes_agree_closely(la, dev):
    g = to_dev(synth.make_layer(4, 5000, 112, 6), dev)
    with la.LinAttn(4, 5000, 112, dev) as ctx:
        hi = run(ctx, g, "high", torch.float32).double()
        lo = run(ctx, g, "lossless", torch.float32).double()
    assert (torch.linalg.norm(hi - lo) / torch.linalg.norm(lo)).item() <= 4e-5


def test_host_buffer_path_matches_device_path(la, dev):
    layer = synth.make_layer(3, 2000, 112, 8)
    pinned = {k: t.pin_memory() for k, t in layer.items()}
    g = to_dev(layer, dev)
    with la.LinAttn(3, 4000, 112, dev) as ctx:
        for mode in MODES:
            for dt in (torch.float32, torch.bfloat16):
                d = run(ctx, g, mode, dt).cpu()
                h = ctx.forward_host(pinned["q_rot"], pinned["k_rot"], pinned["v"], pinned["den"], mode=mode,
                                     out_dtype=dt)
                assert torch.equal(d, h)
        # pageable host memory works too
        h2 = ctx.forward_host(layer["q_rot"], layer["k_rot"], layer["v"], layer["den"], out=torch.empty(
            1, 3, 2000, 112))
        assert torch.equal(h2, run(ctx, g, "high", torch.float32).cpu())


def test_host_pipeline_uneven_chunks_bitwise(la, dev):
    """20 heads run as chunks of 3 (the last one holds 2): the pipelined host path must give
    bitwise what the device path gives, in both tiers."""
    layer = synth.make_layer(20, 3001, 112, 12)
    pinned = {k: t.pin_memory() for k, t in layer.items()}
    g = to_dev(layer, dev)
    with la.LinAttn(20, 3001, 112, dev) as ctx:
        for mode in MODES:
            d = run(ctx, g, mode, torch.float32).cpu()
            for _ in range(2):
                h = ctx.forward_host(pinned["q_rot"], pinned["k_rot"], pinned["v"], pinned["den"], mode=mode)
                assert torch.equal(d, h)
            assert ctx.device_status() == 0


def test_host_pipeline_with_shared_tails_bitwise(la, dev):
    """A length where the KV split hands the tails of all heads to the spare CTAs (152
    chunks at H = 20): the host path launches one head at a time, each launch running the
    body chunks of its head and the tail chunks that touch it, clipped to it; the partial
    sums, so the result, must be bitwise those of the whole-layer call, in both tiers."""
    H, N, D = 20, 120000, 112
    assert la.kv_plan(H, N) == (152, 9)
    g = synth.make_layer(H, N, D, 21, device=dev)
    pinned = {k: t.cpu().pin_memory() for k, t in g.items()}
    with la.LinAttn(H, N, D, dev) as ctx:
        for mode in MODES:
            d = run(ctx, g, mode, torch.float32).cpu()
            h = ctx.forward_host(pinned["q_rot"], pinned["k_rot"], pinned["v"], pinned["den"], mode=mode)
            assert torch.equal(d, h), mode
            assert ctx.device_status() == 0


def test_out_of_range_and_misaligned_calls_are_rejected(la, dev):
    import ctypes
    g = to_dev(synth.make_layer(2, 256, 32, 0), dev)
    with la.LinAttn(2, 256, 32, dev) as ctx:
        out = torch.empty(1, 2, 256, 32, device=dev)
        h = ctx._h
        args = [g["q_rot"].data_ptr(), g["k_rot"].data_ptr(), g["v"].data_ptr(), g["den"].data_ptr(),
                out.data_ptr()]
        s = torch.cuda.current_stream().cuda_stream
        assert la.lib.lin_attn_forward(h, *args, 0, 257, 0, s) == la.ERR_INVALID_ARG
        assert la.lib.lin_attn_forward(h, *args, 0, 0, 0, s) == la.ERR_INVALID_ARG
        assert la.lib.lin_attn_forward(h, *args, 2, 256, 0, s) == la.ERR_INVALID_ARG
        assert la.lib.lin_attn_forward(h, *args, 0, 256, 5, s) == la.ERR_INVALID_ARG
        bad = list(args)
        bad[1] += 2
        assert la.lib.lin_attn_forward(h, *bad, 0, 256, 0, s) == la.ERR_MISALIGNED
        with pytest.raises(ValueError):
            ctx.forward(g["q_rot"].cpu(), g["k_rot"], g["v"], g["den"])
        with pytest.raises(la.LinAttnError) as exc:
            ctx.forward(*(synth.make_layer(2, 257, 32, 0)[k].to(dev) for k in ("q_rot", "k_rot", "v", "den")))
        assert exc.value.status == la.ERR_INVALID_ARG
        # a valid call still works afterwards
        run(ctx, g, "high", torch.float32)
        assert ctx.device_status() == 0


def test_stage_events(la, dev):
    g = to_dev(synth.make_layer(4, 20000, 112, 2), dev)
    with la.LinAttn(4, 20000, 112, dev) as ctx:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ctx.set_stage_events(ev)
        run(ctx, g, "high", torch.float32)
        torch.cuda.synchronize()
        t = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
        assert all(x >= 0 for x in t) and sum(t) > 0


@pytest.mark.parametrize("N", [3000, 1000, 2080, 4127])
def test_ragged_tail_stores_repeated(la, dev, N):
    """Ragged last tiles where whole 32-row boxes lie past the end of a head: the apply
    epilogue must not recycle a staging buffer whose store is still in flight.  The race
    this guards against was intermittent, so the call is repeated."""
    H, D = 24, 112 if N % 2 else 64
    layer = synth.make_layer(H, N, D, seed=N)
    qb, kb, vb, den = oracle.torch_inputs_to_numpy(layer)
    ref = oracle.forward(qb, kb, vb, den)
    g = to_dev(layer, dev)
    with la.LinAttn(H, N, D, dev) as ctx:
        for dt in (torch.float32, torch.bfloat16):
            first = run(ctx, g, "high", dt).clone()
            err = rel_l2(first.double().cpu().numpy()[0], ref)
            assert err <= TOL[dt], f"N={N} {dt}: rel-L2 {err:.3e}"
            for _ in range(8):
                assert torch.equal(run(ctx, g, "high", dt), first)


@pytest.mark.parametrize("shape", [(20, 3001, 112), (3, 777, 64), (2, 256, 32), (5, 129, 128)])
def test_token_major_layout(la, dev, shape):
    """The page-native layout: [1, N, H, D] activations in, [1, N, H*D] out.  Same numbers as
    the head-major call, bitwise, in both tiers and output types; checked against the oracle."""
    H, N, D = shape
    layer = synth.make_layer(H, N, D, seed=N)
    qb, kb, vb, den = oracle.torch_inputs_to_numpy(layer)
    ref = oracle.forward(qb, kb, vb, den)
    g = to_dev(layer, dev)
    tm = {k: to_token_major(g[k]) for k in ("q_rot", "k_rot", "v")}
    with la.LinAttn(H, N, D, dev) as ctx:
        for mode in MODES:
            for dt in (torch.float32, torch.bfloat16):
                hm = run(ctx, g, mode, dt)
                out = ctx.forward(tm["q_rot"], tm["k_rot"], tm["v"], g["den"], mode=mode, out_dtype=dt, layout="nhd")
                assert ctx.device_status() == 0
                assert tuple(out.shape) == (1, N, H * D)
                assert torch.equal(out.view(1, N, H, D), to_token_major(hm)), (mode, dt)
                err = rel_l2(out.view(N, H, D).permute(1, 0, 2).double().cpu().numpy(), ref)
                assert err <= TOL[dt], (mode, dt, err)
