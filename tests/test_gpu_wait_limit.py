"""Bounded barrier waits on the GPU: every wait of the kernels gives up after a limit, winds
the kernel down (copies and tensor-core operations in flight land, tensor memory is freed)
and reports LIN_ATTN_ERR_TIMEOUT through the status word instead of hanging.  The test hook
lin_attn_set_wait_limit shortens the limit to a fraction of a microsecond, so the first
waits for DRAM data run out; nothing faults, traps or spins without a bound.  The context
must stay usable: the next call with the default limit gives bitwise the result of a fresh
context."""
import pytest
import torch

from video_diffusion_dit_gb300 import synth

pytestmark = pytest.mark.gpu

SHORT_NS = 100


@pytest.fixture(scope="module")
def la():
    from video_diffusion_dit_gb300 import lin_attn
    return lin_attn


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def test_wait_limit_argument_checks(la, dev):
    with la.LinAttn(2, 256, 32, dev) as ctx:
        ctx.set_wait_limit(0)
        ctx.set_wait_limit(2_000_000_000)
        with pytest.raises(la.LinAttnError):
            ctx.set_wait_limit(2_000_000_001)
    assert la.lib.lin_attn_set_wait_limit(None, 0) == la.ERR_INVALID_ARG


@pytest.mark.parametrize("call", ["plain", "fused"])
def test_short_wait_limit_reports_timeout_and_context_recovers(la, dev, call):
    w = synth.WORKLOADS["480p_81f"]
    H, N, D = w.heads, w.tokens, w.head_dim
    if call == "plain":
        g = synth.make_workload(w, device=dev)
        run = lambda ctx: ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"])
    else:
        g = synth.make_layer(H, N, D, seed=7, grid=w.grid, device=dev, producer_inputs=True)
        run = lambda ctx: ctx.forward_fused(g["q"], g["k"], g["v"], g["rope_cos"], g["rope_sin"])
    with la.LinAttn(H, N, D, dev) as ctx:
        ctx.set_wait_limit(SHORT_NS)
        run(ctx)
        assert ctx.device_status() == la.ERR_TIMEOUT
        torch.cuda.synchronize()  # no CUDA error: the kernels wound down and exited
        assert ctx.device_status() == la.OK  # the status word was cleared by the read
        ctx.set_wait_limit(0)
        got = run(ctx).clone()
        assert ctx.device_status() == la.OK
    with la.LinAttn(H, N, D, dev) as fresh:
        want = run(fresh)
        assert fresh.device_status() == la.OK
    assert torch.equal(got, want)


def test_short_wait_limit_in_the_anchor_kernel(la, dev):
    H, N, D = 4, 4096, 112
    a = synth.make_anchor_layer(H, N, D, seed=5, logit_scale=2.0)
    g = {k: t.to(dev) for k, t in a.items()}
    with la.LinAttn(H, N, D, dev) as ctx:
        ctx.set_wait_limit(SHORT_NS)
        ctx.anchor_forward(g["q"], g["k"], g["v"])
        assert ctx.device_status() == la.ERR_TIMEOUT
        ctx.set_wait_limit(0)
        got = ctx.anchor_forward(g["q"], g["k"], g["v"]).clone()
        assert ctx.device_status() == la.OK
        want = ctx.anchor_forward(g["q"], g["k"], g["v"])
        assert torch.equal(got, want)
