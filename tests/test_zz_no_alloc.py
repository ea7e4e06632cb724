"""lin_attn_forward_noalloc: the layer call for callers that cannot allocate device memory
(a plugin host that forbids allocation in its execute callback, a process whose device
memory is reserved up front by a caching allocator or a memory cap, a latency-critical
loop that must not pay cudaMalloc's implicit synchronisation).  Its scratch is a fixed
array inside the library.

It is called here through the C ABI on two calls in a row with different shapes (the second
one finds the first one's data still in the shared array).  It runs the same work split,
kernels and grid as the context entry point, so its output must be the same bits; both are
also held to the oracle at the parity tolerance.

This file is named to be collected last, so a failure here comes after every other test
has already run; it also passes alone in a fresh process (its first call sets the
device up)."""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_l2
from video_diffusion_dit_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 2e-5, torch.bfloat16: 4e-3}
SCRATCH_BYTES = 48 << 20


@pytest.fixture(scope="module")
def la():
    from video_diffusion_dit_gb300 import lin_attn
    return lin_attn


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def noalloc_call(la, g, mode, dt):
    _, H, N, D = g["q_rot"].shape
    out = torch.empty(1, H, N, D, dtype=dt, device=g["q_rot"].device)
    st = la.lib.lin_attn_forward_noalloc(
        g["q_rot"].data_ptr(), g["k_rot"].data_ptr(), g["v"].data_ptr(), g["den"].data_ptr(), out.data_ptr(),
        la.OUT_BF16 if dt == torch.bfloat16 else la.OUT_F32, H, N, D,
        la.MODE_HIGH if mode == "high" else la.MODE_LOSSLESS, torch.cuda.current_stream().cuda_stream)
    assert st == la.OK, la.lib.lin_attn_last_error()
    return out


def context_call(la, g, mode, dt, dev):
    _, H, N, D = g["q_rot"].shape
    with la.LinAttn(H, N, D, dev) as ctx:
        out = ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"], mode=mode, out_dtype=dt)
        assert ctx.device_status() == 0
        return out


def scratch_bytes(la, H, N, D):
    """Scratch the call needs: a status word, k partial slots per head of FP32 D x D sums,
    the reduced KV and the three-term KV image, each rounded up to 256 bytes."""
    _, k = la.kv_plan(H, N)
    up = lambda x: (x + 255) // 256 * 256
    return up(4 * D * D * H * k) + up(4 * D * D * H) + up(H * 3 * -(-D // 64) * D * 128) + 256


@pytest.mark.parametrize("mode", ["high", "lossless"])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_two_calls_in_a_row_match_the_context_path(la, dev, mode, dt):
    w = synth.WORKLOADS["480p_81f"]
    layers = [synth.make_workload(w, device=dev), synth.make_layer(6, 3000, 32, seed=1, device=dev)]
    for g in layers:
        got = noalloc_call(la, g, mode, dt)
        torch.cuda.synchronize()
        want = context_call(la, g, mode, dt, dev)
        assert torch.equal(got, want), f"{mode} {dt} {tuple(g['q_rot'].shape)}: not bitwise the context call"
        assert la.noalloc_status(dev) == la.OK  # no kernel of the call gave up waiting
        qb, kb, vb, den = oracle.torch_inputs_to_numpy(g)
        ref = oracle.forward(qb, kb, vb, den)
        err = rel_l2(got.double().cpu().numpy()[0], ref)
        assert err <= TOL[dt], f"{mode} {dt} {tuple(g['q_rot'].shape)}: rel-L2 {err:.3e} against the oracle"


def test_shared_tail_plan_matches_the_context_path(la, dev):
    """A length where the spare CTAs share the tails of all heads (9 partial slots per head):
    the scratch is carved for that many slots and the result is the context call's bits."""
    H, N, D = 20, 120000, 112
    assert la.kv_plan(H, N) == (152, 9)
    g = synth.make_layer(H, N, D, seed=23, device=dev)
    for mode in ("high", "lossless"):
        got = noalloc_call(la, g, mode, torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(got, context_call(la, g, mode, torch.float32, dev)), mode
        assert la.noalloc_status(dev) == la.OK


def test_scratch_limit_boundary(la, dev):
    """At head dim 128 with one partial slot per head the 48 MiB array holds 219 heads: 219 is
    accepted (and gives the context call's bits), 220 is refused before any launch."""
    N, D = 64, 128
    assert scratch_bytes(la, 219, N, D) <= SCRATCH_BYTES < scratch_bytes(la, 220, N, D)
    g = synth.make_layer(219, N, D, seed=3, device=dev)
    got = noalloc_call(la, g, "high", torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(got, context_call(la, g, "high", torch.float32, dev))
    p = torch.empty(16, dtype=torch.uint8, device=dev).data_ptr()
    st = la.lib.lin_attn_forward_noalloc(p, p, p, p, p, la.OUT_F32, 220, N, D, la.MODE_HIGH,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == la.ERR_INVALID_ARG
    assert b"scratch" in la.lib.lin_attn_last_error()


def test_shape_beyond_the_fixed_scratch_is_rejected(la, dev):
    p = torch.empty(16, dtype=torch.uint8, device=dev).data_ptr()
    # 1024 heads get 1 partial slot each (k = max(1, 152 // 1024)); 128^2 FP32 partials x 1024
    # heads are 64 MiB alone.  Nothing is read: the call is refused before any launch.
    assert scratch_bytes(la, 1024, 4096, 128) > SCRATCH_BYTES
    st = la.lib.lin_attn_forward_noalloc(p, p, p, p, p, la.OUT_F32, 1024, 4096, 128, la.MODE_HIGH,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == la.ERR_INVALID_ARG
    assert b"scratch" in la.lib.lin_attn_last_error()


def test_binding_refuses_tensors_off_the_inputs_device(la, dev):
    g = synth.make_layer(2, 256, 32, seed=4, device=dev)
    out = torch.empty(1, 2, 256, 32, device=dev)
    with pytest.raises(ValueError):
        la.forward_noalloc(g["q_rot"], g["k_rot"], g["v"], g["den"].cpu(), out)
    with pytest.raises(ValueError):
        la.forward_noalloc(g["q_rot"], g["k_rot"], g["v"], g["den"], out.cpu())
    with pytest.raises(TypeError):
        la.forward_noalloc(g["q_rot"], g["k_rot"], g["v"], g["den"], out.half())
    got = la.forward_noalloc(g["q_rot"], g["k_rot"], g["v"], g["den"], out)
    torch.cuda.synchronize()
    assert torch.equal(got, context_call(la, g, "high", torch.float32, dev))
