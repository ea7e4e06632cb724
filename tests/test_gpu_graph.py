"""Stream behaviour of the layer calls.  They put only stream work on the caller's stream
(kernel launches with programmatic dependencies, no host synchronisation, no allocation),
so a sequence of them can be captured into a CUDA graph: replayed, the graph gives the
eager calls' bits.  Contexts share no device state, so two of them may run at once."""
import pytest
import torch

from video_diffusion_dit_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    from video_diffusion_dit_gb300 import lin_attn
    return lin_attn


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def test_layer_calls_replay_from_a_cuda_graph(la, dev):
    H, N, D = 4, 20000, 112
    layers = [{k: t.to(dev) for k, t in synth.make_layer(H, N, D, seed, producer_inputs=True).items()}
              for seed in (31, 32)]
    with la.LinAttn(H, N, D, dev) as ctx:
        s = torch.cuda.Stream(dev)

        def calls(outs, stream):
            for g, o in zip(layers, outs[:2]):
                ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"], out=o, stream=stream)
            g = layers[0]
            ctx.forward_fused(g["q"], g["k"], g["v"], g["rope_cos"], g["rope_sin"], out=outs[2], stream=stream)
            ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"], out=outs[3], stream=stream, mode="lossless",
                        layout="hnd")

        want = [torch.empty(1, H, N, D, device=dev) for _ in range(4)]
        with torch.cuda.stream(s):
            calls(want, s)
        torch.cuda.synchronize()
        assert ctx.device_status() == la.OK

        got = [torch.zeros(1, H, N, D, device=dev) for _ in range(4)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            calls(got, torch.cuda.current_stream())
        for o in got:
            o.zero_()
        torch.cuda.synchronize()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        assert ctx.device_status() == la.OK
        for o, w in zip(got, want):
            assert torch.equal(o, w)


def test_two_contexts_on_two_streams_at_once(la, dev):
    """Each context owns its scratch: two contexts running on two streams at the same time
    give the bits each gives alone."""
    H, N, D = 6, 30000, 112
    layers = [{k: t.to(dev) for k, t in synth.make_layer(H, N, D, seed).items()} for seed in (41, 42)]
    with la.LinAttn(H, N, D, dev) as a, la.LinAttn(H, N, D, dev) as b:
        alone = []
        for ctx, g in zip((a, b), layers):
            alone.append(ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"]).clone())
        torch.cuda.synchronize()
        streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        outs = [torch.zeros(1, H, N, D, device=dev) for _ in range(2)]
        for _ in range(3):
            for ctx, g, s, o in zip((a, b), layers, streams, outs):
                ctx.forward(g["q_rot"], g["k_rot"], g["v"], g["den"], out=o, stream=s)
        torch.cuda.synchronize()
        assert a.device_status() == la.OK and b.device_status() == la.OK
        for o, w in zip(outs, alone):
            assert torch.equal(o, w)
