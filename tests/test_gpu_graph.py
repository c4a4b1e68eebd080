"""Layer steps replayed from CUDA graphs (MoELayer.capture_step) against the
same steps run call by call: the outputs, the loads and the bias trajectory
must agree bit for bit, step after step, since a replay launches the same
kernels on the same buffers."""
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("name,steps", [("tiny", 6), ("mid", 4)])
def test_graph_replay_matches_eager_steps(name, steps):
    cfg = synth.CONFIGS[name]
    p = synth.make_params(cfg, "cuda")
    layer = MoELayer(cfg, p)
    xs = [synth.make_tokens(cfg, step=i, device="cuda") for i in range(steps)]
    bias0 = layer.bias.clone()

    eager = []
    for i in range(steps):
        stats = torch.zeros(4, device="cuda")
        y = layer.step(xs[i], stats_out=stats).clone()
        eager.append((y, layer.load.clone(), layer.bias.clone(), stats))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    updates = layer.updates

    layer.bias.copy_(bias0)
    stats = torch.zeros(steps, 4, device="cuda")
    outs = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    graphs = [layer.capture_step(xs[i], stats_out=stats[i], out=outs[i]) for i in range(steps)]
    assert layer.updates == updates          # capturing runs nothing
    for i, g in enumerate(graphs):
        y = g.replay()
        assert y.data_ptr() == outs[i].data_ptr()
        torch.cuda.synchronize()
        ey, eload, ebias, estats = eager[i]
        assert torch.equal(_bits(outs[i]), _bits(ey)), f"output differs at step {i}"
        assert torch.equal(layer.load, eload), f"loads differ at step {i}"
        assert torch.equal(_bits(layer.bias), _bits(ebias)), f"bias differs at step {i}"
        assert torch.equal(_bits(stats[i]), _bits(estats)), f"stats differ at step {i}"
    assert layer.device_status() == 0
    assert layer.updates == updates + steps


def test_graph_replay_reads_the_current_bias():
    """A replay reads the bias buffer as it is at replay time: replaying one
    captured step twice from the same bias gives the same output twice, and
    a bias changed between replays changes the routing like an eager step."""
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cuda")
    layer = MoELayer(cfg, p)
    x = synth.make_tokens(cfg, step=0, device="cuda")
    layer.forward(x)
    bias0 = layer.bias.clone()
    out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    g = layer.capture_step(x, out=out)
    g.replay()
    first = out.clone()
    layer.bias.copy_(bias0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(first))
    # a strongly skewed bias: the replay must route like an eager step with it
    skew = bias0.clone()
    skew[: cfg.E // 2] += 10.0
    layer.bias.copy_(skew)
    g.replay()
    torch.cuda.synchronize()
    got_idx = layer.idx[: cfg.T].clone()
    layer.bias.copy_(skew)
    layer.step(x)
    torch.cuda.synchronize()
    assert torch.equal(got_idx, layer.idx[: cfg.T])
    assert int((got_idx < cfg.E // 2).sum()) == cfg.T * cfg.K
