"""HostPipeline: steps on pinned host activations with overlapped copies give
exactly the eager results (outputs and bias trajectory)."""
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import HostPipeline, MoELayer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_pipeline_matches_eager_steps(name):
    cfg = synth.CONFIGS[name]
    p = synth.make_params(cfg, "cpu")
    xs = [synth.make_tokens(cfg, i, "cpu") for i in range(5)]
    eager = MoELayer(cfg, p)
    want = []
    for x in xs:
        want.append(eager.step(x.cuda()).cpu().clone())
    torch.cuda.synchronize()
    layer = MoELayer(cfg, p)
    pipe = HostPipeline(layer, cfg.T)
    outs = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in xs]
    hx = [x.pin_memory() for x in xs]
    for i in range(len(xs)):
        pipe.step(i, hx[i], outs[i])
    pipe.finish()
    torch.cuda.synchronize()
    for a, b in zip(outs, want):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(layer.bias.cpu(), eager.bias.cpu())


def test_training_pipeline_matches_eager_steps():
    """train=True: x and dy in, dx out, overlapped; dx and the bias trajectory
    equal eager forward + backward + bias update, bit for bit."""
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    xs = [synth.make_tokens(cfg, i, "cpu") for i in range(4)]
    dys = [synth.make_output_grad(cfg, i, "cpu") for i in range(4)]
    eager = MoELayer(cfg, p, training=True)
    want, want_bias = [], []
    for x, dy in zip(xs, dys):
        eager.forward(x.cuda())
        want.append(eager.backward(x.cuda(), dy.cuda())["dx"].cpu().clone())
        eager.bias_update(cfg.T)
        want_bias.append(eager.bias.cpu().clone())
    torch.cuda.synchronize()
    layer = MoELayer(cfg, p, training=True)
    pipe = HostPipeline(layer, cfg.T, train=True)
    outs = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in xs]
    hx = [x.pin_memory() for x in xs]
    hdy = [g.pin_memory() for g in dys]
    for i in range(len(xs)):
        pipe.step(i, hx[i], outs[i], dy_host=hdy[i])
    pipe.finish()
    torch.cuda.synchronize()
    for a, b in zip(outs, want):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(layer.bias.cpu().view(torch.int32), want_bias[-1].view(torch.int32))
