"""Checkpoint / resume of the layer's mutable state (the bias, the update
count and a serving layout's replica plan): a run split by a save and a load
into a fresh layer follows the uninterrupted run bit for bit.  (The pages
describe no checkpoint format; this is the layer's own.)"""
import numpy as np
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer

pytestmark = pytest.mark.gpu


def test_mid_50_steps_equal_25_save_load_25(tmp_path):
    cfg = synth.CONFIGS["mid"]
    p = synth.make_params(cfg, "cpu")
    xs = [synth.make_tokens(cfg, i, "cuda") for i in range(50)]
    straight = MoELayer(cfg, p)
    ys = [straight.step(x).clone() for x in xs]
    first = MoELayer(cfg, p)
    for x in xs[:25]:
        first.step(x)
    first.save_state(str(tmp_path / "moe_state.pt"))
    resumed = MoELayer(cfg, p)
    resumed.load_state(str(tmp_path / "moe_state.pt"))
    assert resumed.updates == 25
    ys2 = [resumed.step(x).clone() for x in xs[25:]]
    torch.cuda.synchronize()
    assert torch.equal(resumed.bias.view(torch.int32), straight.bias.view(torch.int32))
    for a, b in zip(ys2, ys[25:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_replica_plan_survives_save_load(tmp_path):
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cuda")
    a = MoELayer(cfg, p, n_redundant=3)
    a.step(x)
    a.plan_replicas(a.load.cpu())
    ya = a.step(x).clone()
    a.save_state(str(tmp_path / "s.pt"))
    b = MoELayer(cfg, p, n_redundant=3)
    b.load_state(str(tmp_path / "s.pt"))
    a.bias.copy_(b.bias)                       # both from the saved bias
    y1, y2 = a.forward(x).clone(), b.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.slots.cpu(), b.slots.cpu())
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert ya.shape == y1.shape
    with pytest.raises(ValueError):
        MoELayer(cfg, p).load_state_dict({"bias": torch.zeros(cfg.E + 1)})
    assert np.isfinite(y1.float().cpu().numpy()).all()
