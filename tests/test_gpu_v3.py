"""The DeepSeek-V3-shaped layer at full size (T=8192, d=7168, 256 routed
experts, 8 per token, 8 groups / 4 kept, scale 2.5) and its decode and drift
workloads: routing on every token against the fp64 oracle (mismatches only on
counted near-tie tokens), layer output on sampled tokens within 1e-2 relative
L2, and the bias feedback against the oracle's own trajectory."""
import numpy as np
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer
from oracle import moe_ref as ref
from _util import Trajectory, bf16_to_np64, check_pass

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def v3():
    cfg = synth.CONFIGS["v3"]
    p = synth.make_params(cfg, "cuda")
    layer = MoELayer(cfg, p, max_T=16384)
    yield cfg, p, layer
    del layer, p
    torch.cuda.empty_cache()


def test_v3_layer_pass(v3):
    cfg, p, layer = v3
    x = synth.make_tokens(cfg, 0, "cuda")
    out = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    sample = np.random.default_rng(1).choice(cfg.T, 24, replace=False)
    r = check_pass(cfg, p, x, layer, out, sample=sample)
    print(f"v3 rel_l2={r['rel_l2']:.3e} near_tie={r['near_tie']} mismatched={r['mismatched_tokens']}")
    assert int(layer.load.sum().item()) == cfg.T * cfg.K
    groups = layer.idx[:cfg.T].cpu().numpy() // (cfg.E // cfg.n_groups)
    assert max(len(set(g.tolist())) for g in groups) <= cfg.topk_groups


@pytest.mark.parametrize("T", synth.DECODE_T)
def test_v3_decode_sizes(v3, T):
    cfg, p, layer = v3
    c = synth.CONFIGS["v3_decode"].with_T(T)
    x = synth.make_tokens(c, 0, "cuda", seed=100 + T)
    out = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    sample = np.random.default_rng(T).choice(T, 8, replace=False)
    check_pass(c, p, x, layer, out, sample=sample)
    touched = int((layer.load > 0).sum().item())
    assert touched >= 0.8 * 256 * (1 - (1 - 8 / 256) ** T)


def test_v3_drift_steps_across_a_rotation(v3):
    """Clustered tokens, T=16384, steps 23..27 (the mixture rotates at 25)."""
    cfg0, p, layer = v3
    cfg = synth.CONFIGS["v3_drift"]
    layer.cfg = cfg
    layer.bias.copy_(p["bias"])
    traj = Trajectory(cfg, p["bias"].cpu().numpy())
    w_r = p["w_r"].cpu().numpy()
    ratios = []
    for step in range(23, 28):
        x = synth.make_tokens(cfg, step, "cuda")
        b_before = layer.bias.cpu().numpy().copy()
        layer.forward(x)
        layer.bias_update(cfg.T)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        s64 = ref.router_affinity64(bf16_to_np64(x), w_r)
        traj.step(step, cfg.T, s64, layer.idx[:cfg.T].cpu().numpy(), layer.load.cpu().numpy(),
                  b_before, layer.bias.cpu().numpy())
        ratios.append(float(layer.stats[2].item()))
    layer.cfg = cfg0
    print(f"drift max/mean per step {ratios}; near-tie mismatches {traj.near_tie_mismatches}")
    assert all(r >= 1.0 for r in ratios)
