"""The whole layer pass (router GEMM -> selection -> permute -> grouped experts
-> shared experts -> combine -> bias update) against the fp64 oracle on the
tiny and mid workloads."""
import numpy as np
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer
from oracle import moe_ref as ref
from _util import (Trajectory, bf16_to_np64, check_pass, describe, f32_bits, output_sample,
                   route_check, sign_rule_holds)

pytestmark = pytest.mark.gpu


def test_tiny_layer_all_tokens_and_bias_update():
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cpu")
    layer = MoELayer(cfg, p)
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    r = check_pass(cfg, p, x, layer, out)
    # load count and bias update of the step against the oracle's own
    rload = ref.expert_load(r["idx64"], cfg.E)
    layer.bias_update(cfg.T)
    torch.cuda.synchronize()
    gload = layer.load.cpu().numpy()
    assert sign_rule_holds(gload, p["bias"].numpy(), layer.bias.cpu().numpy(), cfg.T, cfg.K,
                           cfg.E, cfg.gamma)
    if r["mismatched_tokens"] == 0:
        np.testing.assert_array_equal(gload, rload)
        want = ref.bias_update(rload, p["bias"].numpy(), cfg.T, cfg.K, cfg.E, cfg.gamma)
        np.testing.assert_array_equal(f32_bits(layer.bias), f32_bits(want))


def test_tiny_layer_deterministic():
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cuda")
    layer = MoELayer(cfg, p)
    a = layer.forward(x).clone()
    b = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_layer_tiled_weights_bit_identical():
    """The forward layer's default box-contiguous expert weights give the
    standard layout's output bit for bit (mid shapes: two shared experts,
    I = 1408)."""
    cfg = synth.CONFIGS["mid"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cuda")
    a = MoELayer(cfg, p)
    b = MoELayer(cfg, p, tiled_weights=False)
    assert a.tiled and not b.tiled
    ya = a.forward(x).clone()
    yb = b.forward(x).clone()
    torch.cuda.synchronize()
    assert a.device_status() == 0 and b.device_status() == 0
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))


def test_tiny_layer_odd_token_counts():
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    layer = MoELayer(cfg, p, max_T=300)
    for T in (1, 3, 129, 300):
        x = synth.make_tokens(cfg, T, "cpu", T=T)
        out = layer.forward(x.cuda()).clone()
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        check_pass(cfg, p, x, layer, out)


@pytest.fixture(scope="module")
def mid():
    cfg = synth.CONFIGS["mid"]
    p = synth.make_params(cfg, "cpu")
    return cfg, p


def test_mid_layer_one_pass_sampled(mid):
    cfg, p = mid
    x = synth.make_tokens(cfg, 0, "cpu")
    layer = MoELayer(cfg, p, shared_stream=True)
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    sample = np.random.default_rng(0).choice(cfg.T, 512, replace=False)
    check_pass(cfg, p, x, layer, out, sample=sample)


MID_OUTPUT_STEPS = (0, 25, 49)


def test_mid_layer_feedback_steps(mid):
    """All 50 bias-feedback steps of the mid workload (Zipf-skewed router,
    fresh tokens every step) through the full layer: the GPU's routing, loads
    and bias against the oracle's own trajectory (see Trajectory) on every
    step, and the layer output on 256 + near-tie tokens at steps 0, 25 and 49
    (with the bias the GPU used at that step)."""
    cfg, p = mid
    layer = MoELayer(cfg, p)
    traj = Trajectory(cfg, p["bias"].numpy())
    ratios, checks = [], []
    for step in range(cfg.steps):
        x = synth.make_tokens(cfg, step, "cpu")
        b_before = layer.bias.clone()
        out = layer.forward(x.cuda())
        if step in MID_OUTPUT_STEPS:
            out = out.clone()
        layer.bias_update(cfg.T)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        s64 = ref.router_affinity64(bf16_to_np64(x), p["w_r"].numpy(), p["logit_offset"].numpy())
        traj.step(step, cfg.T, s64, layer.idx.cpu().numpy(), layer.load.cpu().numpy(),
                  b_before.cpu().numpy(), layer.bias.cpu().numpy())
        ratios.append(float(layer.stats[2].item()))
        if step in MID_OUTPUT_STEPS:
            rc = route_check(cfg, p, x, layer, bias=b_before)
            sample = output_sample(rc, 256, step)
            r = check_pass(cfg, p, x, layer, out, sample=sample, bias=b_before)
            checks.append((step, describe(r)))
    for step, d in checks:
        print(f"mid step {step}: {d}")
    print(f"mid max/mean first {ratios[0]:.4f} last {ratios[-1]:.4f}; near-tie mismatches "
          f"{traj.near_tie_mismatches} (kth {traj.mismatches_kth}); trajectories parted at "
          f"{traj.diverged_at}")
    assert len(ratios) == 50
    assert ratios[0] > 1.5          # the Zipf offset skews the start
