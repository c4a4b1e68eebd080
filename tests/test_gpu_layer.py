"""The whole layer pass (router GEMM -> selection -> permute -> grouped experts
-> shared experts -> combine -> bias update) against the fp64 oracle on the
tiny and mid workloads."""
import numpy as np
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer
from oracle import moe_ref as ref
from _util import bf16_to_np64, f32_bits

pytestmark = pytest.mark.gpu


class HostExperts:
    """Oracle-side view of the expert weights: exact fp64 values fetched one
    expert at a time (the full V3 set does not fit comfortably in host RAM as
    fp64)."""

    def __init__(self, p):
        self.p = p

    def __call__(self, e):
        return (bf16_to_np64(self.p["w1"][e]), bf16_to_np64(self.p["w3"][e]),
                bf16_to_np64(self.p["w2"][e]))

    def shared(self):
        return (bf16_to_np64(self.p["ws1"]), bf16_to_np64(self.p["ws3"]),
                bf16_to_np64(self.p["ws2"]))


def check_pass(cfg, p, x, layer, out, sample=None, bias=None):
    """Compare one pass: routing on every token, output on `sample` tokens."""
    T = x.shape[0]
    x64 = bf16_to_np64(x)
    off = p["logit_offset"].cpu().numpy() if p["logit_offset"] is not None else None
    b = (bias if bias is not None else p["bias"]).cpu().numpy()
    s64 = ref.router_affinity64(x64, p["w_r"].cpu().numpy(), off)
    idx64, gate64 = ref.select_experts(s64, b.astype(np.float64), cfg.K, cfg.n_groups,
                                       cfg.topk_groups, cfg.route_scale, precision="fp64")
    kth, grp = ref.near_tie_tokens(s64, b, cfg.K, cfg.n_groups, cfg.topk_groups)
    gidx = layer.idx[:T].cpu().numpy()
    mism = np.any(np.sort(gidx, 1) != np.sort(idx64, 1), axis=1)
    assert not np.any(mism & ~(kth | grp)), np.nonzero(mism & ~(kth | grp))[0][:10]
    tokens = np.arange(T) if sample is None else sample
    tokens = tokens[~mism[tokens]]
    host = HostExperts(p)
    want = ref.moe_output64(x64, idx64, gate64, host, host.shared(), cfg.n_shared, tokens)
    got = bf16_to_np64(out[torch.from_numpy(tokens).to(out.device)])
    err = ref.rel_l2(got, want)
    assert err < 1e-2, err
    return dict(rel_l2=err, mismatched_tokens=int(mism.sum()), near_tie=int((kth | grp).sum()),
                idx64=idx64)


def test_tiny_layer_all_tokens_and_bias_update():
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cpu")
    layer = MoELayer(cfg, p)
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    r = check_pass(cfg, p, x, layer, out)
    # load and bias update of the step
    rload = ref.expert_load(r["idx64"], cfg.E)
    if r["mismatched_tokens"] == 0:
        np.testing.assert_array_equal(layer.load.cpu().numpy(), rload)
    layer.bias_update(cfg.T)
    torch.cuda.synchronize()
    want = ref.bias_update(layer.load.cpu().numpy(), p["bias"].numpy(), cfg.T, cfg.K, cfg.E,
                           cfg.gamma)
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


def test_mid_layer_feedback_steps(mid):
    """Several bias-feedback steps with fresh tokens; at every step the GPU's
    routing matches the oracle's (up to counted near ties) and the GPU bias
    equals the oracle's sign rule applied to the GPU's loads."""
    cfg, p = mid
    layer = MoELayer(cfg, p)
    b_prev = p["bias"].numpy().copy()
    ratios = []
    for step in range(6):
        x = synth.make_tokens(cfg, step, "cpu")
        layer.forward(x.cuda())
        torch.cuda.synchronize()
        load = layer.load.cpu().numpy()
        x64 = bf16_to_np64(x)
        s64 = ref.router_affinity64(x64, p["w_r"].numpy(), p["logit_offset"].numpy())
        idx64, _ = ref.select_experts(s64, b_prev.astype(np.float64), cfg.K, precision="fp64")
        kth, _ = ref.near_tie_tokens(s64, b_prev, cfg.K)
        gidx = layer.idx.cpu().numpy()
        mism = np.any(np.sort(gidx, 1) != np.sort(idx64, 1), axis=1)
        assert not np.any(mism & ~kth)
        layer.bias_update(cfg.T)
        torch.cuda.synchronize()
        want = ref.bias_update(load, b_prev, cfg.T, cfg.K, cfg.E, cfg.gamma)
        np.testing.assert_array_equal(f32_bits(layer.bias), f32_bits(want))
        b_prev = want
        ratios.append(float(layer.stats[2].item()))
    assert layer.device_status() == 0
    assert ratios[0] > 1.5          # the Zipf offset skews the start
