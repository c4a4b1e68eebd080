"""Serving layouts of the report's deployment (qwbw.cn essay on the report,
"9个专家", "32个冗余专家"): shared experts routed as experts E.. with gate 1,
and redundant copies of hot experts.  Both leave the layer's result unchanged:
checked against the oracle and against the standard layout."""
import numpy as np
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer
from oracle import moe_ref as ref
from _util import bf16_to_np64, check_pass

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["tiny", "mid"])
def case(request):
    cfg = synth.CONFIGS[request.param]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cpu")
    base = MoELayer(cfg, p)
    want = base.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    return cfg, p, x, base, want


def test_shared_as_routed_expert(case):
    cfg, p, x, base, want = case
    layer = MoELayer(cfg, p, shared_as_routed=True)
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    K, E, ns = cfg.K, cfg.E, cfg.n_shared
    idx = layer.idx[:cfg.T].cpu()
    assert torch.equal(idx[:, :K], base.idx[:cfg.T].cpu())
    assert torch.equal(idx[:, K:], torch.arange(E, E + ns, dtype=torch.int32).expand(cfg.T, ns))
    assert torch.all(layer.gate[:cfg.T, K:].cpu() == 1.0)
    assert torch.equal(layer.load.cpu(), base.load.cpu())      # loads count routed experts only
    # same math; each shared expert's output is rounded to bf16 on its own here
    # (the standard layout sums the shared experts inside one GEMM), so the two
    # layouts differ by about one bf16 rounding of the shared terms
    assert ref.rel_l2(bf16_to_np64(out), bf16_to_np64(want)) < 6e-3
    sample = np.arange(0, cfg.T, max(1, cfg.T // 256))
    check_pass(cfg, p, x, layer, out, sample=sample)


def test_redundant_copies_leave_output_unchanged(case):
    cfg, p, x, base, want = case
    n_red = 4
    layer = MoELayer(cfg, p, n_redundant=n_red)
    eo = layer.plan_replicas(base.load.cpu())
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    # the hottest experts got the copies; every copy carries tokens
    load = base.load.cpu().numpy()
    hot = set(np.argsort(-load, kind="stable")[:2].tolist())
    assert hot & set(eo[cfg.E:].tolist())
    K, E = cfg.K, cfg.E
    idx = layer.idx[:cfg.T].cpu().numpy()
    phys = layer.phys_idx[:cfg.T].cpu().numpy()
    ss, sl = layer.slot_start.cpu().numpy(), layer.slots.cpu().numpy()
    for t in range(0, cfg.T, 37):
        for k in range(K):
            e = idx[t, k]
            c = ss[e + 1] - ss[e]
            assert phys[t, k] == sl[ss[e] + t % c]
    counts = np.bincount(phys.reshape(-1), minlength=E + n_red)
    assert np.all(counts[E:E + n_red] > 0)
    # copies hold identical weights and each row's arithmetic is unchanged
    assert torch.equal(out.view(torch.int16).cpu(), want.view(torch.int16).cpu())


def test_both_serving_layouts_together(case):
    cfg, p, x, base, want = case
    layer = MoELayer(cfg, p, shared_as_routed=True, n_redundant=3)
    layer.plan_replicas(base.load.cpu())
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert ref.rel_l2(bf16_to_np64(out), bf16_to_np64(want)) < 6e-3
    phys = layer.phys_idx[:cfg.T].cpu().numpy()
    E_phys = cfg.E + 3 + cfg.n_shared
    assert np.all(phys[:, cfg.K:] == np.arange(cfg.E + 3, E_phys))
