"""The FP8 (E4M3) expert path at the full DeepSeek-V3 layer shape (T=8192,
d=7168, 256 routed experts, 8 per token, I=2048), the configuration
`bench.py --precision fp8` times, against the oracle's FP8 reading:

* routing of every token as in the bf16 path (near-tie mismatches only);
* the routed experts' outputs, row by row in dispatch order, for the least
  and the most loaded expert and two others, against the oracle's FFN on the
  oracle's own 1 x 128 / 128 x 128 quantization of the same rows and weights;
* the shared expert's output on sampled tokens.

Quantizing an expert on the host takes a few seconds, so the check covers
whole experts (every row the GPU sent to them) rather than whole tokens."""
import numpy as np
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer
from oracle import fp8_ref as F8
from oracle import moe_ref as ref
from _util import bf16_to_np64, route_check

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def v3_fp8():
    cfg = synth.CONFIGS["v3"]
    p = synth.make_params(cfg, "cuda")
    layer = MoELayer(cfg, p, precision="fp8")
    x = synth.make_tokens(cfg, 0, "cuda")
    out = layer.forward(x).clone()
    torch.cuda.synchronize()
    yield cfg, p, layer, x, out
    del layer, p
    torch.cuda.empty_cache()


def test_v3_fp8_routing(v3_fp8):
    cfg, p, layer, x, _ = v3_fp8
    assert layer.device_status() == 0
    rc = route_check(cfg, p, x, layer)
    assert len(rc["bad"]) == 0, rc["bad"][:10]
    assert int(layer.load.sum().item()) == cfg.T * cfg.K


def test_v3_fp8_routed_experts_rows(v3_fp8):
    cfg, p, layer, x, _ = v3_fp8
    offs = layer.offsets.cpu().numpy()
    loads = np.diff(offs)
    order = np.argsort(loads, kind="stable")
    experts = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2]), 0})
    tok_of = layer.tok_of.cpu().numpy()
    x64 = bf16_to_np64(x)
    for e in experts:
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r1 == r0:
            continue
        X = x64[tok_of[r0:r1]]
        q = F8.quantize_expert(bf16_to_np64(p["w1"][e]), bf16_to_np64(p["w3"][e]),
                               bf16_to_np64(p["w2"][e]))
        want = F8.swiglu_ffn64_fp8(X, q)
        got = bf16_to_np64(layer.y_perm[r0:r1])
        err = ref.rel_l2(got, want)
        print(f"expert {e}: {r1 - r0} rows, rel_l2 {err:.3e}")
        assert err < 3e-3, (e, err)


def test_v3_fp8_shared_expert_sampled(v3_fp8):
    cfg, p, layer, x, _ = v3_fp8
    tok = np.sort(np.random.default_rng(5).choice(cfg.T, 64, replace=False))
    X = bf16_to_np64(x)[tok]
    q = F8.quantize_expert(bf16_to_np64(p["ws1"]), bf16_to_np64(p["ws3"]), bf16_to_np64(p["ws2"]))
    want = F8.swiglu_ffn64_fp8(X, q)
    got = bf16_to_np64(layer.y_sh[torch.from_numpy(tok).to(layer.y_sh.device)])
    err = ref.rel_l2(got, want)
    print(f"shared expert: rel_l2 {err:.3e}")
    assert err < 3e-3, err
