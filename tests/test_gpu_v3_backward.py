"""Backward pass of the DeepSeek-V3-shaped layer at full size (T=8192,
d=7168, 256 routed experts, 8 per token, 8 groups / 4 kept, scale 2.5) in
the configuration `bench.py --pass train` times, against the fp64 backward
oracle on what it can compute one piece at a time: dx, dgate and du of
sampled tokens (each depends on its own token only, for the chosen experts),
and the full weight gradients of two experts (over all of their rows)."""
import numpy as np
import pytest
import torch

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer
from oracle import moe_bwd_ref as B
from oracle import moe_ref as ref
from _util import HostExperts, bf16_to_np64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_v3_backward_sampled():
    cfg = synth.CONFIGS["v3"]
    p = synth.make_params(cfg, "cuda")
    x = synth.make_tokens(cfg, 0, "cuda")
    dy = synth.make_output_grad(cfg, 0, "cuda")
    x64 = bf16_to_np64(x)
    w_r = p["w_r"].cpu().numpy()
    bias = p["bias"].cpu().numpy()
    s64 = ref.router_affinity64(x64, w_r, None)
    idx64, gate64 = ref.select_experts(s64, bias.astype(np.float64), cfg.K, cfg.n_groups,
                                       cfg.topk_groups, cfg.route_scale, precision="fp64")
    kth, grp = ref.near_tie_tokens(s64, bias, cfg.K, cfg.n_groups, cfg.topk_groups)
    tie = kth | grp
    dy[torch.from_numpy(tie).cuda()] = 0          # near ties: no gradient on either side
    layer = MoELayer(cfg, p, training=True)
    layer.forward(x)
    g = layer.backward(x, dy)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    T = cfg.T
    gidx = layer.idx[:T, :cfg.K].cpu().numpy()
    mism = np.any(np.sort(gidx, 1) != np.sort(idx64, 1), axis=1)
    assert not np.any(mism & ~tie)
    dy64 = bf16_to_np64(dy)
    host = HostExperts(p)                          # one expert at a time to the host

    # per-token gradients of sampled tokens
    tok = np.random.default_rng(3).choice(np.nonzero(~tie)[0], 6, replace=False)
    want = B.moe_layer_bwd64(x64[tok], w_r, None, idx64[tok], cfg.route_scale, host,
                             host.shared(), cfg.n_shared, dy64[tok])
    assert ref.rel_l2(bf16_to_np64(g["dx"][torch.from_numpy(tok).cuda()]), want["dx"]) < 1e-2
    full = np.zeros((len(tok), cfg.E))
    np.put_along_axis(full, idx64[tok], want["dgate"], axis=1)
    got_dg = g["dgate"].cpu().numpy().astype(np.float64)[tok]
    assert ref.rel_l2(got_dg, np.take_along_axis(full, gidx[tok], axis=1)) < 1e-2
    got_du = g["du"].cpu().numpy().astype(np.float64)[tok]
    assert ref.rel_l2(got_du, np.take_along_axis(want["du"], gidx[tok], axis=1)) < 1e-2

    # full weight gradients of the least and the most loaded expert
    load = np.bincount(idx64.ravel(), minlength=cfg.E)
    for e in (int(np.argmin(np.where(load > 0, load, 1 << 30))), int(np.argmax(load))):
        rows, slots = np.nonzero(idx64 == e)
        W1, W3, W2 = host(e)
        dYe = gate64[rows, slots][:, None] * dy64[rows]
        _, dW1, dW3, dW2 = B.swiglu_ffn_bwd64(x64[rows], W1, W3, W2, dYe)
        got13 = g["dw13"][e].cpu().numpy().astype(np.float64)
        assert ref.rel_l2(got13[:cfg.I], dW1) < 1e-2, e
        assert ref.rel_l2(got13[cfg.I:], dW3) < 1e-2, e
        assert ref.rel_l2(g["dw2"][e].cpu().numpy().astype(np.float64), dW2) < 1e-2, e

    # dW_r is the per-expert reduction of du x (a property at any size; du itself
    # is checked against the oracle above)
    du_full = np.zeros((T, cfg.E))
    np.put_along_axis(du_full, gidx, g["du"].cpu().numpy().astype(np.float64), axis=1)
    want_dwr = du_full.T @ x64
    got_dwr = g["dw_r"].cpu().numpy().astype(np.float64)
    assert ref.rel_l2(got_dwr, want_dwr) < 1e-5
    del layer, p, g
    torch.cuda.empty_cache()
