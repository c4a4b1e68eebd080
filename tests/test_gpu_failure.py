"""Failure detection on the GPU without a fault: the bounded wait that every
pipelined kernel uses, made to run out on a barrier nothing arrives on,
records MOE_DEV_TIMEOUT and returns; the context stays usable."""
import time

import pytest
import torch

import expert_ffn_layer_affinity_b300 as moe
from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_with_a_status():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_wait_selftest(20_000_000, status)       # 20 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    v = int(status.item()) & 0xFFFFFFFF
    assert v & moe.MOE_DEV_TIMEOUT
    assert not v & 0x80000000                       # the wait never "succeeded"
    assert 0.015 < dt < 2.0, dt
    # the context is still usable: a layer pass runs and reports no error
    cfg = synth.CONFIGS["tiny"]
    layer = MoELayer(cfg, synth.make_params(cfg, "cpu"))
    out = layer.forward(synth.make_tokens(cfg, 0, "cuda"))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert torch.isfinite(out.float()).all()
