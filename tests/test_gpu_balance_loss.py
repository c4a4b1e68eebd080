"""Sequence-wise balance loss forward value on the GPU against the oracle's
reading of it (one value per sequence, empty sequences included)."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_affinity_b300 as moe
from expert_ffn_layer_affinity_b300 import synth
from oracle import moe_ref as ref

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("E,K,G,M,lens", [
    (16, 2, 1, 1, [256]),
    (64, 6, 1, 1, [1000, 0, 3096]),
    (256, 8, 8, 4, [4096, 4096]),
    (256, 8, 8, 4, [1, 7, 300, 2000]),
])
def test_seq_balance_loss_vs_oracle(E, K, G, M, lens):
    T = sum(lens)
    s = synth.make_affinities(T, E, seed=E + T, skew=0.05)
    b = torch.zeros(E)
    idx, _ = ref.select_experts(s.numpy(), b.numpy(), K, G, M, 1.0)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    loss = torch.empty(len(lens), device="cuda")
    moe.moe_seq_balance_loss(s.cuda(), torch.from_numpy(idx).cuda(), K,
                             torch.from_numpy(offs).cuda(), len(lens), E, K, 1e-3, loss)
    torch.cuda.synchronize()
    want = ref.seq_balance_loss(s.numpy().astype(np.float64), idx, offs, K, 1e-3)
    np.testing.assert_allclose(loss.cpu().numpy(), want, rtol=2e-5, atol=1e-12)


def test_seq_balance_loss_reads_first_K_columns():
    """Serving layout: rows carry K routed ids then the shared ones."""
    E, K, T = 16, 2, 64
    s = synth.make_affinities(T, E, seed=3)
    idx, _ = ref.select_experts(s.numpy(), np.zeros(E, np.float32), K)
    wide = np.concatenate([idx, np.full((T, 1), E, np.int32)], axis=1)
    offs = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    loss = torch.empty(1, device="cuda")
    moe.moe_seq_balance_loss(s.cuda(), torch.from_numpy(wide).cuda(), K + 1, offs, 1, E, K, 1.0,
                             loss)
    torch.cuda.synchronize()
    want = ref.seq_balance_loss(s.numpy().astype(np.float64), idx, [0, T], K, 1.0)
    np.testing.assert_allclose(loss.cpu().numpy(), want, rtol=2e-5)
