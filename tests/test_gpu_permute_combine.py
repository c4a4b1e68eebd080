"""Dispatch (permute) bit-exact and combine within bf16 rounding, against the
oracle."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_affinity_b300 as moe
from expert_ffn_layer_affinity_b300 import synth
from oracle import moe_ref as ref
from _util import bf16_to_np64, sync_status

pytestmark = pytest.mark.gpu


def random_idx(T, K, E, seed, skew=0.0):
    """Expert choices per (token, slot): distinct within a token, optionally
    concentrated on low expert numbers so some experts get nothing."""
    g = torch.Generator().manual_seed(seed)
    w = torch.ones(E)
    if skew:
        w = torch.exp(-skew * torch.arange(E, dtype=torch.float32))
    idx = torch.stack([torch.multinomial(w, K, replacement=False, generator=g) for _ in range(T)]) \
        if T else torch.zeros(0, K, dtype=torch.int64)
    return idx.to(torch.int32)


def run_permute(idx, E, x):
    T, K = idx.shape
    d = x.shape[1] if x is not None else 0
    dev = "cuda"
    R = T * K
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
    row_of = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    tok_of = torch.full((max(R, 1),), -1, dtype=torch.int32, device=dev)
    x_perm = torch.zeros(max(R, 1), max(d, 8), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_b = moe.moe_workspace_bytes(T, d, E, K, 64)
    ws = torch.empty(max(ws_b, 256), dtype=torch.uint8, device=dev)
    moe.moe_permute(idx.to(dev), T, K, E, x.to(dev) if x is not None else None, d, offs, row_of,
                    tok_of, x_perm if x is not None else None, status, ws, ws_b)
    st = sync_status(status)
    return offs.cpu().numpy(), row_of.cpu().numpy(), tok_of.cpu().numpy()[:R], x_perm.cpu()[:R], st


@pytest.mark.parametrize("T,K,E,d,skew", [
    (256, 2, 16, 256, 0.0),
    (4096, 6, 64, 2048, 0.0),
    (8192, 8, 256, 7168, 0.0),
    (1, 8, 256, 64, 0.0),
    (1500, 8, 256, 128, 0.08),     # many empty experts
    (3000, 4, 512, 64, 0.0),
    (333, 3, 8, 512, 0.5),
])
def test_permute_bitexact(T, K, E, d, skew):
    idx = random_idx(T, K, E, seed=T + E, skew=skew)
    x = synth.make_ffn_rows(T, d, seed=T)
    offs, row_of, tok_of, x_perm, st = run_permute(idx, E, x)
    assert st == 0
    r_off, r_row, r_tok = ref.permute(idx.numpy(), E)
    np.testing.assert_array_equal(offs, r_off)
    np.testing.assert_array_equal(row_of, r_row)
    np.testing.assert_array_equal(tok_of, r_tok)
    want = x[torch.from_numpy(r_tok.astype(np.int64))]
    assert torch.equal(x_perm.view(torch.int16), want.view(torch.int16))


def test_permute_maps_only_and_empty():
    idx = random_idx(100, 4, 32, seed=1)
    offs, row_of, tok_of, _, st = run_permute(idx, 32, None)
    r_off, r_row, r_tok = ref.permute(idx.numpy(), 32)
    assert st == 0
    np.testing.assert_array_equal(offs, r_off)
    np.testing.assert_array_equal(row_of, r_row)
    offs, _, _, _, st = run_permute(torch.zeros(0, 4, dtype=torch.int32), 32, None)
    assert st == 0 and np.all(offs == 0)


def test_permute_flags_bad_index():
    idx = random_idx(50, 2, 16, seed=3)
    idx[7, 1] = 99
    _, _, _, _, st = run_permute(idx, 16, None)
    assert st & moe.MOE_DEV_BAD_INDEX


@pytest.mark.parametrize("T,K,d,shared", [
    (256, 2, 256, True),
    (4096, 6, 2048, True),
    (2048, 8, 7168, True),
    (77, 8, 512, False),
    (1, 3, 64, True),
])
def test_combine_vs_oracle(T, K, d, shared):
    E = 64
    idx = random_idx(T, K, E, seed=K + d)
    _, r_row, _ = ref.permute(idx.numpy(), E)
    R = T * K
    y_perm = synth.make_ffn_rows(R, d, seed=5, std=0.5)
    y_sh = synth.make_ffn_rows(T, d, seed=6, std=0.5) if shared else None
    g = torch.Generator().manual_seed(9)
    gate = (torch.rand(T, K, generator=g) * 2.5 / K).float()
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(y_perm.cuda(), torch.from_numpy(r_row).cuda(), gate.cuda(),
                    y_sh.cuda() if shared else None, T, K, d, out)
    torch.cuda.synchronize()
    want = ref.combine64(bf16_to_np64(y_perm), r_row, gate.numpy().astype(np.float64),
                         bf16_to_np64(y_sh) if shared else None)
    got = bf16_to_np64(out)
    # one bf16 rounding of the fp32 sum (2^-9 relative) plus fp32 accumulation
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-5)
    assert ref.rel_l2(got, want) < 3e-3
