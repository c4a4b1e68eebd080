"""The allocation-free dispatch, moe_permute_static, against moe_permute.

moe_permute_static serves callers that cannot allocate device memory at call
time (a plugin inside a host application that owns all device memory, a
serving loop that must never call cudaMalloc once running).  It keeps its
scratch in a fixed array inside the library instead of a caller workspace,
so these tests check that it gives exactly the outputs of the workspace
version, on two calls in a row (the second reuses the array the first one
left behind), and that shapes beyond the array are refused.

Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_affinity_b300 as moe
from expert_ffn_layer_affinity_b300 import synth

pytestmark = pytest.mark.gpu


def seeded_idx(T, K, E, seed):
    g = torch.Generator().manual_seed(seed)
    keys = torch.rand(T, E, generator=g)
    return torch.topk(keys, K, dim=1).indices.to(torch.int32)


def outputs(fn, idx, E, x, **kw):
    T, K = idx.shape
    d = x.shape[1]
    dev = "cuda"
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
    row_of = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    tok_of = torch.full((T * K,), -1, dtype=torch.int32, device=dev)
    x_perm = torch.zeros(T * K, d, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    fn(idx.to(dev), T, K, E, x.to(dev), d, offs, row_of, tok_of, x_perm, status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return [t.cpu() for t in (offs, row_of, tok_of, x_perm.view(torch.int16))]


def workspace_permute(idx, T, K, E, x, d, offs, row_of, tok_of, x_perm, status):
    ws_b = moe.moe_workspace_bytes(T, d, E, K, 64)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    moe.moe_permute(idx, T, K, E, x, d, offs, row_of, tok_of, x_perm, status, ws, ws_b)


@pytest.mark.parametrize("T,K,E,d", [(8192, 8, 256, 7168), (1000, 6, 64, 256), (3, 2, 16, 64)])
def test_static_permute_matches_workspace_permute_on_two_calls(T, K, E, d):
    for call in range(2):
        idx = seeded_idx(T, K, E, seed=100 * call + T)
        x = synth.make_ffn_rows(T, d, seed=call)
        want = outputs(workspace_permute, idx, E, x)
        got = outputs(moe.moe_permute_static, idx, E, x)
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        assert int(got[0][-1]) == T * K


def test_static_permute_refuses_shapes_beyond_its_array():
    """A shape whose per-tile counts exceed the fixed array is refused before
    anything is launched.  Every buffer is a real device tensor of the right
    size, so a weakened size check would give a wrong answer, not a fault."""
    dev = "cuda"
    T, K, E = 40000, 8, 256            # ceil(320000 / 1024) * 256 = 80128 counts > 65536
    idx = torch.zeros(T, K, dtype=torch.int32, device=dev)
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    row_of = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    tok_of = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    r = moe.moe_permute_static(idx, T, K, E, None, 0, offs, row_of, tok_of, None, status,
                               check=False)
    torch.cuda.synchronize()
    assert r == moe.MOE_ERR_SCRATCH_LIMIT
    for t in (offs, row_of, tok_of):
        assert bool(torch.all(t == -7))
    assert int(status.item()) == 0
