"""Grouped SwiGLU experts on the tensor cores against the fp64 oracle:
ragged groups (empty, 1 row, tile edges), column tails, shared-expert form,
rows outside every group left untouched."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_affinity_b300 as moe
from expert_ffn_layer_affinity_b300 import synth
from oracle import moe_ref as ref
from _util import bf16_to_np64, sync_status

pytestmark = pytest.mark.gpu


def weights(G, I, d, seed, std=0.05):
    g = torch.Generator().manual_seed(seed)
    bf = torch.bfloat16
    w1 = (torch.randn(G, I, d, generator=g) * std).to(bf)
    w3 = (torch.randn(G, I, d, generator=g) * std).to(bf)
    w2 = (torch.randn(G, d, I, generator=g) * std).to(bf)
    return w1, w3, w2


def run_grouped(a, offsets, w1, w3, w2, R_buf=None, canary=False):
    R, d = a.shape
    G, I, _ = w1.shape
    dev = "cuda"
    h = torch.zeros(R, I, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(R, d, dtype=torch.bfloat16, device=dev)
    if canary:
        h.fill_(7.0)
        y.fill_(-3.0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_grouped_swiglu(a.to(dev), offsets.to(dev), G, R, d, I, w1.to(dev), w3.to(dev),
                           w2.to(dev), h, y, status)
    st = sync_status(status)
    return h.cpu(), y.cpu(), st


def reference(a, offsets, w1, w3, w2):
    A = bf16_to_np64(a)
    W1, W3, W2 = bf16_to_np64(w1), bf16_to_np64(w3), bf16_to_np64(w2)
    R, d = A.shape
    I = W1.shape[1]
    H = np.zeros((R, I))
    Y = np.zeros((R, d))
    offs = offsets.numpy()
    for g in range(len(offs) - 1):
        r0, r1 = offs[g], offs[g + 1]
        if r1 > r0:
            X = A[r0:r1]
            H[r0:r1] = ref.silu64(X @ W1[g].T) * (X @ W3[g].T)
            Y[r0:r1] = ref.swiglu_ffn64(X, W1[g], W3[g], W2[g])
    return H, Y


@pytest.mark.parametrize("sizes,d,I", [
    ([128], 256, 128),                       # one full tile
    ([1], 256, 128),                         # one row
    ([0, 129, 0, 127, 1, 256, 300], 256, 128),
    ([200, 57, 0, 513], 512, 192),           # I % 128 == 64: column tail in GEMM1
    ([384, 5], 320, 128),                    # d % 256 == 64: column tail in GEMM2
    # every ragged token-tile width: N = 16..256 in steps of 16 (8..128 token
    # rows per CTA, staged as sums of 64/32/16/8-row boxes), alone and as the
    # tail after a full 256-token tile
    (list(range(1, 257, 8)) + [256 + 9, 256 + 100, 256 + 255, 512 + 16], 256, 128),
])
def test_grouped_swiglu_vs_oracle(sizes, d, I):
    G = len(sizes)
    offsets = torch.tensor([0] + list(np.cumsum(sizes)), dtype=torch.int32)
    R = int(offsets[-1])
    a = synth.make_ffn_rows(R, d, seed=R + d)
    w1, w3, w2 = weights(G, I, d, seed=G + I)
    h, y, st = run_grouped(a, offsets, w1, w3, w2)
    assert st == 0
    H, Y = reference(a, offsets, w1, w3, w2)
    hg, yg = bf16_to_np64(h), bf16_to_np64(y)
    assert ref.rel_l2(hg, H) < 4e-3, ref.rel_l2(hg, H)
    assert ref.rel_l2(yg, Y) < 1e-2, ref.rel_l2(yg, Y)
    for g in range(G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 > r0:
            assert ref.rel_l2(hg[r0:r1], H[r0:r1]) < 4e-3, (g, r1 - r0)
            assert ref.rel_l2(yg[r0:r1], Y[r0:r1]) < 1e-2, (g, r1 - r0)


def test_rows_outside_groups_untouched():
    d, I = 256, 128
    sizes = [100, 0, 150]
    offsets = torch.tensor([0, 100, 100, 250], dtype=torch.int32)
    R = 300                                   # last 50 rows belong to no group
    a = synth.make_ffn_rows(R, d, seed=4)
    w1, w3, w2 = weights(3, I, d, seed=2)
    h, y, st = run_grouped(a, offsets, w1, w3, w2, canary=True)
    assert st == 0
    assert torch.all(h[250:].float() == 7.0) and torch.all(y[250:].float() == -3.0)
    H, Y = reference(a[:250], offsets, w1, w3, w2)
    assert ref.rel_l2(bf16_to_np64(y[:250]), Y) < 1e-2


def test_shared_expert_form_equals_sum_of_experts():
    """Two shared experts side by side (width 2I) as one group over all rows."""
    T, d, I = 300, 256, 128
    x = synth.make_ffn_rows(T, d, seed=12)
    w1, w3, w2 = weights(2, I, d, seed=13)
    ws1 = torch.cat([w1[0], w1[1]], 0)[None]
    ws3 = torch.cat([w3[0], w3[1]], 0)[None]
    ws2 = torch.cat([w2[0], w2[1]], 1)[None]
    _, y, st = run_grouped(x, torch.tensor([0, T], dtype=torch.int32), ws1, ws3, ws2)
    assert st == 0
    want = ref.shared_ffn64(bf16_to_np64(x), bf16_to_np64(ws1[0]), bf16_to_np64(ws3[0]),
                            bf16_to_np64(ws2[0]), 2)
    assert ref.rel_l2(bf16_to_np64(y), want) < 1e-2


def test_v3_expert_shape_sampled():
    """One V3-shaped expert (d=7168, I=2048) with 300 rows, plus an empty group."""
    d, I = 7168, 2048
    offsets = torch.tensor([0, 0, 300], dtype=torch.int32)
    a = synth.make_ffn_rows(300, d, seed=3)
    w1, w3, w2 = weights(2, I, d, seed=5, std=0.02)
    h, y, st = run_grouped(a, offsets, w1, w3, w2)
    assert st == 0
    H, Y = reference(a, offsets, w1, w3, w2)
    assert ref.rel_l2(bf16_to_np64(h), H) < 4e-3
    assert ref.rel_l2(bf16_to_np64(y), Y) < 1e-2


@pytest.mark.parametrize("sizes,d,I", [
    ([0, 129, 0, 127, 1, 256, 300], 256, 128),
    ([200, 57, 0, 513], 512, 192),
])
def test_grouped_swiglu_w1_w3_in_one_allocation(sizes, d, I):
    """w1 and w3 as the two halves of one [2, G, I, d] buffer (the layout the
    layer uses): same result as separate tensors, bit for bit."""
    G = len(sizes)
    offsets = torch.tensor([0] + list(np.cumsum(sizes)), dtype=torch.int32)
    R = int(offsets[-1])
    a = synth.make_ffn_rows(R, d, seed=R + d)
    w1, w3, w2 = weights(G, I, d, seed=G + I)
    w13 = torch.stack([w1, w3]).contiguous()
    h_sep, y_sep, st1 = run_grouped(a, offsets, w1, w3, w2)
    dev = "cuda"
    w13d = w13.to(dev)
    h = torch.zeros(R, I, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(R, d, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_grouped_swiglu(a.to(dev), offsets.to(dev), G, R, d, I, w13d[0], w13d[1], w2.to(dev),
                           h, y, status)
    assert sync_status(status) == 0 and st1 == 0
    assert torch.equal(h.cpu().view(torch.int16), h_sep.view(torch.int16))
    assert torch.equal(y.cpu().view(torch.int16), y_sep.view(torch.int16))


def tiled_reference(w1, w3, w2):
    """The box-contiguous arrangement of include/moe.h, written with torch
    reshapes (w1, w3 [G, I, d]; w2 [G, d, I])."""
    G, I, d = w1.shape
    a = w1.reshape(G, I // 64, 64, d // 64, 64).permute(0, 1, 3, 2, 4)
    c = w3.reshape(G, I // 64, 64, d // 64, 64).permute(0, 1, 3, 2, 4)
    # box row 2i = w1 row i, row 2i + 1 = w3 row i
    w13t = torch.stack([a, c], dim=4).reshape(G, I // 64, d // 64, 128, 64).contiguous()
    w2t = w2.reshape(G, d // 128, 128, I // 64, 64).permute(0, 1, 3, 2, 4).contiguous()
    return w13t, w2t


def run_tiled(a, offsets, w1, w3, w2):
    R, d = a.shape
    G, I, _ = w1.shape
    dev = "cuda"
    w13t = torch.empty(G, I // 64, d // 64, 128, 64, dtype=torch.bfloat16, device=dev)
    w2t = torch.empty(G, d // 128, I // 64, 128, 64, dtype=torch.bfloat16, device=dev)
    moe.moe_tile_expert_weights(w1.to(dev), w3.to(dev), w2.to(dev), G, I, d, w13t, w2t)
    h = torch.zeros(R, I, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(R, d, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_grouped_swiglu_tiled(a.to(dev), offsets.to(dev), G, R, d, I, w13t, w2t, h, y, status)
    st = sync_status(status)
    return h.cpu(), y.cpu(), st, w13t.cpu(), w2t.cpu()


@pytest.mark.parametrize("sizes,d,I", [
    ([128], 256, 128),
    ([1], 256, 128),
    ([0, 129, 0, 127, 1, 256, 300], 256, 128),
    ([200, 57, 0, 513], 512, 192),           # I % 128 == 64: column tail in GEMM1
    ([300, 17], 384, 128),                   # d % 256 == 128: column tail in GEMM2
    (list(range(1, 257, 8)) + [256 + 9, 256 + 100, 256 + 255, 512 + 16], 256, 128),
])
def test_grouped_swiglu_tiled_bit_identical(sizes, d, I):
    """Box-contiguous weights: the layout is the one include/moe.h states, and
    h and y equal the standard-layout call's bit for bit (same boxes, same
    order), which the oracle tests above pin."""
    G = len(sizes)
    offsets = torch.tensor([0] + list(np.cumsum(sizes)), dtype=torch.int32)
    R = int(offsets[-1])
    a = synth.make_ffn_rows(R, d, seed=R + d + 1)
    w1, w3, w2 = weights(G, I, d, seed=G + I + 1)
    h0, y0, st0 = run_grouped(a, offsets, w1, w3, w2)
    h1, y1, st1, w13t, w2t = run_tiled(a, offsets, w1, w3, w2)
    assert st0 == 0 and st1 == 0
    r13, r2 = tiled_reference(w1, w3, w2)
    assert torch.equal(w13t.view(torch.int16), r13.view(torch.int16))
    assert torch.equal(w2t.view(torch.int16), r2.view(torch.int16))
    assert torch.equal(h1.view(torch.int16), h0.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16))


def test_grouped_swiglu_tiled_v3_shape():
    """One V3-shaped expert (d=7168, I=2048) with 300 rows and an empty group:
    tiled equals standard bit for bit."""
    d, I = 7168, 2048
    offsets = torch.tensor([0, 0, 300], dtype=torch.int32)
    a = synth.make_ffn_rows(300, d, seed=3)
    w1, w3, w2 = weights(2, I, d, seed=5, std=0.02)
    h0, y0, st0 = run_grouped(a, offsets, w1, w3, w2)
    h1, y1, st1, _, _ = run_tiled(a, offsets, w1, w3, w2)
    assert st0 == 0 and st1 == 0
    assert torch.equal(h1.view(torch.int16), h0.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16))
