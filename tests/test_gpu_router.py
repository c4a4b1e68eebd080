"""Router selection, load count and bias feedback on the GPU against the
oracle: bit-exact when both are fed the same fp32 affinities."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_affinity_b300 as moe
from expert_ffn_layer_affinity_b300 import synth
from oracle import moe_ref as ref
from _util import bf16_to_np64, f32_bits, sync_status

pytestmark = pytest.mark.gpu


def run_topk(s, b, K, G, M, scale):
    T, E = s.shape
    dev = "cuda"
    s_d, b_d = s.to(dev).contiguous(), b.to(dev).contiguous()
    idx = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    gate = torch.zeros(T, K, dtype=torch.float32, device=dev)
    load = torch.full((E,), 12345, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_b = moe.moe_workspace_bytes(T, 64, E, K, 64)
    ws = torch.empty(max(ws_b, 256), dtype=torch.uint8, device=dev)
    moe.moe_router_topk(None, None, s_d, None, b_d, T, 0, E, K, G, M, scale, idx, gate, load,
                        None, status, ws, ws_b)
    st = sync_status(status)
    return idx.cpu().numpy(), gate.cpu().numpy(), load.cpu().numpy(), st


def rand_bias(E, seed, std=0.02, quantum=None):
    g = torch.Generator().manual_seed(seed)
    b = torch.randn(E, generator=g) * std
    if quantum:
        b = torch.round(b / quantum) * quantum
    return b.float()


CASES = [
    # T, E, K, G, M, scale, quantum
    (256, 16, 2, 1, 1, 1.0, None),        # tiny layer routing
    (4096, 64, 6, 1, 1, 1.0, None),       # mid layer routing
    (8192, 256, 8, 8, 4, 2.5, None),      # V3 routing, group limited
    (16384, 256, 8, 8, 4, 2.5, None),     # V3 drift batch size
    (1, 256, 8, 8, 4, 2.5, None),
    (37, 64, 6, 8, 3, 1.0, None),
    (1000, 16, 4, 4, 2, 2.5, 1 / 8),      # forced ties everywhere
    (513, 256, 8, 8, 4, 2.5, 1 / 64),
    (300, 512, 8, 8, 4, 2.5, None),
    (100, 32, 1, 1, 1, 1.0, None),
    (64, 128, 32, 1, 1, 1.0, None),
    (700, 64, 6, 4, 4, 1.0, None),        # M == G: group rule is a no-op
    (333, 8, 3, 4, 2, 2.5, None),
]


@pytest.mark.parametrize("T,E,K,G,M,scale,quantum", CASES)
def test_topk_bitexact_vs_oracle(T, E, K, G, M, scale, quantum):
    s = synth.make_affinities(T, E, seed=T + E, quantum=quantum)
    b = rand_bias(E, seed=K, quantum=quantum)
    idx, gate, load, st = run_topk(s, b, K, G, M, scale)
    assert st == 0
    ridx, rgate = ref.select_experts(s.numpy(), b.numpy(), K, G, M, scale, precision="fp32")
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_array_equal(f32_bits(gate), f32_bits(rgate))
    np.testing.assert_array_equal(load, ref.expert_load(ridx, E))
    assert int(load.sum()) == T * K
    if G > 1:
        assert np.all([len(set((r // (E // G)).tolist())) <= M for r in idx])


def test_topk_empty_batch():
    s = torch.zeros(0, 64)
    idx, gate, load, st = run_topk(s, torch.zeros(64), 4, 1, 1, 1.0)
    assert st == 0 and idx.shape == (0, 4) and np.all(load == 0)


def test_topk_nonfinite_flagged_and_ranked_lowest():
    T, E, K = 64, 64, 6
    s = synth.make_affinities(T, E, seed=5)
    s[3, 10] = float("nan")
    s[3, 11] = float("inf")
    s[7, :] = float("nan")          # a whole row of NaN: lowest indices win
    s[9, 0] = float("-inf")
    b = rand_bias(E, 3)
    idx, gate, load, st = run_topk(s, b, K, 1, 1, 1.0)
    assert st & moe.MOE_DEV_NONFINITE
    ridx, rgate = ref.select_experts(s.numpy(), b.numpy(), K, precision="fp32")
    np.testing.assert_array_equal(idx, ridx)
    assert list(idx[7]) == list(range(K))
    assert idx[3, 0] == 11 and 10 not in idx[3]
    ok = ~np.isnan(rgate)
    np.testing.assert_array_equal(np.isnan(gate), np.isnan(rgate))
    np.testing.assert_array_equal(f32_bits(gate[ok]), f32_bits(rgate[ok]))


def test_gates_do_not_depend_on_bias():
    T, E, K = 4096, 256, 8
    s = synth.make_affinities(T, E, seed=11)
    i0, g0, _, _ = run_topk(s, torch.zeros(E), K, 8, 4, 2.5)
    i1, g1, _, _ = run_topk(s, rand_bias(E, 9, std=0.002), K, 8, 4, 2.5)
    same = np.all(i0 == i1, axis=1)
    assert same.sum() > 0 and (~same).sum() > 0
    np.testing.assert_array_equal(f32_bits(g0[same]), f32_bits(g1[same]))


def test_bias_update_bitexact_single():
    E, T, K = 256, 8192, 8
    g = torch.Generator().manual_seed(2)
    load = torch.randint(0, 2 * T * K // E, (E,), generator=g, dtype=torch.int32)
    load[5] = T * K // E
    b = rand_bias(E, 4, std=0.01)
    b_d = b.cuda()
    stats = torch.zeros(4, device="cuda")
    moe.moe_bias_update(load.cuda(), b_d, T, K, E, 1e-3, stats)
    torch.cuda.synchronize()
    want = ref.bias_update(load.numpy(), b.numpy(), T, K, E, 1e-3)
    np.testing.assert_array_equal(f32_bits(b_d), f32_bits(want))
    np.testing.assert_allclose(stats.cpu().numpy(), ref.load_stats(load.numpy()), rtol=1e-6)


def test_bias_feedback_replay_50_steps():
    """Mid layer shape: 50 steps of selection + load count + bias update fed the
    same skewed fp32 affinities on both sides; every step's loads and bias
    bit-exact, and the feedback lowers the max/mean load."""
    T, E, K, gamma = 4096, 64, 6, 1e-3
    b_gpu = torch.zeros(E, device="cuda")
    b_ref = np.zeros(E, dtype=np.float32)
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    gate = torch.empty(T, K, device="cuda")
    load = torch.empty(E, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stats = torch.zeros(4, device="cuda")
    ws_b = moe.moe_workspace_bytes(T, 64, E, K, 64)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    ratios = []
    for step in range(50):
        s = synth.make_affinities(T, E, step=step, seed=1, skew=0.02)
        moe.moe_router_topk(None, None, s.cuda(), None, b_gpu, T, 0, E, K, 1, 1, 1.0, idx, gate,
                            load, None, status, ws, ws_b)
        moe.moe_bias_update(load, b_gpu, T, K, E, gamma, stats)
        ridx, _ = ref.select_experts(s.numpy(), b_ref, K, precision="fp32")
        rload = ref.expert_load(ridx, E)
        b_ref = ref.bias_update(rload, b_ref, T, K, E, gamma)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(load.cpu().numpy(), rload)
        np.testing.assert_array_equal(f32_bits(b_gpu), f32_bits(b_ref))
        ratios.append(float(stats[2].item()))
    assert int(status.item()) == 0
    assert ratios[-1] < ratios[0]


def test_router_split_is_exact():
    E, d = 64, 512
    g = torch.Generator().manual_seed(8)
    w = torch.randn(E, d, generator=g) * 0.02
    w[0, :4] = torch.tensor([1.0, -3.1415927, 1e-30, 65504.0])
    w_split = torch.empty(E, 3 * d, dtype=torch.bfloat16, device="cuda")
    moe.moe_router_prepare(w.cuda(), E, d, w_split)
    parts = bf16_to_np64(w_split).reshape(E, 3, d)
    np.testing.assert_array_equal(parts.sum(axis=1), w.numpy().astype(np.float64))


@pytest.mark.parametrize("T,d,E,K,G,M,scale,zipf", [
    (256, 256, 16, 2, 1, 1, 1.0, None),
    (1000, 2048, 64, 6, 1, 1, 1.0, 1.2),
    (300, 7168, 256, 8, 8, 4, 2.5, None),
    (129, 512, 8, 3, 4, 2, 2.5, None),
    (1, 1024, 128, 4, 1, 1, 1.0, None),
    # ragged last token tile with four expert tiles; a split V3-width
    # batch; the V3 batch itself (one split)
    (3000, 1024, 512, 8, 8, 4, 2.5, None),
    (2048, 7168, 256, 8, 8, 4, 2.5, None),
    (8192, 7168, 256, 8, 8, 4, 2.5, None),
])
def test_router_gemm_affinity_and_routing(T, d, E, K, G, M, scale, zipf):
    """Tensor-core router logits (exact products, fp32 accumulation) + sigmoid
    against the fp64 oracle; index mismatches only on near-tie tokens."""
    g = torch.Generator().manual_seed(T + d)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, d, generator=g) * 0.02).float()
    b = (torch.randn(E, generator=g) * 0.01).float()
    off = synth.zipf_logit_offset(E, zipf) if zipf else None
    dev = "cuda"
    w_split = torch.empty(E, 3 * d, dtype=torch.bfloat16, device=dev)
    moe.moe_router_prepare(w.to(dev), E, d, w_split)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    gate = torch.empty(T, K, device=dev)
    load = torch.empty(E, dtype=torch.int32, device=dev)
    aff = torch.empty(T, E, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_b = moe.moe_workspace_bytes(T, d, E, K, 64)
    ws = torch.empty(ws_b, dtype=torch.uint8, device=dev)
    moe.moe_router_topk(x.to(dev), w_split, None, off.to(dev) if off is not None else None,
                        b.to(dev), T, d, E, K, G, M, scale, idx, gate, load, aff, status, ws,
                        ws_b)
    assert sync_status(status) == 0
    s64 = ref.router_affinity64(bf16_to_np64(x), w.numpy(), off.numpy() if off is not None else None)
    err = np.abs(aff.cpu().numpy().astype(np.float64) - s64)
    # well inside the 1e-5 near-tie margin, so a gap >= 1e-5 can never flip
    assert err.max() < 4e-6, err.max()
    # end to end against fp64: mismatches only where the K-th/(K+1)-th gap < 1e-5
    ridx64, rgate64 = ref.select_experts(s64, b.numpy().astype(np.float64), K, G, M, scale,
                                         precision="fp64")
    kth, grp = ref.near_tie_tokens(s64, b.numpy(), K, G, M)
    bad = np.any(np.sort(idx.cpu().numpy(), 1) != np.sort(ridx64, 1), axis=1)
    assert not np.any(bad & ~(kth | grp)), np.nonzero(bad & ~(kth | grp))
    good = ~bad
    gi, gg = idx.cpu().numpy()[good], gate.cpu().numpy()[good]
    oi, og = ridx64[good], rgate64[good]
    gg = np.take_along_axis(gg, np.argsort(gi, 1), 1)
    og = np.take_along_axis(og, np.argsort(oi, 1), 1)
    np.testing.assert_allclose(gg, og, rtol=2e-5, atol=1e-6)


@pytest.mark.parametrize("T,d,E,K,G,M,scale", [
    (4096, 2048, 64, 6, 1, 1, 1.0),        # mid layer shape: the reduction is split
    (64, 7168, 256, 8, 8, 4, 2.5),         # decode size of the V3 layer
    (2048, 7168, 256, 8, 8, 4, 2.5),       # 32 tiles at V3 width, each split over 4 CTAs
])
def test_router_split_and_unsplit_reductions_agree(T, d, E, K, G, M, scale):
    """Small batches split each router tile's reduction over several CTAs;
    a workspace with room for the scores only forces the unsplit path.  The
    two sum the same exact products in different orders, so the affinities
    may differ in the last bits (router scores are not batch-invariant
    across split counts), but both stay within the oracle's error bound and
    the chosen experts agree on every token that is not a near tie."""
    assert moe.moe_router_splits(T, d, E) > 1
    g = torch.Generator().manual_seed(T + d + 1)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, d, generator=g) * 0.02).float()
    b = (torch.randn(E, generator=g) * 0.01).float()
    dev = "cuda"
    w_split = torch.empty(E, 3 * d, dtype=torch.bfloat16, device=dev)
    moe.moe_router_prepare(w.to(dev), E, d, w_split)
    scores_only = (T * E * 4 + 255) // 256 * 256
    out = {}
    for name, ws_b in (("split", moe.moe_workspace_bytes(T, d, E, K, 64)), ("unsplit", scores_only)):
        idx = torch.empty(T, K, dtype=torch.int32, device=dev)
        gate = torch.empty(T, K, device=dev)
        load = torch.empty(E, dtype=torch.int32, device=dev)
        aff = torch.empty(T, E, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = torch.empty(ws_b, dtype=torch.uint8, device=dev)
        moe.moe_router_topk(x.to(dev), w_split, None, None, b.to(dev), T, d, E, K, G, M, scale,
                            idx, gate, load, aff, status, ws, ws_b)
        assert sync_status(status) == 0
        out[name] = (idx.cpu().numpy(), aff.cpu().numpy().astype(np.float64))
    s64 = ref.router_affinity64(bf16_to_np64(x), w.numpy())
    for name in out:
        assert np.abs(out[name][1] - s64).max() < 4e-6, name
    kth, grp = ref.near_tie_tokens(s64, b.numpy(), K, G, M)
    diff = np.any(np.sort(out["split"][0], 1) != np.sort(out["unsplit"][0], 1), axis=1)
    assert not np.any(diff & ~(kth | grp)), np.nonzero(diff & ~(kth | grp))[0][:10]
