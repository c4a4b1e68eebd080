"""Backward pass of the layer on the GPU against the fp64 backward oracle:
each kernel on synthetic inputs, then whole passes on the tiny and mid
workloads.

Tolerances.  Weight gradients are fp32 sums of bf16 products (fp32 rounding
only); activation gradients are bf16 and pass through at most six bf16
roundings in sequence (g dy, dh, a, c, [da | dc], dv), unit roundoff 2^-9
each, so a relative L2 error below 1e-2 against the fp64 oracle leaves a
wide margin while a dropped term or a wrong index fails it by far."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_affinity_b300 as moe
from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.layer import MoELayer
from oracle import moe_bwd_ref as B
from oracle import moe_ref as ref
from _util import HostExperts, bf16_to_np64, sync_status

pytestmark = pytest.mark.gpu


def _bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _close(got, want, rel, abs_scale):
    err = np.abs(got - want)
    bound = rel * np.abs(want) + abs_scale
    bad = err > bound
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], want[bad][:5])


# ------------------------------------------------------------------ kernels
@pytest.mark.parametrize("sizes,K,N", [
    ([3, 0, 130, 64, 1, 257], 256, 136),
    ([300, 290, 0, 511, 17, 256, 700, 2], 2048, 1408),
    ([1], 64, 8),
])
def test_grouped_gemm_nt(sizes, K, N):
    G, R = len(sizes), sum(sizes)
    off = _offsets(sizes)
    a = _bf16((R, K), 1)
    w = _bf16((G, N, K), 2, 0.05)
    out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm(a.cuda(), torch.from_numpy(off).cuda(), G, R, K, N, w.cuda(), out, st)
    assert sync_status(st) == 0
    a64, w64, got = bf16_to_np64(a), bf16_to_np64(w), bf16_to_np64(out)
    want = np.concatenate([a64[off[g]:off[g + 1]] @ w64[g].T for g in range(G)])
    rms = np.sqrt(np.mean(want ** 2))
    _close(got, want, 2.0 ** -8, 1e-4 * rms)


@pytest.mark.parametrize("sizes,M,N", [
    ([0, 1, 63, 64, 65, 200], 200, 136),       # ragged tails, empty group, ragged M and N
    ([310, 0, 290, 511, 129], 2048, 1408),
    ([4096], 256, 512),
    ([0, 0, 5], 64, 64),
    ([3] * 40 + [700], 128, 264),              # many tails in a row, one long group
])
def test_grouped_wgrad(sizes, M, N):
    G, R = len(sizes), sum(sizes)
    a, b = _bf16((R, M), 3), _bf16((R, N), 4)
    off = _offsets(sizes)
    out = torch.full((G, M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm_wgrad(a.cuda(), b.cuda(), torch.from_numpy(off).cuda(), G, R, M, N, out,
                               st)
    assert sync_status(st) == 0
    got = out.cpu().numpy().astype(np.float64)
    a64, b64 = bf16_to_np64(a), bf16_to_np64(b)
    for g in range(G):
        A, Bm = a64[off[g]:off[g + 1]], b64[off[g]:off[g + 1]]
        if sizes[g] == 0:
            assert np.all(got[g] == 0.0), g
            continue
        _close(got[g], A.T @ Bm, 0.0, 4e-6 * (np.abs(A).T @ np.abs(Bm)) + 1e-30)


def test_grouped_wgrad_ignores_neighbour_rows():
    """The rows after a group's last token (next group, here huge values)
    must not leak into a ragged tail."""
    sizes = [37, 64, 1]
    G, R, M, N = 3, 102, 64, 64
    a, b = _bf16((R, M), 5), _bf16((R, N), 6)
    a[37:101] = 3.0e4
    b[37:101] = -3.0e4
    off = _offsets(sizes)
    out = torch.empty((G, M, N), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm_wgrad(a.cuda(), b.cuda(), torch.from_numpy(off).cuda(), G, R, M, N, out,
                               st)
    assert sync_status(st) == 0
    a64, b64 = bf16_to_np64(a), bf16_to_np64(b)
    A, Bm = a64[:37], b64[:37]
    _close(out[0].cpu().numpy().astype(np.float64), A.T @ Bm, 0.0,
           4e-6 * (np.abs(A).T @ np.abs(Bm)) + 1e-30)


@pytest.mark.parametrize("sizes,K,N,two", [
    ([3, 0, 130, 64, 1, 257], 256, 136, False),
    ([3, 0, 130, 64, 1, 257], 256, 136, True),
    ([300, 290, 0, 511, 17, 256, 700, 2], 2048, 1408, False),
    ([300, 290, 0, 511, 17, 256, 700, 2], 2816, 2048, True),
    ([1], 128, 8, True),
])
def test_grouped_gemm_kn(sizes, K, N, two):
    """out[r] = a[r] . w[g] with w [G, K, N] (or two stacked halves along K)."""
    G, R = len(sizes), sum(sizes)
    off = _offsets(sizes)
    a = _bf16((R, K), 41)
    K0 = K // 2 if two else K
    w0 = _bf16((G, K0, N), 42, 0.05)
    w1 = _bf16((G, K0, N), 43, 0.05) if two else None
    out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm_kn(a.cuda(), torch.from_numpy(off).cuda(), G, R, K, N, w0.cuda(),
                            w1.cuda() if two else None, out, st)
    assert sync_status(st) == 0
    a64, got = bf16_to_np64(a), bf16_to_np64(out)
    w64 = bf16_to_np64(w0)
    if two:
        w64 = np.concatenate([w64, bf16_to_np64(w1)], axis=1)
    want = np.concatenate([a64[off[g]:off[g + 1]] @ w64[g] for g in range(G)])
    rms = np.sqrt(np.mean(want ** 2))
    _close(got, want, 2.0 ** -8, 1e-4 * rms)


def _routing(T, K, E, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    off, row_of, tok_of = ref.permute(idx, E)
    return idx, off.astype(np.int32), row_of.astype(np.int32), tok_of.astype(np.int32)


def test_combine_backward_and_swiglu_backward():
    T, K, E, d, I = 300, 3, 8, 136, 72
    idx, off, row_of, tok_of = _routing(T, K, E, 7)
    dy, y_perm = _bf16((T, d), 8), _bf16((T * K, d), 9)
    gate = torch.rand(T, K, generator=torch.Generator().manual_seed(10)) * 2.5
    dy_perm = torch.empty(T * K, d, dtype=torch.bfloat16, device="cuda")
    dgate = torch.empty(T, K, dtype=torch.float32, device="cuda")
    moe.moe_combine_backward(dy.cuda(), y_perm.cuda(), torch.from_numpy(row_of).cuda(),
                             gate.cuda(), T, K, d, dy_perm, dgate)
    torch.cuda.synchronize()
    dy64, y64, g64 = bf16_to_np64(dy), bf16_to_np64(y_perm), gate.numpy().astype(np.float64)
    want_perm = np.zeros((T * K, d))
    want_perm[row_of.reshape(-1)] = (g64[:, :, None] * dy64[:, None, :]).reshape(T * K, d)
    _close(bf16_to_np64(dy_perm), want_perm, 2.0 ** -8, 0.0)
    ysel = y64[row_of]                                   # [T, K, d]
    want_dg = np.einsum("td,tkd->tk", dy64, ysel)
    _close(dgate.cpu().numpy().astype(np.float64), want_dg, 0.0,
           1e-5 * np.einsum("td,tkd->tk", np.abs(dy64), np.abs(ysel)))
    # SwiGLU backward
    R = 500
    dh, a, c = _bf16((R, I), 11), _bf16((R, I), 12, 3.0), _bf16((R, I), 13)
    dac = torch.empty(R, 2 * I, dtype=torch.bfloat16, device="cuda")
    h = torch.empty(R, I, dtype=torch.bfloat16, device="cuda")
    moe.moe_swiglu_backward(dh.cuda(), a.cuda(), c.cuda(), R, I, dac, h)
    torch.cuda.synchronize()
    dh64, a64, c64 = bf16_to_np64(dh), bf16_to_np64(a), bf16_to_np64(c)
    da = dh64 * c64 * B.silu_deriv64(a64)
    dc = dh64 * ref.silu64(a64)
    got = bf16_to_np64(dac)
    scale = 1e-6 * np.abs(dh64 * c64).max()
    _close(got[:, :I], da, 2.0 ** -7, scale)
    _close(got[:, I:], dc, 2.0 ** -7, scale)
    _close(bf16_to_np64(h), ref.silu64(a64) * c64, 2.0 ** -7, 1e-6 * np.abs(a64 * c64).max())


@pytest.mark.parametrize("T,K,E,d,scale", [(400, 4, 16, 200, 2.5), (1, 8, 256, 64, 1.0),
                                           (257, 1, 8, 16, 1.0)])
def test_router_backward(T, K, E, d, scale):
    idx, off, row_of, tok_of = _routing(T, K, E, 20 + T)
    rng = np.random.default_rng(21)
    aff = rng.uniform(0.05, 0.95, (T, E)).astype(np.float32)
    dgate = rng.standard_normal((T, K)).astype(np.float32)
    w_r = (rng.standard_normal((E, d)) * 0.1).astype(np.float32)
    x = _bf16((T, d), 22)
    dev = "cuda"
    du = torch.empty(T, K, dtype=torch.float32, device=dev)
    du_row = torch.empty(T * K, dtype=torch.float32, device=dev)
    dx_r = torch.empty(T, d, dtype=torch.float32, device=dev)
    dw_r = torch.full((E, d), float("nan"), dtype=torch.float32, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    moe.moe_router_backward(t(dgate), t(idx), K, t(aff), t(w_r), x.to(dev), t(row_of), t(tok_of),
                            t(off), T, d, E, K, scale, du, du_row, dx_r, dw_r)
    torch.cuda.synchronize()
    s_sel = np.take_along_axis(aff.astype(np.float64), idx, axis=1)
    ds = B.gate_bwd64(s_sel, dgate.astype(np.float64), scale)
    want_du = ds * s_sel * (1.0 - s_sel)
    mag = scale * np.abs(dgate).max() / s_sel.sum(1, keepdims=True)
    _close(du.cpu().numpy().astype(np.float64), want_du, 0.0, 1e-5 * mag)
    du_full = np.zeros((T, E))
    np.put_along_axis(du_full, idx, want_du, axis=1)
    # the error bound of each du entry (s (1 - s) <= 1/4) carried through the sums
    du_abs = np.zeros((T, E))
    np.put_along_axis(du_abs, idx, np.abs(want_du) + 0.25 * mag, axis=1)
    w64, x64 = w_r.astype(np.float64), bf16_to_np64(x)
    _close(dx_r.cpu().numpy().astype(np.float64), du_full @ w64, 0.0,
           1e-5 * (du_abs @ np.abs(w64)) + 1e-30)
    _close(dw_r.cpu().numpy().astype(np.float64), du_full.T @ x64, 0.0,
           1e-5 * (du_abs.T @ np.abs(x64)) + 1e-30)
    if K == 1:   # one chosen expert: its gate is the constant route scale
        assert not du.abs().max().item() and not dw_r.abs().max().item()


def test_combine_dx():
    T, K, E, d = 333, 3, 8, 72
    idx, off, row_of, tok_of = _routing(T, K, E, 30)
    dxp, dxs = _bf16((T * K, d), 31), _bf16((T, d), 32)
    dxr = torch.randn(T, d, generator=torch.Generator().manual_seed(33))
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_combine_dx(dxp.cuda(), torch.from_numpy(row_of).cuda(), K, dxs.cuda(), dxr.cuda(), T, d,
                       out)
    torch.cuda.synchronize()
    want = bf16_to_np64(dxs) + dxr.numpy().astype(np.float64) + bf16_to_np64(dxp)[row_of].sum(1)
    _close(bf16_to_np64(out), want, 2.0 ** -8, 1e-6)
    moe.moe_combine_dx(dxp.cuda(), torch.from_numpy(row_of).cuda(), K, None, None, T, d, out)
    torch.cuda.synchronize()
    _close(bf16_to_np64(out), bf16_to_np64(dxp)[row_of].sum(1), 2.0 ** -8, 1e-6)


# -------------------------------------------------------------------- layer
def _layer_case(cfg, p, T=None, training=True):
    """Forward + backward on the GPU; the oracle's own routing and gates.
    Tokens whose choice is a near tie for the oracle get dy = 0 on both
    sides, so they contribute nothing to any gradient."""
    T = cfg.T if T is None else T
    x = synth.make_tokens(cfg, 0, "cpu", T=T)
    dy = synth.make_output_grad(cfg, 0, "cpu", T=T)
    x64 = bf16_to_np64(x)
    off = p["logit_offset"].numpy() if p["logit_offset"] is not None else None
    s64 = ref.router_affinity64(x64, p["w_r"].numpy(), off)
    b = p["bias"].numpy()
    idx64, gate64 = ref.select_experts(s64, b.astype(np.float64), cfg.K, cfg.n_groups,
                                       cfg.topk_groups, cfg.route_scale, precision="fp64")
    kth, grp = ref.near_tie_tokens(s64, b, cfg.K, cfg.n_groups, cfg.topk_groups)
    tie = kth | grp
    dy[torch.from_numpy(tie)] = 0
    layer = (MoELayer(cfg, p, max_T=T, training=True) if training
             else MoELayer(cfg, p, max_T=T, keep_affinity=True))
    layer.forward(x.cuda())
    g = layer.backward(x.cuda(), dy.cuda())
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    gidx = layer.idx[:T, :cfg.K].cpu().numpy()
    mism = np.any(np.sort(gidx, 1) != np.sort(idx64, 1), axis=1)
    assert not np.any(mism & ~tie)
    return dict(x64=x64, dy64=bf16_to_np64(dy), off=off, idx64=idx64, gate64=gate64, tie=tie,
                gidx=gidx, g={k: v.cpu() for k, v in g.items()})


def _by_gpu_slot(want_tk, idx64, gidx, E):
    """The oracle's per-(token, slot) values, moved to the GPU's slot order
    (the same experts in each token's row, possibly listed differently)."""
    full = np.zeros((want_tk.shape[0], E))
    np.put_along_axis(full, idx64, want_tk, axis=1)
    return np.take_along_axis(full, gidx, axis=1)


def _np(t):
    return bf16_to_np64(t) if t.dtype == torch.bfloat16 else t.numpy().astype(np.float64)


@pytest.mark.parametrize("training", [True, False])
def test_layer_backward_tiny_all_gradients(training):
    """training=True: the pre-activations come from the forward pass;
    False: the backward recomputes them."""
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    c = _layer_case(cfg, p, training=training)
    host = HostExperts(p)
    want = B.moe_layer_bwd64(c["x64"], p["w_r"].numpy(), c["off"], c["idx64"], cfg.route_scale,
                             host, host.shared(), cfg.n_shared, c["dy64"])
    g = c["g"]
    assert ref.rel_l2(_np(g["dx"]), want["dx"]) < 1e-2
    dg_want = _by_gpu_slot(want["dgate"], c["idx64"], c["gidx"], cfg.E)
    assert ref.rel_l2(_np(g["dgate"]), dg_want) < 1e-2
    du_want = np.take_along_axis(want["du"], c["gidx"], axis=1)
    assert ref.rel_l2(_np(g["du"]), du_want) < 1e-2
    assert ref.rel_l2(_np(g["dw_r"]), want["dw_r"]) < 1e-2
    I = cfg.I
    dw13, dw2 = _np(g["dw13"]), _np(g["dw2"])
    for e in range(cfg.E):
        if e in want["experts"]:
            w1, w3, w2 = want["experts"][e]
        else:
            w1 = w3 = np.zeros((I, cfg.d))
            w2 = np.zeros((cfg.d, I))
        got = np.concatenate([dw13[e].ravel(), dw2[e].ravel()])
        ref_e = np.concatenate([w1.ravel(), w3.ravel(), w2.ravel()])
        if not np.any(ref_e):
            assert not np.any(got)
        else:
            assert ref.rel_l2(got, ref_e) < 1e-2, e
    s1, s3, s2 = want["shared"]
    nI = cfg.n_shared * I
    assert ref.rel_l2(_np(g["dws13"])[:nI], s1) < 1e-2
    assert ref.rel_l2(_np(g["dws13"])[nI:], s3) < 1e-2
    assert ref.rel_l2(_np(g["dws2"]), s2) < 1e-2


def test_layer_backward_deterministic():
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cuda")
    dy = synth.make_output_grad(cfg, 0, "cuda")
    layer = MoELayer(cfg, p, training=True)
    runs = []
    for _ in range(2):
        layer.forward(x)
        g = layer.backward(x, dy)
        runs.append({k: v.clone() for k, v in g.items()})
    torch.cuda.synchronize()
    for k in runs[0]:
        assert torch.equal(runs[0][k].view(torch.int16) if runs[0][k].dtype == torch.bfloat16
                           else runs[0][k].view(torch.int32),
                           runs[1][k].view(torch.int16) if runs[1][k].dtype == torch.bfloat16
                           else runs[1][k].view(torch.int32)), k


def test_layer_backward_mid_sampled():
    """mid workload: dx, dgate and du on 256 sampled tokens (each token's
    gradients depend on that token alone for a fixed choice of experts), the
    weight gradients of three experts over all their tokens."""
    cfg = synth.CONFIGS["mid"]
    p = synth.make_params(cfg, "cpu")
    c = _layer_case(cfg, p)
    host = HostExperts(p)
    tok = np.random.default_rng(1).choice(cfg.T, 256, replace=False)
    tok = tok[~c["tie"][tok]]
    want = B.moe_layer_bwd64(c["x64"][tok], p["w_r"].numpy(), c["off"], c["idx64"][tok],
                             cfg.route_scale, host, host.shared(), cfg.n_shared, c["dy64"][tok])
    g = c["g"]
    assert ref.rel_l2(_np(g["dx"])[tok], want["dx"]) < 1e-2
    gidx = c["gidx"][tok]
    assert ref.rel_l2(_np(g["dgate"])[tok],
                      _by_gpu_slot(want["dgate"], c["idx64"][tok], gidx, cfg.E)) < 1e-2
    assert ref.rel_l2(_np(g["du"])[tok], np.take_along_axis(want["du"], gidx, 1)) < 1e-2
    dw13, dw2 = _np(g["dw13"]), _np(g["dw2"])
    for e in (0, 17, 63):
        rows, slots = np.nonzero(c["idx64"] == e)
        W1, W3, W2 = host(e)
        dYe = c["gate64"][rows, slots][:, None] * c["dy64"][rows]
        _, dW1, dW3, dW2 = B.swiglu_ffn_bwd64(c["x64"][rows], W1, W3, W2, dYe)
        assert ref.rel_l2(dw13[e, :cfg.I], dW1) < 1e-2, e
        assert ref.rel_l2(dw13[e, cfg.I:], dW3) < 1e-2, e
        assert ref.rel_l2(dw2[e], dW2) < 1e-2, e


def test_forward_keeps_pre_activations():
    """training=True: the forward writes a = v.W1^T and c = v.W3^T of every
    dispatched row (bf16 of the GEMM's fp32 accumulators), and its output is
    the inference forward's, bit for bit."""
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cpu")
    lt = MoELayer(cfg, p, training=True)
    li = MoELayer(cfg, p)
    yt = lt.forward(x.cuda()).clone()
    yi = li.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert torch.equal(yt.view(torch.int16), yi.view(torch.int16))
    R = cfg.T * cfg.K
    tok = lt.tok_of[:R].cpu().numpy()
    off = lt.offsets.cpu().numpy()
    expert = np.searchsorted(off, np.arange(R), side="right") - 1
    x64 = bf16_to_np64(x)
    host = HostExperts(p)
    got_a, got_c = bf16_to_np64(lt.pre_a[:R]), bf16_to_np64(lt.pre_c[:R])
    for e in np.unique(expert):
        rows = np.nonzero(expert == e)[0]
        W1, W3, _ = host(e)
        want_a, want_c = x64[tok[rows]] @ W1.T, x64[tok[rows]] @ W3.T
        scale = 1e-4 * np.sqrt(np.mean(want_a ** 2))
        _close(got_a[rows], want_a, 2.0 ** -8, scale)
        _close(got_c[rows], want_c, 2.0 ** -8, scale)
    ws1, ws3, _ = host.shared()
    _close(bf16_to_np64(lt.pre_a_sh[:cfg.T]), x64 @ ws1.T, 2.0 ** -8, 1e-4)
    _close(bf16_to_np64(lt.pre_c_sh[:cfg.T]), x64 @ ws3.T, 2.0 ** -8, 1e-4)


@pytest.mark.parametrize("R,I", [(37, 70), (129, 8), (1, 2)])
def test_swiglu_backward_narrow_and_small(R, I):
    """Widths that are not a multiple of 8 take the two-column path."""
    dh, a, c = _bf16((R, I), 51), _bf16((R, I), 52, 3.0), _bf16((R, I), 53)
    dac = torch.empty(R, 2 * I, dtype=torch.bfloat16, device="cuda")
    moe.moe_swiglu_backward(dh.cuda(), a.cuda(), c.cuda(), R, I, dac, None)
    torch.cuda.synchronize()
    dh64, a64, c64 = bf16_to_np64(dh), bf16_to_np64(a), bf16_to_np64(c)
    got = bf16_to_np64(dac)
    scale = 1e-6 * max(np.abs(dh64 * c64).max(), 1e-30)
    _close(got[:, :I], dh64 * c64 * B.silu_deriv64(a64), 2.0 ** -7, scale)
    _close(got[:, I:], dh64 * ref.silu64(a64), 2.0 ** -7, scale)


@pytest.mark.parametrize("T", [1, 3, 129])
def test_layer_backward_odd_token_counts(T):
    """Few tokens: most experts get no rows, the rest ragged tails of 1..3
    rows; every gradient against the oracle."""
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    c = _layer_case(cfg, p, T=T)
    host = HostExperts(p)
    want = B.moe_layer_bwd64(c["x64"], p["w_r"].numpy(), c["off"], c["idx64"], cfg.route_scale,
                             host, host.shared(), cfg.n_shared, c["dy64"])
    g = c["g"]
    assert ref.rel_l2(_np(g["dx"]), want["dx"]) < 1e-2
    assert ref.rel_l2(_np(g["dw_r"]), want["dw_r"]) < 1e-2 or not np.any(want["dw_r"])
    I = cfg.I
    dw13, dw2 = _np(g["dw13"]), _np(g["dw2"])
    for e in range(cfg.E):
        if e in want["experts"]:
            w1, w3, w2 = want["experts"][e]
            assert ref.rel_l2(np.concatenate([dw13[e].ravel(), dw2[e].ravel()]),
                              np.concatenate([w1.ravel(), w3.ravel(), w2.ravel()])) < 1e-2, e
        else:
            assert not np.any(dw13[e]) and not np.any(dw2[e]), e
    s1, s3, s2 = want["shared"]
    nI = cfg.n_shared * I
    assert ref.rel_l2(_np(g["dws13"])[:nI], s1) < 1e-2
    assert ref.rel_l2(_np(g["dws2"]), s2) < 1e-2
