"""Pins of the backward oracle (CPU): central finite differences of the
forward oracle along random directions, PyTorch autograd of the same forward,
and closed forms."""
import numpy as np
import pytest
import torch

from oracle import moe_bwd_ref as B
from oracle import moe_ref as ref


def _problem(seed, T=7, d=16, E=6, K=2, I=8, n_shared=1, offset=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    w_r = rng.standard_normal((E, d)) * 0.3
    off = rng.standard_normal(E) * 0.2 if offset else None
    W1 = rng.standard_normal((E, I, d)) * 0.3
    W3 = rng.standard_normal((E, I, d)) * 0.3
    W2 = rng.standard_normal((E, d, I)) * 0.3
    ws = (rng.standard_normal((n_shared * I, d)) * 0.3, rng.standard_normal((n_shared * I, d)) * 0.3,
          rng.standard_normal((d, n_shared * I)) * 0.3)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    dy = rng.standard_normal((T, d))
    return dict(x=x, w_r=w_r, off=off, W1=W1, W3=W3, W2=W2, ws=ws, idx=idx, dy=dy, n_shared=n_shared)


def _loss(P, scale):
    """<dy, y> with the chosen experts held fixed, from the forward oracle."""
    s = ref.router_affinity64(P["x"], P["w_r"], P["off"])
    s_sel = np.take_along_axis(s, P["idx"], axis=1)
    gate = scale * s_sel / s_sel.sum(axis=1, keepdims=True)
    y = ref.moe_output64(P["x"], P["idx"], gate, lambda e: (P["W1"][e], P["W3"][e], P["W2"][e]),
                         P["ws"], P["n_shared"])
    return float((P["dy"] * y).sum())


def _grads(P, scale):
    return B.moe_layer_bwd64(P["x"], P["w_r"], P["off"], P["idx"], scale,
                             lambda e: (P["W1"][e], P["W3"][e], P["W2"][e]), P["ws"], P["n_shared"],
                             P["dy"])


def _expert_grad(G, E, which, shape):
    out = np.zeros((E,) + shape)
    for e, g in G["experts"].items():
        out[e] = g[which]
    return out


@pytest.mark.parametrize("seed,scale,n_shared", [(0, 1.0, 1), (1, 2.5, 2)])
def test_backward_matches_finite_differences(seed, scale, n_shared):
    P = _problem(seed, n_shared=n_shared)
    G = _grads(P, scale)
    E, I, d = P["W1"].shape
    grads = {
        "x": G["dx"], "w_r": G["dw_r"],
        "W1": _expert_grad(G, E, 0, (I, d)), "W3": _expert_grad(G, E, 1, (I, d)),
        "W2": _expert_grad(G, E, 2, (d, I)),
    }
    rng = np.random.default_rng(100 + seed)
    eps = 1e-6
    for name, g in grads.items():
        for _ in range(3):
            V = rng.standard_normal(P[name].shape)
            Pp = dict(P); Pp[name] = P[name] + eps * V
            Pm = dict(P); Pm[name] = P[name] - eps * V
            fd = (_loss(Pp, scale) - _loss(Pm, scale)) / (2 * eps)
            an = float((g * V).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)
    # the shared experts' weights
    for j, name in enumerate(["ws1", "ws3", "ws2"]):
        V = rng.standard_normal(P["ws"][j].shape)
        wp = list(P["ws"]); wp[j] = P["ws"][j] + eps * V
        wm = list(P["ws"]); wm[j] = P["ws"][j] - eps * V
        Pp = dict(P); Pp["ws"] = tuple(wp)
        Pm = dict(P); Pm["ws"] = tuple(wm)
        fd = (_loss(Pp, scale) - _loss(Pm, scale)) / (2 * eps)
        an = float((G["shared"][j] * V).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_backward_matches_torch_autograd():
    P = _problem(3, T=9, d=12, E=5, K=3, I=6, n_shared=1)
    scale = 2.5
    G = _grads(P, scale)
    t = {k: torch.tensor(P[k], dtype=torch.float64, requires_grad=True)
         for k in ("x", "w_r", "W1", "W3", "W2")}
    ws = [torch.tensor(w, dtype=torch.float64, requires_grad=True) for w in P["ws"]]
    off = torch.tensor(P["off"], dtype=torch.float64)
    idx = torch.tensor(P["idx"])
    s = torch.sigmoid(t["x"] @ t["w_r"].T + off)
    s_sel = torch.gather(s, 1, idx)
    gate = scale * s_sel / s_sel.sum(1, keepdim=True)
    y = torch.nn.functional.silu(t["x"] @ ws[0].T) * (t["x"] @ ws[1].T) @ ws[2].T
    for k in range(idx.shape[1]):
        e = idx[:, k]
        a = torch.einsum("td,tid->ti", t["x"], t["W1"][e])
        c = torch.einsum("td,tid->ti", t["x"], t["W3"][e])
        y = y + gate[:, k:k + 1] * torch.einsum("ti,tdi->td", torch.nn.functional.silu(a) * c, t["W2"][e])
    (y * torch.tensor(P["dy"])).sum().backward()
    np.testing.assert_allclose(G["dx"], t["x"].grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(G["dw_r"], t["w_r"].grad.numpy(), rtol=1e-10, atol=1e-12)
    E, I, d = P["W1"].shape
    for which, name in enumerate(["W1", "W3", "W2"]):
        shape = (I, d) if which < 2 else (d, I)
        np.testing.assert_allclose(_expert_grad(G, E, which, shape), t[name].grad.numpy(),
                                   rtol=1e-10, atol=1e-12)
    for j in range(3):
        np.testing.assert_allclose(G["shared"][j], ws[j].grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_closed_forms():
    # one expert per token: the gate is the constant route scale, so the
    # router gets no gradient at all (R13)
    P = _problem(5, K=1, n_shared=1)
    G = _grads(P, 2.5)
    assert np.abs(G["du"]).max() < 1e-15 and np.abs(G["dw_r"]).max() < 1e-14
    # silu'(0) = 1/2, sigmoid'(0) = 1/4
    assert B.silu_deriv64(0.0) == 0.5
    assert B.sigmoid_deriv64(0.0) == 0.25
    # gate gradient: equal affinities and dgate = e_1 give ds = scale (1/S)(e_1 - 1/K)
    s_sel = np.full((1, 4), 0.5)
    dg = np.array([[1.0, 0.0, 0.0, 0.0]])
    ds = B.gate_bwd64(s_sel, dg, 2.0)
    np.testing.assert_allclose(ds, 2.0 / 2.0 * (np.array([[1.0, 0, 0, 0]]) - 0.25), rtol=0, atol=1e-15)
    # the chosen set's gates sum to scale, so ds is orthogonal to s_sel
    rng = np.random.default_rng(9)
    s_sel = rng.uniform(0.1, 0.9, (5, 3))
    ds = B.gate_bwd64(s_sel, rng.standard_normal((5, 3)), 1.7)
    np.testing.assert_allclose((ds * s_sel).sum(axis=1), 0.0, atol=1e-14)
