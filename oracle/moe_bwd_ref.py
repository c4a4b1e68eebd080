"""Plain CPU reference (the oracle) for the backward pass of the DeepSeekMoE
layer with auxiliary-loss-free balancing.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package's smoke check and
the benchmark's CPU-baseline / reference arm may import this module.  The
product path never imports it and shares no code with it.

What the pages fix: the per-expert bias only chooses experts and never enters
the gate value ("Bias 仅用于路由", deepseekmodel1.org, "公式解密"; chenshi221
notes, "Auxiliary-loss-free 负载均衡": the bias affects only the top-K choice,
not the gating value that multiplies the FFN output).  Hence:

R13  The gradient reaches the router through the gate values only, and the
     gate values depend on the raw affinities only.  The chosen expert set
     (top-K, group limit) is held fixed: the bias, the selection and the
     route scale carry no gradient; a logit offset is a constant input.
     With S = sum_j s_j over the K chosen experts and g_k = scale s_k / S,
       ds_m = scale (dg_m / S - sum_k dg_k s_k / S^2)  for chosen m, else 0,
       du   = ds s (1 - s),   dW_r = du^T x,   dx += du W_r.
     Every FFN is differentiated exactly:
       y = W2 h, h = silu(a) c, a = W1 v, c = W3 v,
       dh = W2^T dy, da = dh c silu'(a), dc = dh silu(a),
       dv = W1^T da + W3^T dc, dW2 = dy h^T, dW1 = da v^T, dW3 = dc v^T,
     with silu'(a) = sig(a) (1 + a (1 - sig(a))).  All in float64.

Parity status: pinned by central finite differences of the forward oracle
(moe_ref) along random directions, and by PyTorch autograd of the same
forward written with torch operations (tests/test_bwd_oracle_pins.py).
"""
from __future__ import annotations

import numpy as np

from . import moe_ref as ref

F64 = np.float64


def sigmoid_deriv64(u):
    s = ref.sigmoid64(u)
    return s * (1.0 - s)


def silu_deriv64(a):
    a = np.asarray(a, dtype=F64)
    sig = ref.sigmoid64(a)
    return sig * (1.0 + a * (1.0 - sig))


def swiglu_ffn_bwd64(X, W1, W3, W2, dY):
    """Gradients of sum(dY * FFN(X)) for FFN(v) = W2 (silu(W1 v) * (W3 v)).
    Returns (dX, dW1, dW3, dW2); X [n, d], W1/W3 [I, d], W2 [d, I]."""
    X, W1, W3, W2, dY = (np.asarray(t, dtype=F64) for t in (X, W1, W3, W2, dY))
    A = X @ W1.T
    C = X @ W3.T
    S = ref.silu64(A)
    H = S * C
    dH = dY @ W2
    dW2 = dY.T @ H
    dA = dH * C * silu_deriv64(A)
    dC = dH * S
    dX = dA @ W1 + dC @ W3
    return dX, dA.T @ X, dC.T @ X, dW2


def gate_bwd64(s_sel, dgate, route_scale):
    """ds for the chosen experts (R13) from the gate gradients; s_sel, dgate
    [T, K]."""
    s_sel = np.asarray(s_sel, dtype=F64)
    dgate = np.asarray(dgate, dtype=F64)
    S = s_sel.sum(axis=1, keepdims=True)
    return route_scale * (dgate / S - (dgate * s_sel).sum(axis=1, keepdims=True) / (S * S))


def moe_layer_bwd64(x, w_r, logit_offset, idx, route_scale, get_expert, shared, n_shared, dy):
    """Backward of the layer output of reading R6 for a fixed choice `idx`.

    x [T, d], w_r [E, d], dy [T, d]; get_expert(e) -> (W1, W3, W2);
    shared = (ws1, ws3, ws2) side by side or None.
    Returns dict: dx [T, d], dw_r [E, d], experts {e: (dW1, dW3, dW2)},
    shared (dws1, dws3, dws2) or None, dgate [T, K], du [T, E]."""
    x = np.asarray(x, dtype=F64)
    dy = np.asarray(dy, dtype=F64)
    w_r = np.asarray(w_r, dtype=F64)
    idx = np.asarray(idx)
    T, K = idx.shape
    E = w_r.shape[0]
    u = x @ w_r.T
    if logit_offset is not None:
        u = u + np.asarray(logit_offset, dtype=F64)[None, :]
    s = ref.sigmoid64(u)
    s_sel = np.take_along_axis(s, idx, axis=1)
    gate = route_scale * s_sel / s_sel.sum(axis=1, keepdims=True)
    dx = np.zeros_like(x)
    dgate = np.zeros((T, K), dtype=F64)
    experts = {}
    for e in np.unique(idx):
        W1, W3, W2 = (np.asarray(t, dtype=F64) for t in get_expert(int(e)))
        rows, slots = np.nonzero(idx == e)
        Y = ref.swiglu_ffn64(x[rows], W1, W3, W2)
        dgate[rows, slots] = (dy[rows] * Y).sum(axis=1)
        dXe, dW1, dW3, dW2 = swiglu_ffn_bwd64(x[rows], W1, W3, W2, gate[rows, slots][:, None] * dy[rows])
        dx[rows] += dXe
        experts[int(e)] = (dW1, dW3, dW2)
    shared_grads = None
    if shared is not None:
        ws1, ws3, ws2 = (np.asarray(t, dtype=F64) for t in shared)
        I = ws1.shape[0] // n_shared
        g1 = np.zeros_like(ws1)
        g3 = np.zeros_like(ws3)
        g2 = np.zeros_like(ws2)
        for j in range(n_shared):
            sl = slice(j * I, (j + 1) * I)
            dXs, dW1, dW3, dW2 = swiglu_ffn_bwd64(x, ws1[sl], ws3[sl], ws2[:, sl], dy)
            dx += dXs
            g1[sl], g3[sl], g2[:, sl] = dW1, dW3, dW2
        shared_grads = (g1, g3, g2)
    ds_sel = gate_bwd64(s_sel, dgate, route_scale)
    ds = np.zeros((T, E), dtype=F64)
    np.put_along_axis(ds, idx, ds_sel, axis=1)
    du = ds * s * (1.0 - s)
    dx += du @ w_r
    return dict(dx=dx, dw_r=du.T @ x, experts=experts, shared=shared_grads, dgate=dgate, du=du)
