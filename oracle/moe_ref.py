"""Plain CPU reference (the oracle) for the DeepSeekMoE layer forward pass with
auxiliary-loss-free load balancing.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package's smoke check and
the benchmark's CPU-baseline / reference arm may import this module.  The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.

Everything here is written from the method's statement, not from any kernel:

* Selection score = affinity + per-expert bias; the bias only steers the top-K
  choice and never enters the gate value.  Sources: "DeepSeek-V3 Technical
  Report" reading notes (chenshi221.pages.dev), section "Auxiliary-loss-free
  负载均衡"; "DeepSeek-V3 Technical Report：中英对照解读" (weigao.cc), §3
  table row "DeepSeek-V3 uses an expert-level routing bias"; "DeepSeek V3"
  (deepseekmodel1.org), "公式解密: Score = Affinity + Bias".
* Loads are counted over the whole batch after the step; an overloaded expert
  has its bias lowered by gamma, an underloaded one raised by gamma.  Sources:
  the chenshi221 notes, same section (b_i <- b_i - gamma / + gamma); weigao.cc
  §3 row "The bias is updated from observed expert load"; qwbw.cn essay on the
  report, passage "训练的每一步结束之后统计整批样本各个专家的负载情况".
* Node (group) limited routing: each token reaches at most M nodes (M = 4 in
  the report).  Sources: chenshi221 notes, same section ("每个 token 最多发往
  M 个节点"); qwbw.cn essay, "每一个token最多被分发到4个节点".
* Shared experts see every token, routed experts are chosen per token.
  Source: weigao.cc §2 table rows "DeepSeekMoE" and "Shared experts and routed
  experts".

The task specification fixes what the pages leave open: the affinity is a
sigmoid, gates are normalised over the selected experts and then multiplied by
a route scale, groups are contiguous blocks of E/G experts, experts are SwiGLU
FFNs.  Readings of points the pages leave open (each also listed in the design
notes):

R1  Group score = sum of the ceil(K/M) largest biased scores of the group,
    added largest first.  Groups are ranked by that score, highest first,
    lower group index first on equal scores; the first M groups are kept.
R2  Expert order is the biased score, highest first, lower expert index first
    on equal scores.  -0.0 and +0.0 compare equal.  NaN ranks below every
    number (below -inf); experts of dropped groups rank below NaN.  The K
    selected experts are reported in that rank order.
R3  "Overloaded" means load_i > T*K/E, "underloaded" load_i < T*K/E, compared
    exactly as integers E*load_i vs T*K; at equality the bias is unchanged.
R4  Gate g_k = scale * s_k / sum_j s_j over the K selected experts, the sum
    taken in rank order.  In the fp32 rule every operation is one IEEE fp32
    operation: z = s + b; group score = top1 + top2 (+ ...); denominator
    accumulated in rank order; g = (s_k / denom) * scale.
R5  No capacity limit, no token dropping; no residual is added to the output.
R6  Layer output y(t) = sum over shared experts FFN_j(x_t)
                       + sum_k g_k * FFN_{idx_k}(x_t),
    FFN(v) = W2 (silu(W1 v) * (W3 v)), silu(a) = a / (1 + exp(-a)).
R7  Dispatch order: the rows sent to expert e are the (token, slot) pairs with
    idx == e in ascending (token, slot) order; experts are laid out in
    ascending expert order.
R8  Sequence-wise balance loss (the pages keep "a tiny-weight sequence-wise
    balance loss" next to the bias feedback -- chenshi221 notes, same section;
    weigao.cc §3 row "A small sequence-wise auxiliary loss is still used" --
    but print no formula).  Reading: for a sequence of T_s tokens,
      f_i = E / (K T_s) * #{(t, k): idx[t, k] = i},
      P_i = (1 / T_s) * sum_t s[t, i] / sum_j s[t, j],
      L   = alpha * sum_i f_i P_i.
    Its formula is therefore not fixed by the pages (parity unpinned against
    them); the pins fix the function against this reading.

Function-level parity status: every function below is pinned by the CPU test
suite (brute force, closed forms, invariants, hand-worked cases: load_stats
and both branches of near_tie_tokens included).  seq_balance_loss follows a
reading (R8) whose formula the pages do not print: parity unpinned against
the pages, pinned against the reading.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32
F64 = np.float64


# ---------------------------------------------------------------------------
# Step 1: affinities (sigmoid of the router logits).  Task spec step (1).
# ---------------------------------------------------------------------------
def sigmoid64(u):
    """s = 1 / (1 + exp(-u)) in float64."""
    u = np.asarray(u, dtype=F64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-u))


def router_logits64(x, w_r, logit_offset=None):
    """u[t, e] = sum_j x[t, j] * w_r[e, j] (+ o[e]) in float64.

    x holds the exact values of the bf16 activations, w_r the exact fp32
    router weights (the report keeps MoE gating in high precision: qwbw.cn
    essay, "MoE门控...依然保留BF16或者FP32高精度")."""
    u = np.asarray(x, dtype=F64) @ np.asarray(w_r, dtype=F64).T
    if logit_offset is not None:
        u = u + np.asarray(logit_offset, dtype=F64)[None, :]
    return u


def router_affinity64(x, w_r, logit_offset=None):
    return sigmoid64(router_logits64(x, w_r, logit_offset))


# ---------------------------------------------------------------------------
# Steps 2-3: biased, group-limited top-K and gates.
# ---------------------------------------------------------------------------
def _rank_desc(values, eligible):
    """Permutation along the last axis that lists entries in the order of
    readings R1/R2: eligible before ineligible, numbers before NaN, larger
    value first, lower index first among equals (+0.0 == -0.0)."""
    values = np.asarray(values)
    nan = np.isnan(values)
    klass = np.where(eligible, np.where(nan, 1, 2), 0)
    v = np.where(nan, 0.0, values).astype(F64)
    idx = np.broadcast_to(np.arange(values.shape[-1]), values.shape)
    # np.lexsort: the last key is the primary one, all keys ascending.
    return np.lexsort((idx, -v, -klass), axis=-1)


def select_experts(s, bias, K, n_groups=1, topk_groups=1, route_scale=1.0,
                   precision="fp32", return_detail=False):
    """Auxiliary-loss-free top-K routing for every token.

    s     [T, E] affinities; bias [E].  precision "fp32": every arithmetic
    operation is a single IEEE fp32 operation (the bit-exact rule R4);
    "fp64": the same steps in float64 (the end-to-end reference).
    Returns idx int32 [T, K] (rank order) and gate [T, K] in that precision.
    """
    dt = F32 if precision == "fp32" else F64
    s = np.asarray(s, dtype=dt)
    T, E = s.shape
    b = np.asarray(bias, dtype=dt)
    if not (1 <= K <= E):
        raise ValueError("need 1 <= K <= E")
    if E % n_groups or not (1 <= topk_groups <= n_groups):
        raise ValueError("bad group configuration")
    # score = affinity + bias (selection only)
    z = (s + b[None, :]).astype(dt)
    eligible = np.ones((T, E), dtype=bool)
    kept_groups = None
    if n_groups > 1:
        gsz = E // n_groups
        if K > topk_groups * gsz:
            raise ValueError("K larger than the experts in the kept groups")
        n_top = -(-K // topk_groups)  # ceil(K / M), reading R1
        if n_top > gsz:
            raise ValueError("ceil(K/M) larger than a group")
        zg = z.reshape(T, n_groups, gsz)
        order_in_group = _rank_desc(zg, np.ones_like(zg, dtype=bool))
        top = np.take_along_axis(zg, order_in_group[..., :n_top], axis=-1)
        gscore = top[..., 0].copy()
        for j in range(1, n_top):          # added largest first, in dt
            gscore = (gscore + top[..., j]).astype(dt)
        gorder = _rank_desc(gscore, np.ones_like(gscore, dtype=bool))
        kept_groups = np.sort(gorder[:, :topk_groups], axis=1)
        keep = np.zeros((T, n_groups), dtype=bool)
        np.put_along_axis(keep, gorder[:, :topk_groups], True, axis=1)
        eligible = np.repeat(keep, gsz, axis=1)
    order = _rank_desc(z, eligible)
    idx = order[:, :K].astype(np.int32)
    s_sel = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    denom = s_sel[:, 0].copy()
    for k in range(1, K):                  # rank order, in dt
        denom = (denom + s_sel[:, k]).astype(dt)
    gate = (s_sel / denom[:, None]).astype(dt)
    gate = (gate * dt(route_scale)).astype(dt)
    if return_detail:
        return idx, gate, dict(z=z, eligible=eligible, kept_groups=kept_groups)
    return idx, gate


def near_tie_tokens(s64, bias, K, n_groups=1, topk_groups=1, eps=1e-5):
    """Tokens whose selection is numerically fragile, in float64.

    Returns (kth_gap_mask, group_gap_mask): the K-th vs (K+1)-th biased-score
    gap among eligible experts is below eps, resp. (with a group limit) the
    M-th vs (M+1)-th group-score gap is below eps."""
    s64 = np.asarray(s64, dtype=F64)
    T, E = s64.shape
    idx, _, det = select_experts(s64, bias, K, n_groups, topk_groups, 1.0,
                                 precision="fp64", return_detail=True)
    z = det["z"]
    order = _rank_desc(z, det["eligible"])
    zs = np.take_along_axis(z, order, axis=1)
    elig = np.take_along_axis(det["eligible"], order, axis=1)
    kth = np.zeros(T, dtype=bool)
    if K < E:
        valid = elig[:, K]
        kth = valid & (np.abs(zs[:, K - 1] - zs[:, K]) < eps)
    grp = np.zeros(T, dtype=bool)
    if n_groups > 1 and topk_groups < n_groups:
        gsz = E // n_groups
        n_top = -(-K // topk_groups)
        zg = np.sort(z.reshape(T, n_groups, gsz), axis=-1)[..., ::-1]
        gscore = zg[..., :n_top].sum(axis=-1)
        gs = np.sort(gscore, axis=1)[:, ::-1]
        grp = np.abs(gs[:, topk_groups - 1] - gs[:, topk_groups]) < eps
    return kth, grp


# ---------------------------------------------------------------------------
# Step 5: load count and bias feedback.
# ---------------------------------------------------------------------------
def expert_load(idx, E):
    """load[e] = number of (token, slot) selections of expert e in the batch."""
    idx = np.asarray(idx)
    load = np.zeros(E, dtype=np.int64)
    for e in range(E):
        load[e] = int(np.count_nonzero(idx == e))
    return load.astype(np.int32)


def bias_update(load, bias, T, K, E, gamma):
    """b_i - gamma if overloaded, b_i + gamma if underloaded (reading R3),
    each a single fp32 operation."""
    load = np.asarray(load, dtype=np.int64)
    b = np.asarray(bias, dtype=F32)
    g = F32(gamma)
    over = E * load > T * K
    under = E * load < T * K
    out = b.copy()
    out[over] = (b[over] - g).astype(F32)
    out[under] = (b[under] + g).astype(F32)
    return out


def seq_balance_loss(s, idx, seq_offsets, K, alpha):
    """Reading R8, one value per sequence (float64)."""
    s = np.asarray(s, dtype=F64)
    idx = np.asarray(idx)
    T, E = s.shape
    out = []
    for a, b in zip(seq_offsets[:-1], seq_offsets[1:]):
        Ts = b - a
        if Ts == 0:
            out.append(0.0)
            continue
        count = np.zeros(E)
        for t in range(a, b):
            for k in range(K):
                count[idx[t, k]] += 1
        f = E / (K * Ts) * count
        P = (s[a:b] / s[a:b].sum(axis=1, keepdims=True)).sum(axis=0) / Ts
        out.append(alpha * float((f * P).sum()))
    return np.array(out, dtype=F64)


def load_stats(load):
    """(max, mean, max/mean, coefficient of variation) of the loads, taken
    over all E experts (untouched ones count as load 0).  The coefficient of
    variation is the population standard deviation (divide by E) over the
    mean; with no load at all every statistic is 0."""
    l = np.asarray(load, dtype=F64)
    mean = l.mean()
    mx = l.max()
    cv = l.std() / mean if mean > 0 else 0.0
    return np.array([mx, mean, mx / mean if mean > 0 else 0.0, cv], dtype=F64)


# ---------------------------------------------------------------------------
# Step 4: dispatch, experts, combine.
# ---------------------------------------------------------------------------
def silu64(a):
    a = np.asarray(a, dtype=F64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def swiglu_ffn64(X, W1, W3, W2):
    """FFN(v) = W2 (silu(W1 v) * (W3 v)) for every row v of X, in float64.
    W1, W3: [I, d]; W2: [d, I]."""
    X = np.asarray(X, dtype=F64)
    A = X @ np.asarray(W1, dtype=F64).T
    C = X @ np.asarray(W3, dtype=F64).T
    return (silu64(A) * C) @ np.asarray(W2, dtype=F64).T


def permute(idx, E):
    """Dispatch maps of reading R7.

    Returns offsets [E+1] (exclusive scan of the loads), row_of [T, K] (the
    row of x_perm holding (t, k)) and tok_of [T*K] (the token of each row)."""
    idx = np.asarray(idx)
    T, K = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")      # (t, k) ascending inside an expert
    load = expert_load(idx, E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + load[e]
    row_of = np.empty(T * K, dtype=np.int64)
    row_of[order] = np.arange(T * K)
    tok_of = order // K
    return (offsets.astype(np.int32), row_of.reshape(T, K).astype(np.int32),
            tok_of.astype(np.int32))


def combine64(y_perm, row_of, gate, y_shared=None):
    """out[t] = y_shared[t] + sum_k gate[t, k] * y_perm[row_of[t, k]] (fp64)."""
    y_perm = np.asarray(y_perm, dtype=F64)
    T, K = row_of.shape
    out = np.zeros((T, y_perm.shape[1]), dtype=F64)
    if y_shared is not None:
        out += np.asarray(y_shared, dtype=F64)
    for k in range(K):
        out += np.asarray(gate[:, k], dtype=F64)[:, None] * y_perm[row_of[:, k]]
    return out


def shared_ffn64(X, ws1, ws3, ws2, n_shared):
    """Sum of the n_shared shared experts.  Shared expert j owns rows
    j*I..(j+1)*I of ws1/ws3 ([n_shared*I, d]) and the same columns of ws2
    ([d, n_shared*I])."""
    ws1 = np.asarray(ws1)
    I = ws1.shape[0] // n_shared
    y = 0.0
    for j in range(n_shared):
        sl = slice(j * I, (j + 1) * I)
        y = y + swiglu_ffn64(X, ws1[sl], np.asarray(ws3)[sl], np.asarray(ws2)[:, sl])
    return np.asarray(y, dtype=F64)


def moe_output64(x, idx, gate, get_expert, shared, n_shared, tokens=None):
    """Layer output (reading R6) for the tokens `tokens` (default: all).

    get_expert(e) -> (W1 [I,d], W3 [I,d], W2 [d,I]) as arrays;
    shared = (ws1, ws3, ws2) or None.  Experts are evaluated once per expert
    on the rows routed to it (a sparse evaluation; the dense masked form
    below is its independent check)."""
    x = np.asarray(x, dtype=F64)
    T = x.shape[0]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    xs = x[tokens]
    out = np.zeros_like(xs)
    if shared is not None:
        out += shared_ffn64(xs, *shared, n_shared)
    sub_idx = np.asarray(idx)[tokens]
    sub_gate = np.asarray(gate, dtype=F64)[tokens]
    K = sub_idx.shape[1]
    for e in np.unique(sub_idx):
        w1, w3, w2 = get_expert(int(e))
        rows, slots = np.nonzero(sub_idx == e)
        y = swiglu_ffn64(xs[rows], w1, w3, w2)
        out[rows] += sub_gate[rows, slots][:, None] * y
    return out


def dense_masked_output64(x, idx, gate, W1, W3, W2, shared, n_shared):
    """Every routed expert on every token, masked by the gate matrix: the
    dense form of dispatch + combine, for tiny inputs only."""
    x = np.asarray(x, dtype=F64)
    T = x.shape[0]
    E = np.asarray(W1).shape[0]
    G = np.zeros((T, E), dtype=F64)
    idx = np.asarray(idx)
    gate = np.asarray(gate, dtype=F64)
    for t in range(T):
        for k in range(idx.shape[1]):
            G[t, idx[t, k]] += gate[t, k]
    out = np.zeros_like(x)
    if shared is not None:
        out += shared_ffn64(x, *shared, n_shared)
    for e in range(E):
        out += G[:, e:e + 1] * swiglu_ffn64(x, W1[e], W3[e], W2[e])
    return out


def bf16_to_f64(a):
    """Exact values of a bf16 array given as its uint16 bit patterns."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(F64)


def rel_l2(a, b):
    a = np.asarray(a, dtype=F64)
    b = np.asarray(b, dtype=F64)
    den = math.sqrt(float((b * b).sum()))
    return math.sqrt(float(((a - b) ** 2).sum())) / (den if den > 0 else 1.0)
