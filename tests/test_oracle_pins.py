"""Pins for the CPU oracle: checks against what the method's statement and
plain mathematics fix, written independently of the oracle's own code
(brute-force enumeration, closed forms, hand-worked cases, invariants).

Runs on CPU only."""
import itertools
import json
import math
import os
import struct

import numpy as np
import pytest

from oracle import moe_ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(x: float) -> float:
    """Round a Python float to the nearest fp32 value (ties to even)."""
    return struct.unpack("f", struct.pack("f", x))[0]


def beats(zi, i, zj, j):
    """Total order of the selection rule: numbers above NaN, larger first,
    lower index first on equal values (+0 == -0)."""
    ni, nj = math.isnan(zi), math.isnan(zj)
    if ni or nj:
        if ni and nj:
            return i < j
        return nj
    if zi != zj:
        return zi > zj
    return i < j


def brute_topk(z, cand, K):
    """Enumerate all K-subsets of `cand`; return the unique one whose every
    member beats every non-member, ordered by the rule."""
    winners = []
    for S in itertools.combinations(cand, K):
        rest = [j for j in cand if j not in S]
        if all(beats(z[i], i, z[j], j) for i in S for j in rest):
            winners.append(S)
    assert len(winners) == 1
    S = list(winners[0])
    # order inside the set by pairwise wins
    return sorted(S, key=lambda i: -sum(beats(z[i], i, z[j], j) for j in S))


def brute_route_token(s, b, K, G, M, scale):
    E = len(s)
    z = [f32(s[e] + b[e]) for e in range(E)]
    cand = list(range(E))
    if G > 1:
        gsz = E // G
        n_top = -(-K // M)
        gscore = []
        for g in range(G):
            members = list(range(g * gsz, (g + 1) * gsz))
            top = brute_topk(z, members, n_top)
            acc = z[top[0]]
            for e in top[1:]:
                acc = f32(acc + z[e])
            gscore.append(acc)
        kept = brute_topk(gscore, list(range(G)), M)
        cand = [e for g in sorted(kept) for e in range(g * gsz, (g + 1) * gsz)]
    sel = brute_topk(z, cand, K)
    den = s[sel[0]]
    for e in sel[1:]:
        den = f32(den + s[e])
    gates = [f32(f32(s[e] / den) * f32(scale)) for e in sel]
    return sel, gates


def rand_scores(rng, T, E, quantum=None):
    s = rng.random((T, E)).astype(np.float32)
    if quantum:
        s = (np.round(s / quantum) * quantum).astype(np.float32)
    return s


@pytest.mark.parametrize("E,K,G,M,scale,quantum", [
    (16, 2, 1, 1, 1.0, None),
    (16, 2, 1, 1, 1.0, 1 / 8),      # many exact ties
    (12, 4, 1, 1, 1.0, None),
    (8, 3, 4, 2, 2.5, None),
    (16, 3, 4, 2, 2.5, 1 / 16),
    (16, 4, 8, 4, 2.5, None),
    (16, 4, 8, 4, 1.0, 1 / 4),
])
def test_selection_matches_bruteforce(E, K, G, M, scale, quantum):
    rng = np.random.default_rng(E * 100 + K * 10 + G)
    T = 24
    s = rand_scores(rng, T, E, quantum)
    b = (rng.standard_normal(E) * 0.05).astype(np.float32)
    if quantum:
        b = (np.round(b / quantum) * quantum).astype(np.float32)
    idx, gate = ref.select_experts(s, b, K, G, M, scale, precision="fp32")
    for t in range(T):
        sel, gates = brute_route_token([float(v) for v in s[t]],
                                       [float(v) for v in b], K, G, M, scale)
        assert list(idx[t]) == sel, (t, s[t], b)
        assert [float(g) for g in gate[t]] == gates


def test_signed_zero_and_nan_ordering():
    # z = -0.0 and +0.0 are equal: lower index wins; NaN ranks below -inf.
    s = np.array([[0.0, 0.0, 0.5, np.nan, 0.25]], dtype=np.float32)
    b = np.array([-0.0, 0.0, -0.5, 0.0, -np.inf], dtype=np.float32)
    # z = [-0.0, 0.0, 0.0, nan, -inf]
    idx, _ = ref.select_experts(s, b, 5, precision="fp32")
    assert list(idx[0]) == [0, 1, 2, 4, 3]
    sel, _ = brute_route_token([float(v) for v in s[0]], [float(v) for v in b],
                               5, 1, 1, 1.0)
    assert sel == [0, 1, 2, 4, 3]


def test_group_limit_at_most_M_groups():
    rng = np.random.default_rng(7)
    T, E, K, G, M = 500, 64, 6, 8, 3
    s = rand_scores(rng, T, E)
    b = (rng.standard_normal(E) * 0.1).astype(np.float32)
    idx, _ = ref.select_experts(s, b, K, G, M, 1.0)
    groups = idx // (E // G)
    for t in range(T):
        assert len(set(groups[t].tolist())) <= M


def test_gate_independent_of_bias():
    rng = np.random.default_rng(3)
    T, E, K = 2000, 32, 4
    s = rand_scores(rng, T, E)
    b0 = np.zeros(E, dtype=np.float32)
    b1 = (rng.standard_normal(E) * 0.02).astype(np.float32)
    i0, g0 = ref.select_experts(s, b0, K, 4, 2, 2.5)
    i1, g1 = ref.select_experts(s, b1, K, 4, 2, 2.5)
    same = np.all(i0 == i1, axis=1)
    assert same.sum() > 100 and (~same).sum() > 100
    assert np.array_equal(g0[same].view(np.uint32), g1[same].view(np.uint32))
    # and the gate is always the normalised raw affinity, whatever the bias
    for t in range(0, T, 97):
        den = float(s[t, i1[t, 0]])
        for e in i1[t, 1:]:
            den = f32(den + float(s[t, e]))
        want = [f32(f32(float(s[t, e]) / den) * 2.5) for e in i1[t]]
        assert [float(v) for v in g1[t]] == want


def test_gates_sum_to_scale():
    rng = np.random.default_rng(11)
    s = rand_scores(rng, 1000, 256)
    b = (rng.standard_normal(256) * 0.01).astype(np.float32)
    _, g = ref.select_experts(s, b, 8, 8, 4, 2.5)
    np.testing.assert_allclose(g.astype(np.float64).sum(1), 2.5, rtol=1e-6)


def test_loads_sum_and_count():
    rng = np.random.default_rng(5)
    T, E, K = 300, 16, 3
    idx, _ = ref.select_experts(rand_scores(rng, T, E), np.zeros(E, np.float32), K)
    load = ref.expert_load(idx, E)
    assert int(load.sum()) == T * K
    for e in range(E):
        assert load[e] == sum(1 for t in range(T) for k in range(K) if idx[t, k] == e)


def test_bias_update_sign_rule():
    rng = np.random.default_rng(9)
    E, T, K, gamma = 64, 4096, 6, 1e-3
    load = rng.integers(0, 2 * T * K // E, size=E).astype(np.int32)
    load[3] = T * K // E          # exactly on target: unchanged
    b = (rng.standard_normal(E) * 0.01).astype(np.float32)
    nb = ref.bias_update(load, b, T, K, E, gamma)
    for e in range(E):
        diff = T * K - E * int(load[e])
        want = float(b[e]) if diff == 0 else f32(float(b[e]) + (1 if diff > 0 else -1) * f32(gamma))
        assert float(nb[e]) == want
    assert nb[3] == b[3]
    d = nb.astype(np.float64) - b.astype(np.float64)
    assert np.all(np.isclose(np.abs(d[d != 0]), 1e-3, rtol=1e-3))


def test_sigmoid_closed_forms():
    assert ref.sigmoid64(0.0) == 0.5
    assert abs(ref.sigmoid64(math.log(3.0)) - 0.75) < 1e-15
    assert abs(ref.sigmoid64(-math.log(3.0)) - 0.25) < 1e-15
    u = np.linspace(-30, 30, 101)
    np.testing.assert_allclose(ref.sigmoid64(u) + ref.sigmoid64(-u), 1.0, atol=1e-15)
    assert ref.sigmoid64(-1000.0) == 0.0 and ref.sigmoid64(1000.0) == 1.0


def silu(a):
    return a / (1.0 + math.exp(-a))


def test_swiglu_closed_form():
    # d = 2, I = 3: W1, W3 are [I, d], W2 is [d, I]; none square or symmetric,
    # so a transposed operand or a swapped W1/W3 changes the numbers.
    W1 = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    W3 = np.array([[2.0, 0.0], [0.0, 3.0], [1.0, -1.0]])
    W2 = np.array([[1.0, 0.0, 2.0], [0.0, 1.0, -1.0]])
    x = np.array([[1.0, -2.0]])
    a = [1.0, -2.0, -1.0]
    c = [2.0, -6.0, 3.0]
    h = [silu(a[i]) * c[i] for i in range(3)]
    want = [h[0] + 2.0 * h[2], h[1] - h[2]]
    got = ref.swiglu_ffn64(x, W1, W3, W2)[0]
    np.testing.assert_allclose(got, want, rtol=1e-14)


def test_silu_closed_forms():
    assert ref.silu64(0.0) == 0.0
    assert abs(ref.silu64(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert ref.silu64(-1000.0) == 0.0 or abs(ref.silu64(-1000.0)) < 1e-300


def tiny_layer(rng, T=16, d=8, E=6, K=2, I=4, ns=2):
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((E, I, d)) * 0.3
    W3 = rng.standard_normal((E, I, d)) * 0.3
    W2 = rng.standard_normal((E, d, I)) * 0.3
    shared = (rng.standard_normal((ns * I, d)) * 0.3, rng.standard_normal((ns * I, d)) * 0.3,
              rng.standard_normal((d, ns * I)) * 0.3)
    return x, W1, W3, W2, shared


def test_sparse_dispatch_combine_equals_dense_masked_sum():
    rng = np.random.default_rng(21)
    T, d, E, K, I, ns = 16, 8, 6, 2, 4, 2
    x, W1, W3, W2, shared = tiny_layer(rng, T, d, E, K, I, ns)
    s = ref.sigmoid64(x @ rng.standard_normal((E, d)).T)
    b = rng.standard_normal(E) * 0.05
    idx, gate = ref.select_experts(s, b, K, precision="fp64", route_scale=2.5)
    sparse = ref.moe_output64(x, idx, gate, lambda e: (W1[e], W3[e], W2[e]), shared, ns)
    dense = ref.dense_masked_output64(x, idx, gate, W1, W3, W2, shared, ns)
    np.testing.assert_allclose(sparse, dense, rtol=1e-12, atol=1e-12)
    # permute + per-expert FFN + combine reaches the same output
    off, row_of, tok_of = ref.permute(idx, E)
    y_perm = np.zeros((T * K, d))
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        y_perm[r0:r1] = ref.swiglu_ffn64(x[tok_of[r0:r1]], W1[e], W3[e], W2[e])
    y_sh = ref.shared_ffn64(x, *shared, ns)
    out = ref.combine64(y_perm, row_of, gate, y_sh)
    np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-12)


def test_shared_experts_sum_separately():
    rng = np.random.default_rng(2)
    x, _, _, _, (a, b, c) = tiny_layer(rng, ns=2)
    I = a.shape[0] // 2
    want = (ref.swiglu_ffn64(x, a[:I], b[:I], c[:, :I]) +
            ref.swiglu_ffn64(x, a[I:], b[I:], c[:, I:]))
    np.testing.assert_allclose(ref.shared_ffn64(x, a, b, c, 2), want, rtol=1e-14)


def test_permute_definition():
    rng = np.random.default_rng(4)
    T, E, K = 200, 16, 3
    idx, _ = ref.select_experts(rand_scores(rng, T, E), np.zeros(E, np.float32), K)
    off, row_of, tok_of = ref.permute(idx, E)
    load = ref.expert_load(idx, E)
    assert off[0] == 0 and off[E] == T * K
    assert np.all(np.diff(off) == load)
    assert sorted(row_of.reshape(-1).tolist()) == list(range(T * K))
    prev = {}
    for t in range(T):
        for k in range(K):
            r = row_of[t, k]
            e = idx[t, k]
            assert off[e] <= r < off[e + 1]
            assert tok_of[r] == t
            if e in prev:
                assert r == prev[e] + 1     # stable (t, k) order inside an expert
            prev[e] = r


def test_handworked_golden_cases():
    with open(os.path.join(GOLDEN, "handworked_routing.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        s = np.array(c["s"], dtype=np.float32)
        b = np.array(c["bias"], dtype=np.float32)
        T = s.shape[0]
        idx, gate = ref.select_experts(s, b, c["K"], c["n_groups"], c["topk_groups"],
                                       c["route_scale"], precision="fp32")
        assert idx.tolist() == c["idx"], c["name"]
        for t in range(T):
            for k in range(c["K"]):
                num, den = c["gate_frac"][t][k]
                want = f32(num / den)
                ulp = abs(f32(want * (1 + 2 ** -23)) - want)
                assert abs(float(gate[t, k]) - want) <= 2 * ulp, c["name"]
        load = ref.expert_load(idx, c["E"])
        assert load.tolist() == c["load"], c["name"]
        nb = ref.bias_update(load, b, T, c["K"], c["E"], c["gamma"])
        assert nb.tolist() == c["bias_after"], c["name"]


def test_bf16_decode():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F80], dtype=np.uint16)
    v = ref.bf16_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -1.0 and v[3] == 0.0 and math.isinf(v[5])
    assert abs(v[2] - 3.140625) == 0.0


def test_near_tie_detection():
    s = np.array([[0.5, 0.5 + 1e-6, 0.1, 0.9]])
    kth, grp = ref.near_tie_tokens(s, np.zeros(4), 2)
    assert kth[0]          # 2nd vs 3rd: 0.5+1e-6 vs 0.5
    kth, _ = ref.near_tie_tokens(s, np.zeros(4), 1)
    assert not kth[0]


# Hand-built biased scores z for the group-limited rule with E = 12 experts in
# G = 4 groups of 3, M = 2 groups kept, K = 4 (so a group's score is the sum of
# its 2 largest z, reading R1).  Every value is dyadic, so each sum and gap
# below is exact in fp64 and the group scores are worked out by hand:
#   token 0  group scores 0.75, 0.1875, 1.8125, 0.75 - 2^-18 -> 2nd vs 3rd
#            group gap 2^-18 (< 1e-5): group near-tie.  The kept groups are 2
#            and 0; among their experts the 4th and 5th z are 0.25 and 0.125.
#   token 1  the same with the gap 2^-15 (> 1e-5): no group near-tie, although
#            the two groups' LARGEST members tie exactly (0.5 and 0.5).
#   token 2  kept groups 0 and 1; 4th vs 5th among their experts 0.5 vs
#            0.0625, while the best expert of a DROPPED group (group 2) is
#            0.5 - 2^-18: that candidate must not count as the (K+1)-th.
#   token 3  4th vs 5th among the kept groups' experts 0.5 vs 0.5 - 2^-18.
_NT_Z = np.array([
    [0.5, 0.25, 0.125, 0.125, 0.0625, 0.03125, 0.9375, 0.875, 0.0625,
     0.5, 0.25 - 2.0**-18, 0.0078125],
    [0.5, 0.25, 0.0, 0.125, 0.0625, 0.03125, 0.9375, 0.875, 0.0,
     0.5, 0.25 - 2.0**-15, 0.0],
    [0.9375, 0.875, 0.0625, 0.75, 0.5, 0.0, 0.5 - 2.0**-18, 0.125, 0.0,
     0.25, 0.125, 0.0],
    [0.9375, 0.875, 0.0625, 0.75, 0.5, 0.5 - 2.0**-18, 0.25, 0.125, 0.0,
     0.125, 0.0625, 0.0],
])


def test_near_tie_group_gap_and_eligible_kth_gap():
    """The group-gap branch and the K-th gap among eligible experts only
    (node-limited routing: at most M groups per token -- chenshi221 notes,
    "Auxiliary-loss-free 负载均衡")."""
    want_grp = [True, False, False, False]
    want_kth = [False, False, False, True]
    kth, grp = ref.near_tie_tokens(_NT_Z, np.zeros(12), 4, n_groups=4, topk_groups=2)
    assert grp.tolist() == want_grp
    assert kth.tolist() == want_kth
    # the masks look at z = s + b: a dyadic bias moved into s gives the same z
    b = np.tile(np.array([0.03125, -0.0625, 0.0]), 4)
    kth_b, grp_b = ref.near_tie_tokens(_NT_Z - b[None, :], b.astype(np.float32), 4,
                                       n_groups=4, topk_groups=2)
    assert grp_b.tolist() == want_grp and kth_b.tolist() == want_kth
    # the kept groups of tokens 0 and 2 are the hand-worked ones
    idx, _ = ref.select_experts(_NT_Z, np.zeros(12), 4, 4, 2, precision="fp64")
    assert sorted({int(e) // 3 for e in idx[0]}) == [0, 2]
    assert sorted({int(e) // 3 for e in idx[2]}) == [0, 1]
    # without a group limit only the plain K-th gap exists: for token 2 the
    # 5th-best z overall is the 0.5 - 2^-18 that the group limit had excluded
    kth1, grp1 = ref.near_tie_tokens(_NT_Z, np.zeros(12), 4)
    assert kth1[2] and not grp1.any()


def test_load_stats_handworked():
    """max, mean, max/mean and the coefficient of variation (population
    standard deviation over the mean, over ALL experts, untouched ones too)
    of per-expert loads."""
    # [0, 2, 2, 4]: mean 2, max 4, deviations -2, 0, 0, 2 -> variance 8/4 = 2
    np.testing.assert_allclose(ref.load_stats([0, 2, 2, 4]),
                               [4.0, 2.0, 2.0, math.sqrt(2.0) / 2.0], rtol=0, atol=1e-15)
    # all load on one of E experts: mean 3/E, max/mean = E, CV = sqrt(E - 1)
    for E in (2, 6, 256):
        load = np.zeros(E, dtype=np.int32)
        load[E // 2] = 3
        np.testing.assert_allclose(ref.load_stats(load), [3.0, 3.0 / E, E, math.sqrt(E - 1)],
                                   rtol=1e-14, atol=0)
    # perfectly even loads: max/mean 1, CV 0; no load at all: zeros, not NaN
    np.testing.assert_array_equal(ref.load_stats([5, 5, 5]), [5.0, 5.0, 1.0, 0.0])
    np.testing.assert_array_equal(ref.load_stats([0, 0, 0, 0]), [0.0, 0.0, 0.0, 0.0])


def test_seq_balance_loss_closed_forms():
    rng = np.random.default_rng(13)
    E, K, alpha = 8, 2, 1e-4
    # perfectly even routing: f_i = 1 for every expert, so L = alpha * sum_i P_i = alpha
    T = 16
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)])
    s = rng.random((T, E))
    assert abs(ref.seq_balance_loss(s, idx, [0, T], K, alpha)[0] - alpha) < 1e-18
    # everything on expert 0 with all affinity there: f_0 = E, P_0 = 1 -> L = alpha * E
    idx1 = np.zeros((4, 1), dtype=int)
    s1 = np.zeros((4, E))
    s1[:, 0] = 1.0
    assert abs(ref.seq_balance_loss(s1, idx1, [0, 4], 1, alpha)[0] - alpha * E) < 1e-18


def test_seq_balance_loss_handworked_and_per_sequence():
    # E=4, K=1, one sequence of 2 tokens: token 0 picks expert 0, token 1 picks 2.
    # s rows (sums): [1,1,1,1] (4) and [2,0,1,1] (4)
    # f = 4/(1*2) * [1,0,1,0] = [2,0,2,0];  P = ([.25,.25,.25,.25] + [.5,0,.25,.25]) / 2
    #   = [.375, .125, .25, .25];  L = a * (2*.375 + 2*.25) = 1.25 a
    s = np.array([[1.0, 1, 1, 1], [2, 0, 1, 1]])
    idx = np.array([[0], [2]])
    assert abs(ref.seq_balance_loss(s, idx, [0, 2], 1, 1.0)[0] - 1.25) < 1e-15
    # two sequences are independent; an empty sequence gives 0
    s2 = np.vstack([s, s])
    idx2 = np.vstack([idx, idx])
    got = ref.seq_balance_loss(s2, idx2, [0, 2, 2, 4], 1, 1.0)
    assert np.allclose(got, [1.25, 0.0, 1.25], atol=1e-15)
