"""The redundant-expert planner (a host call of the C ABI, no GPU needed):
the greedy placement reaches the smallest possible largest load per copy,
checked by brute force over all placements on small cases."""
import itertools

import numpy as np
import pytest

import expert_ffn_layer_affinity_b300 as moe


def best_max_load(load, n_extra):
    E = len(load)
    best = None
    for extra in itertools.combinations_with_replacement(range(E), n_extra):
        c = np.ones(E)
        for e in extra:
            c[e] += 1
        m = max(load[e] / c[e] for e in range(E))
        best = m if best is None else min(best, m)
    return best


@pytest.mark.parametrize("E,n,seed", [(4, 3, 0), (6, 4, 1), (5, 5, 2), (8, 2, 3), (3, 0, 4)])
def test_plan_is_optimal_and_consistent(E, n, seed):
    rng = np.random.default_rng(seed)
    load = rng.integers(0, 500, size=E).astype(np.int32)
    load[0] = load.max()            # a tie for the largest
    ss, sl, eo = moe.moe_replica_plan(load, E, n)
    ss, sl, eo = ss.numpy(), sl.numpy(), eo.numpy()
    assert ss[0] == 0 and ss[E] == E + n and np.all(np.diff(ss) >= 1)
    assert sorted(sl.tolist()) == list(range(E + n))
    for e in range(E):
        mine = sl[ss[e]:ss[e + 1]]
        assert mine[0] == e and all(eo[s] == e for s in mine)
    copies = np.diff(ss)
    got = max(load[e] / copies[e] for e in range(E))
    assert abs(got - best_max_load(load, n)) < 1e-12


def test_plan_rejects_bad_arguments():
    assert moe.moe_replica_plan(np.zeros(4, np.int32), 4, -1, check=False) == moe.MOE_ERR_INVALID_ARG
