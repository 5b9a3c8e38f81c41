"""Host-side work order of the tensor-core Newton-Schulz launches (no GPU).

The library hands each launch's work units to its clusters longest-processing-
time first (a unit costs k / 64 + 6 k-steps; each unit, in launch order, to the
least-loaded cluster, ties to the lowest index) and lays the result out round
by round. These tests pin the properties the kernel relies on: every unit once,
a cluster's units before its padding, the plain round-robin order when all
units cost the same, and the balance bound of list scheduling.
"""
import heapq

import pytest

import muon_adamw_hybrid_grad_gb300 as mx


def _lib_or_skip():
    try:
        mx.load_library()
    except Exception as e:  # pragma: no cover - the build step makes it
        pytest.skip(f"library not built: {e}")


def _cost(k):
    return k // 64 + 6


def _per_cluster(order, ncl):
    rounds = len(order) // ncl
    return [[order[r * ncl + c] for r in range(rounds)] for c in range(ncl)]


def _loads(order, ncl, unit_cost):
    return [sum(unit_cost[u] for u in lst if u >= 0) for lst in _per_cluster(order, ncl)]


def _unit_costs(k, units):
    out = []
    for kk, n in zip(k, units):
        out += [_cost(kk)] * n
    return out


CASES = [
    ([1024], [1120], 76),                  # A A of the 1024-wide workload: one length
    ([4096, 1024], [480, 640], 76),        # X X^T of the same: two lengths
    ([8192, 2048], [2592, 3456], 76),      # X X^T of the 2048-wide workload
    ([512, 128], [40, 24], 152),           # fewer units than clusters
    ([1024, 256, 64], [7, 300, 1], 13),    # three problems, odd cluster count
    ([64], [0], 8),                        # an empty problem
]


@pytest.mark.parametrize("k,units,ncl", CASES)
def test_every_unit_exactly_once_and_padding_last(k, units, ncl):
    _lib_or_skip()
    order = mx.muon_adamw_plan_work_order(k, units, ncl)
    total = sum(units)
    assert len(order) % ncl == 0
    got = sorted(u for u in order if u >= 0)
    assert got == list(range(total))
    assert all(u == -1 for u in order if u < 0)
    for lst in _per_cluster(order, ncl):
        valid = [u for u in lst if u >= 0]
        assert lst[:len(valid)] == valid  # a cluster's padding follows its units
    # no position row is entirely padding
    assert len(order) // ncl == max(len([u for u in lst if u >= 0]) for lst in _per_cluster(order, ncl))


@pytest.mark.parametrize("n,ncl", [(1120, 76), (4096, 76), (75, 76), (77, 76), (1, 1), (300, 152)])
def test_equal_costs_give_round_robin(n, ncl):
    _lib_or_skip()
    order = mx.muon_adamw_plan_work_order([1024], [n], ncl)
    rounds = -(-n // ncl)
    assert len(order) == rounds * ncl
    assert order == [i if i < n else -1 for i in range(rounds * ncl)]


@pytest.mark.parametrize("k,units,ncl", CASES[1:3] + CASES[4:5])
def test_list_scheduling_balance_bound(k, units, ncl):
    """Greedy list scheduling ends within one unit of the mean load, and here
    beats the plain round-robin assignment of the same units."""
    _lib_or_skip()
    order = mx.muon_adamw_plan_work_order(k, units, ncl)
    cost = _unit_costs(k, units)
    loads = _loads(order, ncl, cost)
    mean = sum(cost) / ncl
    assert max(loads) <= mean + max(cost) + 1e-9
    rr = [0] * ncl
    for u, c in enumerate(cost):
        rr[u % ncl] += c
    assert max(loads) <= max(rr)


def test_matches_a_direct_statement_of_the_rule():
    """Small case against the rule written out with a heap."""
    _lib_or_skip()
    k, units, ncl = [2048, 512, 128], [5, 9, 4], 4
    cost = _unit_costs(k, units)
    heap = [(0, c) for c in range(ncl)]
    lists = [[] for _ in range(ncl)]
    for u, cst in enumerate(cost):
        load, c = heapq.heappop(heap)
        lists[c].append(u)
        heapq.heappush(heap, (load + cst, c))
    rounds = max(len(x) for x in lists)
    want = [-1] * (rounds * ncl)
    for c, lst in enumerate(lists):
        for r, u in enumerate(lst):
            want[r * ncl + c] = u
    assert mx.muon_adamw_plan_work_order(k, units, ncl) == want


@pytest.mark.parametrize("k,units,ncl", [
    ([], [], 4),               # no problem
    ([64] * 5, [1] * 5, 4),    # more than four problems
    ([96], [4], 4),            # k not a multiple of 64
    ([0], [4], 4),             # k not positive
    ([64], [-1], 4),           # negative unit count
    ([64], [4], 0),            # no cluster
])
def test_invalid_arguments(k, units, ncl):
    _lib_or_skip()
    with pytest.raises(mx.MuonAdamWError):
        mx.muon_adamw_plan_work_order(k, units, ncl)
