"""The sharded step's host side on the CPU: the partition of the C ABI
(muon_adamw_plan_shards, a host-only call) and, with two gloo ranks, the
norm all-reduce and the exchange of updated parameters, with the fp64 oracle
doing each rank's arithmetic.

OpenDM article, 核心揭秘一 / 为 FSDP 分片量身定制的细节 (Muon under FSDP on 8
GPUs): here Muon matrices go whole to one owner rank each and AdamW elements
are split into contiguous ranges; every element is updated by exactly one
rank and the global norm is the square root of the summed per-rank sums of
squares.
"""
import heapq
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

from conftest import ROOT

MUON, ADAMW, FROZEN = 1, 2, 3


@pytest.fixture(scope="module")
def mx():
    from muon_adamw_hybrid_grad_gb300 import build

    build.build()
    import muon_adamw_hybrid_grad_gb300 as m

    m.load_library()
    return m


def _model():
    """A mixed parameter list: Muon matrices of several shapes, AdamW vectors
    and matrices of ragged lengths, a frozen embedding and an empty tensor."""
    rng = np.random.default_rng(7)
    params = []
    for k in range(23):
        r, c = [(1024, 1024), (4096, 1024), (1024, 4096), (256, 512), (40, 1000)][k % 5]
        params.append((MUON, r * c, r, c))
    for k in range(40):
        n = int(rng.integers(1, 70000))
        params.append((ADAMW, n, n, 1))
    params.append((ADAMW, 2048 * 2048, 2048, 2048))
    params.append((FROZEN, 1000 * 64, 1000, 64))
    params.append((ADAMW, 0, 0, 1))
    return params


def _plan(mx, params, world):
    g, n, r, c = zip(*params)
    return mx.muon_adamw_plan_shards(g, n, r, c, world)


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_every_element_is_updated_by_exactly_one_rank(mx, world):
    params = _model()
    owner, ranges = _plan(mx, params, world)
    for i, (grp, n, _, _) in enumerate(params):
        rr = ranges[i]
        assert len(rr) == world
        if grp == FROZEN or n == 0:
            assert all(b == e for b, e in rr) and owner[i] == -1
            continue
        if grp == MUON:
            assert 0 <= owner[i] < world
            assert rr[owner[i]] == (0, n)
            assert all(b == e for r, (b, e) in enumerate(rr) if r != owner[i])
            continue
        assert owner[i] == -1
        covered = np.zeros(n, dtype=np.int32)
        for b, e in rr:
            assert 0 <= b <= e <= n
            covered[b:e] += 1
        assert (covered == 1).all()


@pytest.mark.parametrize("world", [2, 3, 8])
def test_adamw_ranges_are_contiguous_balanced_and_aligned(mx, world):
    params = _model()
    _, ranges = _plan(mx, params, world)
    adam = [i for i, p in enumerate(params) if p[0] == ADAMW and p[1] > 0]
    start = np.cumsum([0] + [params[i][1] for i in adam])
    total = int(start[-1])
    pieces = []  # (global begin, global end, rank)
    for k, i in enumerate(adam):
        for r, (b, e) in enumerate(ranges[i]):
            if e > b:
                # a range starts at the parameter's start or at a multiple of 64 of it
                assert b % 64 == 0
                pieces.append((int(start[k]) + b, int(start[k]) + e, r))
    pieces.sort()
    # ranks own consecutive stretches of the concatenation, in rank order
    assert [r for _, _, r in pieces] == sorted(r for _, _, r in pieces)
    assert pieces[0][0] == 0 and pieces[-1][1] == total
    for (b0, e0, _), (b1, _, _) in zip(pieces, pieces[1:]):
        assert e0 == b1
    per_rank = [sum(e - b for b, e, r in pieces if r == q) for q in range(world)]
    # each cut moves by less than 64 elements from total * r / world
    assert max(per_rank) - min(per_rank) <= 2 * 64 + world


@pytest.mark.parametrize("world", [2, 3, 8])
def test_muon_owners_follow_longest_first_list_scheduling(mx, world):
    params = _model()
    owner, _ = _plan(mx, params, world)
    cost = {i: 5.0 * (4.0 * min(r, c) ** 2 * max(r, c) + 2.0 * min(r, c) ** 3)
            for i, (g, n, r, c) in enumerate(params) if g == MUON}
    # the same rule restated with a heap: longest first, least-loaded rank, ties to the lower rank
    heap = [(0.0, r) for r in range(world)]
    want = {}
    for i in sorted(cost, key=lambda i: (-cost[i], i)):
        load, r = heapq.heappop(heap)
        want[i] = r
        heapq.heappush(heap, (load + cost[i], r))
    assert {i: owner[i] for i in cost} == want
    loads = [sum(cost[i] for i in cost if owner[i] == r) for r in range(world)]
    # list scheduling bound: no rank exceeds the mean by more than the largest matrix
    assert max(loads) <= sum(loads) / world + max(cost.values()) + 1e-6


def test_plan_shards_errors(mx):
    with pytest.raises(mx.MuonAdamWError) as ei:
        mx.muon_adamw_plan_shards([MUON], [6], [2], [3], 0)
    assert ei.value.status == mx.MA_ERR_ARG
    with pytest.raises(mx.MuonAdamWError) as ei:
        mx.muon_adamw_plan_shards([7], [6], [2], [3], 2)
    assert ei.value.status == mx.MA_ERR_ARG
    with pytest.raises(mx.MuonAdamWError) as ei:
        mx.muon_adamw_plan_shards([MUON], [7], [2], [3], 2)
    assert ei.value.status == mx.MA_ERR_SHAPE
    with pytest.raises(mx.MuonAdamWError) as ei:
        mx.muon_adamw_plan_shards([ADAMW], [-1], [1], [1], 2)
    assert ei.value.status == mx.MA_ERR_SHAPE
    assert mx.muon_adamw_plan_shards([], [], [], [], 4) == ([], [])


# ---- two gloo ranks: norm all-reduce and exchange, oracle arithmetic ----

WORKER = r"""
import json, math, os, sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
import torch.distributed as dist
import muon_adamw_hybrid_grad_gb300 as mx
import oracle
import workloads
from workloads import TensorSpec

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
base = workloads.get_workload("tiny")
t = list(base.tensors) + [TensorSpec("model.vlm.v.weight", (100003,)), TensorSpec("model.vlm.b.bias", (77,))]
w = workloads.custom_workload("tiny_shard", t, policy="fp32_mixed", steps=2)
names = [x.name for x in w.tensors]
shapes = [x.shape for x in w.tensors]
groups = [oracle.route(n, len(s)) for n, s in zip(names, shapes)]
code = {{"muon": mx.MA_GROUP_MUON, "adamw": mx.MA_GROUP_ADAMW, "frozen": mx.MA_GROUP_FROZEN}}
owner, ranges = mx.muon_adamw_plan_shards(
    [code[g] for g in groups], [x.numel for x in w.tensors],
    [s[0] if len(s) == 2 else int(np.prod(s)) for s in shapes], [s[1] if len(s) == 2 else 1 for s in shapes],
    world)
masters = workloads.master_weights(w)
# this rank's oracle: its Muon matrices whole, its pieces of the AdamW parameters
mine = [(i, ranges[i][rank]) for i in range(len(names)) if ranges[i][rank][1] > ranges[i][rank][0]]
orc = oracle.HybridOracle([names[i] for i, _ in mine],
                          [shapes[i] if groups[i] == "muon" else (e - b,) for i, (b, e) in mine])
assert [orc.groups[k] for k in range(len(mine))] == [groups[i] for i, _ in mine]
full = [torch.from_numpy(m.astype(np.float64)).clone() for m in masters]
pieces = [full[i].view(-1)[b:e].clone().numpy() if groups[i] != "muon" else full[i].clone().numpy()
          for i, (b, e) in mine]
out = {{"norms": [], "rank": rank}}
for step in (1, 2):
    grads = workloads.gradients(w, step)
    local = sum(float(np.sum(np.square(grads[i].reshape(-1)[b:e].astype(np.float64)))) for i, (b, e) in mine)
    tot = torch.tensor([local], dtype=torch.float64)
    dist.all_reduce(tot)
    total = math.sqrt(float(tot.item()))
    out["norms"].append([total, oracle.global_grad_norm(grads)])
    g_mine = [grads[i] if groups[i] == "muon" else grads[i].reshape(-1)[b:e] for i, (b, e) in mine]
    orc.step(pieces, g_mine, w.lr, total_override=total)
    for (i, (b, e)), v in zip(mine, pieces):
        full[i].view(-1)[b:e] = torch.from_numpy(np.ascontiguousarray(v).reshape(-1))
    mx.shard_exchange(full, ranges, rank, world, dist)
np.save(os.path.join({outdir!r}, f"rank{{rank}}.npy"), np.concatenate([f.view(-1).numpy() for f in full]))
print(json.dumps(out), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_sharded_step_with_two_gloo_ranks_matches_the_whole_oracle_step(mx, tmp_path):
    import oracle
    import workloads
    from workloads import TensorSpec

    world = 2
    port = _free_port()
    code = WORKER.format(root=ROOT, outdir=str(tmp_path))
    procs = []
    for r in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(r),
                   LOCAL_RANK=str(r), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=300)
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    # the all-reduced norm is the norm over every gradient
    for o in outs:
        for got, want in o["norms"]:
            assert got == pytest.approx(want, rel=1e-12)
    # both ranks end with the same parameters, those of one oracle step over everything
    a, b = (np.load(tmp_path / f"rank{r}.npy") for r in range(world))
    assert np.array_equal(a, b)
    base = workloads.get_workload("tiny")
    t = list(base.tensors) + [TensorSpec("model.vlm.v.weight", (100003,)), TensorSpec("model.vlm.b.bias", (77,))]
    w = workloads.custom_workload("tiny_shard", t, policy="fp32_mixed", steps=2)
    params = [m.astype(np.float64) for m in workloads.master_weights(w)]
    orc = oracle.HybridOracle([x.name for x in w.tensors], [x.shape for x in w.tensors])
    for step in (1, 2):
        orc.step(params, workloads.gradients(w, step), w.lr)
    want = np.concatenate([p.reshape(-1) for p in params])
    np.testing.assert_allclose(a, want, rtol=1e-12, atol=1e-15)
