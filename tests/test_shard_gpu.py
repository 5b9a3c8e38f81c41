"""The sharded step on one GPU: two or three handles act as the ranks of a
world of that size, one after the other on the same stream (no kernel waits
for another). The matrices take every Newton-Schulz path: tensor-core,
fused small-matrix (128 x 512) and narrow (1000 x 40). Each has its own copy of the parameters and reads the same
gradients; the host sums their local sums of squares (what an all-reduce
does) and copies each rank's updated parts to the others (what the exchange
does). Checked against the
fp64 oracle's whole step at the parity suite's tolerances: the norm, O of
every Muon matrix, AdamW p, m and v (each rank's state holds its range), the
bf16 shadows; each rank's local sum of squares against the fp64 sum over the
elements it owns; and that a rank writes nothing outside what it owns.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from harness import NORM_TOL, O_TOL, StateBounds, _f32, compare_state, relative_frobenius
from workloads import TensorSpec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    from muon_adamw_hybrid_grad_gb300 import build

    build.build()
    import muon_adamw_hybrid_grad_gb300 as m

    m.load_library()
    return m


def _workload():
    base = workloads.get_workload("tiny")
    t = list(base.tensors) + [TensorSpec("model.action_expert.layers.2.wq.weight", (384, 640), rank8=True),
                              TensorSpec("model.action_expert.layers.2.w_small.weight", (128, 512), rank8=True),
                              TensorSpec("model.action_expert.layers.2.w_narrow.weight", (1000, 40), rank8=True),
                              TensorSpec("model.vlm.v.weight", (100003,)), TensorSpec("model.vlm.b.bias", (77,))]
    return workloads.custom_workload("tiny_shard", t, policy="bf16_mixed", steps=2)


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_step_ranks_on_one_gpu(mx, world):
    import torch

    w = _workload()
    dev = torch.device("cuda")
    n = len(w.tensors)
    names = [t.name for t in w.tensors]
    shapes = [t.shape for t in w.tensors]
    masters = workloads.master_weights(w)
    G = [torch.zeros(t.shape, dtype=torch.bfloat16, device=dev) for t in w.tensors]
    P = [[torch.from_numpy(m).to(dev) for m in masters] for _ in range(world)]
    S = [[torch.zeros(t.shape, dtype=torch.bfloat16, device=dev) for t in w.tensors] for _ in range(world)]
    opts = [mx.MuonAdamW([(names[i], P[r][i], G[i], S[r][i]) for i in range(n)], shard=(r, world),
                         precision=mx.MA_BF16_MIXED) for r in range(world)]
    try:
        ranges = opts[0].shard_ranges()
        assert all(o.shard_ranges() == ranges for o in opts[1:])
        groups = opts[0].groups
        orc = oracle.HybridOracle(names, shapes)
        assert orc.groups == groups
        cfg = opts[0].cfg
        orc_p = [m.astype(np.float64) for m in masters]
        beta1, beta2 = (float(b) for b in orc.cfg["adam_betas"])
        bounds = StateBounds()
        assert any(b > 0 for rr in ranges for b, _ in rr)  # an AdamW parameter is cut mid-way
        for step in (1, 2):
            grads = workloads.gradients(w, step)
            for g_dev, g in zip(G, grads):
                g_dev.copy_(torch.from_numpy(g).to(torch.bfloat16))
            before = [[p.cpu().numpy() for p in P[r]] for r in range(world)]
            local = [torch.zeros(1, dtype=torch.float64, device=dev) for _ in range(world)]
            for r in range(world):
                opts[r].step_begin(w.lr, local[r])
            total = sum(local[1:], local[0].clone())
            norms = [opts[r].step_end(total, want_norm=True) for r in range(world)]
            m_prev = dict(orc.m)
            res = orc.step(orc_p, grads, w.lr)
            for r in range(world):
                own = sum(float(np.sum(np.square(grads[i].reshape(-1)[b:e].astype(np.float64))))
                          for i, rr in enumerate(ranges) for b, e in [rr[r]])
                assert local[r].item() == pytest.approx(own, rel=1e-6)
                assert math.isclose(norms[r], res["total"], rel_tol=NORM_TOL)
            # a rank writes nothing outside what it owns
            for r in range(world):
                for i in range(n):
                    b, e = ranges[i][r]
                    now = P[r][i].cpu().numpy().reshape(-1)
                    was = before[r][i].reshape(-1)
                    assert np.array_equal(np.delete(now, np.s_[b:e]), np.delete(was, np.s_[b:e])), (r, names[i])
            # the exchange: every rank gets every updated part
            for i in range(n):
                for src in range(world):
                    b, e = ranges[i][src]
                    for dst in range(world):
                        if dst != src and e > b:
                            P[dst][i].view(-1)[b:e].copy_(P[src][i].view(-1)[b:e])
                            S[dst][i].view(-1)[b:e].copy_(S[src][i].view(-1)[b:e])
            coef = res["coef"]
            for i in range(n):
                p_gpu = P[0][i].cpu().numpy()
                assert all(np.array_equal(p_gpu, P[r][i].cpu().numpy()) for r in range(1, world))
                assert np.array_equal(S[0][i].float().cpu().numpy(), workloads.bf16_round(p_gpu)), names[i]
                if groups[i] == "muon":
                    m_, n_ = shapes[i]
                    decay = _f32(1.0 - w.lr * cfg.muon_weight_decay)
                    lr_mult = _f32(cfg.muon_lr_scale * cfg.moonlight_coef * math.sqrt(max(m_, n_)))
                    O_gpu = (before[0][i].astype(np.float64) * decay - p_gpu) / (_f32(w.lr) * lr_mult)
                    err = relative_frobenius(O_gpu, res["O"][i])
                    assert err <= O_TOL, (names[i], err)
                elif groups[i] == "adamw":
                    ghat = coef * grads[i].astype(np.float64)
                    s_m = bounds.recurrence(("m", i), orc.m[i], m_prev[i], beta1, (1.0 - beta1) * ghat)
                    s_p = bounds.adamw_param(("p", i), orc_p[i], s_m, orc.v[i], res["t"], w.lr, beta1, beta2,
                                             float(orc.cfg["adam_eps"]))
                    compare_state(f"step {step} p[{names[i]}]", p_gpu, orc_p[i], s_p)
                    for r in range(world):
                        b, e = ranges[i][r]
                        if e <= b:
                            continue
                        sl = np.s_[b:e]
                        m_gpu = opts[r].state(i, 0).numpy().reshape(-1)
                        v_gpu = opts[r].state(i, 1).numpy().reshape(-1)
                        assert m_gpu.size == e - b
                        compare_state(f"step {step} m[{names[i]}] rank {r}", m_gpu, orc.m[i].reshape(-1)[sl],
                                      s_m.reshape(-1)[sl])
                        compare_state(f"step {step} v[{names[i]}] rank {r}", v_gpu, orc.v[i].reshape(-1)[sl],
                                      np.abs(orc.v[i].reshape(-1)[sl]))
    finally:
        for o in opts:
            o.close()


def test_sharded_handle_call_order(mx):
    import torch

    dev = torch.device("cuda")
    p = torch.zeros(300, dtype=torch.float32, device=dev)
    g = torch.ones(300, dtype=torch.bfloat16, device=dev)
    opt = mx.MuonAdamW([("model.vlm.v.weight", p, g, None)], shard=(1, 2), precision=mx.MA_FP32_MIXED)
    try:
        buf = torch.zeros(1, dtype=torch.float64, device=dev)
        with pytest.raises(mx.MuonAdamWError) as ei:
            opt.step(1e-3)  # a sharded handle steps in two halves
        assert ei.value.status == mx.MA_ERR_STATE
        with pytest.raises(mx.MuonAdamWError) as ei:
            opt.step_end(buf)
        assert ei.value.status == mx.MA_ERR_STATE
        opt.step_begin(1e-3, buf)
        with pytest.raises(mx.MuonAdamWError) as ei:
            opt.step_begin(1e-3, buf)
        assert ei.value.status == mx.MA_ERR_STATE
        b, e = opt.shard_range(0)
        assert (b, e) == (128, 300)  # the cut at 150 moves down to 128
        assert buf.item() == pytest.approx(float(e - b))  # gradients of ones: the owned count
        buf.fill_(300.0)  # all ranks' sum
        norm = opt.step_end(buf, want_norm=True)
        assert norm == pytest.approx(math.sqrt(300.0), rel=1e-6)
        with pytest.raises(mx.MuonAdamWError) as ei:
            mx.muon_adamw_set_shard(opt.handle, 0, 2)  # after the first step
        assert ei.value.status == mx.MA_ERR_STATE
        assert opt.state(0, 0).numel() == e - b
        assert torch.count_nonzero(p[:b]).item() == 0 and torch.count_nonzero(p[b:]).item() == e - b
    finally:
        opt.close()
