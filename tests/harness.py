"""Run the CUDA optimizer and the fp64 oracle side by side on the same inputs.

Inputs come from ``workloads`` (seeded, synthetic). The GPU side goes
through the C ABI (via the ctypes binding); the oracle side is ``oracle``.
Nothing computed by the CUDA path is ever fed to the oracle.

Tolerances (derived from the arithmetic; see the assertions below):
  * global norm: relative 1e-5 (fp32 partial sums, Kahan-compensated);
  * optimizer state, 1e-6 relative to the terms of its own recurrence (the
    hyperparameters are doubles on both sides and the kernels round each
    operation once in fp32, about 6e-8 each; the oracle never takes a value
    from the GPU, so an error made at one step is carried into the next by
    the recurrence's own decay, and the bound carries it the same way):
      v (AdamW second moment): 1e-6 |v| -- every term of
        v = beta2 v_prev + (1 - beta2) g^2 is non-negative, so nothing cancels
        and the relative error grows by at most a few roundings per step;
      m (AdamW first moment): 1e-6 S_m with
        S_m = |m| + beta1 |m_prev| + (1 - beta1) |g| + beta1 S_m_prev;
      buf (Muon momentum): 1e-6 S_buf with
        S_buf = |buf| + mu |buf_prev| + w |g| + mu S_buf_prev, w = 1, or
        1 - mu for the exponential-average form;
      p (AdamW parameter): 1e-6 S_p with
        S_p = S_p_prev + |p| + (lr / bc1) S_m / (sqrt(v / bc2) + eps):
        the parameter's own rounding plus the update's terms, summed over the
        steps (an error in p is never decayed away);
    g is the clipped gradient and every S starts at 0; each bound also has a
    floor of 1e-37, below fp32's smallest normal number, for states that are
    exactly zero;
  * the orthogonalised update O (bf16 Newton-Schulz): relative Frobenius
    error <= 2e-2 per matrix, every shape included. O is recovered from the
    fp32 parameter update: O = (p_before * decay - p_after) / (lr * lr_mult),
    with decay and lr_mult rounded to fp32 as the kernel uses them.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

import oracle
import workloads

O_TOL = 2e-2
STATE_TOL = 1e-6
STATE_FLOOR = 1e-37
NORM_TOL = 1e-5


def _f32(x: float) -> float:
    return float(np.float32(x))


class GpuSide:
    """GPU tensors of a workload registered with one optimizer handle."""

    def __init__(self, w: workloads.Workload, masters: List[np.ndarray], *, config: Optional[dict] = None):
        import torch

        import muon_adamw_hybrid_grad_gb300 as mx

        self.torch = torch
        self.mx = mx
        self.w = w
        dev = torch.device("cuda")
        gdt = torch.bfloat16 if w.grad_dtype == "bf16" else torch.float32
        cfg = dict(config or {})
        cfg.setdefault("precision", mx.MA_BF16_MIXED if w.policy == "bf16_mixed" else mx.MA_FP32_MIXED)
        self.P, self.G, self.S = [], [], []
        entries = []
        for i, t in enumerate(w.tensors):
            p = torch.from_numpy(masters[i]).to(dev) if masters[i] is not None else None
            g = None if t.frozen else torch.zeros(t.shape, dtype=gdt, device=dev)
            s = (torch.zeros(t.shape, dtype=torch.bfloat16, device=dev)
                 if (w.policy == "bf16_mixed" and not t.frozen) else None)
            if p is None:
                p = torch.zeros(t.shape, dtype=torch.float32, device=dev)
            self.P.append(p)
            self.G.append(g)
            self.S.append(s)
            entries.append((t.name, p, g, s, mx.MA_GROUP_FROZEN if t.frozen else None))
        self.opt = mx.MuonAdamW(entries, **cfg)

    def load_grads(self, grads: Sequence[Optional[np.ndarray]]) -> None:
        for g_dev, g in zip(self.G, grads):
            if g_dev is not None:
                g_dev.copy_(self.torch.from_numpy(np.ascontiguousarray(g)).to(g_dev.dtype))

    def step(self, lr: float) -> float:
        return self.opt.step(lr, want_norm=True)

    def param(self, i: int) -> np.ndarray:
        return self.P[i].cpu().numpy()

    def close(self):
        self.opt.close()


def compare_state(name: str, got: np.ndarray, want: np.ndarray, scale: np.ndarray, tol: float = STATE_TOL):
    err = np.abs(got.astype(np.float64) - want)
    bound = tol * scale + STATE_FLOOR
    bad = err > bound
    if bad.any():
        k = int(np.argmax(err - bound))
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {bad.size} elements out of tolerance; worst at flat index {k}: "
            f"got {got.flat[k]!r} want {want.flat[k]!r} scale {scale.flat[k]!r}")


class StateBounds:
    """Per-element error scales of the optimizer states, carried from step to
    step as the recurrences carry their errors (see the module docstring)."""

    def __init__(self):
        self.s: Dict[object, np.ndarray] = {}

    def recurrence(self, key, new: np.ndarray, prev: np.ndarray, decay: float, drive: np.ndarray) -> np.ndarray:
        """S = |new| + decay |prev| + |drive| + decay S_prev for new = decay prev + drive."""
        sc = np.abs(new) + decay * np.abs(prev) + np.abs(drive)
        if key in self.s:
            sc = sc + decay * self.s[key]
        self.s[key] = sc
        return sc

    def adamw_param(self, key, p: np.ndarray, s_m: np.ndarray, v: np.ndarray, t: int, lr: float, beta1: float,
                    beta2: float, eps: float) -> np.ndarray:
        """S_p = S_p_prev + |p| + (lr / bc1) S_m / (sqrt(v / bc2) + eps)."""
        bc1, bc2 = 1.0 - beta1 ** t, 1.0 - beta2 ** t
        sc = np.abs(p) + (lr / bc1) * s_m / (np.sqrt(v / bc2) + eps)
        if key in self.s:
            sc = sc + self.s[key]
        self.s[key] = sc
        return sc


def momentum_weight(cfg: dict) -> float:
    """Weight of the clipped gradient in the Muon momentum recurrence."""
    return 1.0 - float(cfg["muon_momentum"]) if cfg["muon_momentum_form"] == "ema" else 1.0


def relative_frobenius(got: np.ndarray, want: np.ndarray) -> float:
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / den) if den > 0 else float(np.linalg.norm(got))


def run_parity(w: workloads.Workload, *, steps: Optional[int] = None, config: Optional[dict] = None,
               oracle_overrides: Optional[dict] = None, muon_sample: Optional[Sequence[int]] = None,
               grad_scale: float = 1.0, lr: Optional[float] = None, check_states: bool = True,
               optim: str = "muon_adamw",
               param_options: Optional[Dict[int, Sequence[float]]] = None) -> Dict[str, object]:
    """Run ``steps`` optimizer steps on both sides and assert parity.

    ``muon_sample``: Muon parameter indices whose Newton-Schulz output is
    checked (all when None). Every AdamW/momentum element is checked when
    ``check_states`` is set. ``param_options``: {index: (lr_scale,
    weight_decay_scale)} given to both sides.
    """
    steps = steps or w.steps
    lr = w.lr if lr is None else lr
    masters = workloads.master_weights(w)
    gpu = GpuSide(w, masters, config=config)
    try:
        for i, (ls, ws) in (param_options or {}).items():
            gpu.opt.set_param_options(i, ls, ws)
        cfg = gpu.opt.cfg
        names = [t.name for t in w.tensors]
        shapes = [t.shape for t in w.tensors]
        frozen = [t.frozen for t in w.tensors]
        ov = dict(oracle_overrides or {})
        orc = oracle.HybridOracle(names, shapes, frozen, optim=optim, param_options=param_options, **ov)
        groups = orc.groups
        assert groups == gpu.opt.groups, "routing differs between the C ABI and the oracle"
        muon_idx = [i for i, g in enumerate(groups) if g == "muon"]
        adam_idx = [i for i, g in enumerate(groups) if g == "adamw"]
        sample = muon_idx if muon_sample is None else list(muon_sample)
        orc_p = [m.astype(np.float64) for m in masters]
        worst_o = 0.0
        o_errors: Dict[int, float] = {}
        beta1, beta2 = (float(b) for b in orc.cfg["adam_betas"])
        adam_eps = float(orc.cfg["adam_eps"])
        mu = float(orc.cfg["muon_momentum"])
        w_mom = momentum_weight(orc.cfg)
        bounds = StateBounds()
        for step in range(1, steps + 1):
            grads = workloads.gradients(w, step, scale=grad_scale)
            gpu.load_grads(grads)
            before = {i: gpu.param(i) for i in sample}
            # the oracle replaces its state arrays each step: these stay the previous step's
            buf_prev, m_prev = dict(orc.buf), dict(orc.m)
            total_gpu = gpu.step(lr)
            res = orc.step(orc_p, grads, lr, muon_indices=sample)
            # --- norm ---
            assert math.isclose(total_gpu, res["total"], rel_tol=NORM_TOL, abs_tol=1e-30), \
                f"step {step}: norm {total_gpu} vs {res['total']}"
            coef = res["coef"]
            # --- Muon: momentum (all elements) and O (sampled) ---
            for i in muon_idx:
                if check_states:
                    ghat = coef * grads[i].astype(np.float64)
                    buf = gpu.opt.state(i, 0).numpy()
                    compare_state(f"step {step} buf[{names[i]}]", buf, orc.buf[i],
                                  bounds.recurrence(("buf", i), orc.buf[i], buf_prev[i], mu, w_mom * ghat))
            for i in sample:
                m_, n_ = shapes[i]
                ls, ws = orc.options[i]
                decay = _f32(1.0 - lr * ls * cfg.muon_weight_decay * ws)
                lr_mult = _f32(ls * cfg.muon_lr_scale * cfg.moonlight_coef * math.sqrt(max(m_, n_)))
                after = gpu.param(i).astype(np.float64)
                O_gpu = (before[i].astype(np.float64) * decay - after) / (_f32(lr) * lr_mult)
                err = relative_frobenius(O_gpu, res["O"][i])
                worst_o = max(worst_o, err)
                o_errors[i] = max(o_errors.get(i, 0.0), err)
                assert err <= O_TOL, f"step {step} {names[i]} {shapes[i]}: O rel. Frobenius error {err:.3e}"
                if gpu.S[i] is not None:
                    sh = gpu.S[i].float().cpu().numpy()
                    want = workloads.bf16_round(after.astype(np.float32))
                    assert np.array_equal(sh, want), f"{names[i]}: bf16 shadow != bf16(p)"
            # --- AdamW ---
            if check_states:
                for i in adam_idx:
                    ghat = coef * grads[i].astype(np.float64)
                    m_gpu = gpu.opt.state(i, 0).numpy()
                    v_gpu = gpu.opt.state(i, 1).numpy()
                    s_m = bounds.recurrence(("m", i), orc.m[i], m_prev[i], beta1, (1.0 - beta1) * ghat)
                    compare_state(f"step {step} m[{names[i]}]", m_gpu, orc.m[i], s_m)
                    compare_state(f"step {step} v[{names[i]}]", v_gpu, orc.v[i], np.abs(orc.v[i]))
                    p_gpu = gpu.param(i)
                    compare_state(f"step {step} p[{names[i]}]", p_gpu, orc_p[i],
                                  bounds.adamw_param(("p", i), orc_p[i], s_m, orc.v[i], res["t"],
                                                     lr * orc.options[i][0], beta1, beta2, adam_eps))
                    if gpu.S[i] is not None:
                        sh = gpu.S[i].float().cpu().numpy()
                        assert np.array_equal(sh, workloads.bf16_round(p_gpu)), f"{names[i]}: shadow"
                    # keep the oracle on the same footing as the GPU for the
                    # next step's parameters (p is compared, not inherited)
            # frozen params are never written
            for i, fz in enumerate(frozen):
                if fz:
                    assert np.array_equal(gpu.param(i), masters[i]), f"frozen {names[i]} was modified"
        return {"worst_o": worst_o, "o_errors": o_errors, "steps": steps, "groups": groups}
    finally:
        gpu.close()


def _batches(idx: Sequence[int], size: int = 16):
    idx = list(idx)
    for k in range(0, len(idx), size):
        yield idx[k:k + size]


def run_parity_sampled(w: workloads.Workload, sample: Sequence[int], *, steps: int = 1,
                       o_sample: Optional[Sequence[int]] = None, lr: Optional[float] = None,
                       config: Optional[dict] = None) -> Dict[str, object]:
    """A whole workload on the GPU, the oracle on a sample of its tensors.

    Every master and gradient comes from the seeded generators (in batches,
    uploaded as they are made, so that full-size workloads fit in host
    memory). The expected global norm is ``oracle.global_grad_norm`` over
    every gradient of the model; an oracle over the sampled tensors steps
    with that norm (``total_override``). Compared each step: the norm, and
    for every sampled tensor its optimizer state and parameters at the
    tolerances of ``run_parity``; O of the Muon matrices in ``o_sample``
    (default: every sampled Muon matrix); frozen tensors stay unwritten.
    """
    import torch

    import muon_adamw_hybrid_grad_gb300 as mx

    lr = w.lr if lr is None else lr
    dev = torch.device("cuda")
    gdt = torch.bfloat16 if w.grad_dtype == "bf16" else torch.float32
    n = len(w.tensors)
    sample = sorted(set(sample))
    P: List = [None] * n
    G: List = [None] * n
    S: List = [None] * n
    m0: Dict[int, np.ndarray] = {}
    for batch in _batches(range(n)):
        for i, m in zip(batch, workloads.master_weights(w, batch)):
            t = w.tensors[i]
            P[i] = torch.from_numpy(m).to(dev)
            if not t.frozen:
                G[i] = torch.zeros(t.shape, dtype=gdt, device=dev)
                if w.policy == "bf16_mixed":
                    S[i] = torch.zeros(t.shape, dtype=torch.bfloat16, device=dev)
            if i in sample or t.frozen:
                m0[i] = m
    entries = [(t.name, P[i], G[i], S[i], mx.MA_GROUP_FROZEN if t.frozen else None)
               for i, t in enumerate(w.tensors)]
    cfg_kw = dict(config or {})
    cfg_kw.setdefault("precision", mx.MA_BF16_MIXED if w.policy == "bf16_mixed" else mx.MA_FP32_MIXED)
    opt = mx.MuonAdamW(entries, **cfg_kw)
    try:
        cfg = opt.cfg
        names = [w.tensors[i].name for i in sample]
        shapes = [w.tensors[i].shape for i in sample]
        frozen = [w.tensors[i].frozen for i in sample]
        orc = oracle.HybridOracle(names, shapes, frozen)
        for k, i in enumerate(sample):
            assert orc.groups[k] == opt.groups[i], f"routing of {names[k]} differs"
        local = {i: k for k, i in enumerate(sample)}
        o_idx = [i for i in (sample if o_sample is None else o_sample) if opt.groups[i] == "muon"]
        orc_p = [m0[i].astype(np.float64) for i in sample]
        beta1, beta2 = (float(b) for b in orc.cfg["adam_betas"])
        adam_eps = float(orc.cfg["adam_eps"])
        mu = float(orc.cfg["muon_momentum"])
        w_mom = momentum_weight(orc.cfg)
        bounds = StateBounds()
        worst_o = 0.0
        for step in range(1, steps + 1):
            sq = 0.0
            gs: Dict[int, np.ndarray] = {}
            for batch in _batches(range(n)):
                for i, g in zip(batch, workloads.gradients(w, step, batch)):
                    if g is None:
                        continue
                    G[i].copy_(torch.from_numpy(g).to(dev).to(gdt))
                    sq += float(np.sum(np.square(g, dtype=np.float64)))
                    if i in local:
                        gs[i] = g
            total = math.sqrt(sq)
            before = {i: P[i].cpu().numpy() for i in o_idx}
            buf_prev, m_prev = dict(orc.buf), dict(orc.m)
            total_gpu = opt.step(lr, want_norm=True)
            grads_local = [gs.get(i) for i in sample]
            res = orc.step(orc_p, grads_local, lr, muon_indices=[local[i] for i in o_idx], total_override=total)
            assert math.isclose(total_gpu, total, rel_tol=NORM_TOL), f"step {step}: norm {total_gpu} vs {total}"
            coef = res["coef"]
            for i in sample:
                k = local[i]
                grp = opt.groups[i]
                if grp == "frozen":
                    continue
                ghat = coef * gs[i].astype(np.float64)
                if grp == "muon":
                    compare_state(f"step {step} buf[{names[k]}]", opt.state(i, 0).numpy(), orc.buf[k],
                                  bounds.recurrence(("buf", k), orc.buf[k], buf_prev[k], mu, w_mom * ghat))
                else:
                    s_m = bounds.recurrence(("m", k), orc.m[k], m_prev[k], beta1, (1.0 - beta1) * ghat)
                    compare_state(f"step {step} m[{names[k]}]", opt.state(i, 0).numpy(), orc.m[k], s_m)
                    compare_state(f"step {step} v[{names[k]}]", opt.state(i, 1).numpy(), orc.v[k], np.abs(orc.v[k]))
                    p_gpu = P[i].cpu().numpy()
                    compare_state(f"step {step} p[{names[k]}]", p_gpu, orc_p[k],
                                  bounds.adamw_param(("p", k), orc_p[k], s_m, orc.v[k], res["t"], lr, beta1, beta2,
                                                     adam_eps))
                    if S[i] is not None:
                        assert np.array_equal(S[i].float().cpu().numpy(), workloads.bf16_round(p_gpu))
            for i in o_idx:
                k = local[i]
                m_, n_ = w.tensors[i].shape
                decay = _f32(1.0 - lr * cfg.muon_weight_decay)
                lr_mult = _f32(cfg.muon_lr_scale * cfg.moonlight_coef * math.sqrt(max(m_, n_)))
                after = P[i].cpu().numpy().astype(np.float64)
                O_gpu = (before[i].astype(np.float64) * decay - after) / (_f32(lr) * lr_mult)
                err = relative_frobenius(O_gpu, res["O"][k])
                worst_o = max(worst_o, err)
                assert err <= O_TOL, f"step {step} {names[k]} {(m_, n_)}: O rel. Frobenius error {err:.3e}"
                if S[i] is not None:
                    assert np.array_equal(S[i].float().cpu().numpy(), workloads.bf16_round(after.astype(np.float32)))
            for i, t in enumerate(w.tensors):
                if t.frozen:
                    assert torch.equal(P[i], torch.from_numpy(m0[i]).to(dev)), f"frozen {t.name} was modified"
        return {"worst_o": worst_o, "steps": steps, "o_checked": len(o_idx)}
    finally:
        opt.close()
