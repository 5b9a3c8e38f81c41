"""fp64 oracle of the hybrid Muon + AdamW step (test infrastructure; see package doc).

Citations name the article "VLA训练栈深度揭秘：OpenDM的Muon+AdamW优化器、FSDP分布式
训练与混合精度策略" (OpenDM VLA training stack, gsyq.cn/news/451971) and its
sections; "LeRobot multi-GPU training guide, notes" is the huggingface LeRobot
page on multi-GPU training, section 注意/Примечания.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

GROUP_MUON = "muon"
GROUP_ADAMW = "adamw"
GROUP_FROZEN = "frozen"

# Hyperparameters. Page values cite the article; the others are the workload
# definition's values (the article does not print them).
DEFAULTS: Dict[str, object] = {
    # OpenDM article, 核心揭秘一 / 关键超参默认值 (key hyperparameter defaults)
    "muon_momentum": 0.95,
    "muon_nesterov": True,
    "muon_ns_steps": 5,
    "muon_moonlight_coefficient": 0.2,
    "base_lr": 2.5e-5,
    # muon_lr_scale is named in the same section without a value: reading 1.0
    "muon_lr_scale": 1.0,
    # OpenDM article, 训练栈默认参数速查表 (defaults table)
    "max_grad_norm": 1.0,
    "lr_scheduler": "cosine_with_min_lr",
    "min_lr_rate": 0.1,
    "optim": "adamw",
    "precision_policy": "bf16_mixed",
    # Not printed on the page: the standard Muon quintic, as given by the
    # workload definition, and that definition's AdamW settings.
    "ns_coefficients": (3.4445, -4.7750, 2.0315),
    "ns_eps": 1e-7,
    "adam_betas": (0.9, 0.999),
    "adam_eps": 1e-8,
    "weight_decay": 0.1,
    "muon_weight_decay": 0.1,
    "clip_eps": 1e-6,
    # Variants off by default (the page's step uses none of them): the
    # exponential-average form of the momentum, a per-iteration coefficient
    # schedule, and no weight decay on biases and normalisation weights.
    "muon_momentum_form": "sgd",
    "ns_schedule": None,
    "adam_decay_exempt_bias_norm": False,
}

READINGS = {
    "routing": "2-D, name contains 'action_expert', a dotted component equals 'layers', "
               "name ends with '.weight', lower-cased name contains none of 'embed', "
               "'lm_head', 'norm'",
    "nesterov": "buf = mu*buf + g; update = g + mu*buf (SGD-Nesterov form)",
    "ns_coefficients": "the same (a, b, c) in all five iterations",
    "short_side": "transpose iff rows > cols; square matrices are not transposed",
    "normalise": "X0 = G / (||G||_F + 1e-7)",
    "lr_scale": "lr * muon_lr_scale * 0.2 * sqrt(max(rows, cols)) of the full matrix",
    "muon_weight_decay": "decoupled p *= 1 - lr*wd with the base lr, wd 0.1",
    "adamw": "PyTorch AdamW: decoupled decay first, eps outside sqrt of bias-corrected v",
    "clip": "coef = min(1, max_norm/(total+1e-6)) over both groups' gradients, before either update; "
            "a NaN norm gives a NaN coefficient, an infinite norm gives 0",
    "schedule": "HF cosine_with_min_lr, num_cycles 0.5, lr = base*(min + (1-min)*0.5*(1+cos(pi*p)))",
    "momentum_form_ema": "variant: buf = mu*buf + (1-mu)*g; update = (1-mu)*g + mu*buf (Nesterov) or buf",
    "ns_schedule": "variant: iteration i uses its own (a_i, b_i, c_i) in the same three products",
    "param_options": "per parameter, like a PyTorch parameter group: lr_i = lr*lr_scale and "
                     "wd_i = wd*wd_scale, used in both the step and the decoupled decay",
    "decay_exempt": "variant: an AdamW parameter whose lower-cased name ends with 'bias' or contains "
                    "'norm' has wd_scale 0 unless set explicitly",
}


# ---------------------------------------------------------------------------
# Routing -- OpenDM article, 核心揭秘一 / 参数如何分流 (how parameters are routed)
# ---------------------------------------------------------------------------

def is_muon_parameter(name: str, ndim: int) -> bool:
    """The article's rule for is_default_muon_parameter.

    A parameter goes to Muon when it is a matrix (2-D), its path holds
    ``action_expert`` and sits under ``layers``, it ends with ``.weight``, and
    it is neither an embedding, ``lm_head`` nor a norm layer.
    """
    if ndim != 2:
        return False
    if "action_expert" not in name:
        return False
    if "layers" not in name.split("."):
        return False
    if not name.endswith(".weight"):
        return False
    low = name.lower()
    for excluded in ("embed", "lm_head", "norm"):
        if excluded in low:
            return False
    return True


def route(name: str, ndim: int, *, frozen: bool = False, optim: str = "muon_adamw") -> str:
    """Group of one parameter. ``optim='adamw'`` sends everything to AdamW
    (article, end of 参数如何分流: the optim switch falls back to pure AdamW)."""
    if frozen:
        return GROUP_FROZEN
    if optim == "muon_adamw" and is_muon_parameter(name, ndim):
        return GROUP_MUON
    return GROUP_ADAMW


# ---------------------------------------------------------------------------
# Gradient clipping -- OpenDM article, defaults table: max_grad_norm 1.0
# ---------------------------------------------------------------------------

def global_grad_norm(grads: Sequence[np.ndarray]) -> float:
    """Euclidean norm of all gradients taken together, in fp64."""
    total_sq = 0.0
    for g in grads:
        g64 = np.asarray(g, dtype=np.float64)
        total_sq += float(np.sum(g64 * g64))
    return math.sqrt(total_sq)


def clip_coefficient(total: float, max_norm: float, eps: float = 1e-6) -> float:
    """Factor applied to every gradient: min(1, max_norm / (total + eps)).

    The article gives no rule for a non-finite norm. Reading: no step is
    skipped; a NaN norm gives a NaN factor (every update becomes NaN, as
    multiplying the gradients by the unclamped ratio would), and an infinite
    norm gives the factor 0.
    """
    if max_norm <= 0.0:
        return 1.0
    if math.isnan(total):
        return float("nan")
    return min(1.0, max_norm / (total + eps))


# ---------------------------------------------------------------------------
# Muon -- OpenDM article, 核心揭秘一 / Muon 的工作原理 and 关键超参默认值
# ---------------------------------------------------------------------------

def nesterov_momentum(buf: np.ndarray, g: np.ndarray, mu: float, nesterov: bool = True,
                      form: str = "sgd"):
    """Momentum buffer update and the update direction fed to Newton-Schulz.

    form "sgd" (the step's reading of muon_nesterov): buf <- mu * buf + g,
    and the Nesterov look-ahead direction is g + mu * buf.
    form "ema" (a variant): the buffer is an exponential average,
    buf <- mu * buf + (1 - mu) * g, and the look-ahead direction is
    (1 - mu) * g + mu * buf.
    Without Nesterov the direction is the buffer itself. Returns
    (new_buf, direction).
    """
    if form == "sgd":
        w = 1.0
    elif form == "ema":
        w = 1.0 - mu
    else:
        raise ValueError(f"unknown momentum form {form!r}")
    new_buf = mu * buf + w * g
    direction = w * g + mu * new_buf if nesterov else new_buf.copy()
    return new_buf, direction


def zeropower_newton_schulz5(G: np.ndarray, steps: int = 5,
                             coefficients=(3.4445, -4.7750, 2.0315),
                             eps: float = 1e-7) -> np.ndarray:
    """Newton-Schulz approximation of the orthogonal factor of ``G`` (fp64).

    Works on the short side: a tall matrix is transposed first and the
    result transposed back. The matrix is scaled to unit Frobenius norm, then
    each iteration forms A = X X^T, B = b A + c A A and X <- a X + B X.
    ``coefficients`` is one (a, b, c) used in every iteration, or a sequence
    of ``steps`` triples, the i-th used in iteration i (a schedule).
    """
    coeffs = np.asarray(coefficients, dtype=np.float64)
    if coeffs.ndim == 1:
        schedule = [tuple(coeffs)] * steps
    else:
        if coeffs.shape != (steps, 3):
            raise ValueError(f"a schedule needs {steps} triples, got shape {coeffs.shape}")
        schedule = [tuple(row) for row in coeffs]
    X = np.array(G, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = X / (np.linalg.norm(X) + eps)
    for a, b, c in schedule:
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    if tall:
        X = X.T
    return X


def decay_exempt(name: str) -> bool:
    """Biases and normalisation weights take no weight decay when the
    exemption variant is on (the convention of HF Trainer's selection of
    decay parameters; the defaults table lists one weight_decay for all)."""
    low = name.lower()
    return low.endswith("bias") or "norm" in low


def muon_lr(lr: float, rows: int, cols: int, muon_lr_scale: float = 1.0,
            moonlight_coefficient: float = 0.2) -> float:
    """Effective Muon lr: lr * muon_lr_scale * 0.2 * sqrt(max(shape))."""
    return lr * muon_lr_scale * moonlight_coefficient * math.sqrt(max(rows, cols))


def muon_apply(p: np.ndarray, O: np.ndarray, lr: float, weight_decay: float, lr_eff: float) -> np.ndarray:
    """Decoupled weight decay with the base lr, then the scaled orthogonal step."""
    return p * (1.0 - lr * weight_decay) - lr_eff * O


# ---------------------------------------------------------------------------
# AdamW -- every parameter not routed to Muon (article, 参数如何分流)
# ---------------------------------------------------------------------------

def adamw_update(p, g, m, v, t: int, lr: float, beta1: float, beta2: float,
                 eps: float, weight_decay: float):
    """One decoupled-weight-decay Adam step at step count ``t`` (1-based).

    Returns (p, m, v). The bias-corrected second moment's square root is
    taken before eps is added.
    """
    p = p * (1.0 - lr * weight_decay)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * (g * g)
    bc1 = 1.0 - beta1 ** t
    bc2 = 1.0 - beta2 ** t
    denom = np.sqrt(v) / math.sqrt(bc2) + eps
    p = p - (lr / bc1) * (m / denom)
    return p, m, v


# ---------------------------------------------------------------------------
# Schedule -- defaults table: cosine_with_min_lr, min_lr_rate 0.1; stepped once
# per optimizer step (LeRobot multi-GPU guide, notes)
# ---------------------------------------------------------------------------

def cosine_with_min_lr(step: int, total_steps: int, warmup_steps: int, min_lr_rate: float) -> float:
    """Multiplier of the base lr at ``step``: linear warmup, then a half cosine
    from 1 down to ``min_lr_rate``."""
    if step < warmup_steps:
        return step / max(1, warmup_steps)
    progress = (step - warmup_steps) / max(1, total_steps - warmup_steps)
    cosine = 0.5 * (1.0 + math.cos(math.pi * progress))
    return max(0.0, cosine * (1.0 - min_lr_rate) + min_lr_rate)


# ---------------------------------------------------------------------------
# The whole hybrid step
# ---------------------------------------------------------------------------

class HybridOracle:
    """fp64 state and step of the hybrid optimizer over a list of parameters.

    ``names``/``shapes``/``frozen`` describe the parameters in registration
    order. ``step(params, grads, lr)`` updates ``params`` (a list of fp64
    arrays, modified in place) and returns a dict with the global norm, the
    clip coefficient and the orthogonalised update O of every Muon matrix.
    """

    def __init__(self, names: Sequence[str], shapes: Sequence[Sequence[int]],
                 frozen: Optional[Sequence[bool]] = None, *, optim: str = "muon_adamw",
                 param_options: Optional[Dict[int, Sequence[float]]] = None, **overrides):
        cfg = dict(DEFAULTS)
        cfg.update(overrides)
        self.cfg = cfg
        self.names = list(names)
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        fz = list(frozen) if frozen is not None else [False] * len(self.names)
        self.groups = [route(n, len(s), frozen=f, optim=optim)
                       for n, s, f in zip(self.names, self.shapes, fz)]
        # per parameter (lr_scale, wd_scale): explicit options win over the exemption rule
        self.options = []
        for i, (n, grp) in enumerate(zip(self.names, self.groups)):
            ls, ws = 1.0, 1.0
            if cfg["adam_decay_exempt_bias_norm"] and grp == GROUP_ADAMW and decay_exempt(n):
                ws = 0.0
            if param_options and i in param_options:
                ls, ws = (float(x) for x in param_options[i])
            self.options.append((ls, ws))
        self.t = 0
        self.buf: Dict[int, np.ndarray] = {}
        self.m: Dict[int, np.ndarray] = {}
        self.v: Dict[int, np.ndarray] = {}
        for i, (grp, shp) in enumerate(zip(self.groups, self.shapes)):
            if grp == GROUP_MUON:
                self.buf[i] = np.zeros(shp, dtype=np.float64)
            elif grp == GROUP_ADAMW:
                self.m[i] = np.zeros(shp, dtype=np.float64)
                self.v[i] = np.zeros(shp, dtype=np.float64)

    def step(self, params: List[np.ndarray], grads: List[Optional[np.ndarray]], lr: float,
             muon_indices: Optional[Sequence[int]] = None, total_override: Optional[float] = None) -> dict:
        """One optimizer step. ``muon_indices`` limits the (expensive) Muon
        orthogonalisation to a subset; the other Muon matrices still get their
        momentum update but no parameter update (used for sampled checks).
        ``total_override``: the global gradient norm when this oracle holds
        only a sample of a model's parameters (computed by ``global_grad_norm``
        over every gradient of the model); the clip coefficient follows from it."""
        cfg = self.cfg
        self.t += 1
        t = self.t
        active = [i for i, g in enumerate(self.groups) if g != GROUP_FROZEN]
        total = global_grad_norm([grads[i] for i in active]) if total_override is None else float(total_override)
        coef = clip_coefficient(total, float(cfg["max_grad_norm"]), float(cfg["clip_eps"]))
        a_b_c = cfg["ns_schedule"] if cfg["ns_schedule"] is not None else tuple(cfg["ns_coefficients"])
        beta1, beta2 = cfg["adam_betas"]
        out_O: Dict[int, np.ndarray] = {}
        for i in active:
            g = coef * np.asarray(grads[i], dtype=np.float64)
            ls, ws = self.options[i]
            lr_i = lr * ls
            if self.groups[i] == GROUP_MUON:
                self.buf[i], direction = nesterov_momentum(
                    self.buf[i], g, float(cfg["muon_momentum"]), bool(cfg["muon_nesterov"]),
                    str(cfg["muon_momentum_form"]))
                if muon_indices is not None and i not in muon_indices:
                    continue
                O = zeropower_newton_schulz5(direction, int(cfg["muon_ns_steps"]), a_b_c,
                                             float(cfg["ns_eps"]))
                rows, cols = self.shapes[i]
                lr_eff = muon_lr(lr_i, rows, cols, float(cfg["muon_lr_scale"]),
                                 float(cfg["muon_moonlight_coefficient"]))
                params[i][...] = muon_apply(params[i], O, lr_i, float(cfg["muon_weight_decay"]) * ws, lr_eff)
                out_O[i] = O
            else:
                p, m, v = adamw_update(params[i], g, self.m[i], self.v[i], t, lr_i, float(beta1),
                                       float(beta2), float(cfg["adam_eps"]), float(cfg["weight_decay"]) * ws)
                params[i][...] = p
                self.m[i], self.v[i] = m, v
        return {"total": total, "coef": coef, "O": out_O, "t": t}
