"""fp64 CPU oracle of the hybrid Muon + AdamW optimizer step (test infrastructure).

This package is test infrastructure. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. The product path (the
CUDA library and its Python binding) never imports, links or runs anything
here, and this package imports nothing from the product: the two share only
the seeded input generators in ``workloads``.

Source of the method: the article "VLA训练栈深度揭秘：OpenDM的Muon+AdamW优化器、
FSDP分布式训练与混合精度策略" (gsyq.cn/news/451971), section 核心揭秘一 (the
MuonAdamW hybrid optimizer): parameter routing (参数如何分流), Newton-Schulz
orthogonalisation (Muon 的工作原理), the default hyperparameters
(关键超参默认值), and the training-stack defaults table (训练栈默认参数速查表:
cosine_with_min_lr with min_lr_rate 0.1, max_grad_norm 1.0).

Every function is plain fp64 numpy, written step by step; the readings taken
where the article is silent are listed in ``hybrid.READINGS``.

Pins (tests marked ``not gpu``): NS5 against the SVD closed form
U diag(phi^5(sigma)) V^T, the quintic's singular-value band, the polar factor,
transpose and scale invariance, rank-1 closed forms of the full Muon update,
closed-form AdamW trajectories (t = 1 sign step, constant gradient, zero
gradient, unrolled EMAs), hand-computed clip factors and lr scalings, the
schedule's closed-form points and the routing table; the variants (exponential-
average momentum, coefficient schedules, per-parameter lr / weight-decay
multipliers, the bias/norm decay exemption) against unrolled sums, composed
SVD closed forms and hand-solved steps. No function here is "parity unpinned".
"""
from .hybrid import (  # noqa: F401
    DEFAULTS,
    READINGS,
    GROUP_MUON,
    GROUP_ADAMW,
    GROUP_FROZEN,
    is_muon_parameter,
    route,
    global_grad_norm,
    clip_coefficient,
    nesterov_momentum,
    zeropower_newton_schulz5,
    decay_exempt,
    muon_lr,
    muon_apply,
    adamw_update,
    cosine_with_min_lr,
    HybridOracle,
)
