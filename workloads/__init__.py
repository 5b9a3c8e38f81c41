"""Seeded synthetic inputs for the hybrid Muon + AdamW optimizer step.

This module is shared by the CUDA-path tests/bench and by the fp64 oracle
tests. It holds parameter lists (names, shapes), the seeded random draws for
master weights and gradients, and the fp32 -> bf16 storage rounding of those
draws. It holds none of the optimizer's arithmetic.

Workloads (all synthetic; no dataset is involved):

``tiny``        2 action-expert layers {wq 256x256, w_up 1024x256,
                w_down 256x1024}; AdamW group = 4 RMSNorm weights [256] and a
                trainable 1000x256 embedding; 3 steps.
``h1024``       action expert, hidden 1024, MLP 4096, 16 layers:
                q,k,v,o 1024x1024, gate/up 4096x1024, down 1024x4096 (Muon);
                per layer 2 RMSNorms + q/k/v biases, plus a final norm (AdamW);
                grads = N(0, 1e-3) + rank-8 component of element std 5e-3;
                bf16 shadow written (bf16_mixed policy); 10 steps.
``h2048``       as h1024 at hidden 2048, MLP 8192, 24 layers (Muon group
                1.611 G elements); fp32_mixed policy (no shadow); 10 steps.
``many_small``  512 Muon matrices 128x512 and 256 of 512x128, plus 4096 1-D
                AdamW tensors with lengths drawn from
                ``default_rng(0).integers(128, 4097, 4096)``; 10 steps.
``narrow``      320 Muon matrices with a short side of 40 (128 of 1000x40,
                128 of 40x1000, 64 of 2000x40; rank-8 + noise gradients), which
                take the fp32 Newton-Schulz path, plus 8 norm vectors; 10 steps.
``full_vla``    Muon group of h2048 plus a 1.69 G-element AdamW backbone
                (28 layers of hidden 2048 with GQA k/v 1024x2048, MLP 6144,
                two norms; 67 vision stand-in blocks 2048x2048) and a frozen
                151936x2048 embedding; run at step 1000 of a 2000-step
                cosine_with_min_lr schedule (the schedule itself is computed by
                the optimizer side, not here); 5 steps.

Random draws: every tensor has its own ``numpy.random.PCG64`` stream keyed by
``SeedSequence([seed, kind, tensor_index, step])`` (kind 0 = master weight,
kind 1 = gradient). Masters ~ N(0, 0.02) in fp32. Gradients ~ N(0, 1e-3) in
fp32; Muon gradients of h1024/h2048/full_vla add ``s * P @ Q.T`` with P (m x 8),
Q (n x 8) ~ N(0, 1) and s = 5e-3 / sqrt(8). bf16 gradients are the fp32 draw
rounded to nearest-even bf16; both the GPU and the oracle consume exactly
those values.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional, Sequence, Tuple

import numpy as np

KIND_PARAM = 0
KIND_GRAD = 1

MASTER_STD = 0.02
GRAD_STD = 1e-3
RANK8_STD = 5e-3
RANK8 = 8


@dataclasses.dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: Tuple[int, ...]
    frozen: bool = False
    rank8: bool = False  # add the low-rank gradient component

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape)) if self.shape else 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tensors: Tuple[TensorSpec, ...]
    policy: str            # "bf16_mixed" (bf16 shadow written) or "fp32_mixed"
    grad_dtype: str        # "bf16" or "fp32"
    steps: int
    lr: float              # base learning rate
    seed: int = 0
    # (step, total_steps, warmup_steps, min_lr_rate) of a cosine_with_min_lr
    # schedule at which the workload is run; None = constant ``lr``.
    schedule: Optional[Tuple[int, int, int, float]] = None
    note: str = ""

    def trainable(self) -> List[int]:
        return [i for i, t in enumerate(self.tensors) if not t.frozen]


BASE_LR = 2.5e-5


def _expert_layers(hidden: int, mlp: int, layers: int, *, rank8: bool) -> List[TensorSpec]:
    out: List[TensorSpec] = []
    for i in range(layers):
        pre = f"model.action_expert.layers.{i}"
        for p in ("q", "k", "v", "o"):
            out.append(TensorSpec(f"{pre}.self_attn.{p}_proj.weight", (hidden, hidden), rank8=rank8))
        out.append(TensorSpec(f"{pre}.mlp.gate_proj.weight", (mlp, hidden), rank8=rank8))
        out.append(TensorSpec(f"{pre}.mlp.up_proj.weight", (mlp, hidden), rank8=rank8))
        out.append(TensorSpec(f"{pre}.mlp.down_proj.weight", (hidden, mlp), rank8=rank8))
    return out


def _expert_vectors(hidden: int, layers: int) -> List[TensorSpec]:
    out: List[TensorSpec] = []
    for i in range(layers):
        pre = f"model.action_expert.layers.{i}"
        out.append(TensorSpec(f"{pre}.input_layernorm.weight", (hidden,)))
        out.append(TensorSpec(f"{pre}.post_attention_layernorm.weight", (hidden,)))
        for p in ("q", "k", "v"):
            out.append(TensorSpec(f"{pre}.self_attn.{p}_proj.bias", (hidden,)))
    out.append(TensorSpec("model.action_expert.norm.weight", (hidden,)))
    return out


def _tiny() -> Workload:
    t: List[TensorSpec] = []
    for i in range(2):
        pre = f"model.action_expert.layers.{i}"
        t.append(TensorSpec(f"{pre}.wq.weight", (256, 256)))
        t.append(TensorSpec(f"{pre}.w_up.weight", (1024, 256)))
        t.append(TensorSpec(f"{pre}.w_down.weight", (256, 1024)))
    for i in range(2):
        pre = f"model.action_expert.layers.{i}"
        t.append(TensorSpec(f"{pre}.input_layernorm.weight", (256,)))
        t.append(TensorSpec(f"{pre}.post_attention_layernorm.weight", (256,)))
    t.append(TensorSpec("model.vlm.embed_tokens.weight", (1000, 256)))
    return Workload("tiny", tuple(t), policy="fp32_mixed", grad_dtype="bf16", steps=3, lr=BASE_LR)


def _h1024() -> Workload:
    t = _expert_layers(1024, 4096, 16, rank8=True) + _expert_vectors(1024, 16)
    return Workload("h1024", tuple(t), policy="bf16_mixed", grad_dtype="bf16", steps=10, lr=BASE_LR)


def _h2048(grad_dtype: str = "bf16") -> Workload:
    t = _expert_layers(2048, 8192, 24, rank8=True) + _expert_vectors(2048, 24)
    return Workload("h2048" if grad_dtype == "bf16" else "h2048_fp32grad", tuple(t),
                    policy="fp32_mixed", grad_dtype=grad_dtype, steps=10, lr=BASE_LR)


def many_small_lengths() -> np.ndarray:
    return np.random.default_rng(0).integers(128, 4097, 4096)


def _many_small() -> Workload:
    t: List[TensorSpec] = []
    for k in range(768):
        if k < 512:
            t.append(TensorSpec(f"model.action_expert.layers.{k}.w_a.weight", (128, 512)))
        else:
            t.append(TensorSpec(f"model.action_expert.layers.{k}.w_b.weight", (512, 128)))
    for k, n in enumerate(many_small_lengths()):
        t.append(TensorSpec(f"model.vlm.layers.{k}.ln.weight", (int(n),)))
    return Workload("many_small", tuple(t), policy="fp32_mixed", grad_dtype="bf16", steps=10, lr=BASE_LR)


def _narrow() -> Workload:
    t: List[TensorSpec] = []
    shapes = [(1000, 40)] * 128 + [(40, 1000)] * 128 + [(2000, 40)] * 64
    for k, sh in enumerate(shapes):
        t.append(TensorSpec(f"model.action_expert.layers.{k}.mlp.w_narrow.weight", sh, rank8=True))
    for k in range(8):
        t.append(TensorSpec(f"model.action_expert.layers.{k}.input_layernorm.weight", (1000,)))
    return Workload("narrow", tuple(t), policy="bf16_mixed", grad_dtype="bf16", steps=10, lr=BASE_LR)


FULL_VLA_VISION_BLOCKS = 67


def _full_vla() -> Workload:
    t = _expert_layers(2048, 8192, 24, rank8=True) + _expert_vectors(2048, 24)
    t.append(TensorSpec("model.vlm.embed_tokens.weight", (151936, 2048), frozen=True))
    for i in range(28):
        pre = f"model.vlm.language_model.layers.{i}"
        t.append(TensorSpec(f"{pre}.self_attn.q_proj.weight", (2048, 2048)))
        t.append(TensorSpec(f"{pre}.self_attn.k_proj.weight", (1024, 2048)))
        t.append(TensorSpec(f"{pre}.self_attn.v_proj.weight", (1024, 2048)))
        t.append(TensorSpec(f"{pre}.self_attn.o_proj.weight", (2048, 2048)))
        t.append(TensorSpec(f"{pre}.mlp.gate_proj.weight", (6144, 2048)))
        t.append(TensorSpec(f"{pre}.mlp.up_proj.weight", (6144, 2048)))
        t.append(TensorSpec(f"{pre}.mlp.down_proj.weight", (2048, 6144)))
        t.append(TensorSpec(f"{pre}.input_layernorm.weight", (2048,)))
        t.append(TensorSpec(f"{pre}.post_attention_layernorm.weight", (2048,)))
    for i in range(FULL_VLA_VISION_BLOCKS):
        t.append(TensorSpec(f"model.vlm.vision_tower.blocks.{i}.proj.weight", (2048, 2048)))
    return Workload("full_vla", tuple(t), policy="fp32_mixed", grad_dtype="bf16", steps=5, lr=BASE_LR,
                    schedule=(1000, 2000, 0, 0.1),
                    note="lr from cosine_with_min_lr at step 1000 of 2000 (no warmup), min_lr_rate 0.1")


_BUILDERS = {
    "tiny": _tiny,
    "h1024": _h1024,
    "h2048": _h2048,
    "h2048_fp32grad": lambda: _h2048("fp32"),
    "many_small": _many_small,
    "narrow": _narrow,
    "full_vla": _full_vla,
}

WORKLOADS = tuple(_BUILDERS)


def get_workload(name: str) -> Workload:
    """A named workload, or ``expert:<hidden>:<mlp>:<layers>[:<policy>]`` for
    an action expert of that size built like h1024 (bf16 grads with the
    rank-8 part; policy bf16_mixed unless ``fp32_mixed`` is given, as the
    2048-hidden expert of h2048 and full_vla uses)."""
    if name.startswith("expert:"):
        parts = name.split(":")[1:]
        hidden, mlp, layers = (int(x) for x in parts[:3])
        policy = parts[3] if len(parts) > 3 else "bf16_mixed"
        if policy not in ("bf16_mixed", "fp32_mixed"):
            raise KeyError(f"unknown policy {policy!r} in {name!r}")
        t = _expert_layers(hidden, mlp, layers, rank8=True) + _expert_vectors(hidden, layers)
        return Workload(name, tuple(t), policy=policy, grad_dtype="bf16", steps=10, lr=BASE_LR)
    try:
        return _BUILDERS[name]()
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {', '.join(WORKLOADS)} or expert:H:M:L") from None


def scaled_workload(name: str, *, layers: int, hidden: int, mlp: int, vectors: bool = True) -> Workload:
    """An action-expert workload of arbitrary size (parity tests at small sizes)."""
    t = _expert_layers(hidden, mlp, layers, rank8=True)
    if vectors:
        t += _expert_vectors(hidden, layers)
    return Workload(name, tuple(t), policy="bf16_mixed", grad_dtype="bf16", steps=3, lr=BASE_LR)


def custom_workload(name: str, tensors: Sequence[TensorSpec], *, policy: str = "bf16_mixed",
                    grad_dtype: str = "bf16", steps: int = 3, lr: float = BASE_LR) -> Workload:
    return Workload(name, tuple(tensors), policy=policy, grad_dtype=grad_dtype, steps=steps, lr=lr)


# ---------------------------------------------------------------------------
# Seeded draws
# ---------------------------------------------------------------------------

def _rng(seed: int, kind: int, index: int, step: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, kind, index, step])))


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32 holding bf16 values."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    rounded = (bits + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    # NaN stays NaN (quiet it); inf stays inf through the add above.
    nan = np.isnan(x)
    if nan.any():
        rounded = np.where(nan, np.uint32(0x7FC00000), rounded)
    return rounded.view(np.float32)


def bf16_bits(x_bf16_valued: np.ndarray) -> np.ndarray:
    """Upper 16 bits of fp32 values that are exactly bf16-representable."""
    return (np.ascontiguousarray(x_bf16_valued, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def master_weight(w: Workload, index: int) -> np.ndarray:
    spec = w.tensors[index]
    r = _rng(w.seed, KIND_PARAM, index, 0)
    return (r.standard_normal(spec.numel, dtype=np.float32) * np.float32(MASTER_STD)).reshape(spec.shape)


def gradient(w: Workload, index: int, step: int, scale: float = 1.0) -> np.ndarray:
    """Gradient of tensor ``index`` at optimizer step ``step`` (1-based), fp32 array.

    For bf16 workloads the values are already rounded to bf16.
    """
    spec = w.tensors[index]
    r = _rng(w.seed, KIND_GRAD, index, step)
    g = r.standard_normal(spec.numel, dtype=np.float32) * np.float32(GRAD_STD)
    if spec.rank8 and len(spec.shape) == 2:
        m, n = spec.shape
        p = r.standard_normal((m, RANK8), dtype=np.float32)
        q = r.standard_normal((n, RANK8), dtype=np.float32)
        g = g.reshape(m, n) + np.float32(RANK8_STD / math.sqrt(RANK8)) * (p @ q.T)
    g = g.reshape(spec.shape)
    if scale != 1.0:
        g = g * np.float32(scale)
    if w.grad_dtype == "bf16":
        g = bf16_round(g)
    return g.astype(np.float32, copy=False)


def _pool_workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def master_weights(w: Workload, indices: Optional[Sequence[int]] = None) -> List[np.ndarray]:
    idx = list(range(len(w.tensors))) if indices is None else list(indices)
    with ThreadPoolExecutor(_pool_workers()) as ex:
        return list(ex.map(lambda i: master_weight(w, i), idx))


def gradients(w: Workload, step: int, indices: Optional[Sequence[int]] = None,
              scale: float = 1.0) -> List[Optional[np.ndarray]]:
    idx = list(range(len(w.tensors))) if indices is None else list(indices)

    def one(i: int):
        return None if w.tensors[i].frozen else gradient(w, i, step, scale)

    with ThreadPoolExecutor(_pool_workers()) as ex:
        return list(ex.map(one, idx))
