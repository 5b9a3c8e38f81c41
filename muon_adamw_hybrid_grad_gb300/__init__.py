"""Python binding of the GB300 hybrid Muon + AdamW optimizer library.

Argument marshalling only: every step of the optimizer runs in the CUDA
kernels of ``lib/libmuon_adamw_gb300.so`` behind the C ABI declared in
``include/muon_adamw.h``. The functions below carry the C names; the
``MuonAdamW`` class is a convenience wrapper that takes torch tensors and
passes their device pointers and the current CUDA stream.

There is no fallback: if the shared library has not been built, every call
raises ``LibraryNotBuilt`` (run ``muon_adamw_hybrid_grad_gb300.build.build()``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import build as _build

# ---- enums (mirror include/muon_adamw.h) ----
MA_OK = 0
MA_ERR_ARG = 1
MA_ERR_SHAPE = 2
MA_ERR_DTYPE = 3
MA_ERR_ALIGN = 4
MA_ERR_STATE = 5
MA_ERR_OOM = 6
MA_ERR_CUDA = 7
MA_ERR_DEVICE_CHECK = 8
MA_ERR_UNSUPPORTED = 9
STATUS_NAMES = {0: "MA_OK", 1: "MA_ERR_ARG", 2: "MA_ERR_SHAPE", 3: "MA_ERR_DTYPE", 4: "MA_ERR_ALIGN",
                5: "MA_ERR_STATE", 6: "MA_ERR_OOM", 7: "MA_ERR_CUDA", 8: "MA_ERR_DEVICE_CHECK",
                9: "MA_ERR_UNSUPPORTED"}

MA_MODE_MUON_ADAMW = 0
MA_MODE_ADAMW_ONLY = 1
MA_BF16_MIXED = 0
MA_FP32_MIXED = 1
MA_GROUP_AUTO = 0
MA_GROUP_MUON = 1
MA_GROUP_ADAMW = 2
MA_GROUP_FROZEN = 3
MA_DT_F32 = 0
MA_DT_BF16 = 1
MA_NS_TCGEN05 = 0
MA_NS_SIMT = 1
MA_MOMENTUM_SGD = 0
MA_MOMENTUM_EMA = 1
MA_NS_SCHEDULE_MAX = 16
MA_MAX_OPTION_GROUPS = 8

KERNEL_KINDS = ("grad_norm", "clip", "momentum", "ns_prep", "ns_gram", "ns_poly", "ns_update", "adamw", "ns_apply",
                "ns_fused", "ns_narrow")
MA_K_COUNT = len(KERNEL_KINDS)
GROUP_NAMES = {MA_GROUP_MUON: "muon", MA_GROUP_ADAMW: "adamw", MA_GROUP_FROZEN: "frozen"}


class MuonAdamWConfig(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int32),
        ("precision", ctypes.c_int32),
        ("muon_nesterov", ctypes.c_int32),
        ("ns_steps", ctypes.c_int32),
        ("ns_kernel", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 4),
        ("muon_momentum_form", ctypes.c_int32),
        ("adam_decay_exempt_bias_norm", ctypes.c_int32),
        ("ns_schedule_len", ctypes.c_int32),
        ("muon_momentum", ctypes.c_double),
        ("ns_a", ctypes.c_double),
        ("ns_b", ctypes.c_double),
        ("ns_c", ctypes.c_double),
        ("ns_eps", ctypes.c_double),
        ("moonlight_coef", ctypes.c_double),
        ("muon_lr_scale", ctypes.c_double),
        ("muon_weight_decay", ctypes.c_double),
        ("adam_beta1", ctypes.c_double),
        ("adam_beta2", ctypes.c_double),
        ("adam_eps", ctypes.c_double),
        ("adam_weight_decay", ctypes.c_double),
        ("max_grad_norm", ctypes.c_double),
        ("clip_eps", ctypes.c_double),
        ("ns_schedule", (ctypes.c_double * 3) * MA_NS_SCHEDULE_MAX),
    ]


class Profile(ctypes.Structure):
    _fields_ = [
        ("launches", ctypes.c_int64 * MA_K_COUNT),
        ("ms", ctypes.c_double * MA_K_COUNT),
        ("units", ctypes.c_double * MA_K_COUNT),
        ("steps", ctypes.c_int64),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("n_params", ctypes.c_int32),
        ("n_muon", ctypes.c_int32),
        ("n_adamw", ctypes.c_int32),
        ("n_frozen", ctypes.c_int32),
        ("n_buckets", ctypes.c_int32),
        ("muon_elems", ctypes.c_int64),
        ("adamw_elems", ctypes.c_int64),
        ("grad_elems", ctypes.c_int64),
        ("state_bytes", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
        ("ns_flops_per_step", ctypes.c_double),
        ("ns_dense_flops_per_step", ctypes.c_double),
        ("stream_bytes_per_step", ctypes.c_double),
    ]


class LibraryNotBuilt(RuntimeError):
    pass


class MuonAdamWError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


# Exported symbols and their ctypes signatures: (restype, argtypes).
_P = ctypes.c_void_p
_SIGNATURES = {
    "muon_adamw_config_init": (None, [ctypes.POINTER(MuonAdamWConfig)]),
    "muon_adamw_is_muon_param": (ctypes.c_int, [ctypes.c_char_p, ctypes.c_int]),
    "muon_adamw_cosine_with_min_lr": (ctypes.c_double, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                        ctypes.c_double]),
    "muon_adamw_create": (ctypes.c_int, [ctypes.POINTER(MuonAdamWConfig), _P, ctypes.POINTER(_P)]),
    "muon_adamw_register_param": (ctypes.c_int, [_P, ctypes.c_char_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                                                 _P, _P, ctypes.c_int, _P, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "muon_adamw_step": (ctypes.c_int, [_P, ctypes.c_double, ctypes.POINTER(ctypes.c_float)]),
    "muon_adamw_sync": (ctypes.c_int, [_P]),
    "muon_adamw_test_arm_stall": (ctypes.c_int, [_P]),
    "muon_adamw_plan_work_order": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                                                  ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                                  ctypes.POINTER(ctypes.c_int32), ctypes.c_int64,
                                                  ctypes.POINTER(ctypes.c_int64)]),
    "muon_adamw_record_grads_consumed": (ctypes.c_int, [_P, _P]),
    "muon_adamw_set_graph_mode": (ctypes.c_int, [_P, ctypes.c_int]),
    "muon_adamw_set_param_options": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_double, ctypes.c_double]),
    "muon_adamw_get_state": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _P]),
    "muon_adamw_set_state": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _P]),
    "muon_adamw_get_step": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int64)]),
    "muon_adamw_set_step": (ctypes.c_int, [_P, ctypes.c_int64]),
    "muon_adamw_last_norm": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]),
    "muon_adamw_plan_info": (ctypes.c_int, [_P, ctypes.POINTER(PlanInfo)]),
    "muon_adamw_set_profiling": (ctypes.c_int, [_P, ctypes.c_int]),
    "muon_adamw_get_profile": (ctypes.c_int, [_P, ctypes.POINTER(Profile)]),
    "muon_adamw_reset_profile": (ctypes.c_int, [_P]),
    "muon_adamw_destroy": (ctypes.c_int, [_P]),
    "muon_adamw_plan_shards": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                              ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                              ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64),
                                              ctypes.POINTER(ctypes.c_int64)]),
    "muon_adamw_set_shard": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int]),
    "muon_adamw_shard_range": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                                              ctypes.POINTER(ctypes.c_int64)]),
    "muon_adamw_step_begin": (ctypes.c_int, [_P, ctypes.c_double, _P]),
    "muon_adamw_step_end": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_float)]),
    "muon_adamw_grad_norm_noalloc": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_int64),
                                                    ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_double,
                                                    ctypes.c_double, _P, _P]),
    "muon_adamw_last_error": (ctypes.c_char_p, []),
    "muon_adamw_version": (ctypes.c_char_p, []),
}

_LIB: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.lib_path()


def load_library() -> ctypes.CDLL:
    """Load the shared library (once). Raises LibraryNotBuilt if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise LibraryNotBuilt(f"{path} is missing: build it with muon_adamw_hybrid_grad_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != MA_OK:
        msg = load_library().muon_adamw_last_error().decode("utf-8", "replace")
        raise MuonAdamWError(status, msg)


# ---- C-named functions ----

def muon_adamw_config_init() -> MuonAdamWConfig:
    cfg = MuonAdamWConfig()
    load_library().muon_adamw_config_init(ctypes.byref(cfg))
    return cfg


def muon_adamw_is_muon_param(name: str, ndim: int) -> bool:
    return bool(load_library().muon_adamw_is_muon_param(name.encode("utf-8"), int(ndim)))


def muon_adamw_cosine_with_min_lr(step: int, total: int, warmup: int, min_lr_rate: float) -> float:
    return float(load_library().muon_adamw_cosine_with_min_lr(int(step), int(total), int(warmup), float(min_lr_rate)))


def muon_adamw_create(cfg: MuonAdamWConfig, cuda_stream: int = 0) -> int:
    h = _P()
    _check(load_library().muon_adamw_create(ctypes.byref(cfg), _P(cuda_stream or None), ctypes.byref(h)))
    return h.value


def muon_adamw_register_param(h: int, name: str, shape: Sequence[int], param_ptr: int, grad_ptr: int,
                              grad_dtype: int, shadow_ptr: int = 0, group: int = MA_GROUP_AUTO):
    """Returns (index, assigned_group)."""
    arr = (ctypes.c_int64 * max(1, len(shape)))(*[int(d) for d in shape])
    assigned = ctypes.c_int(-1)
    index = ctypes.c_int(-1)
    _check(load_library().muon_adamw_register_param(
        _P(h), name.encode("utf-8"), len(shape), arr, _P(param_ptr or None), _P(grad_ptr or None),
        int(grad_dtype), _P(shadow_ptr or None), int(group), ctypes.byref(assigned), ctypes.byref(index)))
    return index.value, assigned.value


def muon_adamw_step(h: int, lr: float, want_norm: bool = False) -> Optional[float]:
    if want_norm:
        out = ctypes.c_float()
        _check(load_library().muon_adamw_step(_P(h), float(lr), ctypes.byref(out)))
        return float(out.value)
    _check(load_library().muon_adamw_step(_P(h), float(lr), None))
    return None


def muon_adamw_sync(h: int) -> None:
    _check(load_library().muon_adamw_sync(_P(h)))


def muon_adamw_set_param_options(h: int, index: int, lr_scale: float, weight_decay_scale: float) -> None:
    _check(load_library().muon_adamw_set_param_options(_P(h), int(index), float(lr_scale),
                                                       float(weight_decay_scale)))


def muon_adamw_set_graph_mode(h: int, enable: bool) -> None:
    _check(load_library().muon_adamw_set_graph_mode(_P(h), 1 if enable else 0))


def muon_adamw_record_grads_consumed(h: int, cuda_event: int) -> None:
    _check(load_library().muon_adamw_record_grads_consumed(_P(h), _P(cuda_event)))


def muon_adamw_test_arm_stall(h: int) -> None:
    _check(load_library().muon_adamw_test_arm_stall(_P(h)))


def muon_adamw_plan_work_order(k, units, nclusters: int) -> list:
    """Position -> unit table of one tensor-core launch (host only); -1 = no unit."""
    n = len(k)
    ka = (ctypes.c_int64 * n)(*k)
    ua = (ctypes.c_int64 * n)(*units)
    npos = ctypes.c_int64()
    lib = load_library()
    st = lib.muon_adamw_plan_work_order(n, ka, ua, nclusters, None, 0, ctypes.byref(npos))
    if st not in (0, MA_ERR_SHAPE):
        _check(st)
    buf = (ctypes.c_int32 * max(1, npos.value))()
    _check(lib.muon_adamw_plan_work_order(n, ka, ua, nclusters, buf, npos.value, ctypes.byref(npos)))
    return list(buf)[:npos.value]


def muon_adamw_get_state(h: int, index: int, which: int, dst_ptr: int) -> None:
    _check(load_library().muon_adamw_get_state(_P(h), int(index), int(which), _P(dst_ptr)))


def muon_adamw_set_state(h: int, index: int, which: int, src_ptr: int) -> None:
    _check(load_library().muon_adamw_set_state(_P(h), int(index), int(which), _P(src_ptr)))


def muon_adamw_get_step(h: int) -> int:
    t = ctypes.c_int64()
    _check(load_library().muon_adamw_get_step(_P(h), ctypes.byref(t)))
    return t.value


def muon_adamw_set_step(h: int, t: int) -> None:
    _check(load_library().muon_adamw_set_step(_P(h), int(t)))


def muon_adamw_last_norm(h: int):
    total = ctypes.c_float()
    coef = ctypes.c_float()
    _check(load_library().muon_adamw_last_norm(_P(h), ctypes.byref(total), ctypes.byref(coef)))
    return float(total.value), float(coef.value)


def muon_adamw_plan_info(h: int) -> PlanInfo:
    info = PlanInfo()
    _check(load_library().muon_adamw_plan_info(_P(h), ctypes.byref(info)))
    return info


def muon_adamw_set_profiling(h: int, enable: bool) -> None:
    _check(load_library().muon_adamw_set_profiling(_P(h), 1 if enable else 0))


def muon_adamw_get_profile(h: int) -> Profile:
    prof = Profile()
    _check(load_library().muon_adamw_get_profile(_P(h), ctypes.byref(prof)))
    return prof


def muon_adamw_reset_profile(h: int) -> None:
    _check(load_library().muon_adamw_reset_profile(_P(h)))


def muon_adamw_destroy(h: int) -> None:
    _check(load_library().muon_adamw_destroy(_P(h)))


MA_SHARD_MAX_WORLD = 4096


def muon_adamw_plan_shards(groups: Sequence[int], numels: Sequence[int], rows: Sequence[int],
                           cols: Sequence[int], world: int):
    """The sharded step's partition (host only). Returns (owner, ranges):
    owner[i] is the rank that updates Muon matrix i (-1 otherwise), ranges[i]
    a list of `world` (begin, end) element ranges of parameter i."""
    n = len(groups)
    g = (ctypes.c_int32 * max(1, n))(*[int(x) for x in groups])
    nu = (ctypes.c_int64 * max(1, n))(*[int(x) for x in numels])
    r = (ctypes.c_int64 * max(1, n))(*[int(x) for x in rows])
    c = (ctypes.c_int64 * max(1, n))(*[int(x) for x in cols])
    owner = (ctypes.c_int32 * max(1, n))()
    b = (ctypes.c_int64 * max(1, n * world))()
    e = (ctypes.c_int64 * max(1, n * world))()
    _check(load_library().muon_adamw_plan_shards(n, g, nu, r, c, int(world), owner, b, e))
    return ([int(owner[i]) for i in range(n)],
            [[(int(b[i * world + k]), int(e[i * world + k])) for k in range(world)] for i in range(n)])


def muon_adamw_set_shard(h: int, rank: int, world: int) -> None:
    _check(load_library().muon_adamw_set_shard(_P(h), int(rank), int(world)))


def muon_adamw_shard_range(h: int, index: int, rank: int):
    b, e = ctypes.c_int64(), ctypes.c_int64()
    _check(load_library().muon_adamw_shard_range(_P(h), int(index), int(rank), ctypes.byref(b), ctypes.byref(e)))
    return int(b.value), int(e.value)


def muon_adamw_step_begin(h: int, lr: float, local_sumsq_ptr: int) -> None:
    _check(load_library().muon_adamw_step_begin(_P(h), float(lr), _P(local_sumsq_ptr or None)))


def muon_adamw_step_end(h: int, global_sumsq_ptr: int, want_norm: bool = False) -> Optional[float]:
    if want_norm:
        out = ctypes.c_float()
        _check(load_library().muon_adamw_step_end(_P(h), _P(global_sumsq_ptr or None), ctypes.byref(out)))
        return float(out.value)
    _check(load_library().muon_adamw_step_end(_P(h), _P(global_sumsq_ptr or None), None))
    return None


def shard_exchange(tensors, ranges, rank: int, world: int, dist, group=None) -> None:
    """After a sharded step, give every rank the parts the others updated:
    for each tensor i (None is skipped) and each rank r, the elements
    ranges[i][r] = (begin, end) of its flattened view are broadcast from r.
    Collectives only (torch.distributed): gloo for CPU tensors, NCCL for CUDA
    ones."""
    for t, rr in zip(tensors, ranges):
        if t is None:
            continue
        flat = t.view(-1)
        for src in range(world):
            b, e = rr[src]
            if e > b:
                dist.broadcast(flat[b:e], src=src, group=group)


MA_NOALLOC_MAX_TENSORS = 64


def muon_adamw_grad_norm_noalloc(grad_ptrs: Sequence[int], numels: Sequence[int], dtypes: Sequence[int],
                                 max_norm: float, clip_eps: float, out_ptr: int, cuda_stream: int = 0) -> None:
    """Allocation-free global norm + clip factor into 2 device floats at out_ptr."""
    n = len(grad_ptrs)
    ptrs = (_P * max(1, n))(*[_P(p or None) for p in grad_ptrs])
    nums = (ctypes.c_int64 * max(1, n))(*[int(x) for x in numels])
    dts = (ctypes.c_int32 * max(1, n))(*[int(x) for x in dtypes])
    _check(load_library().muon_adamw_grad_norm_noalloc(ptrs, nums, dts, n, float(max_norm), float(clip_eps),
                                                       _P(out_ptr), _P(cuda_stream or None)))


def muon_adamw_last_error() -> str:
    return load_library().muon_adamw_last_error().decode("utf-8", "replace")


def muon_adamw_version() -> str:
    return load_library().muon_adamw_version().decode()


# ---- convenience wrapper over torch tensors ----

class MuonAdamW:
    """Owns one optimizer handle; parameters and gradients are torch tensors.

    ``params``: list of (name, fp32 CUDA parameter, CUDA gradient (bf16 or
    fp32), optional bf16 shadow or None, optional group override or None).
    Tensors must stay alive and keep their storage until ``close()``.
    """

    def __init__(self, params, *, stream=None, shard=None, **config):
        import torch

        cfg = muon_adamw_config_init()
        for k, v in config.items():
            if k == "reserved":
                for i, x in enumerate(v):
                    cfg.reserved[i] = int(x)
                continue
            if k == "ns_schedule":
                # a list of (a, b, c) per iteration, or None for the constant triple
                rows = [] if v is None else [tuple(float(x) for x in r) for r in v]
                if len(rows) > MA_NS_SCHEDULE_MAX or any(len(r) != 3 for r in rows):
                    raise ValueError(f"ns_schedule: at most {MA_NS_SCHEDULE_MAX} triples")
                cfg.ns_schedule_len = len(rows)
                for i, r in enumerate(rows):
                    for j in range(3):
                        cfg.ns_schedule[i][j] = r[j]
                continue
            if k == "muon_momentum_form" and isinstance(v, str):
                v = {"sgd": MA_MOMENTUM_SGD, "ema": MA_MOMENTUM_EMA}[v]
            if not hasattr(cfg, k):
                raise TypeError(f"unknown config field {k!r}")
            setattr(cfg, k, v)
        self.cfg = cfg
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.handle = muon_adamw_create(cfg, self.stream.cuda_stream)
        self.rank, self.world = (0, 1) if shard is None else (int(shard[0]), int(shard[1]))
        if self.world > 1:
            try:
                muon_adamw_set_shard(self.handle, self.rank, self.world)
            except Exception:
                self.close()
                raise
        self._keep = []
        self.indices = []
        self.groups = []
        try:
            for entry in params:
                name, p, g = entry[0], entry[1], entry[2]
                shadow = entry[3] if len(entry) > 3 else None
                group = entry[4] if len(entry) > 4 and entry[4] is not None else MA_GROUP_AUTO
                if p is not None and (p.dtype != torch.float32 or not p.is_contiguous()):
                    raise TypeError(f"{name}: parameter must be a contiguous fp32 tensor")
                if g is not None:
                    if g.dtype not in (torch.bfloat16, torch.float32) or not g.is_contiguous():
                        raise TypeError(f"{name}: gradient must be a contiguous bf16 or fp32 tensor")
                    if p is not None and g.shape != p.shape:
                        raise ValueError(f"{name}: gradient shape {tuple(g.shape)} != parameter {tuple(p.shape)}")
                if shadow is not None and (shadow.dtype != torch.bfloat16 or not shadow.is_contiguous()):
                    raise TypeError(f"{name}: shadow must be a contiguous bf16 tensor")
                shape = tuple(p.shape) if p is not None else tuple(g.shape) if g is not None else ()
                gdt = MA_DT_BF16 if (g is None or g.dtype == torch.bfloat16) else MA_DT_F32
                idx, grp = muon_adamw_register_param(
                    self.handle, name, shape, p.data_ptr() if p is not None else 0,
                    g.data_ptr() if g is not None else 0, gdt,
                    shadow.data_ptr() if shadow is not None else 0, group)
                self._keep.append((p, g, shadow))
                self.indices.append(idx)
                self.groups.append(GROUP_NAMES.get(grp, grp))
        except Exception:
            self.close()
            raise

    def record_grads_consumed(self, event=None):
        """A torch.cuda.Event that completes once the latest step has read
        every gradient (the gradient buffers may then be overwritten)."""
        import torch

        ev = event if event is not None else torch.cuda.Event()
        if not ev.cuda_event:
            ev.record()  # torch creates the underlying CUDA event on its first record
        muon_adamw_record_grads_consumed(self.handle, ev.cuda_event)
        return ev

    def set_param_options(self, index: int, lr_scale: float = 1.0, weight_decay_scale: float = 1.0) -> None:
        muon_adamw_set_param_options(self.handle, index, lr_scale, weight_decay_scale)

    def step(self, lr: float, want_norm: bool = False):
        return muon_adamw_step(self.handle, lr, want_norm)

    def shard_range(self, index: int, rank: Optional[int] = None):
        """(begin, end): the elements of parameter `index` that `rank` (this
        handle's rank by default) updates."""
        return muon_adamw_shard_range(self.handle, index, self.rank if rank is None else rank)

    def shard_ranges(self):
        """Per parameter, the (begin, end) range of every rank."""
        return [[self.shard_range(i, r) for r in range(self.world)] for i in range(len(self._keep))]

    def step_begin(self, lr: float, local_sumsq) -> None:
        """First half of a step: this rank's gradient sum of squares into the
        one-element fp64 CUDA tensor `local_sumsq`."""
        muon_adamw_step_begin(self.handle, lr, local_sumsq.data_ptr())

    def step_end(self, global_sumsq, want_norm: bool = False):
        """Second half: clip with the summed `global_sumsq` and update this
        rank's parameters."""
        return muon_adamw_step_end(self.handle, global_sumsq.data_ptr(), want_norm)

    def sharded_step(self, lr: float, dist, group=None, want_norm: bool = False):
        """One step of rank `self.rank` of `self.world`: step_begin, an
        all-reduce (sum) of the local sums of squares, step_end, then the
        exchange of every rank's updated parameters and shadows."""
        import torch

        if not hasattr(self, "_sumsq"):
            self._sumsq = torch.zeros(1, dtype=torch.float64, device=self._device())
        self.step_begin(lr, self._sumsq)
        dist.all_reduce(self._sumsq, group=group)
        norm = self.step_end(self._sumsq, want_norm)
        ranges = self.shard_ranges()
        shard_exchange([k[0] for k in self._keep], ranges, self.rank, self.world, dist, group)
        shard_exchange([k[2] for k in self._keep], ranges, self.rank, self.world, dist, group)
        return norm

    def _device(self):
        for p, g, _ in self._keep:
            if p is not None:
                return p.device
        import torch

        return torch.device("cuda")

    def state(self, index: int, which: int = 0):
        """The optimizer state of parameter `index` on the host (for a sharded
        handle: this rank's range of it, flattened, where that is not the
        whole parameter)."""
        import torch

        p = self._keep[index][0]
        b, e = self.shard_range(index) if self.world > 1 else (0, p.numel())
        shape = p.shape if e - b == p.numel() else (e - b,)
        out = torch.empty(shape, dtype=torch.float32)
        muon_adamw_get_state(self.handle, index, which, out.data_ptr())
        return out

    def set_state(self, index: int, which: int, value) -> None:
        import torch

        src = value.detach().to(device="cpu", dtype=torch.float32).contiguous()
        muon_adamw_set_state(self.handle, index, which, src.data_ptr())

    def profile(self) -> dict:
        prof = muon_adamw_get_profile(self.handle)
        return {k: {"launches": int(prof.launches[i]), "ms": float(prof.ms[i]), "units": float(prof.units[i])}
                for i, k in enumerate(KERNEL_KINDS)} | {"steps": int(prof.steps)}

    def plan_info(self) -> dict:
        info = muon_adamw_plan_info(self.handle)
        return {f: getattr(info, f) for f, _ in PlanInfo._fields_}

    def close(self) -> None:
        if getattr(self, "handle", None):
            muon_adamw_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
