"""Host-side checks of the C ABI library (no GPU needed, no compute calls).

The library is built from source here if needed; these tests load it, check
that every entry point ``include/muon_adamw.h`` declares is exported, and
exercise the pure host functions (routing predicate, schedule helper,
config defaults) and the argument checks that return before any CUDA call.
"""
import ctypes
import json
import math
import os
import re

import pytest

import oracle
from conftest import GOLDEN, ROOT

HEADER = os.path.join(ROOT, "include", "muon_adamw.h")


@pytest.fixture(scope="session")
def mx():
    from muon_adamw_hybrid_grad_gb300 import build

    build.build()
    import muon_adamw_hybrid_grad_gb300 as m

    m.load_library()
    return m


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MA_API\s+[\w\s\*]+?\b(muon_adamw_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_four_core_entry_points():
    names = declared_functions()
    for core in ("muon_adamw_create", "muon_adamw_register_param", "muon_adamw_step", "muon_adamw_destroy"):
        assert core in names
    assert len(names) >= 19


def test_every_declared_symbol_is_exported(mx):
    lib = ctypes.CDLL(mx.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding covers each of them with a signature
    from muon_adamw_hybrid_grad_gb300 import _SIGNATURES

    assert set(declared_functions()) == set(_SIGNATURES)


def test_library_links_no_cuda_shared_runtime(mx):
    # the static CUDA runtime is linked in and the driver is resolved lazily:
    # the dynamic section needs no CUDA shared library (read from readelf's
    # listing of the NEEDED entries)
    import shutil
    import subprocess

    readelf = shutil.which("readelf")
    if readelf is None:
        pytest.skip("readelf not available")
    listing = subprocess.run([readelf, "-d", mx.library_path()], capture_output=True, text=True, check=True).stdout
    needed = [ln.split("[", 1)[1].split("]", 1)[0] for ln in listing.splitlines() if "(NEEDED)" in ln]
    assert needed, listing
    assert not [n for n in needed if n.startswith(("libcudart", "libcuda.so", "libcublas"))], needed


def _routing_cases():
    rows = []
    for line in open(os.path.join(GOLDEN, "routing_cases.tsv")):
        if line.startswith("#") or not line.strip():
            continue
        name, ndim, expected, _ = line.rstrip("\n").split("\t")
        rows.append((name, int(ndim), expected))
    return rows


@pytest.mark.parametrize("name,ndim,expected", _routing_cases())
def test_routing_predicate_matches_page_table(mx, name, ndim, expected):
    assert mx.muon_adamw_is_muon_param(name, ndim) == (expected == "muon")


def test_routing_predicate_agrees_with_oracle_on_workload_names(mx):
    import workloads

    for wname in ("tiny", "h1024", "many_small", "full_vla"):
        w = workloads.get_workload(wname)
        for t in w.tensors:
            assert mx.muon_adamw_is_muon_param(t.name, len(t.shape)) == oracle.is_muon_parameter(t.name, len(t.shape))


def test_routing_null_name(mx):
    assert mx.load_library().muon_adamw_is_muon_param(None, 2) == 0


def test_cosine_schedule_helper(mx):
    f = mx.muon_adamw_cosine_with_min_lr
    assert f(0, 2000, 0, 0.1) == 1.0
    assert f(2000, 2000, 0, 0.1) == pytest.approx(0.1, abs=1e-15)
    assert f(1000, 2000, 0, 0.1) == pytest.approx(0.55, abs=1e-15)
    assert f(500, 2000, 0, 0.1) == pytest.approx(0.1 + 0.9 * (0.5 + math.sqrt(2) / 4), abs=1e-15)
    assert f(5, 2000, 10, 0.1) == 0.5
    for s in (0, 1, 17, 999, 1000, 1999, 2000, 2500):
        assert f(s, 2000, 0, 0.1) == pytest.approx(oracle.cosine_with_min_lr(s, 2000, 0, 0.1), abs=1e-15)


def test_config_defaults_match_page(mx):
    page = json.load(open(os.path.join(GOLDEN, "hparams_page.json")))
    spec = json.load(open(os.path.join(GOLDEN, "hparams_workload.json")))
    c = mx.muon_adamw_config_init()
    f32 = float
    assert c.muon_momentum == f32(page["muon_momentum"]["value"])
    assert bool(c.muon_nesterov) == page["muon_nesterov"]["value"]
    assert c.ns_steps == page["muon_ns_steps"]["value"]
    assert c.moonlight_coef == f32(page["muon_moonlight_coefficient"]["value"])
    assert c.max_grad_norm == f32(page["max_grad_norm"]["value"])
    assert c.precision == mx.MA_BF16_MIXED and page["precision_policy"]["value"] == "bf16_mixed"
    assert (c.ns_a, c.ns_b, c.ns_c) == tuple(f32(x) for x in spec["ns_coefficients"])
    assert (c.adam_beta1, c.adam_beta2) == tuple(f32(x) for x in spec["adam_betas"])
    assert c.adam_eps == f32(spec["adam_eps"]) and c.adam_weight_decay == f32(spec["weight_decay"])
    assert c.muon_lr_scale == 1.0 and c.ns_kernel == mx.MA_NS_TCGEN05


def test_null_handle_calls_return_errors(mx):
    lib = mx.load_library()
    assert lib.muon_adamw_destroy(None) == mx.MA_ERR_ARG
    assert "NULL" in mx.muon_adamw_last_error()
    assert lib.muon_adamw_step(None, 1e-3, None) == mx.MA_ERR_ARG
    assert lib.muon_adamw_sync(None) == mx.MA_ERR_ARG
    assert lib.muon_adamw_set_profiling(None, 1) == mx.MA_ERR_ARG
    assert lib.muon_adamw_register_param(None, b"x", 0, None, None, None, 0, None, 0, None, None) == mx.MA_ERR_ARG
    lib.muon_adamw_config_init(None)  # must not crash
    assert lib.muon_adamw_create(None, None, None) == mx.MA_ERR_ARG
    with pytest.raises(mx.MuonAdamWError) as ei:
        mx.muon_adamw_destroy(0)
    assert ei.value.status == mx.MA_ERR_ARG


def test_invalid_config_rejected_before_device_use(mx):
    lib = mx.load_library()
    h = ctypes.c_void_p()
    for field, value in (("ns_steps", 0), ("mode", 7), ("adam_beta1", 1.0), ("ns_kernel", 5), ("adam_eps", -1.0)):
        c = mx.muon_adamw_config_init()
        setattr(c, field, value)
        assert lib.muon_adamw_create(ctypes.byref(c), None, ctypes.byref(h)) == mx.MA_ERR_ARG, field


def test_create_without_gpu_fails_cleanly(mx):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    c = mx.muon_adamw_config_init()
    with pytest.raises(mx.MuonAdamWError) as ei:
        mx.muon_adamw_create(c, 0)
    assert ei.value.status in (mx.MA_ERR_CUDA, mx.MA_ERR_UNSUPPORTED)


def test_binding_fails_loudly_without_library(monkeypatch, mx):
    import muon_adamw_hybrid_grad_gb300 as m

    monkeypatch.setattr(m, "_LIB", None)
    monkeypatch.setattr(m, "library_path", lambda: "/nonexistent/libmuon_adamw_gb300.so")
    with pytest.raises(m.LibraryNotBuilt):
        m.muon_adamw_config_init()


def test_version(mx):
    assert "sm_103a" in mx.muon_adamw_version()


def test_config_struct_matches_c_layout(mx):
    """config_init zero-fills the C struct and then sets fields: with canary
    bytes around the Python mirror, every byte of the mirror is rewritten
    (the C struct is not shorter) and none beyond it (not longer)."""
    import ctypes

    n = ctypes.sizeof(mx.MuonAdamWConfig)
    buf = (ctypes.c_ubyte * (n + 64))(*([0xAB] * (n + 64)))
    mx.load_library().muon_adamw_config_init(ctypes.cast(buf, ctypes.POINTER(mx.MuonAdamWConfig)))
    assert all(b == 0xAB for b in bytes(buf)[n:]), "C config struct is larger than the Python mirror"
    cfg = mx.MuonAdamWConfig.from_buffer_copy(bytes(buf)[:n])
    assert bytes(cfg.ns_schedule[mx.MA_NS_SCHEDULE_MAX - 1]) == bytes(24), "C config struct is shorter"
    assert cfg.ns_steps == 5 and cfg.clip_eps == 1e-6
    assert cfg.muon_momentum_form == mx.MA_MOMENTUM_SGD
    assert cfg.adam_decay_exempt_bias_norm == 0 and cfg.ns_schedule_len == 0


@pytest.mark.parametrize("field,value", [
    ("muon_momentum_form", 2),
    ("adam_decay_exempt_bias_norm", 3),
    ("ns_schedule_len", 4),          # != ns_steps
    ("ns_schedule_len", 17),
    ("reserved1", 1),
    ("reserved0_bit0", 1),
    ("schedule_nan", 0),
])
def test_invalid_variant_config_is_rejected(mx, field, value):
    import ctypes

    c = mx.muon_adamw_config_init()
    if field == "reserved1":
        c.reserved[1] = value
    elif field == "reserved0_bit0":
        c.reserved[0] = value
    elif field == "schedule_nan":
        c.ns_schedule_len = 5
        c.ns_schedule[2][1] = float("nan")
    else:
        setattr(c, field, value)
    h = ctypes.c_void_p()
    st = mx.load_library().muon_adamw_create(ctypes.byref(c), None, ctypes.byref(h))
    assert st == mx.MA_ERR_ARG, mx.muon_adamw_last_error()
    assert not h.value


def test_set_param_options_null_handle(mx):
    assert mx.load_library().muon_adamw_set_param_options(None, 0, 1.0, 1.0) == mx.MA_ERR_ARG


def test_record_grads_consumed_argument_errors(mx):
    lib = mx.load_library()
    assert lib.muon_adamw_record_grads_consumed(None, None) == mx.MA_ERR_ARG


def test_set_graph_mode_null_handle(mx):
    assert mx.load_library().muon_adamw_set_graph_mode(None, 1) == mx.MA_ERR_ARG
