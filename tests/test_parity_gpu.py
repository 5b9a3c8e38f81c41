"""GPU parity of the CUDA optimizer step against the fp64 oracle (via the C ABI).

Tolerances are those of ``tests/harness.py``: norm 1e-5 relative; AdamW
p/m/v and Muon momentum 1e-6 relative to the magnitude of their terms;
orthogonalised update 2e-2 relative Frobenius per matrix.
"""
import math

import numpy as np
import pytest

import workloads
from harness import O_TOL, GpuSide, relative_frobenius, run_parity, run_parity_sampled
from workloads import TensorSpec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    from muon_adamw_hybrid_grad_gb300 import build

    build.build()
    import muon_adamw_hybrid_grad_gb300 as m

    m.load_library()
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


KERNELS = [0, 1]  # MA_NS_TCGEN05, MA_NS_SIMT
KNAMES = {0: "tcgen05", 1: "simt"}


@pytest.mark.parametrize("ns_kernel", KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("policy", ["fp32_mixed", "bf16_mixed"])
def test_tiny_three_steps(mx, ns_kernel, policy):
    w = workloads.get_workload("tiny")
    w = workloads.custom_workload("tiny", w.tensors, policy=policy, steps=3)
    r = run_parity(w, config={"ns_kernel": ns_kernel})
    assert r["worst_o"] <= O_TOL


def test_twenty_steps_every_path(mx):
    """Twenty steps of the tiny workload plus a small and a narrow matrix (the
    tensor-core, small-matrix and narrow paths), against the oracle at every
    step: each step's rounding is carried into the next by the recurrences,
    and the state bounds carry it the same way, so a drift that a few steps
    would not show fails here."""
    tiny = workloads.get_workload("tiny")
    extra = [TensorSpec("model.action_expert.layers.2.mlp.w_small.weight", (128, 512), rank8=True),
             TensorSpec("model.action_expert.layers.2.mlp.w_narrow.weight", (1000, 40), rank8=True)]
    w = workloads.custom_workload("tiny20", list(tiny.tensors) + extra, policy="bf16_mixed", steps=20)
    r = run_parity(w)
    assert r["worst_o"] <= O_TOL


def _many_small_reduced():
    lens = workloads.many_small_lengths()[:256]
    t = [TensorSpec(f"model.action_expert.layers.{k}.w_a.weight", (128, 512)) for k in range(64)]
    t += [TensorSpec(f"model.action_expert.layers.{64 + k}.w_b.weight", (512, 128)) for k in range(32)]
    t += [TensorSpec(f"model.vlm.layers.{k}.ln.weight", (int(n),)) for k, n in enumerate(lens)]
    return workloads.custom_workload("many_small_reduced", t, policy="fp32_mixed", steps=2)


@pytest.mark.parametrize("ns_kernel", KERNELS, ids=lambda k: KNAMES[k])
def test_many_small_mixed_orientation(mx, ns_kernel):
    r = run_parity(_many_small_reduced(), config={"ns_kernel": ns_kernel})
    assert r["worst_o"] <= O_TOL


def _ragged():
    shapes = [(100, 300), (300, 100), (37, 53), (53, 37), (1, 129), (129, 1), (200, 200), (640, 384),
              (384, 640), (130, 258), (8, 8)]
    t = [TensorSpec(f"model.action_expert.layers.{k}.mlp.w{k}.weight", s) for k, s in enumerate(shapes)]
    t += [TensorSpec(f"model.vlm.v{k}.weight", (n,)) for k, n in enumerate((1, 7, 65535, 65537, 131073))]
    t += [TensorSpec("model.vlm.mat.weight", (33, 65))]
    return workloads.custom_workload("ragged", t, policy="bf16_mixed", steps=2)


@pytest.mark.parametrize("ns_kernel", KERNELS, ids=lambda k: KNAMES[k])
def test_ragged_shapes_and_chunk_tails(mx, ns_kernel):
    r = run_parity(_ragged(), config={"ns_kernel": ns_kernel})
    assert r["worst_o"] <= O_TOL


def _random_shapes_workload(policy):
    """Seeded random matrix shapes (1..699 per side) that reach every
    Newton-Schulz path: narrow fp32 (short side < 64), the fused small-matrix
    kernel, single-CTA and paired tensor-core launches; plus AdamW vectors of
    random lengths across chunk boundaries."""
    rng = np.random.default_rng(20261202)
    t = []
    for k in range(14):
        m, n = int(rng.integers(1, 700)), int(rng.integers(1, 700))
        t.append(TensorSpec(f"model.action_expert.layers.{k}.mlp.w{k}.weight", (m, n), rank8=True))
    for k in range(6):
        t.append(TensorSpec(f"model.vlm.layers.{k}.norm.weight", (int(rng.integers(1, 200000)),)))
    return workloads.custom_workload(f"random_{policy}", t, policy=policy, steps=2)


@pytest.mark.parametrize("policy", ["bf16_mixed", "fp32_mixed"])
def test_random_shapes_every_path(mx, policy):
    w = _random_shapes_workload(policy)
    r = run_parity(w)
    assert r["worst_o"] <= O_TOL
    gpu = GpuSide(w, workloads.master_weights(w))
    try:
        gpu.load_grads(workloads.gradients(w, 1))
        gpu.mx.muon_adamw_set_profiling(gpu.opt.handle, True)
        gpu.step(w.lr)
        prof = gpu.opt.profile()
        for k in ("ns_narrow", "ns_fused", "ns_gram", "ns_poly", "ns_update", "ns_apply"):
            assert prof[k]["launches"] > 0, k
    finally:
        gpu.close()


def test_without_cta_clusters(mx):
    """Cross-check switch: every Newton-Schulz product on single CTAs
    (cta_group::1) instead of CTA pairs, against the oracle."""
    w = workloads.get_workload("tiny")
    w = workloads.custom_workload("tiny", w.tensors, policy="bf16_mixed", steps=2)
    r = run_parity(w, config={"reserved": [2]})
    assert r["worst_o"] <= O_TOL


def test_small_matrices_through_per_product_launches(mx):
    """Cross-check switch: matrices of 128 canonical rows or fewer (here with
    padding, both orientations and several widths) through the per-product
    tensor-core launches instead of the fused small-matrix kernel, against
    the oracle."""
    r = run_parity(_ragged(), config={"reserved": [8]})
    assert r["worst_o"] <= O_TOL


def test_fused_small_matrix_kernel(mx):
    """Buckets of small matrices run their whole Newton-Schulz chain and the
    update in one launch each (two buckets here: 128 x 512 in both
    orientations, and 64 x 200), checked against the oracle; no per-product
    launch is made for them."""
    shapes = [(128, 512), (512, 128), (64, 200), (200, 64), (128, 512)]
    t = [TensorSpec(f"model.action_expert.layers.{k}.mlp.w.weight", sh) for k, sh in enumerate(shapes)]
    t.append(TensorSpec("model.vlm.norm.weight", (300,)))
    w = workloads.custom_workload("small_fused", t, policy="bf16_mixed", steps=3)
    r = run_parity(w)
    assert r["worst_o"] <= O_TOL
    gpu = GpuSide(w, workloads.master_weights(w))
    try:
        gpu.load_grads(workloads.gradients(w, 1))
        gpu.mx.muon_adamw_set_profiling(gpu.opt.handle, True)
        gpu.step(w.lr)
        prof = gpu.opt.profile()
        assert prof["ns_fused"]["launches"] == 2
        for k in ("ns_gram", "ns_poly", "ns_update", "ns_apply"):
            assert prof[k]["launches"] == 0
        assert prof["ns_fused"]["units"] > 0
    finally:
        gpu.close()


def _small_workload(steps=3):
    shapes = [(128, 512), (512, 128), (100, 384), (96, 96)]
    t = [TensorSpec(f"model.action_expert.layers.{k}.mlp.w.weight", sh) for k, sh in enumerate(shapes)]
    t.append(TensorSpec("model.action_expert.layers.0.mlp.w.bias", (96,)))
    return workloads.custom_workload("small", t, policy="bf16_mixed", steps=steps)


@pytest.mark.parametrize("steps_ns", [1, 3])
def test_fused_small_matrix_step_counts(mx, steps_ns):
    """The fused small-matrix kernel with one iteration (first and last at
    once: both Frobenius scales and the update in the same launch) and
    three, against the oracle."""
    r = run_parity(_small_workload(2), config={"ns_steps": steps_ns}, oracle_overrides={"muon_ns_steps": steps_ns})
    assert r["worst_o"] <= O_TOL


def test_fused_small_matrix_ema_and_schedule(mx):
    """Per-iteration coefficients and the exponential-average momentum through
    the fused small-matrix kernel, against the oracle."""
    r = run_parity(_small_workload(3), config={"muon_momentum_form": "ema", "ns_schedule": SCHEDULE},
                   oracle_overrides={"muon_momentum_form": "ema", "ns_schedule": SCHEDULE})
    assert r["worst_o"] <= O_TOL


NARROW_SHAPES = [(1000, 40), (520, 40), (2000, 40), (40, 1000), (8, 8), (1, 129), (129, 1), (37, 53), (63, 200),
                 (200, 63), (300, 24), (17, 400), (9000, 40), (60, 7000)]


@pytest.mark.parametrize("ns_kernel", KERNELS, ids=lambda k: KNAMES[k])
def test_narrow_matrices_fp32_newton_schulz(mx, ns_kernel):
    """Matrices whose short side is below 64 run Newton-Schulz in fp32 on the
    CUDA cores. With bf16 storage the 40-wide rank-8-plus-noise matrices
    (1000 x 40, 520 x 40, 2000 x 40) come out 2.2-2.3e-2 from the exact
    iteration; here every matrix meets the 2e-2 bound, and the narrow ones
    meet 1e-4, which only fp32 arithmetic does (a larger lr makes the
    recovery of O from the fp32 parameter update precise to ~1e-6). A 64-wide
    matrix stays on the bf16 tensor-core path. The narrow matrices go in one
    launch per cluster size of the resident kernel (8 CTAs for 2000 x 40, 4
    for the 520- to 1000-long ones, 2 for 300 x 24 and 17 x 400, 1 for the
    short ones) and one of the streaming kernel (9000 x 40 and 60 x 7000,
    whose slices would not fit in 8 CTAs' shared memory); none of the
    per-product launches takes them."""
    t = [TensorSpec(f"model.action_expert.layers.{k}.mlp.w{k}.weight", sh, rank8=True)
         for k, sh in enumerate(NARROW_SHAPES)]
    t.append(TensorSpec("model.action_expert.layers.99.mlp.w.weight", (64, 200), rank8=True))
    t.append(TensorSpec("model.action_expert.layers.0.input_layernorm.weight", (40,)))
    w = workloads.custom_workload("narrow", t, policy="bf16_mixed", steps=3)
    r = run_parity(w, config={"ns_kernel": ns_kernel}, lr=2e-3)
    assert r["worst_o"] <= O_TOL
    for i, sh in enumerate(NARROW_SHAPES):
        assert r["o_errors"][i] <= 1e-4, (sh, r["o_errors"][i])
    assert r["o_errors"][len(NARROW_SHAPES)] > 1e-4  # bf16 path: its error is the bf16 rounding
    gpu = GpuSide(w, workloads.master_weights(w), config={"ns_kernel": ns_kernel})
    try:
        gpu.load_grads(workloads.gradients(w, 1))
        gpu.mx.muon_adamw_set_profiling(gpu.opt.handle, True)
        gpu.step(w.lr)
        prof = gpu.opt.profile()
        assert prof["ns_narrow"]["launches"] == 5
    finally:
        gpu.close()


def test_narrow_plans_of_two_handles_share_the_device(mx):
    """The resident narrow kernel's shared-memory ceiling is a per-device
    attribute: a handle whose narrow matrices need less (1000 x 40, 85 KB per
    CTA) must not lower it under another's (40 x 8000 in clusters of 8 at
    227 KB per CTA). The big handle, stepped around the small one's plan and
    step, matches bit for bit the same steps on a handle of its own."""
    big = workloads.custom_workload(
        "narrow_big", [TensorSpec("model.action_expert.layers.0.mlp.w_big.weight", (40, 8000), rank8=True)],
        policy="bf16_mixed", steps=2)
    small = workloads.custom_workload(
        "narrow_small", [TensorSpec("model.action_expert.layers.0.mlp.w_small.weight", (1000, 40), rank8=True)],
        policy="bf16_mixed", steps=1)

    def run(interleave):
        g = GpuSide(big, workloads.master_weights(big))
        try:
            g.load_grads(workloads.gradients(big, 1))
            g.step(big.lr)
            if interleave:
                o = GpuSide(small, workloads.master_weights(small))
                try:
                    o.load_grads(workloads.gradients(small, 1))
                    o.step(small.lr)
                finally:
                    o.close()
            g.load_grads(workloads.gradients(big, 2))
            g.step(big.lr)
            return g.param(0)
        finally:
            g.close()

    alone, shared = run(False), run(True)
    assert not np.array_equal(alone, workloads.master_weights(big)[0])
    assert np.array_equal(alone, shared)


def test_gpu_orthogonalised_update_singular_values_in_band(mx):
    """OpenDM article, Muon 的工作原理: the quintic X <- a X + (b A + c A A) X
    maps each singular value x of the normalised update to phi(x) = a x +
    b x^3 + c x^5 and keeps the singular vectors, so five steps give
    phi^5(x). On x in [0.003, 1] phi^5 lies in a band near 1 (computed here
    on a fine grid); the GPU's O, recovered from the fp32 parameter update,
    keeps its singular values inside that band up to the 2e-2 that bf16
    storage allows, for inputs whose smallest normalised singular value is
    at least 0.003 (rectangular matrices, both orientations, on the
    tensor-core, small-matrix and narrow paths)."""
    import torch  # noqa: F401  (GpuSide holds torch tensors)

    a, b, c = 3.4445, -4.7750, 2.0315
    x = np.concatenate([np.linspace(0.003, 0.05, 20001), np.linspace(0.05, 1.0, 20001)])
    y = x.copy()
    for _ in range(5):
        y = a * y + b * y ** 3 + c * y ** 5
    lo, hi = float(y.min()), float(y.max())
    assert 0.6 < lo < 0.75 and 1.1 < hi < 1.3
    shapes = [(1024, 256), (256, 1024), (640, 384), (128, 512), (512, 128), (1000, 40)]
    t = [TensorSpec(f"model.action_expert.layers.{k}.mlp.w{k}.weight", sh) for k, sh in enumerate(shapes)]
    w = workloads.custom_workload("band", t, policy="fp32_mixed", steps=1)
    masters = workloads.master_weights(w)
    gpu = GpuSide(w, masters)
    try:
        grads = workloads.gradients(w, 1)
        gpu.load_grads(grads)
        gpu.step(w.lr)
        cfg = gpu.opt.cfg
        f32 = np.float32
        for i, (m_, n_) in enumerate(shapes):
            g = grads[i].astype(np.float64)
            sg = np.linalg.svd(g, compute_uv=False)
            assert sg.min() / np.linalg.norm(g) >= 0.003, shapes[i]  # the band's premise
            decay = float(f32(1.0 - w.lr * cfg.muon_weight_decay))
            lr_mult = float(f32(cfg.muon_lr_scale * cfg.moonlight_coef * math.sqrt(max(m_, n_))))
            O = (masters[i].astype(np.float64) * decay - gpu.param(i)) / (float(f32(w.lr)) * lr_mult)
            so = np.linalg.svd(O, compute_uv=False)
            assert lo - 2e-2 <= so.min() and so.max() <= hi + 2e-2, (shapes[i], so.min(), so.max(), lo, hi)
    finally:
        gpu.close()


def test_large_matrices_norm_and_band(mx):
    """Larger than any configuration: Muon matrices of 4096 x 16384 and
    16384 x 4096 (67 M elements each; 16 x 16 output units of the symmetric
    products, K up to 16384), where the fp64 oracle's Newton-Schulz would
    take minutes. Checked by what holds at any size: the step's norm against
    the fp64 sum over the gradients, and every singular value of the
    orthogonalised update (recovered from the fp32 parameter update; SVD on
    the GPU in fp32) inside phi^5([0.003, 1]) with the 2e-2 bf16 slack
    (OpenDM article, Muon 的工作原理; the inputs' smallest normalised singular
    value is about 0.008)."""
    import torch

    a, b, c = 3.4445, -4.7750, 2.0315
    x = np.concatenate([np.linspace(0.003, 0.05, 20001), np.linspace(0.05, 1.0, 20001)])
    y = x.copy()
    for _ in range(5):
        y = a * y + b * y ** 3 + c * y ** 5
    lo, hi = float(y.min()), float(y.max())
    shapes = [(4096, 16384), (16384, 4096)]
    t = [TensorSpec(f"model.action_expert.layers.{k}.mlp.w{k}.weight", sh) for k, sh in enumerate(shapes)]
    w = workloads.custom_workload("large", t, policy="fp32_mixed", steps=1)
    masters = workloads.master_weights(w)
    gpu = GpuSide(w, masters)
    try:
        grads = workloads.gradients(w, 1)
        gpu.load_grads(grads)
        norm = gpu.step(w.lr)
        want = math.sqrt(sum(float(np.sum(np.square(g.astype(np.float64)))) for g in grads))
        assert math.isclose(norm, want, rel_tol=1e-5)
        cfg = gpu.opt.cfg
        f32 = np.float32
        for i, (m_, n_) in enumerate(shapes):
            decay = float(f32(1.0 - w.lr * cfg.muon_weight_decay))
            lr_mult = float(f32(cfg.muon_lr_scale * cfg.moonlight_coef * math.sqrt(max(m_, n_))))
            p0 = torch.from_numpy(masters[i]).to("cuda", torch.float64)
            O = (p0 * decay - gpu.P[i].to(torch.float64)) / (float(f32(w.lr)) * lr_mult)
            so = torch.linalg.svdvals(O.to(torch.float32)).cpu().numpy()
            assert lo - 2e-2 <= so.min() and so.max() <= hi + 2e-2, (shapes[i], so.min(), so.max())
    finally:
        gpu.close()


def test_fp32_gradients(mx):
    w = workloads.get_workload("tiny")
    w = workloads.custom_workload("tiny_fp32g", w.tensors, grad_dtype="fp32", policy="fp32_mixed", steps=2)
    run_parity(w)


def test_fp32_gradients_small_and_narrow(mx):
    """fp32 gradients into the fused small-matrix kernel's momentum pass and
    into the narrow kernels, which read the gradient themselves: 16-byte
    words where the rows allow (1000 x 40, 37 x 300), single elements where
    they do not (300 x 37), and the streaming kernel (9000 x 40); the narrow
    ones within 1e-4."""
    t = [TensorSpec("model.action_expert.layers.0.mlp.w_s.weight", (128, 512), rank8=True),
         TensorSpec("model.action_expert.layers.0.mlp.w_a.weight", (1000, 40), rank8=True),
         TensorSpec("model.action_expert.layers.0.mlp.w_b.weight", (37, 300), rank8=True),
         TensorSpec("model.action_expert.layers.0.mlp.w_c.weight", (300, 37), rank8=True),
         TensorSpec("model.action_expert.layers.0.mlp.w_d.weight", (9000, 40), rank8=True),
         TensorSpec("model.action_expert.layers.0.input_layernorm.weight", (40,))]
    w = workloads.custom_workload("small_narrow_fp32g", t, grad_dtype="fp32", policy="bf16_mixed", steps=2)
    r = run_parity(w, lr=2e-3)
    assert r["worst_o"] <= O_TOL
    for i in range(1, 5):
        assert r["o_errors"][i] <= 1e-4, (t[i].shape, r["o_errors"][i])


def test_h1024_full_size_sampled(mx):
    """The benchmark workload at full size (16 layers, 268 M Muon elements):
    every momentum and AdamW element checked; O checked on layers 0, 8, 15
    for every shape (1024x1024, 4096x1024, 1024x4096)."""
    w = workloads.get_workload("h1024")
    per_layer = 7
    sample = [layer * per_layer + k for layer in (0, 8, 15) for k in (0, 4, 6)]
    r = run_parity(w, steps=2, muon_sample=sample)
    assert r["worst_o"] <= O_TOL


def _layer_sample(w, layers, per_layer=7, extra=()):
    """Indices of the matrices of the given expert layers plus ``extra``."""
    return [layer * per_layer + k for layer in layers for k in range(per_layer)] + list(extra)


def test_h2048_full_size_sampled(mx):
    """The 2048-hidden expert at full size (24 layers, 1.61 G Muon elements,
    fp32 masters): the norm over every gradient; momentum, parameters and O of
    every matrix of layers 0 and 23 (2048x2048, 8192x2048, 2048x8192); AdamW
    state of layer 0's norms and biases."""
    w = workloads.get_workload("h2048")
    vec0 = 24 * 7  # first vector tensor (layer 0's input_layernorm)
    sample = _layer_sample(w, (0, 23), extra=range(vec0, vec0 + 5))
    o_sample = [0, 4, 6, 23 * 7, 23 * 7 + 4, 23 * 7 + 6]
    r = run_parity_sampled(w, sample, steps=2, o_sample=o_sample)
    assert r["o_checked"] == 6 and r["worst_o"] <= O_TOL


def test_h2048_fp32_gradients_full_size_sampled(mx):
    """The 2048-hidden expert with fp32 gradients (fp32 weights give fp32
    gradients under the fp32_mixed policy) at full size: the norm over every
    gradient; momentum, parameters and O of layer 12's matrices (2048x2048,
    8192x2048, 2048x8192); AdamW state of layer 12's norms and biases."""
    w = workloads.get_workload("h2048_fp32grad")
    assert w.grad_dtype == "fp32"
    vec12 = 24 * 7 + 12 * 5
    sample = _layer_sample(w, (12,), extra=range(vec12, vec12 + 5))
    r = run_parity_sampled(w, sample, steps=1, o_sample=[12 * 7, 12 * 7 + 4, 12 * 7 + 6])
    assert r["o_checked"] == 3 and r["worst_o"] <= O_TOL


def test_full_vla_full_size_sampled(mx):
    """The full VLA workload at full size (1.61 G Muon + 1.69 G AdamW elements,
    a frozen 151936x2048 embedding), lr from the cosine schedule at step 1000:
    the norm over every gradient; one expert layer (O of its 2048x2048 and
    8192x2048 matrices), one language-model layer (AdamW, every shape) and one
    vision block sampled; the frozen embedding unwritten."""
    w = workloads.get_workload("full_vla")
    names = [t.name for t in w.tensors]
    emb = names.index("model.vlm.embed_tokens.weight")
    lm0 = names.index("model.vlm.language_model.layers.0.self_attn.q_proj.weight")
    vis = names.index("model.vlm.vision_tower.blocks.0.proj.weight")
    sample = _layer_sample(w, (11,)) + list(range(lm0, lm0 + 9)) + [vis]
    lr = w.lr * mx.muon_adamw_cosine_with_min_lr(1000, 2000, 0, 0.1)
    r = run_parity_sampled(w, sample, steps=1, o_sample=[11 * 7, 11 * 7 + 4], lr=lr)
    assert r["o_checked"] == 2 and r["worst_o"] <= O_TOL
    assert w.tensors[emb].frozen


def test_many_small_full_size(mx):
    """The many-small workload at full size (768 matrices of 128x512 and
    512x128, 4096 AdamW vectors): every state element and O of 64 matrices."""
    w = workloads.get_workload("many_small")
    sample = list(range(0, 512, 16)) + list(range(512, 768, 8))
    r = run_parity(w, steps=2, muon_sample=sample)
    assert r["worst_o"] <= O_TOL


def test_zero_gradients(mx):
    w = workloads.get_workload("tiny")
    run_parity(w, steps=2, grad_scale=0.0)


def test_large_gradients_clip(mx):
    # grads scaled by 1e3: the clip coefficient is far below 1
    w = workloads.get_workload("tiny")
    run_parity(w, steps=2, grad_scale=1e3)


def test_clipping_disabled(mx):
    w = workloads.get_workload("tiny")
    run_parity(w, steps=2, config={"max_grad_norm": 0.0}, oracle_overrides={"max_grad_norm": 0.0})


def test_adamw_only_mode(mx):
    w = workloads.get_workload("tiny")
    r = run_parity(w, steps=2, config={"mode": mx.MA_MODE_ADAMW_ONLY}, optim="adamw")
    assert set(r["groups"]) == {"adamw"}


@pytest.mark.parametrize("steps_ns", [1, 2, 3])
@pytest.mark.parametrize("ns_kernel", KERNELS, ids=lambda k: KNAMES[k])
def test_other_newton_schulz_step_counts(mx, steps_ns, ns_kernel):
    w = workloads.get_workload("tiny")
    run_parity(w, steps=2, config={"ns_steps": steps_ns, "ns_kernel": ns_kernel},
               oracle_overrides={"muon_ns_steps": steps_ns})


def test_frozen_and_empty_parameters(mx):
    t = [TensorSpec("model.action_expert.layers.0.q.weight", (256, 512)),
         TensorSpec("model.vlm.embed_tokens.weight", (500, 64), frozen=True),
         TensorSpec("model.action_expert.layers.0.k.weight", (0, 64)),
         TensorSpec("model.vlm.empty.bias", (0,)),
         TensorSpec("model.vlm.ln.weight", (64,))]
    w = workloads.custom_workload("frozen", t, policy="bf16_mixed", steps=2)
    r = run_parity(w)
    assert r["groups"] == ["muon", "frozen", "muon", "adamw", "adamw"]


def test_nan_gradient_propagates(mx):
    import torch

    w = workloads.get_workload("tiny")
    masters = workloads.master_weights(w)
    gpu = GpuSide(w, masters)
    try:
        grads = workloads.gradients(w, 1)
        grads[0] = grads[0].copy()
        grads[0][3, 5] = np.nan
        gpu.load_grads(grads)
        total = gpu.step(w.lr)
        assert math.isnan(total)
        for i in range(len(w.tensors)):
            assert torch.isnan(gpu.P[i]).all(), w.tensors[i].name
    finally:
        gpu.close()


def test_inf_gradient_zero_clip(mx):
    w = workloads.get_workload("tiny")
    masters = workloads.master_weights(w)
    gpu = GpuSide(w, masters)
    try:
        grads = workloads.gradients(w, 1)
        # an infinite entry in an AdamW tensor: norm inf, clip factor 0
        idx = len(w.tensors) - 1
        grads[idx] = grads[idx].copy()
        grads[idx][0, 0] = np.inf
        gpu.load_grads(grads)
        assert gpu.step(w.lr) == math.inf
        total, coef = gpu.mx.muon_adamw_last_norm(gpu.opt.handle)
        assert coef == 0.0
        # a finite Muon matrix gets a zero direction: O = 0, pure decay
        p0 = masters[0].astype(np.float64)
        decay = float(np.float32(1.0 - w.lr * 0.1))
        assert np.allclose(gpu.param(0), p0 * decay, rtol=1e-7, atol=0)
    finally:
        gpu.close()


def _all_paths_workload():
    """Small matrices of both orientations, tensor-core matrices (single CTAs
    and CTA pairs), narrow matrices in clusters of 4 and 8 and one for the
    streaming kernel, and AdamW vectors."""
    lens = workloads.many_small_lengths()[:64]
    t = [TensorSpec(f"model.action_expert.layers.{k}.w_a.weight", (128, 512)) for k in range(8)]
    t += [TensorSpec(f"model.action_expert.layers.{8 + k}.w_b.weight", (512, 128)) for k in range(4)]
    t += [TensorSpec("model.action_expert.layers.20.wq.weight", (384, 640), rank8=True),
          TensorSpec("model.action_expert.layers.20.wk.weight", (512, 1024), rank8=True),
          TensorSpec("model.action_expert.layers.20.w_n1.weight", (1000, 40), rank8=True),
          TensorSpec("model.action_expert.layers.20.w_n2.weight", (40, 2000), rank8=True),
          TensorSpec("model.action_expert.layers.20.w_n3.weight", (9000, 40), rank8=True)]
    t += [TensorSpec(f"model.vlm.layers.{k}.ln.weight", (int(n),)) for k, n in enumerate(lens)]
    return workloads.custom_workload("all_paths", t, policy="bf16_mixed", steps=2)


def test_deterministic(mx):
    """Two runs of the same steps give bitwise-identical parameters on every
    Newton-Schulz path (no atomics; the narrow clusters add their partial
    Gram tiles in rank order)."""
    w = _all_paths_workload()
    outs = []
    for _ in range(2):
        masters = workloads.master_weights(w)
        gpu = GpuSide(w, masters)
        try:
            for s in (1, 2):
                gpu.load_grads(workloads.gradients(w, s))
                gpu.step(w.lr)
            outs.append([gpu.param(i) for i in range(len(w.tensors))])
        finally:
            gpu.close()
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_tcgen05_matches_simt_kernel(mx):
    """Same inputs through the tensor-core and the CUDA-core GEMM: both are
    bf16-in/fp32-accumulate, so their O agree far more closely than either
    agrees with the fp64 oracle."""
    w = workloads.scaled_workload("mid", layers=2, hidden=512, mlp=1536)
    res = []
    for k in KERNELS:
        masters = workloads.master_weights(w)
        gpu = GpuSide(w, masters, config={"ns_kernel": k})
        try:
            gpu.load_grads(workloads.gradients(w, 1))
            gpu.step(w.lr)
            res.append([gpu.param(i).astype(np.float64) - masters[i] for i in range(len(w.tensors))])
        finally:
            gpu.close()
    for i, t in enumerate(w.tensors):
        if len(t.shape) == 2:
            assert relative_frobenius(res[0][i], res[1][i]) < 5e-3, t.name


@pytest.mark.parametrize("policy", ["bf16_mixed", "fp32_mixed"])
def test_tma_writeback_matches_register_writeback(mx, policy):
    """The last iteration's parameter update leaves through TMA for aligned
    parameters and from registers otherwise (cross-check switch bit 2 forces
    the latter). Both evaluate the same fp32 expression on the same
    accumulator, so parameters and shadows agree bit for bit, including
    blocks cut by the parameter's edges in both orientations."""
    shapes = [(200, 136), (136, 200), (256, 1024), (1024, 256), (96, 1000), (1000, 72), (33, 64), (640, 384)]
    t = [TensorSpec(f"model.action_expert.layers.{k}.mlp.w{k}.weight", sh) for k, sh in enumerate(shapes)]
    t.append(TensorSpec("model.vlm.ln.weight", (64,)))
    w = workloads.custom_workload("edges", t, policy=policy, steps=2)
    masters = workloads.master_weights(w)
    outs = []
    for reserved in ([0], [4]):
        gpu = GpuSide(w, masters, config={"reserved": reserved})
        try:
            for st in (1, 2):
                gpu.load_grads(workloads.gradients(w, st))
                gpu.step(w.lr)
            outs.append(([gpu.param(i) for i in range(len(t))],
                         [None if x is None else x.float().cpu().numpy() for x in gpu.S]))
        finally:
            gpu.close()
    (pa, sa), (pb, sb) = outs
    for i in range(len(t)):
        assert np.array_equal(pa[i], pb[i]), t[i].name
        if sa[i] is not None:
            assert np.array_equal(sa[i], sb[i]), t[i].name
    # and the TMA path itself is right against the oracle
    r = run_parity(w)
    assert r["worst_o"] <= O_TOL


def test_checkpoint_roundtrip_bitwise(mx):
    """get_state/set_state/set_step resume: a restored optimizer continues
    bit for bit like the original, on every Newton-Schulz path."""
    import torch

    w = _all_paths_workload()
    masters = workloads.master_weights(w)
    a = GpuSide(w, masters)
    try:
        for s in (1, 2):
            a.load_grads(workloads.gradients(w, s))
            a.step(w.lr)
        snap_p = [a.param(i) for i in range(len(w.tensors))]
        b = GpuSide(w, snap_p)
        try:
            for i, grp in enumerate(a.opt.groups):
                if grp == "muon":
                    b.opt.set_state(i, 0, a.opt.state(i, 0))
                elif grp == "adamw":
                    b.opt.set_state(i, 0, a.opt.state(i, 0))
                    b.opt.set_state(i, 1, a.opt.state(i, 1))
            mxm = a.mx
            mxm.muon_adamw_set_step(b.opt.handle, mxm.muon_adamw_get_step(a.opt.handle))
            g3 = workloads.gradients(w, 3)
            a.load_grads(g3)
            b.load_grads(g3)
            a.step(w.lr)
            b.step(w.lr)
            for i in range(len(w.tensors)):
                assert np.array_equal(a.param(i), b.param(i)), w.tensors[i].name
        finally:
            b.close()
    finally:
        a.close()


def test_error_paths(mx):
    import torch

    dev = torch.device("cuda")
    cfg = mx.muon_adamw_config_init()
    h = mx.muon_adamw_create(cfg, torch.cuda.current_stream().cuda_stream)
    try:
        p = torch.zeros(64, 64, device=dev)
        g = torch.zeros(64, 64, device=dev, dtype=torch.bfloat16)
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_register_param(h, "x.weight", (64, 64), p.data_ptr(), g.data_ptr(), 7)
        assert e.value.status == mx.MA_ERR_DTYPE
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_register_param(h, "x.weight", (64, 64), p.data_ptr(), g.data_ptr() + 1, mx.MA_DT_BF16)
        assert e.value.status == mx.MA_ERR_ALIGN
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_register_param(h, "v", (64,), p.data_ptr(), g.data_ptr(), mx.MA_DT_BF16, 0,
                                         mx.MA_GROUP_MUON)
        assert e.value.status == mx.MA_ERR_SHAPE
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_register_param(h, "x.weight", (64, 64), 0, g.data_ptr(), mx.MA_DT_BF16)
        assert e.value.status == mx.MA_ERR_ARG
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_plan_info(h)
        assert e.value.status == mx.MA_ERR_STATE
        idx, grp = mx.muon_adamw_register_param(h, "model.action_expert.layers.0.q.weight", (64, 64),
                                                p.data_ptr(), g.data_ptr(), mx.MA_DT_BF16)
        assert (idx, grp) == (0, mx.MA_GROUP_MUON)
        out = torch.empty(64, 64)
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_get_state(h, 0, 0, out.data_ptr())
        assert e.value.status == mx.MA_ERR_STATE
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_step(h, float("nan"))
        assert e.value.status == mx.MA_ERR_ARG
        assert mx.muon_adamw_step(h, 1e-3, want_norm=True) == 0.0
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_register_param(h, "late.weight", (64, 64), p.data_ptr(), g.data_ptr(), mx.MA_DT_BF16)
        assert e.value.status == mx.MA_ERR_STATE
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_get_state(h, 0, 1, out.data_ptr())  # Muon has no second moment
        assert e.value.status == mx.MA_ERR_ARG
        with pytest.raises(mx.MuonAdamWError) as e:
            mx.muon_adamw_get_state(h, 5, 0, out.data_ptr())
        assert e.value.status == mx.MA_ERR_ARG
        mx.muon_adamw_sync(h)
        info = mx.muon_adamw_plan_info(h)
        assert info.n_muon == 1 and info.n_buckets == 1
    finally:
        mx.muon_adamw_destroy(h)


def test_profiling_counts_launches(mx):
    w = workloads.get_workload("tiny")
    masters = workloads.master_weights(w)
    gpu = GpuSide(w, masters)
    try:
        gpu.load_grads(workloads.gradients(w, 1))
        gpu.mx.muon_adamw_set_profiling(gpu.opt.handle, True)
        gpu.step(w.lr)
        gpu.step(w.lr)
        prof = gpu.opt.profile()
        assert prof["steps"] == 2
        assert prof["ns_gram"]["launches"] == 2 * 5
        assert prof["adamw"]["launches"] == 2 and prof["momentum"]["launches"] == 2
        assert prof["ns_update"]["launches"] == 2 * 4 and prof["ns_apply"]["launches"] == 2
        for k in ("grad_norm", "momentum", "ns_gram", "ns_poly", "ns_update", "ns_apply", "adamw"):
            assert prof[k]["ms"] > 0 and prof[k]["units"] > 0
    finally:
        gpu.close()


# a schedule: the standard triple three times, then two polishing steps with
# phi(1) = 1 (the last one also has phi'(1) = 0)
SCHEDULE = [(3.4445, -4.7750, 2.0315)] * 3 + [(3.0, -3.2, 1.2), (1.875, -1.25, 0.375)]


@pytest.mark.parametrize("ns_kernel", KERNELS, ids=lambda k: KNAMES[k])
def test_every_hyperparameter_off_its_default(mx, ns_kernel):
    """Every numeric hyperparameter of the configuration away from its
    default at once (momentum, the 0.2 coefficient, muon_lr_scale, both
    weight decays, both betas, both epsilons, the clip threshold and the
    quintic's coefficients), on every Newton-Schulz path, against the oracle
    given the same values: no kernel holds a default of its own."""
    tiny = workloads.get_workload("tiny")
    extra = [TensorSpec("model.action_expert.layers.2.mlp.w_small.weight", (128, 512), rank8=True),
             TensorSpec("model.action_expert.layers.2.mlp.w_narrow.weight", (1000, 40), rank8=True)]
    w = workloads.custom_workload("tiny_hp", list(tiny.tensors) + extra, policy="bf16_mixed", steps=3)
    abc = (3.0, -3.2, 1.2)
    config = {"ns_kernel": ns_kernel, "muon_momentum": 0.9, "moonlight_coef": 0.3, "muon_lr_scale": 1.5,
              "muon_weight_decay": 0.05, "adam_beta1": 0.85, "adam_beta2": 0.99, "adam_eps": 1e-6,
              "adam_weight_decay": 0.02, "ns_eps": 1e-6, "max_grad_norm": 0.5,
              "ns_a": abc[0], "ns_b": abc[1], "ns_c": abc[2]}
    overrides = {"muon_momentum": 0.9, "muon_moonlight_coefficient": 0.3, "muon_lr_scale": 1.5,
                 "muon_weight_decay": 0.05, "adam_betas": (0.85, 0.99), "adam_eps": 1e-6, "weight_decay": 0.02,
                 "ns_eps": 1e-6, "max_grad_norm": 0.5, "ns_coefficients": abc}
    r = run_parity(w, config=config, oracle_overrides=overrides, grad_scale=50.0, lr=2e-3)
    assert r["worst_o"] <= O_TOL
    assert r["o_errors"][len(w.tensors) - 1] <= 1e-4  # the narrow matrix: fp32 throughout (either setting)


@pytest.mark.parametrize("ns_kernel", KERNELS, ids=lambda k: KNAMES[k])
def test_plain_momentum_without_nesterov(mx, ns_kernel):
    """muon_nesterov off (OpenDM article, 关键超参默认值 names the switch):
    the update is the momentum buffer itself, u = mu buf + g; through the
    momentum pass, the fused small-matrix kernel and the narrow kernel (which
    recompute u from buf), against the oracle over three steps."""
    tiny = workloads.get_workload("tiny")
    extra = [TensorSpec("model.action_expert.layers.2.mlp.w_small.weight", (128, 512), rank8=True),
             TensorSpec("model.action_expert.layers.2.mlp.w_narrow.weight", (1000, 40), rank8=True)]
    w = workloads.custom_workload("tiny_plain", list(tiny.tensors) + extra, policy="bf16_mixed", steps=3)
    r = run_parity(w, config={"ns_kernel": ns_kernel, "muon_nesterov": 0},
                   oracle_overrides={"muon_nesterov": False})
    assert r["worst_o"] <= O_TOL


@pytest.mark.parametrize("variant", ["ema_schedule", "one_step", "three_steps"])
def test_narrow_kernels_variants(mx, variant):
    """The narrow kernels (resident, in clusters of 4 and 2, and streaming)
    with the exponential-average momentum and a per-iteration coefficient
    schedule, and with one and three iterations (one: the first iteration's
    scale and the parameter update in the same pass), against the oracle
    within 1e-4."""
    t = [TensorSpec("model.action_expert.layers.0.mlp.w_a.weight", (1000, 40), rank8=True),
         TensorSpec("model.action_expert.layers.0.mlp.w_b.weight", (40, 300), rank8=True),
         TensorSpec("model.action_expert.layers.0.mlp.w_c.weight", (9000, 40), rank8=True),
         TensorSpec("model.action_expert.layers.0.input_layernorm.weight", (40,))]
    w = workloads.custom_workload("narrow_variants", t, policy="bf16_mixed", steps=3)
    if variant == "ema_schedule":
        config = {"muon_momentum_form": "ema", "ns_schedule": SCHEDULE}
        overrides = {"muon_momentum_form": "ema", "ns_schedule": SCHEDULE}
    else:
        k = 1 if variant == "one_step" else 3
        config, overrides = {"ns_steps": k}, {"muon_ns_steps": k}
    r = run_parity(w, config=config, oracle_overrides=overrides, lr=2e-3)
    for i in range(3):
        assert r["o_errors"][i] <= 1e-4, (variant, t[i].shape, r["o_errors"][i])


@pytest.mark.parametrize("ns_kernel", KERNELS, ids=lambda k: KNAMES[k])
def test_ema_momentum_and_coefficient_schedule(mx, ns_kernel):
    w = workloads.get_workload("tiny")
    w = workloads.custom_workload("tiny", w.tensors, policy="bf16_mixed", steps=3)
    r = run_parity(w, config={"ns_kernel": ns_kernel, "muon_momentum_form": "ema", "ns_schedule": SCHEDULE},
                   oracle_overrides={"muon_momentum_form": "ema", "ns_schedule": SCHEDULE})
    assert r["worst_o"] <= O_TOL


def _options_workload():
    t = [TensorSpec("model.action_expert.layers.0.mlp.up_proj.weight", (512, 256)),
         TensorSpec("model.action_expert.layers.0.mlp.down_proj.weight", (256, 512)),
         TensorSpec("model.action_expert.layers.0.self_attn.q_proj.weight", (256, 256)),
         TensorSpec("model.action_expert.layers.0.self_attn.q_proj.bias", (256,)),
         TensorSpec("model.action_expert.layers.0.input_layernorm.weight", (256,)),
         TensorSpec("model.vlm.proj.weight", (96, 200)),
         TensorSpec("model.vlm.proj.bias", (200,)),
         TensorSpec("model.vlm.final_norm.weight", (200,))]
    return workloads.custom_workload("options", t, policy="bf16_mixed", steps=3)


def test_param_options_on_small_and_narrow_matrices(mx):
    """Per-parameter (lr_scale, weight_decay_scale) on matrices of the fused
    small-matrix kernel and of the narrow kernel (clusters of 4 and of 2),
    which apply the update in their own epilogues, against the oracle given
    the same options; the narrow ones within 1e-4 (fp32 throughout)."""
    t = [TensorSpec("model.action_expert.layers.0.mlp.w_small.weight", (128, 512), rank8=True),
         TensorSpec("model.action_expert.layers.0.mlp.w_narrow.weight", (1000, 40), rank8=True),
         TensorSpec("model.action_expert.layers.0.mlp.w_narrow2.weight", (40, 300), rank8=True),
         TensorSpec("model.action_expert.layers.0.self_attn.q_proj.weight", (256, 256)),
         TensorSpec("model.action_expert.layers.0.input_layernorm.weight", (256,))]
    w = workloads.custom_workload("options_small", t, policy="bf16_mixed", steps=3)
    opts = {0: (2.0, 0.0), 1: (0.5, 3.0), 2: (1.5, 2.0), 3: (0.25, 1.0)}
    r = run_parity(w, param_options=opts, lr=2e-3)
    assert r["worst_o"] <= O_TOL
    assert r["o_errors"][1] <= 1e-4 and r["o_errors"][2] <= 1e-4, r["o_errors"]


def test_param_options_and_decay_exemption(mx):
    """Per-parameter (lr_scale, weight_decay_scale) on Muon and AdamW
    parameters, the bias/norm exemption rule, and an explicit option that
    overrides the rule (the q_proj bias)."""
    w = _options_workload()
    opts = {0: (2.0, 0.0), 2: (0.5, 3.0), 3: (1.0, 1.0), 5: (3.0, 0.5)}
    r = run_parity(w, config={"adam_decay_exempt_bias_norm": 1},
                   oracle_overrides={"adam_decay_exempt_bias_norm": True}, param_options=opts)
    assert r["worst_o"] <= O_TOL


def test_param_options_errors(mx):
    w = _options_workload()
    gpu = GpuSide(w, workloads.master_weights(w))
    try:
        opt = gpu.opt
        for bad in ((99, 1.0, 1.0), (0, -1.0, 1.0), (0, 1.0, float("inf")), (0, float("nan"), 1.0)):
            with pytest.raises(mx.MuonAdamWError) as ei:
                opt.set_param_options(*bad)
            assert ei.value.status == mx.MA_ERR_ARG
        # seven more distinct pairs fill the table of eight; the next one is refused
        for i in range(7):
            opt.set_param_options(i, 2.0 + i, 1.0)
        with pytest.raises(mx.MuonAdamWError) as ei:
            opt.set_param_options(7, 9.0, 1.0)
        assert ei.value.status == mx.MA_ERR_UNSUPPORTED
        opt.set_param_options(7, 1.0, 1.0)   # the default pair is always available
        gpu.load_grads(workloads.gradients(w, 1))
        gpu.step(w.lr)
        with pytest.raises(mx.MuonAdamWError) as ei:
            opt.set_param_options(0, 1.0, 1.0)
        assert ei.value.status == mx.MA_ERR_STATE
    finally:
        gpu.close()


def test_grads_consumed_event_allows_overwriting_gradients(mx):
    """Gradient buffers overwritten on another stream as soon as the event of
    muon_adamw_record_grads_consumed completes leave that step's result bit
    for bit unchanged; the event is refused before the first step."""
    import torch

    w = _options_workload()
    masters = workloads.master_weights(w)
    g1 = workloads.gradients(w, 1)
    ref = GpuSide(w, masters)
    try:
        ref.load_grads(g1)
        ref.step(w.lr)
        want = [ref.param(i) for i in range(len(w.tensors))]
    finally:
        ref.close()
    gpu = GpuSide(w, masters)
    try:
        with pytest.raises(mx.MuonAdamWError) as ei:
            gpu.opt.record_grads_consumed()
        assert ei.value.status == mx.MA_ERR_STATE
        gpu.load_grads(g1)
        side = torch.cuda.Stream()
        gpu.opt.step(w.lr)
        ev = gpu.opt.record_grads_consumed()
        side.wait_event(ev)
        with torch.cuda.stream(side):
            for g in gpu.G:
                if g is not None:
                    g.fill_(1e6)
        torch.cuda.synchronize()
        for i in range(len(w.tensors)):
            assert np.array_equal(gpu.param(i), want[i]), w.tensors[i].name
    finally:
        gpu.close()


@pytest.mark.parametrize("which", ["options", "small", "all_paths"])
def test_graph_mode_matches_direct_launches(mx, which):
    """Steps replayed from the captured CUDA graph (the default) and steps
    launched one kernel at a time give bitwise-identical parameters and
    shadows, with a different lr every step (the step's scalars are read from
    HBM) and with profiling (which forces direct launches) on for one step;
    for per-product launches, the fused small-matrix kernel and the narrow
    kernels' cluster launches."""
    w = {"options": _options_workload, "small": _small_workload, "all_paths": _all_paths_workload}[which]()
    masters = workloads.master_weights(w)
    lrs = (w.lr, 0.5 * w.lr, 2.0 * w.lr)
    outs = []
    for graph in (False, True):
        gpu = GpuSide(w, masters)
        try:
            mx.muon_adamw_set_graph_mode(gpu.opt.handle, graph)
            for st, lr in enumerate(lrs, start=1):
                gpu.load_grads(workloads.gradients(w, st))
                if graph and st == 2:
                    mx.muon_adamw_set_profiling(gpu.opt.handle, True)
                gpu.step(lr)
                if graph and st == 2:
                    mx.muon_adamw_set_profiling(gpu.opt.handle, False)
            outs.append(([gpu.param(i) for i in range(len(w.tensors))],
                         [None if x is None else x.float().cpu().numpy() for x in gpu.S]))
        finally:
            gpu.close()
    (pa, sa), (pb, sb) = outs
    for i, t in enumerate(w.tensors):
        assert np.array_equal(pa[i], pb[i]), t.name
        if sa[i] is not None:
            assert np.array_equal(sa[i], sb[i]), t.name


def test_bounded_wait_runs_out_and_reports(mx):
    """Failure path without a fault: the armed test hook starves one CTA of
    its operand loads, its bounded mbarrier wait runs out (2 s), and the step
    reports MA_ERR_DEVICE_CHECK; the handle then steps normally again."""
    import time

    t = [TensorSpec("model.action_expert.layers.0.w.weight", (128, 512)), TensorSpec("model.vlm.ln.weight", (64,))]
    w = workloads.custom_workload("stall", t, policy="fp32_mixed", steps=2)
    gpu = GpuSide(w, workloads.master_weights(w))
    try:
        gpu.load_grads(workloads.gradients(w, 1))
        gpu.mx.muon_adamw_test_arm_stall(gpu.opt.handle)
        t0 = time.time()
        with pytest.raises(gpu.mx.MuonAdamWError) as ei:
            gpu.step(w.lr)
        assert ei.value.status == gpu.mx.MA_ERR_DEVICE_CHECK
        assert time.time() - t0 < 60
        # the flag was consumed; the next steps run normally and stay finite
        assert math.isfinite(gpu.step(w.lr))
        gpu.mx.muon_adamw_sync(gpu.opt.handle)
        assert np.isfinite(gpu.param(1)).all()
    finally:
        gpu.close()
