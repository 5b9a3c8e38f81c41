"""Pins of the fp64 oracle against closed forms, invariants and page values.

Nothing here re-types an oracle formula: each check compares the oracle with
a different route to the same number (an SVD closed form, an unrolled sum, a
trajectory solved by hand, a value printed on the page or worked by hand).
The last section plants mistakes in copies of the oracle functions and checks
that at least one pin catches each.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import hybrid as H

from conftest import GOLDEN

PAGE = json.load(open(os.path.join(GOLDEN, "hparams_page.json")))
SPEC = json.load(open(os.path.join(GOLDEN, "hparams_workload.json")))
COEF = tuple(SPEC["ns_coefficients"])


def phi(x):
    a, b, c = COEF
    return a * x + b * x ** 3 + c * x ** 5


def phi_n(x, n=5):
    for _ in range(n):
        x = phi(x)
    return x


def ns_closed_form(G, steps=5, eps=1e-7):
    """U diag(phi^steps(sigma / (||G||_F + eps))) V^T from an SVD."""
    U, S, Vt = np.linalg.svd(np.asarray(G, dtype=np.float64), full_matrices=False)
    x = S / (np.linalg.norm(S) + eps)
    return (U * phi_n(x, steps)) @ Vt


def random_orthogonal(rng, n):
    q, r = np.linalg.qr(rng.standard_normal((n, n)))
    return q * np.sign(np.diag(r))


def well_conditioned(rng, m, n, lo=1.0, hi=10.0):
    k = min(m, n)
    U = random_orthogonal(rng, m)[:, :k]
    V = random_orthogonal(rng, n)[:, :k]
    s = rng.uniform(lo, hi, k)
    return (U * s) @ V.T, U, V


# ---------------------------------------------------------------------------
# Page values
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("key", [k for k in PAGE if not k.startswith("_")])
def test_defaults_match_page(key):
    assert oracle.DEFAULTS[key] == PAGE[key]["value"], PAGE[key]["cite"]


def test_workload_constants():
    assert tuple(oracle.DEFAULTS["ns_coefficients"]) == COEF
    assert tuple(oracle.DEFAULTS["adam_betas"]) == tuple(SPEC["adam_betas"])
    assert oracle.DEFAULTS["adam_eps"] == SPEC["adam_eps"]
    assert oracle.DEFAULTS["weight_decay"] == SPEC["weight_decay"]


def _routing_cases():
    rows = []
    for line in open(os.path.join(GOLDEN, "routing_cases.tsv")):
        if line.startswith("#") or not line.strip():
            continue
        name, ndim, expected, why = line.rstrip("\n").split("\t")
        rows.append((name, int(ndim), expected, why))
    return rows


@pytest.mark.parametrize("name,ndim,expected,why", _routing_cases())
def test_routing_table(name, ndim, expected, why):
    assert oracle.route(name, ndim) == expected, why
    # optim='adamw' sends every trainable parameter to AdamW
    assert oracle.route(name, ndim, optim="adamw") == "adamw"
    assert oracle.route(name, ndim, frozen=True) == "frozen"


def test_lr_scaling_hand_values():
    data = json.load(open(os.path.join(GOLDEN, "lr_scaling.json")))
    for case in data["cases"]:
        m, n = case["shape"]
        got = oracle.muon_lr(data["lr"], m, n)
        assert got == pytest.approx(case["lr_eff"], rel=1e-8), case


# ---------------------------------------------------------------------------
# Newton-Schulz
# ---------------------------------------------------------------------------

SHAPES = [(8, 8), (16, 64), (64, 16), (64, 256), (256, 64), (33, 47), (47, 33), (1, 12), (12, 1)]


@pytest.mark.parametrize("shape", SHAPES)
def test_ns5_equals_svd_closed_form(shape):
    rng = np.random.default_rng(hash(shape) % 2**32)
    G = rng.standard_normal(shape)
    O = oracle.zeropower_newton_schulz5(G, 5, COEF, 1e-7)
    ref = ns_closed_form(G)
    assert np.linalg.norm(O - ref) <= 1e-10 * np.linalg.norm(ref)


@pytest.mark.parametrize("steps", [1, 2, 3, 7])
def test_ns_other_step_counts_closed_form(steps):
    rng = np.random.default_rng(steps)
    G = rng.standard_normal((24, 40))
    O = oracle.zeropower_newton_schulz5(G, steps, COEF, 1e-7)
    assert np.allclose(O, ns_closed_form(G, steps), rtol=0, atol=1e-11)


def test_ns5_rank_deficient_closed_form():
    rng = np.random.default_rng(7)
    G = rng.standard_normal((40, 3)) @ rng.standard_normal((3, 24))
    O = oracle.zeropower_newton_schulz5(G, 5, COEF, 1e-7)
    assert np.linalg.norm(O - ns_closed_form(G)) <= 1e-10 * np.linalg.norm(O)
    # rank is preserved: 3 non-zero singular values
    s = np.linalg.svd(O, compute_uv=False)
    assert np.sum(s > 1e-8) == 3


def _band(xmin):
    xs = np.linspace(xmin, 1.0, 200001)
    y = phi_n(xs)
    return float(y.min()), float(y.max())


def test_band_values():
    lo, hi = _band(0.003)
    assert 0.68 < lo < 0.69 and 1.19 < hi < 1.21
    assert phi_n(1e-9) / 1e-9 == pytest.approx(COEF[0] ** 5, rel=1e-6)


@pytest.mark.parametrize("shape", [(64, 64), (32, 128), (128, 32), (96, 160)])
def test_ns5_singular_values_in_band_and_near_polar(shape):
    rng = np.random.default_rng(shape[0] * 1000 + shape[1])
    G, U, V = well_conditioned(rng, *shape)
    s = np.linalg.svd(G, compute_uv=False)
    xmin = s.min() / np.linalg.norm(G)
    assert xmin >= 0.003
    lo, hi = _band(xmin)
    O = oracle.zeropower_newton_schulz5(G)
    so = np.linalg.svd(O, compute_uv=False)
    assert so.min() >= lo - 1e-9 and so.max() <= hi + 1e-9
    polar = U @ V.T
    dev = max(abs(lo - 1.0), abs(hi - 1.0))
    assert np.linalg.norm(O - polar) <= dev * np.linalg.norm(polar) + 1e-9


@pytest.mark.parametrize("shape", [(20, 50), (50, 20), (30, 30)])
def test_ns5_transpose_invariance(shape):
    G = np.random.default_rng(3).standard_normal(shape)
    a = oracle.zeropower_newton_schulz5(G)
    b = oracle.zeropower_newton_schulz5(G.T).T
    assert np.allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("k", [0.1, 3.0, 1e3])
def test_ns5_scale_invariance(k):
    G = np.random.default_rng(4).standard_normal((24, 36))
    G /= np.linalg.norm(G)
    a = oracle.zeropower_newton_schulz5(G)
    b = oracle.zeropower_newton_schulz5(k * G)
    # eps = 1e-7 enters as ||kG|| + eps; its effect is below 1e-5 here
    assert np.allclose(a, b, rtol=0, atol=1e-5)


def test_ns5_zero_matrix():
    O = oracle.zeropower_newton_schulz5(np.zeros((5, 7)))
    assert np.all(O == 0.0)


# ---------------------------------------------------------------------------
# Momentum
# ---------------------------------------------------------------------------

def test_momentum_unrolled_sum():
    rng = np.random.default_rng(11)
    mu = 0.95
    gs = [rng.standard_normal(6) for _ in range(7)]
    buf = np.zeros(6)
    for t, g in enumerate(gs, start=1):
        buf, d = oracle.nesterov_momentum(buf, g, mu)
        unrolled = sum(mu ** (t - k) * gs[k - 1] for k in range(1, t + 1))
        assert np.allclose(buf, unrolled, atol=1e-13)
        # Nesterov look-ahead: the direction is the next buffer if g repeated
        assert np.allclose(d, mu * unrolled + g, atol=1e-13)


def test_momentum_constant_gradient():
    g = np.array([0.5, -2.0])
    buf = np.zeros(2)
    mu = 0.95
    for t in range(1, 4):
        buf, d = oracle.nesterov_momentum(buf, g, mu)
    assert np.allclose(buf, g * (1 + mu + mu ** 2))
    assert np.allclose(d, g * (1 + mu + mu ** 2 + mu ** 3))


# ---------------------------------------------------------------------------
# AdamW
# ---------------------------------------------------------------------------

B1, B2 = SPEC["adam_betas"]
EPS = SPEC["adam_eps"]
WD = SPEC["weight_decay"]
LR = SPEC["lr"]


def test_adamw_first_step_is_sign_step():
    g = np.array([0.5, -0.25, 1.0, 3e-9, 0.0])
    p0 = np.array([1.0, 1.0, -2.0, 0.5, 0.25])
    p, m, v = oracle.adamw_update(p0, g, np.zeros(5), np.zeros(5), 1, LR, B1, B2, EPS, WD)
    expect = p0 * (1 - LR * WD) - LR * g / (np.abs(g) + EPS)
    assert np.allclose(p, expect, rtol=0, atol=1e-18)
    assert np.allclose(m, (1 - B1) * g) and np.allclose(v, (1 - B2) * g * g)


def test_adamw_constant_gradient_trajectory():
    # With a constant gradient, bias-corrected moments equal g and g^2 at
    # every t, so each Adam step is lr*g/(|g|+eps): p_t has a closed form.
    g = np.array([0.5, -0.25, 1.0])
    p0 = np.array([1.0, -1.0, 0.3])
    p, m, v = p0.copy(), np.zeros(3), np.zeros(3)
    T = 12
    for t in range(1, T + 1):
        p, m, v = oracle.adamw_update(p, g, m, v, t, LR, B1, B2, EPS, WD)
        assert np.allclose(m, (1 - B1 ** t) * g, rtol=1e-13)
        assert np.allclose(v, (1 - B2 ** t) * g * g, rtol=1e-13)
    d = 1 - LR * WD
    s = g / (np.abs(g) + EPS)
    closed = p0 * d ** T - LR * s * sum(d ** k for k in range(T))
    assert np.allclose(p, closed, rtol=1e-12, atol=1e-15)


def test_adamw_zero_gradient_pure_decay():
    p0 = np.array([0.7, -0.1])
    p, m, v = p0.copy(), np.zeros(2), np.zeros(2)
    for t in range(1, 6):
        p, m, v = oracle.adamw_update(p, np.zeros(2), m, v, t, LR, B1, B2, EPS, WD)
    assert np.all(m == 0) and np.all(v == 0)
    assert np.allclose(p, p0 * (1 - LR * WD) ** 5, rtol=1e-14)


def test_adamw_unrolled_moments_and_scale_invariance():
    rng = np.random.default_rng(5)
    gs = [rng.standard_normal(4) for _ in range(6)]
    p = np.ones(4)
    m = np.zeros(4)
    v = np.zeros(4)
    q = np.ones(4)
    mq = np.zeros(4)
    vq = np.zeros(4)
    for t, g in enumerate(gs, start=1):
        p, m, v = oracle.adamw_update(p, g, m, v, t, LR, B1, B2, 0.0, WD)
        q, mq, vq = oracle.adamw_update(q, 1000.0 * g, mq, vq, t, LR, B1, B2, 0.0, WD)
        mu_ = sum((1 - B1) * B1 ** (t - k) * gs[k - 1] for k in range(1, t + 1))
        nu_ = sum((1 - B2) * B2 ** (t - k) * gs[k - 1] ** 2 for k in range(1, t + 1))
        assert np.allclose(m, mu_, rtol=1e-12) and np.allclose(v, nu_, rtol=1e-12)
    # with eps = 0 Adam's step does not depend on the gradient's scale
    assert np.allclose(p, q, rtol=1e-12)


# ---------------------------------------------------------------------------
# Clip
# ---------------------------------------------------------------------------

def test_clip_hand_values():
    ones = [np.ones(1024)]
    assert oracle.global_grad_norm(ones) == 32.0
    assert oracle.clip_coefficient(32.0, 1.0) == 1.0 / (32.0 + 1e-6)
    assert oracle.clip_coefficient(0.5, 1.0) == 1.0
    assert oracle.global_grad_norm([np.zeros(7), np.zeros((3, 3))]) == 0.0
    assert oracle.clip_coefficient(0.0, 1.0) == 1.0
    # a 3-4-5 triangle split across two tensors
    assert oracle.global_grad_norm([np.array([3.0]), np.array([[4.0]])]) == 5.0
    assert oracle.clip_coefficient(5.0, 1.0) == 1.0 / (5.0 + 1e-6)
    assert oracle.clip_coefficient(5.0, 0.0) == 1.0  # max_norm <= 0 disables


def test_clip_non_finite():
    assert math.isnan(oracle.clip_coefficient(float("nan"), 1.0))
    assert oracle.clip_coefficient(float("inf"), 1.0) == 0.0
    assert math.isnan(oracle.global_grad_norm([np.array([1.0, np.nan])]))
    assert oracle.global_grad_norm([np.array([np.inf, 1.0])]) == float("inf")


# ---------------------------------------------------------------------------
# Schedule
# ---------------------------------------------------------------------------

def test_cosine_with_min_lr_points():
    f = oracle.cosine_with_min_lr
    assert f(0, 2000, 0, 0.1) == 1.0
    assert f(2000, 2000, 0, 0.1) == pytest.approx(0.1, abs=1e-15)
    assert f(1000, 2000, 0, 0.1) == pytest.approx(0.55, abs=1e-15)
    assert f(500, 2000, 0, 0.1) == pytest.approx(0.1 + 0.9 * (0.5 + math.sqrt(2) / 4), abs=1e-15)
    assert f(5, 2000, 10, 0.1) == 0.5
    assert 2.5e-5 * f(1000, 2000, 0, 0.1) == pytest.approx(1.375e-5, rel=1e-14)


# ---------------------------------------------------------------------------
# The whole step against closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(6, 10), (10, 6), (8, 8)])
def test_full_step_rank1_muon_and_constant_adamw(shape):
    m_, n_ = shape
    rng = np.random.default_rng(m_ * n_)
    u = rng.standard_normal(m_)
    u /= np.linalg.norm(u)
    v = rng.standard_normal(n_)
    v /= np.linalg.norm(v)
    sigma = 4.0
    names = ["model.action_expert.layers.0.mlp.w.weight", "model.action_expert.layers.0.ln.weight",
             "model.vlm.embed_tokens.weight"]
    shapes = [shape, (3,), (2, 2)]
    orc = oracle.HybridOracle(names, shapes, frozen=[False, False, True])
    assert orc.groups == ["muon", "adamw", "frozen"]
    p0 = [rng.standard_normal(shape) * 0.02, np.array([1.0, -1.0, 0.5]), np.ones((2, 2))]
    params = [x.copy() for x in p0]
    gm = sigma * np.outer(u, v)
    ga = np.array([3.0, 0.0, 0.0])     # with gm: total^2 = 16 + 9 -> total 5
    gf = np.full((2, 2), 100.0)        # frozen: ignored by the norm
    res = orc.step(params, [gm, ga, gf], LR)
    assert res["total"] == pytest.approx(5.0, rel=1e-14)
    coef = 1.0 / (5.0 + 1e-6)
    assert res["coef"] == pytest.approx(coef, rel=1e-14)
    # Muon: direction (1 + mu) * coef * gm is rank one, so NS5 maps it to
    # phi^5(||d|| / (||d|| + 1e-7)) * u v^T
    d = (1 + 0.95) * coef * sigma
    O = phi_n(d / (d + 1e-7)) * np.outer(u, v)
    assert np.allclose(res["O"][0], O, rtol=0, atol=1e-12)
    lr_eff = LR * 0.2 * math.sqrt(max(shape))
    assert np.allclose(params[0], p0[0] * (1 - LR * 0.1) - lr_eff * O, rtol=0, atol=1e-15)
    # AdamW at t = 1: a sign step on non-zero coordinates, decay only on zeros
    ghat = coef * ga
    expect = p0[1] * (1 - LR * WD) - LR * ghat / (np.abs(ghat) + EPS)
    assert np.allclose(params[1], expect, rtol=0, atol=1e-17)
    assert np.array_equal(params[2], p0[2])


def test_full_step_three_steps_constant_grads():
    # constant grads over 3 steps: Muon buffer is a geometric sum, AdamW follows
    # the closed-form trajectory, and NS5 of a rank-1 direction stays rank-1.
    names = ["model.action_expert.layers.1.w_up.weight", "model.action_expert.layers.1.post_norm.weight"]
    shapes = [(4, 6), (5,)]
    orc = oracle.HybridOracle(names, shapes)
    u = np.array([1.0, 0, 0, 0])
    v = np.array([0, 1.0, 0, 0, 0, 0])
    gm = 0.1 * np.outer(u, v)
    ga = np.full(5, 0.02)
    params = [np.zeros((4, 6)), np.ones(5)]
    for _ in range(3):
        res = orc.step(params, [gm, ga], LR)
    total = math.sqrt(0.1 ** 2 + 5 * 0.02 ** 2)
    assert res["total"] == pytest.approx(total, rel=1e-14)
    assert res["coef"] == 1.0
    assert np.allclose(orc.buf[0], gm * (1 + 0.95 + 0.95 ** 2), rtol=1e-14)
    d = 1 - LR * WD
    s = 0.02 / (0.02 + EPS)
    assert np.allclose(params[1], d ** 3 - LR * s * (1 + d + d * d), rtol=1e-13)


def test_adamw_only_mode_routes_everything_to_adamw():
    names = ["model.action_expert.layers.0.q.weight", "model.action_expert.layers.0.ln.weight"]
    orc = oracle.HybridOracle(names, [(3, 3), (3,)], optim="adamw")
    assert orc.groups == ["adamw", "adamw"]
    g = [np.full((3, 3), 0.5), np.full(3, -0.5)]
    params = [np.ones((3, 3)), np.ones(3)]
    res = orc.step(params, g, LR)
    assert res["coef"] == pytest.approx(1.0 / (math.sqrt(12 * 0.25) + 1e-6))
    ghat = res["coef"] * 0.5
    assert np.allclose(params[0], (1 - LR * WD) - LR * ghat / (ghat + EPS), rtol=1e-14)


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by the closed forms above
# ---------------------------------------------------------------------------

def _ns_wrong_sign(G, steps=5, coefficients=COEF, eps=1e-7):
    a, b, c = coefficients
    return H.zeropower_newton_schulz5(G, steps, (a, -b, c), eps)


def _ns_dropped_quintic(G, steps=5, coefficients=COEF, eps=1e-7):
    X = np.array(G, dtype=np.float64)
    X = X / (np.linalg.norm(X) + eps)
    a, b, c = coefficients
    for _ in range(steps):
        A = X @ X.T
        X = a * X + b * A @ X          # c A^2 X term dropped
    return X


def _ns_transposed_operand(G, steps=5, coefficients=COEF, eps=1e-7):
    X = np.array(G, dtype=np.float64)
    X = X / (np.linalg.norm(X) + eps)
    a, b, c = coefficients
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * A @ A
        X = a * X + (B @ X.T.T if X.shape[0] == X.shape[1] else B @ X)
        X = X.T if X.shape[0] == X.shape[1] else X   # transposes square iterates
    return X


@pytest.mark.parametrize("bad", [_ns_wrong_sign, _ns_dropped_quintic, _ns_transposed_operand])
def test_planted_ns_mistakes_are_caught(bad):
    G = np.random.default_rng(9).standard_normal((16, 16))
    ref = ns_closed_form(G)
    with np.errstate(all="ignore"):
        diff = np.linalg.norm(bad(G) - ref)
    assert not diff <= 1e-3 * np.linalg.norm(ref)   # also true when diff is inf/nan


def test_planted_momentum_and_adam_mistakes_are_caught():
    g = np.array([0.5, -0.25])
    # heavy-ball direction instead of Nesterov: direction would equal buf
    buf = np.zeros(2)
    for _ in range(3):
        buf = 0.95 * buf + g
    assert not np.allclose(buf, g * (1 + 0.95 + 0.95 ** 2 + 0.95 ** 3))
    # Adam without bias correction breaks the t = 1 sign step
    m = (1 - B1) * g
    v = (1 - B2) * g * g
    p_no_bc = 1.0 - LR * m / (np.sqrt(v) + EPS)
    assert not np.allclose(p_no_bc, 1.0 - LR * g / (np.abs(g) + EPS), rtol=1e-6)
    # clip without eps: 1/32 differs from the hand value 1/(32 + 1e-6)
    assert 1.0 / 32.0 != oracle.clip_coefficient(32.0, 1.0)
