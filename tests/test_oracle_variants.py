"""Pins of the oracle's configuration variants: the exponential-average form of
the momentum, per-iteration Newton-Schulz coefficient schedules, per-parameter
lr / weight-decay multipliers and the bias/norm decay exemption.

As in the main pin file, each check reaches the same number by another route
(an unrolled sum, an SVD closed form with the composed scalar polynomials, a
hand-solved AdamW step, a rank-one Muon update) and planted mistakes in copies
of the oracle are caught.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import hybrid as H

MU = 0.95
LR = 2.5e-5
B1, B2, EPS, WD = 0.9, 0.999, 1e-8, 0.1

# Five distinct triples: the closed form below composes them in order, so the
# order of application matters (the odd polynomials do not commute).
SCHEDULE = [(3.0, -3.2, 1.2), (3.4445, -4.7750, 2.0315), (2.2, -1.1, 0.1),
            (1.875, -1.25, 0.375), (1.5, -0.5, 0.0)]


def composed_closed_form(G, schedule, eps=1e-7):
    """U diag(phi_T(...phi_1(sigma / (||G||_F + eps)))) V^T from an SVD."""
    U, S, Vt = np.linalg.svd(np.asarray(G, dtype=np.float64), full_matrices=False)
    x = S / (np.linalg.norm(S) + eps)
    for a, b, c in schedule:
        x = a * x + b * x ** 3 + c * x ** 5
    return (U * x) @ Vt


# ---------------------------------------------------------------------------
# Exponential-average momentum
# ---------------------------------------------------------------------------

def test_ema_momentum_unrolled_sum():
    rng = np.random.default_rng(21)
    gs = [rng.standard_normal(5) for _ in range(8)]
    buf = np.zeros(5)
    for t, g in enumerate(gs, start=1):
        buf, d = oracle.nesterov_momentum(buf, g, MU, True, "ema")
        unrolled = (1 - MU) * sum(MU ** (t - k) * gs[k - 1] for k in range(1, t + 1))
        assert np.allclose(buf, unrolled, atol=1e-14)
        # look-ahead: the average the buffer would reach if g came once more
        assert np.allclose(d, MU * unrolled + (1 - MU) * g, atol=1e-14)


def test_ema_momentum_constant_gradient_and_plain():
    g = np.array([2.0, -0.5, 1e-3])
    buf = np.zeros(3)
    for t in range(1, 6):
        buf, d = oracle.nesterov_momentum(buf, g, MU, True, "ema")
        assert np.allclose(buf, (1 - MU ** t) * g, rtol=1e-14)
        assert np.allclose(d, (1 - MU ** (t + 1)) * g, rtol=1e-14)
    b2, d2 = oracle.nesterov_momentum(np.zeros(3), g, MU, False, "ema")
    assert np.array_equal(d2, b2)
    with pytest.raises(ValueError):
        oracle.nesterov_momentum(np.zeros(3), g, MU, True, "lerp2")


def test_ema_and_sgd_forms_differ_in_direction_not_only_scale():
    # SGD form: (1+mu) g + mu^2 b; EMA form: (1-mu)(1+mu) g + mu^2 b. With a
    # non-zero history the two directions are not parallel.
    b0 = np.array([1.0, 0.0])
    g = np.array([0.0, 1.0])
    _, ds = oracle.nesterov_momentum(b0, g, MU, True, "sgd")
    _, de = oracle.nesterov_momentum(b0, g, MU, True, "ema")
    cos = ds @ de / (np.linalg.norm(ds) * np.linalg.norm(de))
    assert cos < 0.9
    assert np.allclose(ds, (1 + MU) * g + MU * MU * b0)
    assert np.allclose(de, (1 - MU) * (1 + MU) * g + MU * MU * b0)


# ---------------------------------------------------------------------------
# Coefficient schedules
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(12, 20), (20, 12), (9, 9)])
def test_schedule_equals_composed_closed_form(shape):
    G = np.random.default_rng(sum(shape)).standard_normal(shape)
    O = oracle.zeropower_newton_schulz5(G, 5, SCHEDULE, 1e-7)
    ref = composed_closed_form(G, SCHEDULE)
    assert np.linalg.norm(O - ref) <= 1e-11 * np.linalg.norm(ref)


def test_constant_schedule_is_the_default():
    G = np.random.default_rng(4).standard_normal((10, 16))
    coef = (3.4445, -4.7750, 2.0315)
    a = oracle.zeropower_newton_schulz5(G, 5, [coef] * 5, 1e-7)
    b = oracle.zeropower_newton_schulz5(G, 5, coef, 1e-7)
    assert np.array_equal(a, b)


def test_schedule_length_must_match_steps():
    with pytest.raises(ValueError):
        oracle.zeropower_newton_schulz5(np.eye(3), 5, SCHEDULE[:4])


def test_planted_reversed_schedule_is_caught():
    G = np.random.default_rng(8).standard_normal((14, 14))
    ref = composed_closed_form(G, SCHEDULE)
    bad = oracle.zeropower_newton_schulz5(G, 5, SCHEDULE[::-1], 1e-7)
    assert not np.linalg.norm(bad - ref) <= 1e-6 * np.linalg.norm(ref)


# ---------------------------------------------------------------------------
# Per-parameter multipliers and the decay exemption
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,exempt", [
    ("model.vlm.layers.0.self_attn.q_proj.bias", True),
    ("model.action_expert.layers.0.input_layernorm.weight", True),
    ("model.action_expert.norm.weight", True),
    ("model.vlm.RMSNorm.scale", True),
    ("model.vlm.layers.0.mlp.up_proj.weight", False),
    ("model.vlm.biased_gate.weight", False),
    ("model.vlm.embed_tokens.weight", False),
])
def test_decay_exempt_rule(name, exempt):
    assert oracle.decay_exempt(name) is exempt


def _adamw_two_params(**kw):
    names = ["model.vlm.proj.weight", "model.vlm.proj.bias"]
    return oracle.HybridOracle(names, [(2, 2), (3,)], **kw)


def test_adamw_options_first_step_closed_form():
    # t = 1 with a tiny gradient (no clipping): p * (1 - lr*ls*wd*ws) - lr*ls*g/(|g|+eps)
    orc = _adamw_two_params(param_options={0: (3.0, 0.0), 1: (0.5, 2.0)})
    p0 = [np.full((2, 2), 0.7), np.array([1.0, -2.0, 0.3])]
    g = [np.full((2, 2), 1e-3), np.array([-1e-3, 2e-3, 0.0])]
    params = [x.copy() for x in p0]
    res = orc.step(params, g, LR)
    assert res["coef"] == 1.0
    assert np.allclose(params[0], 0.7 - 3 * LR * 1e-3 / (1e-3 + EPS), rtol=0, atol=1e-16)
    expect = p0[1] * (1 - 0.5 * LR * WD * 2.0) - 0.5 * LR * g[1] / (np.abs(g[1]) + EPS)
    assert np.allclose(params[1], expect, rtol=0, atol=1e-16)


def test_exemption_flag_and_explicit_override():
    p0 = [np.full((2, 2), 0.7), np.array([1.0, -2.0, 0.3])]
    zero = [np.zeros((2, 2)), np.zeros(3)]
    # with the flag, the bias keeps its value under a zero gradient; the weight decays
    orc = _adamw_two_params(adam_decay_exempt_bias_norm=True)
    params = [x.copy() for x in p0]
    orc.step(params, zero, LR)
    assert np.array_equal(params[1], p0[1])
    assert np.allclose(params[0], 0.7 * (1 - LR * WD), rtol=1e-15)
    # an explicit option wins over the rule
    orc = _adamw_two_params(adam_decay_exempt_bias_norm=True, param_options={1: (1.0, 1.0)})
    params = [x.copy() for x in p0]
    orc.step(params, zero, LR)
    assert np.allclose(params[1], p0[1] * (1 - LR * WD), rtol=1e-15)
    # off by default
    orc = _adamw_two_params()
    params = [x.copy() for x in p0]
    orc.step(params, zero, LR)
    assert np.allclose(params[1], p0[1] * (1 - LR * WD), rtol=1e-15)


def test_muon_options_rank1_closed_form():
    # rank-one gradient: O = phi^5(x) u v^T; with (lr_scale, wd_scale) = (2, 0)
    # p' = p - 2*lr*0.2*sqrt(max(m,n)) * O and no decay.
    m_, n_ = 6, 10
    rng = np.random.default_rng(3)
    u = rng.standard_normal(m_)
    u /= np.linalg.norm(u)
    v = rng.standard_normal(n_)
    v /= np.linalg.norm(v)
    names = ["model.action_expert.layers.0.mlp.w.weight"]
    orc = oracle.HybridOracle(names, [(m_, n_)], param_options={0: (2.0, 0.0)})
    p0 = rng.standard_normal((m_, n_)) * 0.02
    params = [p0.copy()]
    g = 0.5 * np.outer(u, v)          # norm 0.5: no clipping
    res = orc.step(params, [g], LR)
    d = (1 + MU) * 0.5
    x = d / (d + 1e-7)
    for _ in range(5):
        x = 3.4445 * x - 4.7750 * x ** 3 + 2.0315 * x ** 5
    O = x * np.outer(u, v)
    assert np.allclose(res["O"][0], O, rtol=0, atol=1e-12)
    assert np.allclose(params[0], p0 - 2 * LR * 0.2 * math.sqrt(10) * O, rtol=0, atol=1e-15)


def test_full_step_variants_compose():
    # EMA momentum + schedule through the whole step equal the pieces
    names = ["model.action_expert.layers.0.mlp.w.weight"]
    orc = oracle.HybridOracle(names, [(8, 12)], muon_momentum_form="ema", ns_schedule=SCHEDULE)
    rng = np.random.default_rng(12)
    g1, g2 = rng.standard_normal((8, 12)) * 0.01, rng.standard_normal((8, 12)) * 0.01
    params = [np.zeros((8, 12))]
    orc.step(params, [g1], LR)
    res = orc.step(params, [g2], LR)
    buf = (1 - MU) * (MU * g1 + g2)
    d = (1 - MU) * g2 + MU * buf
    assert np.allclose(orc.buf[0], buf, rtol=1e-14)
    assert np.allclose(res["O"][0], composed_closed_form(d, SCHEDULE), rtol=0, atol=1e-11)


def test_planted_option_mistakes_are_caught():
    # decay with the unscaled lr (ignoring lr_scale) breaks the closed form above
    p = 0.7
    ls, ws = 0.5, 2.0
    right = p * (1 - ls * LR * WD * ws)
    wrong = p * (1 - LR * WD * ws)
    assert not math.isclose(right, wrong, rel_tol=1e-9)
    # exempting by substring "bias" would exempt 'biased_gate'
    assert "bias" in "model.vlm.biased_gate.weight" and not oracle.decay_exempt("model.vlm.biased_gate.weight")


def test_total_override_sets_the_clip_coefficient():
    # a sampled oracle takes the model's global norm from outside: with its own
    # norm nothing changes; with a larger one the momentum is the gradient times
    # max_norm / (total + 1e-6) (first step: buf = coef * g)
    names = ["model.action_expert.layers.0.mlp.w.weight", "model.vlm.ln.weight"]
    shapes = [(6, 8), (5,)]
    rng = np.random.default_rng(31)
    g = [rng.standard_normal((6, 8)), rng.standard_normal(5)]
    own = math.sqrt(sum(float(np.sum(x * x)) for x in g))
    a = oracle.HybridOracle(names, shapes)
    b = oracle.HybridOracle(names, shapes)
    pa = [np.zeros((6, 8)), np.ones(5)]
    pb = [x.copy() for x in pa]
    ra = a.step(pa, g, LR)
    rb = b.step(pb, g, LR, total_override=own)
    assert ra["coef"] == rb["coef"] and all(np.array_equal(x, y) for x, y in zip(pa, pb))
    c = oracle.HybridOracle(names, shapes)
    rc = c.step([np.zeros((6, 8)), np.ones(5)], g, LR, total_override=1000.0)
    assert rc["total"] == 1000.0 and rc["coef"] == pytest.approx(1.0 / (1000.0 + 1e-6), rel=1e-15)
    assert np.allclose(c.buf[0], g[0] / (1000.0 + 1e-6), rtol=1e-15)
