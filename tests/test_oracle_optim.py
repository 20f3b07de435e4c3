"""Pins the oracle's optimiser step: global gradient norm (canonical-order sum
of squares), clip coefficient, bias-correction powers and the AdamW update.

The recipe (Open-1B review, onedev.kr/papers/92, section "Premises and limits")
names AdamW with beta1 0.9, beta2 0.95, eps 1e-8, decoupled weight decay 0.1 and
clipping at global L2 norm 1.0, without an operation order; the oracle fixes one
(oracle.h).  Pins: closed forms, the textbook left fold for short sums, the
exact-rational bound for the binary powers, and a float64 evaluation of the
textbook AdamW formulas from the same binary32 state within a rounding bound
that a wrong sign, a missing bias correction or a swapped moment would break.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import exact_binary32 as E
from golden_io import f32_to_bits

U = 2.0 ** -24
HP = dict(lr=4.5e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0)


def _f(x):
    return float(np.float32(x))


@pytest.mark.parametrize("n", [1, 64, 65, 1000, 4097])
def test_sumsq_closed_form(orc, n):
    g = np.full(n, 2.0 ** -4, np.float32)
    g[::3] = -2.0 ** -4
    assert float(orc.sumsq(g)) == n * 2.0 ** -8


def test_sumsq_short_is_textbook_left_fold(orc):
    rng = np.random.default_rng(1)
    for n in [1, 5, 64]:
        g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
        terms = [E.mul(E.f(float(x)), E.f(float(x))) for x in g]
        acc = terms[0]
        for t in terms[1:]:
            acc = E.add(acc, t)
        assert f32_to_bits(orc.sumsq(g)) == acc.bits()


def test_sumsq_within_bound_of_exact(orc):
    rng = np.random.default_rng(2)
    n = 20000
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    exact = sum(Fraction(float(x)) ** 2 for x in g)
    C = (n + 63) // 64
    d = 64 + math.ceil(math.log2(C))
    assert abs(Fraction(float(orc.sumsq(g))) - exact) <= Fraction(d * U / (1 - d * U)) * exact


def test_pow_t_closed_form_and_bound(orc):
    for t in range(0, 127):
        assert float(orc.pow_t(0.5, t)) == 2.0 ** -t        # powers of two are exact
    for b in [0.9, 0.95, 0.999]:
        bf = Fraction(_f(b))
        for t in [1, 2, 3, 7, 10, 100, 667, 5000]:
            got = Fraction(float(orc.pow_t(b, t)))
            # squaring doubles the accumulated relative error at every level:
            # base_k carries (2^k - 1) units, so the product carries < t + 2 log2 t
            k = t + 2 * t.bit_length()
            exact = bf ** t
            if exact < Fraction(1, 2 ** 120):
                assert got == 0                    # underflows and is flushed to +0
                continue
            assert abs(got - exact) <= Fraction(k * U / (1 - k * U)) * exact, (b, t)
    assert float(orc.pow_t(0.9, 1)) == _f(0.9)


def test_pow_t_sequence(orc):
    # right-to-left binary exponentiation, each multiply rounded (t = 13 = 0b1101)
    b = E.f(0.95)
    r, base = E.f(1.0), b
    for bit in [1, 0, 1, 1]:
        if bit:
            r = E.mul(r, base)
        base = E.mul(base, base)
    assert f32_to_bits(orc.pow_t(0.95, 13)) == r.bits()


def test_clip_coefficient(orc):
    assert float(orc.clip_coef(0.25, 1.0)) == 1.0          # norm 0.5: no clipping
    at_one = E.div(E.f(1.0), E.add(E.f(1.0), E.f(1e-6)))    # norm == max_norm: 1/(1+1e-6) < 1
    assert f32_to_bits(orc.clip_coef(1.0, 1.0)) == at_one.bits() and at_one.to_float() < 1.0
    exp = E.div(E.f(1.0), E.add(E.f(10.0), E.f(1e-6)))
    assert f32_to_bits(orc.clip_coef(100.0, 1.0)) == exp.bits()


def test_zero_gradient_only_decays(orc):
    rng = np.random.default_rng(3)
    p = (rng.standard_normal(100) * 0.02).astype(np.float32)
    z = np.zeros(100, np.float32)
    p2, m2, v2 = orc.adamw_step(p, z, z, z, 0.0, 1, **HP)
    decay = E.add(E.f(1.0), E.f(-float(E.mul(E.f(HP["lr"]), E.f(HP["weight_decay"])).to_float())))
    for i in range(100):
        assert f32_to_bits(p2[i]) == E.mul(E.f(float(p[i])), decay).bits()
    assert not m2.any() and not v2.any()


def test_zero_lr_leaves_parameters(orc):
    rng = np.random.default_rng(4)
    p = (rng.standard_normal(100) * 0.02).astype(np.float32)
    g = (rng.standard_normal(100) * 1e-3).astype(np.float32)
    hp = dict(HP, lr=0.0)
    p2, m2, v2 = orc.adamw_step(p, np.zeros_like(p), np.zeros_like(p), g, orc.sumsq(g), 1, **hp)
    assert np.array_equal(p2.view(np.uint32), p.view(np.uint32))
    assert m2.any() and v2.any()


@pytest.mark.parametrize("t", [1, 2, 10, 700])
@pytest.mark.parametrize("scale", [1e-4, 1.0])
def test_adamw_matches_textbook_in_float64(orc, t, scale):
    # one step from an arbitrary binary32 state; the float64 evaluation of the
    # textbook formulas bounds every rounding the oracle takes
    rng = np.random.default_rng(t)
    n = 2000
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3 * scale).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-6 * scale * scale).astype(np.float32)
    g = (rng.standard_normal(n) * 0.03 * scale).astype(np.float32)
    s = orc.sumsq(g)
    p2, m2, v2 = orc.adamw_step(p, m, v, g, s, t, **HP)
    b1, b2 = _f(HP["beta1"]), _f(HP["beta2"])
    lr, wd, eps = _f(HP["lr"]), _f(HP["weight_decay"]), _f(HP["eps"])
    norm = math.sqrt(float(s))
    coef = min(_f(HP["max_norm"]) / (norm + _f(1e-6)), 1.0)
    gc = g.astype(np.float64) * coef
    m64 = b1 * m.astype(np.float64) + (1 - b1) * gc
    v64 = b2 * v.astype(np.float64) + (1 - b2) * gc * gc
    mh = m64 / (1 - b1 ** t)
    vh = v64 / (1 - b2 ** t)
    upd = lr * mh / (np.sqrt(vh) + eps)
    p64 = p.astype(np.float64) * (1 - lr * wd) - upd
    tol_m = 8 * U * (np.abs(b1 * m) + np.abs((1 - b1) * gc)) + 1e-45
    tol_v = 8 * U * (np.abs(b2 * v) + np.abs((1 - b2) * gc * gc)) + 1e-45
    tol_p = 4 * U * np.abs(p) + 40 * U * np.abs(upd) + 1e-45
    assert np.all(np.abs(m2 - m64) <= tol_m)
    assert np.all(np.abs(v2 - v64) <= tol_v)
    assert np.all(np.abs(p2 - p64) <= tol_p)
    # the update is not negligible here, so a sign or bias-correction slip shows
    assert np.median(np.abs(upd) / (4 * U * np.abs(p))) > 10


def test_clipping_scales_the_gradient(orc):
    g = np.full(400, 0.5, np.float32)                 # global norm 10
    z = np.zeros_like(g)
    p = np.zeros_like(g)
    s = orc.sumsq(g)
    assert float(s) == 100.0
    _, m2, _ = orc.adamw_step(p, z, z, g, s, 1, **HP)
    coef = orc.clip_coef(s, 1.0)
    exp = E.mul(E.add(E.f(1.0), E.f(-_f(0.9))), E.mul(E.f(0.5), E.f(float(coef))))
    assert f32_to_bits(m2[0]) == exp.bits()
    assert abs(float(m2[0]) - 0.1 * 0.05) < 1e-8
