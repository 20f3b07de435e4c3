"""Pins the oracle's canonical sum (chunks of 64, left to right, then the
stride-doubling pairwise tree) and the weight/activation scales.

Pins: hand-worked discriminators (tests/golden/canon_discriminators.txt) that
fail for another chunk size, another in-chunk order or another tree shape; the
textbook sequential sum for L <= 64; closed forms; the error bound of a
summation tree against the exact rational sum; an independent streaming
(binary-counter) formulation of the same tree; the aligned power-of-two split
property the GPU kernels rely on.  Fixed order: Open-1B review,
onedev.kr/papers/92, section "How it works"; scale formula 2*mean|w|/sqrt(q_max):
sections "How to use" and "Premises and limits".
"""
import functools
import math
from fractions import Fraction

import numpy as np
import pytest

import exact_binary32 as E
from golden_io import canon_cases, f32_to_bits

U = Fraction(1, 2 ** 24)


def _emu_add_f(a, b):
    return E.add(E.f(float(a)), E.f(float(b))).to_float()


def test_discriminators(orc):
    for p, exp in canon_cases():
        got = f32_to_bits(orc.canon_sum(p))
        assert got == exp, (p.size, hex(got), hex(exp))


def test_short_sums_are_the_textbook_left_fold(orc):
    rng = np.random.default_rng(11)
    for L in [1, 2, 3, 7, 31, 63, 64]:
        for _ in range(5):
            p = (rng.standard_normal(L) * 10.0 ** rng.integers(-3, 4, L)).astype(np.float32)
            ref = functools.reduce(_emu_add_f, p[1:], float(p[0]))
            assert f32_to_bits(orc.canon_sum(p)) == f32_to_bits(ref)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 127, 128, 129, 320, 384, 448, 1000, 4097, 65536])
def test_equal_powers_of_two_sum_exactly(orc, L):
    p = np.full(L, 2.0 ** -8, dtype=np.float32)
    assert float(orc.canon_sum(p)) == L * 2.0 ** -8


def _exact(p):
    return sum(Fraction(float(x)) for x in p)


@pytest.mark.parametrize("L", [100, 1000, 5000, 20000])
def test_error_within_summation_tree_bound(orc, L):
    # Every term passes through at most 63 in-chunk adds plus ceil(log2 C)
    # tree adds, so |error| <= gamma_d * sum|p| with d = 63 + ceil(log2 C).
    rng = np.random.default_rng(L)
    p = (rng.standard_normal(L) * np.exp(rng.uniform(-3, 3, L))).astype(np.float32)
    C = (L + 63) // 64
    d = 63 + max(0, math.ceil(math.log2(C)))
    gamma = d * U / (1 - d * U)
    err = abs(Fraction(float(orc.canon_sum(p))) - _exact(p))
    assert err <= gamma * sum(abs(Fraction(float(x))) for x in p)


def _stride_tree(t):
    t = list(t)
    C = len(t)
    s = 1
    while s < C:
        for j in range(0, C - s, 2 * s):
            t[j] = _emu_add_f(t[j], t[j + s])
        s *= 2
    return t[0]


def _chunk_sums(p):
    out = []
    for lo in range(0, len(p), 64):
        out.append(functools.reduce(_emu_add_f, p[lo + 1:lo + 64], float(p[lo])))
    return out


def _streaming_stack(t):
    """Binary-counter evaluation of the same tree: push each partial, merge
    while the count has trailing ones, then fold remaining levels right to left."""
    stack = {}
    for c, v in enumerate(t):
        lvl = 0
        while (c >> lvl) & 1:
            v = _emu_add_f(stack.pop(lvl), v)
            lvl += 1
        stack[lvl] = v
    acc = None
    for lvl in sorted(stack):
        acc = stack[lvl] if acc is None else _emu_add_f(stack[lvl], acc)
    return acc


@pytest.mark.parametrize("L", [65, 130, 320, 448, 640, 1000, 1025, 3000])
def test_streaming_formulation_agrees(orc, L):
    rng = np.random.default_rng(L + 1)
    p = (rng.standard_normal(L) * 10.0 ** rng.integers(-2, 3, L)).astype(np.float32)
    chunks = _chunk_sums(p)
    ref = _streaming_stack(chunks)
    assert f32_to_bits(orc.canon_sum(p)) == f32_to_bits(ref)
    assert f32_to_bits(_stride_tree(chunks)) == f32_to_bits(ref)


@pytest.mark.parametrize("blk_chunks", [1, 2, 4, 8, 16])
def test_aligned_power_of_two_split(orc, blk_chunks):
    # canon over aligned blocks of 2^b chunks, then the tree over block results
    rng = np.random.default_rng(blk_chunks)
    for L in [700, 1024, 1600, 2049]:
        p = (rng.standard_normal(L) * 10.0 ** rng.integers(-2, 3, L)).astype(np.float32)
        B = 64 * blk_chunks
        parts = [orc.canon_sum(p[lo:lo + B]) for lo in range(0, L, B)]
        assert f32_to_bits(_stride_tree(parts)) == f32_to_bits(orc.canon_sum(p))


def test_order_is_observable(orc):
    # reversing a chunk changes the bits: the fixed order is not a formality
    p = np.array([2.0 ** 24] + [1.0] * 63, dtype=np.float32)
    assert orc.canon_sum(p) != orc.canon_sum(p[::-1].copy())


# ----------------------------------------------------------------- scales

def _sqrt127():
    return E.sqrt(E.i2f(127))


@pytest.mark.parametrize("n", [1, 2, 64, 65, 1000, 4096, 1 << 16, 100000])
def test_weight_scale_closed_form(orc, n):
    # |w| = 2^-8 everywhere: S = n 2^-8 exactly, mean = 2^-8,
    # s_w = RN(2^-7 / RN(sqrt(127)))
    rng = np.random.default_rng(n)
    w = np.where(rng.integers(0, 2, n) == 1, 2.0 ** -8, -2.0 ** -8).astype(np.float32)
    ref = E.div(E.f(2.0 ** -7), _sqrt127())
    assert f32_to_bits(orc.wscale(w, 0)) == ref.bits()


def test_weight_scale_within_bound_of_exact_formula(orc):
    rng = np.random.default_rng(3)
    n = 50000
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    got = Fraction(float(orc.wscale(w, 0)))
    exact_mean = sum(abs(Fraction(float(x))) for x in w) / n
    # compare s^2 with the exact (2 mean)^2 / 127 to avoid an irrational sqrt
    exact_sq = (2 * exact_mean) ** 2 / 127
    C = (n + 63) // 64
    d = 63 + math.ceil(math.log2(C))
    rel = d * U / (1 - d * U) + 4 * U       # sum, mean, 2x, sqrt, divide
    assert abs(got * got - exact_sq) <= (2 * rel + rel * rel) * exact_sq


def test_activation_scale_is_exact_max_over_127(orc):
    rng = np.random.default_rng(4)
    for n in [1, 5, 64, 1000, 77777]:
        x = (rng.standard_normal(n) * 3).astype(np.float32)
        amax = max(abs(Fraction(float(v))) for v in x)
        ref = E.div(E.round_to_f32(False, amax), E.i2f(127))
        assert f32_to_bits(orc.wscale(x, 1)) == ref.bits()


def test_activation_scale_flushes_subnormals(orc):
    x = np.array([1e-40, -3e-39, 0.0], dtype=np.float32)   # all subnormal or zero
    assert f32_to_bits(orc.wscale(x, 1)) == 0
    x = np.array([1e-40, 2.0 ** -100], dtype=np.float32)
    ref = E.div(E.f(2.0 ** -100), E.i2f(127))
    assert f32_to_bits(orc.wscale(x, 1)) == ref.bits()
