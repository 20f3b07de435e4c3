"""Pins the oracle's elementary binary32 operations and quantiser.

Each operation of the C oracle is compared bit for bit with an exact-rational
emulation written from IEEE 754 (tests/exact_binary32.py) and with the
hand-worked cases in tests/golden/ (flush-to-zero rule: Open-1B review,
onedev.kr/papers/92, section "How it works"; quantiser: sections "How to use"
and "Premises and limits").
"""
import numpy as np
import pytest

import exact_binary32 as E
from golden_io import bits_to_f32, f32_to_bits, ftz_cases, quant_cases


def _rand_bits(rng, n):
    """Bit patterns spread over the interesting binary32 ranges."""
    out = []
    for _ in range(n):
        kind = rng.integers(0, 8)
        sign = int(rng.integers(0, 2)) << 31
        if kind == 0:      # subnormal
            out.append(sign | int(rng.integers(1, 1 << 23)))
        elif kind == 1:    # just above FLT_MIN
            out.append(sign | (1 << 23) | int(rng.integers(0, 1 << 10)))
        elif kind == 2:    # small normals
            e = int(rng.integers(1, 20))
            out.append(sign | (e << 23) | int(rng.integers(0, 1 << 23)))
        elif kind == 3:    # zero
            out.append(sign)
        elif kind == 4:    # near 1 and powers of two
            e = int(rng.integers(120, 135))
            m = int(rng.choice([0, 1, (1 << 23) - 1, int(rng.integers(0, 1 << 23))]))
            out.append(sign | (e << 23) | m)
        else:              # general normals, moderate exponents
            e = int(rng.integers(60, 190))
            out.append(sign | (e << 23) | int(rng.integers(0, 1 << 23)))
    return out


def test_ftz_golden(orc):
    ops = {"add": orc.add, "mul": orc.mul, "div": orc.div}
    emu = {"add": E.add, "mul": E.mul, "div": E.div}
    for op, a, b, exp in ftz_cases():
        fa, fb = bits_to_f32(a), bits_to_f32(b)
        if op == "sqrt":
            got = orc.sqrt(float(fa))
            em = E.sqrt(E.F32.from_bits(a))
        else:
            got = ops[op](float(fa), float(fb))
            em = emu[op](E.F32.from_bits(a), E.F32.from_bits(b))
        assert f32_to_bits(got) == exp, (op, hex(a), hex(b), hex(f32_to_bits(got)))
        assert em.bits() == exp, (op, hex(a), hex(b), em)


@pytest.mark.parametrize("op", ["add", "mul", "div"])
def test_binary_ops_match_exact_rounding(orc, op):
    rng = np.random.default_rng(1234 + ["add", "mul", "div"].index(op))
    A = _rand_bits(rng, 1500)
    B = _rand_bits(rng, 1500)
    fn = getattr(orc, op)
    em = getattr(E, op)
    for a, b in zip(A, B):
        ea, eb = E.F32.from_bits(a), E.F32.from_bits(b)
        if op == "div" and E.flush(eb).is_zero():
            continue
        ref = em(ea, eb)
        if ref.kind != "fin":
            continue
        got = f32_to_bits(fn(float(bits_to_f32(a)), float(bits_to_f32(b))))
        assert got == ref.bits(), (op, hex(a), hex(b), hex(got), ref)


def test_add_of_close_values_cancels_exactly(orc):
    # Sterbenz: b/2 <= a <= 2b makes a - b exact; covers the add alignment path
    rng = np.random.default_rng(7)
    for _ in range(500):
        a = np.float32(rng.uniform(1, 2))
        b = np.float32(rng.uniform(float(a) / 2, float(a)))
        got = orc.add(float(a), -float(b))
        assert np.float32(got) == np.float32(float(a) - float(b))


def test_sqrt_matches_exact_rounding(orc):
    rng = np.random.default_rng(99)
    for b in _rand_bits(rng, 1500):
        b &= 0x7FFFFFFF
        got = f32_to_bits(orc.sqrt(float(bits_to_f32(b))))
        assert got == E.sqrt(E.F32.from_bits(b)).bits(), hex(b)


def test_i2f_rounds_to_nearest_even(orc):
    vals = [0, 1, -1, 2**24, 2**24 + 1, 2**24 + 2, 2**24 + 3, -(2**24 + 3), 2**25 + 2,
            2**25 + 6, 16129 * 2048, 16129 * 5632, -16129 * 5632 - 1, 2**31 - 1, -2**31,
            2**40 + 2**16, 2**62 + 2**38]
    rng = np.random.default_rng(5)
    vals += [int(v) for v in rng.integers(-2**40, 2**40, 400)]
    for v in vals:
        assert f32_to_bits(orc.i2f(v)) == E.i2f(v).bits(), v


def test_quant_golden(orc):
    for xb, sb, q in quant_cases():
        x, s = bits_to_f32(xb), bits_to_f32(sb)
        assert orc.quant_one(float(x), float(s)) == q, (hex(xb), hex(sb))
        assert E.quant(E.F32.from_bits(xb), E.F32.from_bits(sb)) == q, (hex(xb), hex(sb))
        arr = orc.quant_i8(np.array([x], dtype=np.float32), float(s))
        assert int(arr[0]) == q


def test_quant_matches_exact_rounding(orc):
    rng = np.random.default_rng(2024)
    xs = rng.standard_normal(3000).astype(np.float32) * np.float32(3.0)
    # include exact half-integer multiples of the scale
    s = np.float32(0.0284)
    xs[:200] = (np.arange(200, dtype=np.float32) - 100 + 0.5) * s
    q = orc.quant_i8(xs, float(s))
    es = E.F32.from_float(float(s))
    for i, x in enumerate(xs):
        assert int(q[i]) == E.quant(E.F32.from_float(float(x)), es), (i, float(x))
    assert q.min() >= -127 and q.max() <= 127


def test_no_contraction_in_mul_then_add(orc):
    # a*b+c where a fused multiply-add would keep the 2^-24 term
    a = np.float32(1 + 2**-12)
    c = -np.float32(1 + 2**-11)
    p = orc.mul(float(a), float(a))
    r = orc.add(p, float(c))
    assert r == 0.0
    assert E.add(E.mul(E.f(float(a)), E.f(float(a))), E.f(float(c))).to_float() == 0.0
