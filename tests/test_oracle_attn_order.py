"""Bit-level pins of the attention oracle (oracle.c, int8 P.V attention with a
64-bit fixed-point dQ; Open-1B review, onedev.kr/papers/92, section "How to
use"), against things other than the oracle itself:

* e^x: the library defines its exponential as Cody-Waite range reduction with
  ln 2 split in two, the degree-7 Taylor polynomial in Horner form and an
  exact scaling by 2^k.  Here those steps are replayed in the exact-rational
  binary32 emulator (tests/exact_binary32.py), with every constant derived from
  its mathematical definition (RN(1/n!), RN(1/ln 2), the 9-bit head 355/512 of
  ln 2 and RN of the remainder), so a wrong coefficient, a dropped term or a
  different reduction fails bit for bit.
* the reduction orders of the forward and backward: hand-worked inputs in
  tests/golden/attn_order.txt on which another tile width (32 or 128 instead
  of 64), window-relative instead of absolute tiles, per-key or end-of-row
  fixed-point conversion, tile-major instead of head-major folding, a plain
  left fold, or a left fold instead of the canonical sum over d, each give
  other bits (each line states the alternatives).
* the reading that a zero row maximum is stored as +0.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import exact_binary32 as E
from golden_io import attn_order_cases

# --------------------------------------------------------------- e^x replay


def _ln2(terms: int = 120) -> Fraction:
    """ln 2 = sum_{k>=1} 1 / (k 2^k), to within 2^-terms."""
    return sum((Fraction(1, k * 2 ** k) for k in range(1, terms + 1)), Fraction(0))


def _exp_constants():
    ln2 = _ln2()
    log2e = E.round_to_f32(False, 1 / ln2)                # RN(1/ln 2)
    c1 = Fraction(355, 512)                                 # 9-bit head of ln 2
    assert abs(ln2 - c1) < Fraction(1, 2 ** 12)
    c2 = E.round_to_f32(True, abs(ln2 - c1))                # RN(ln 2 - C1), negative
    coef = [E.round_to_f32(False, Fraction(1, math.factorial(n))) for n in range(8)]
    return log2e, E.round_to_f32(False, c1), c2, coef


_CONST = None


def exp_replay(x: float) -> int:
    """Bits of the library's e^x, every step rounded and flushed exactly."""
    global _CONST
    if _CONST is None:
        _CONST = _exp_constants()
    log2e, c1, c2, coef = _CONST
    xf = E.f(x)
    k = E.rint_half_even(E.mul(xf, log2e))
    kf = E.i2f(k)
    t1 = E.mul(kf, c1)
    t2 = E.mul(kf, c2)
    r = E.add(E.add(xf, E.F32(not t1.neg, t1.mag)), E.F32(not t2.neg, t2.mag))
    p = coef[7]
    for n in range(6, -1, -1):
        p = E.add(E.mul(p, r), coef[n])
    if k < -126:
        return 0
    scaled = E.round_to_f32(p.neg, p.mag * Fraction(2) ** k)
    return E.flush(scaled).bits()


def _bits(v) -> int:
    return int(np.array([v], dtype=np.float32).view(np.uint32)[0])


def test_exp_constants_are_their_definitions():
    log2e, c1, c2, coef = _exp_constants()
    # the stated values of the definitions (binary32 hex), derived here from
    # the series for ln 2 and exact factorials
    assert log2e.bits() == _bits(float.fromhex("0x1.715476p+0"))
    assert c1.bits() == _bits(float.fromhex("0x1.63p-1"))
    assert c2.bits() == _bits(float.fromhex("-0x1.bd0106p-13"))
    assert [c.bits() for c in coef[3:]] == [_bits(float.fromhex(h)) for h in
                                            ("0x1.555556p-3", "0x1.555556p-5", "0x1.111112p-7",
                                             "0x1.6c16c2p-10", "0x1.a01a02p-13")]


def test_exp_bits_match_the_exact_replay(orc):
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        -rng.random(1500) * 88.0,                       # the softmax's range: x <= 0
        -rng.random(300) * 1e-3, -rng.random(100) * 1e-6,
        -np.arange(0, 127) * math.log(2),                 # near the reduction's k boundaries
        -(np.arange(0, 127) + 0.5) * math.log(2),         # midway: k ties
        [0.0, -0.0, -1e-30, -0.5, -1.0, -10.0, -87.3, -87.33654, -88.0, -103.0, -104.0],
        rng.random(200) * 10.0,                         # positive arguments, same algorithm
    ]).astype(np.float32)
    for x in xs:
        got = _bits(orc.exp(float(x)))
        exp = exp_replay(float(x))
        assert got == exp, (float(x), hex(got), hex(exp))


@pytest.mark.parametrize("slip", ["coef5", "drop_c2", "degree6", "k_floor"])
def test_exp_replay_discriminates_plausible_slips(slip):
    """The replay is sharp: each of these variants of the algorithm gives other
    bits on a few thousand of the arguments above (so the bit-exact test
    would catch the same slip in the oracle)."""
    log2e, c1, c2, coef = _exp_constants()

    def variant(x):
        xf = E.f(x)
        v = E.mul(xf, log2e).value()
        k = math.floor(v) if slip == "k_floor" else E.rint_half_even(E.mul(xf, log2e))
        kf = E.i2f(k)
        t1 = E.mul(kf, c1)
        r = E.add(xf, E.F32(not t1.neg, t1.mag))
        if slip != "drop_c2":
            t2 = E.mul(kf, c2)
            r = E.add(r, E.F32(not t2.neg, t2.mag))
        cf = list(coef)
        if slip == "coef5":
            cf[5] = E.round_to_f32(False, Fraction(1, 100))
        top = 6 if slip == "degree6" else 7
        p = cf[top]
        for n in range(top - 1, -1, -1):
            p = E.add(E.mul(p, r), cf[n])
        if k < -126:
            return 0
        return E.flush(E.round_to_f32(p.neg, p.mag * Fraction(2) ** k)).bits()

    rng = np.random.default_rng(11)
    xs = (-rng.random(400) * 80.0).astype(np.float32)
    differ = sum(variant(float(x)) != exp_replay(float(x)) for x in xs)
    assert differ > 20, (slip, differ)


# ------------------------------------------------- hand-worked order cases

def _c_bits() -> E.F32:
    """c = 1 (/) sqrt(128), the logit and dQ/dK scale."""
    return E.div(E.f(1.0), E.sqrt(E.f(128.0)))


def _build(case):
    T, W, Hq, Hkv, D = case["T"], case["W"], case["Hq"], case["Hkv"], 128
    q = np.zeros((1, T, Hq, D), np.float32)
    k = np.zeros((1, T, Hkv, D), np.float32)
    vq = np.zeros((1, T, Hkv, D), np.int8)
    dout = np.zeros((1, T, Hq, D), np.float32)
    o = np.zeros((1, T, Hq, D), np.float32)
    if case["kind"] in ("dq", "dk", "dv"):
        dout[..., 0] = 1.0
        vq[..., 0] = 1
    arrs = {"q": q, "k": k, "vq": vq, "dout": dout, "o": o}
    for name, i_lo, i_hi, h, d_lo, d_hi, val in case["assign"]:
        arrs[name][0, i_lo:i_hi + 1, h, d_lo:d_hi + 1] = val
    return q, k, vq, dout, o


@pytest.mark.parametrize("case", list(attn_order_cases()), ids=lambda c: c["name"])
def test_attention_order_cases(orc, case):
    q, k, vq, dout, o = _build(case)
    T, W, Hq, Hkv = case["T"], case["W"], case["Hq"], case["Hkv"]
    row, col = case["row"], case["col"]
    expected = E.F32.from_bits(case["bits"])
    if case["times_c"]:
        expected = E.mul(expected, _c_bits())
    if case["kind"] in ("m", "l", "o"):
        om, mm, lm = orc.attn_fwd(q, k, vq, 1.0, W)
        got = {"m": mm.reshape(-1), "l": lm.reshape(-1), "o": om.reshape(-1, 128)[:, col]}[
            case["kind"]][row]
    else:
        m = np.zeros((1, T, Hq), np.float32)          # +0 maxima, unit sums: a = p = 1
        lsum = np.ones((1, T, Hq), np.float32)
        one = np.array([row], dtype=np.int64)
        zero = np.array([0], dtype=np.int64)
        qrows, krows = (one, zero) if case["kind"] == "dq" else (zero, one)
        dq, dk, dv = orc.attn_bwd_rows(q, k, vq, 1.0, o, dout, m, lsum, W, qrows, krows)
        got = {"dq": dq, "dk": dk, "dv": dv}[case["kind"]].reshape(-1, 128)[0, col]
    assert _bits(got) == expected.bits(), (case["name"], hex(_bits(got)), hex(expected.bits()))


def _canon_exact(terms):
    """The canonical sum in the exact emulator: chunks of 64 left to right from
    the first term, then the stride-doubling tree over the chunk partials."""
    t = []
    for c0 in range(0, len(terms), 64):
        a = terms[c0]
        for x in terms[c0 + 1:c0 + 64]:
            a = E.add(a, x)
        t.append(a)
    s = 1
    while s < len(t):
        for j in range(0, len(t) - s, 2 * s):
            t[j] = E.add(t[j], t[j + s])
        s *= 2
    return t[0]


def test_row_sum_order(orc):
    # row i = 127 of a causal row: key 0 has logit +0 (the maximum, p = 1) and
    # keys 1..127 the logit RN(-192 c) ~ -16.97, p ~ 0.72 * 2^-24, below half
    # the spacing at 1.  A left fold over the keys loses every small p (l = 1);
    # the canonical order sums the second 64-key chunk on its own first.
    T = 128
    q = np.zeros((1, T, 1, 128), np.float32)
    k = np.zeros((1, T, 1, 128), np.float32)
    q[0, 127, 0, 0] = 1.0
    k[0, 1:, 0, 0] = -192.0
    vq = np.zeros((1, T, 1, 128), np.int8)
    _, m, l = orc.attn_fwd(q, k, vq, 1.0, 0)
    s = E.mul(E.f(-192.0), _c_bits())
    p = E.F32.from_bits(exp_replay(s.to_float()))
    terms = [E.f(1.0)] + [p] * 127
    expected = _canon_exact(terms)
    left = terms[0]
    for x in terms[1:]:
        left = E.add(left, x)
    assert left.bits() == E.f(1.0).bits() != expected.bits()   # the case discriminates
    assert _bits(m[0, 127, 0]) == 0
    assert _bits(l[0, 127, 0]) == expected.bits()


def test_zero_row_maximum_is_positive_zero(orc):
    # q = 0 and every k negative: every product q (x) k is -0, so every logit
    # is -0 and the exact maximum over {-0} is -0; the reading stores it as
    # +0, which makes m independent of the order in which a kernel compares
    # +0 and -0 (IEEE max leaves that choice open)
    T, D = 70, 128
    q = np.zeros((1, T, 2, D), np.float32)
    k = -np.ones((1, T, 1, D), np.float32)
    vq = np.ones((1, T, 1, D), np.int8)
    o, m, l = orc.attn_fwd(q, k, vq, 1.0, 0)
    assert np.all(m.view(np.uint32) == 0)
    assert np.array_equal(l[0, :, 0], np.arange(1, T + 1, dtype=np.float32))   # p = e^0 = 1


# ------------------------------------------- planted mistakes are caught

# Each entry copies oracle.c to a temporary directory, plants one plausible
# mistake by a textual substitution, builds it, and checks that the pins above
# fail on it: the named golden cases, and/or the e^x replay.
_LEFT_FOLD = """
static float planted_left_fold(const float* p, int64_t n)
{
    float a = p[0];
    for (int64_t i = 1; i < n; ++i)
        a = oracle_add(a, p[i]);
    return a;
}
"""
MUTATIONS = {
    "key_and_query_tiles_of_32": ("#define ATTN_TILE 64", "#define ATTN_TILE 32",
                                  ["dq_tiles", "dk_groups", "dv_groups", "dk_window"]),
    "key_and_query_tiles_of_128": ("#define ATTN_TILE 64", "#define ATTN_TILE 128",
                                   ["dq_tiles", "dq_window", "dk_groups", "dv_groups", "dk_window"]),
    "key_tiles_from_the_window_start": (
        "    for (int64_t t0 = (lo / ATTN_TILE) * ATTN_TILE; t0 <= i; t0 += ATTN_TILE) {",
        "    for (int64_t t0 = lo; t0 <= i; t0 += ATTN_TILE) {", ["dq_window"]),
    "query_tiles_from_the_key": (
        "        for (int64_t t0 = (j / ATTN_TILE) * ATTN_TILE; t0 <= ihi; t0 += ATTN_TILE) {",
        "        for (int64_t t0 = j; t0 <= ihi; t0 += ATTN_TILE) {", ["dk_window"]),
    "tile_major_fold": (
        "    for (int64_t hh = 0; hh < G; ++hh) {\n"
        "        const int64_t h = g * G + hh;\n"
        "        for (int64_t t0 = (j / ATTN_TILE) * ATTN_TILE; t0 <= ihi; t0 += ATTN_TILE) {",
        "    for (int64_t t0 = (j / ATTN_TILE) * ATTN_TILE; t0 <= ihi; t0 += ATTN_TILE) {\n"
        "        for (int64_t hh = 0; hh < G; ++hh) {\n"
        "        const int64_t h = g * G + hh;", ["dk_groups", "dv_groups"]),
    "logit_left_fold": ("    return oracle_mul(oracle_canon_sum(tmp, D), c);",
                        "    return oracle_mul(planted_left_fold(tmp, D), c);", ["m_logit"]),
    "drow_left_fold": ("        tmp[d] = oracle_mul(dout[r * D + d], o[r * D + d]);\n"
                       "    return oracle_canon_sum(tmp, D);",
                       "        tmp[d] = oracle_mul(dout[r * D + d], o[r * D + d]);\n"
                       "    return planted_left_fold(tmp, D);", ["dq_drow"]),
    "fixed_point_per_key": ("            for (int64_t d = 0; d < D; ++d) {\n"
                            "                const float t = oracle_mul(ds, kj[d]);\n"
                            "                part[d] = j == jb ? t : oracle_add(part[d], t);\n"
                            "            }",
                            "            for (int64_t d = 0; d < D; ++d)\n"
                            "                acc[d] += oracle_attn_fx(oracle_mul(ds, kj[d]));\n"
                            "            for (int64_t d = 0; d < D; ++d)\n"
                            "                part[d] = 0.0f;", ["dq_tiles", "dq_window"]),
    "row_sum_left_fold": ("    const float l = oracle_canon_sum(tmp, n);",
                          "    const float l = planted_left_fold(tmp, n);", "row_sum"),
    "zero_maximum_kept_negative": ("        m = 0.0f; /* a zero maximum is stored as +0 */",
                                   "        (void)0;", "zero_max"),
    "exp_coefficients_swapped": ("0x1.555556p-5f, 0x1.111112p-7f", "0x1.111112p-7f, 0x1.555556p-5f",
                                 "exp"),
    "exp_coefficient_typo": ("0x1.6c16c2p-10f", "0x1.6c16c2p-11f", "exp"),
    "exp_without_c2": ("    const float r = oracle_add(oracle_add(x, -oracle_mul(kf, EXP_C1)), "
                       "-oracle_mul(kf, EXP_C2));",
                       "    const float r = oracle_add(x, -oracle_mul(kf, EXP_C1));", "exp"),
}


def _build_planted(tmp_path, old, new):
    import shutil
    import subprocess
    import oracle
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) == 1, old
    src = src.replace(old, new)
    src = src.replace('#include "oracle.h"\n', '#include "oracle.h"\n' + _LEFT_FOLD, 1)
    d = tmp_path / "planted"
    d.mkdir()
    shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "oracle.h"), d / "oracle.h")
    (d / "oracle.c").write_text(src)
    so = str(d / "liboracle_planted.so")
    cc = shutil.which("gcc") or shutil.which("cc")
    r = subprocess.run([cc, *oracle.CFLAGS, str(d / "oracle.c"), "-o", so, "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return oracle.load(so)


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistakes_fail_the_pins(orc, tmp_path, name):
    old, new, caught_by = MUTATIONS[name]
    planted = _build_planted(tmp_path, old, new)
    saved = orc._lib
    orc._lib = planted
    try:
        if caught_by in ("row_sum", "zero_max"):
            fn = test_row_sum_order if caught_by == "row_sum" else test_zero_row_maximum_is_positive_zero
            with pytest.raises(AssertionError):
                fn(orc)
            return
        if caught_by == "exp":
            rng = np.random.default_rng(3)
            xs = (-rng.random(300) * 80.0).astype(np.float32)
            assert any(_bits(orc.exp(float(x))) != exp_replay(float(x)) for x in xs)
            return
        cases = {c["name"]: c for c in attn_order_cases()}
        for cname in caught_by:
            with pytest.raises(AssertionError):
                test_attention_order_cases(orc, cases[cname])
    finally:
        orc._lib = saved
