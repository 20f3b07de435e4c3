"""Pins of the attention oracle (oracle.c, int8 P.V attention) against things
other than itself: float64 e^x within an error bound, an independent float64
attention forward (standard softmax attention with the int8 quantisation of P
and V) within rounding bounds, exact special cases (one-key windows), the
causal and window masks, a float64 analytic backward checked in turn by finite
differences, and the fixed-point conversions."""
import math

import numpy as np
import pytest


def ulps(a: np.float32, b: float) -> float:
    """|a - b| in units of the binary32 spacing at b (b exact, float64)."""
    a = float(a)
    if a == b:
        return 0.0
    return abs(a - b) / float(np.spacing(np.float32(abs(b))))


def test_exp_special_arguments(orc):
    # the scaling by 2^k decides these: k < -126 gives 0, k > 254 overflows
    # whatever the polynomial gave (at +inf the reduction itself is NaN), and a
    # NaN argument stays NaN
    assert orc.exp(float("inf")) == np.inf
    assert orc.exp(1e38) == np.inf and orc.exp(177.0) == np.inf
    assert orc.exp(float("-inf")) == 0.0 and orc.exp(-1e38) == 0.0
    assert np.isnan(orc.exp(float("nan")))
    assert orc.exp(0.0) == 1.0 and orc.exp(-0.0) == 1.0


def test_exp_within_two_ulp(orc):
    rng = np.random.default_rng(0)
    xs = np.concatenate([-rng.random(20000) * 87.0, -rng.random(2000) * 1e-3,
                         -np.arange(0, 60) * math.log(2), [-1e-30, -0.5, -1.0, -10.0]])
    worst = 0.0
    for x in xs.astype(np.float32):
        got = orc.exp(float(x))
        ref = math.exp(float(x))
        if ref < 1.1754944e-38:      # subnormal true value: flushed
            assert got == 0.0
            continue
        worst = max(worst, ulps(got, ref))
    assert worst <= 2.0, worst
    assert orc.exp(0.0) == 1.0 and orc.exp(-0.0) == 1.0
    assert orc.exp(-104.0) == 0.0 and orc.exp(-1000.0) == 0.0


def test_quant_p_and_fixed_point(orc):
    assert orc.attn_quant_p(1.0) == 127 and orc.attn_quant_p(0.0) == 0
    assert orc.attn_quant_p(0.5 / 127) == 0          # tie -> even
    assert orc.attn_quant_p(1.5 / 127 + 1e-6) == 2
    assert orc.attn_quant_p(float("nan")) == 0       # the clamp's lower bound
    assert orc.attn_quant_p(float("inf")) == 127 and orc.attn_quant_p(-1.0) == 0
    assert orc.attn_fx(1.0) == 1 << 48
    assert orc.attn_fx(-1.0) == -(1 << 48)
    assert orc.attn_fx(2.0 ** -49) == 0               # 0.5 -> even
    assert orc.attn_fx(3 * 2.0 ** -49) == 2           # 1.5 -> even
    assert orc.attn_fx(5 * 2.0 ** -49) == 2           # 2.5 -> even
    assert orc.attn_fx(2.0 ** 16) == (1 << 63) - 1    # saturates
    assert orc.attn_fx(2.0 ** 15) == (1 << 63) - 1    # 2^63 itself is out of range
    assert orc.attn_fx(-(2.0 ** 15)) == -(1 << 63)    # -2^63 is the minimum
    assert orc.attn_fx(np.float32(2.0 ** 15) * np.float32(1 - 2.0 ** -24)) == (1 << 63) - (1 << 39)
    assert orc.attn_fx(np.inf) == (1 << 63) - 1 and orc.attn_fx(-np.inf) == -(1 << 63)
    assert orc.attn_fx(np.nan) == 0                   # a NaN partial adds nothing
    assert orc.attn_fx(1e-30) == 0
    assert orc.attn_fix2f(1 << 48) == 1.0
    assert orc.attn_fix2f(3) == np.float32(3 * 2.0 ** -48)
    assert orc.attn_fix2f(-(1 << 50)) == -4.0


def _case(seed, B, T, Hq, Hkv, D):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    vq = rng.integers(-127, 128, (B, T, Hkv, D)).astype(np.int8)
    return q, k, vq


def _ref_fwd(q, k, vq, s_v, W):
    """float64 softmax attention with P quantised as rint(127 p); returns o, m, l."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    vh = vq.astype(np.float64) * np.float64(np.float32(s_v))
    o = np.zeros((B, T, Hq, D))
    m = np.zeros((B, T, Hq))
    l = np.zeros((B, T, Hq))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            s = q[b, :, h].astype(np.float64) @ k[b, :, g].astype(np.float64).T / math.sqrt(D)
            for i in range(T):
                lo = max(0, i - W + 1) if W > 0 else 0
                row = s[i, lo:i + 1]
                m[b, i, h] = row.max()
                p = np.exp(row - row.max())
                l[b, i, h] = p.sum()
                pq = np.clip(np.rint(p * 127), 0, 127)
                o[b, i, h] = pq @ vh[b, lo:i + 1, g] / (127 * p.sum())
    return o, m, l


@pytest.mark.parametrize("W", [0, 1, 5, 64, 100])
def test_forward_matches_float64_attention(orc, W):
    B, T, Hq, Hkv, D = 2, 150, 4, 2, 128
    q, k, vq = _case(W, B, T, Hq, Hkv, D)
    s_v = 0.0123
    o, m, l = orc.attn_fwd(q, k, vq, s_v, W)
    ro, rm, rl = _ref_fwd(q, k, vq, s_v, W)
    assert np.allclose(m, rm, rtol=2e-6, atol=2e-6)
    assert np.allclose(l, rl, rtol=2e-5)
    # two P codes off by one (rounding-boundary cases) at most, plus rounding
    tol = 2 * 127 * s_v / (127 * rl[..., None]) + 1e-5 * np.abs(ro)
    assert np.all(np.abs(o - ro) <= tol)


def test_one_key_window_is_exact(orc):
    q, k, vq = _case(1, 1, 80, 4, 4, 128)
    o, m, l = orc.attn_fwd(q, k, vq, 2.0 ** -5, 1)
    assert np.all(l == 1.0)
    assert np.array_equal(o, vq.astype(np.float32) * np.float32(2.0 ** -5))


def test_masks(orc):
    B, T, Hq, Hkv, D = 1, 130, 4, 2, 128
    q, k, vq = _case(2, B, T, Hq, Hkv, D)
    for W in (0, 40):
        o, m, l = orc.attn_fwd(q, k, vq, 0.01, W)
        k2, v2 = k.copy(), vq.copy()
        k2[:, 100:] = 0.0          # the future of rows < 100
        v2[:, 100:] = 1
        o2, _, _ = orc.attn_fwd(q, k2, v2, 0.01, W)
        assert np.array_equal(o[:, :100], o2[:, :100])
        if W:
            k3, v3 = k.copy(), vq.copy()
            k3[:, :30] = 0.0       # outside the window of rows >= 69
            v3[:, :30] = 1
            o3, _, _ = orc.attn_fwd(q, k3, v3, 0.01, W)
            assert np.array_equal(o[:, 69:], o3[:, 69:])
            assert not np.array_equal(o[:, :69], o3[:, :69])


def test_gqa_head_mapping(orc):
    B, T, Hq, Hkv, D = 1, 20, 8, 2, 128
    q, k, _ = _case(3, B, T, Hq, Hkv, D)
    vq = np.zeros((B, T, Hkv, D), np.int8)
    vq[:, :, 0] = 10
    vq[:, :, 1] = 100
    o, _, _ = orc.attn_fwd(q, k, vq, 1.0, 0)
    # heads 0-3 read kv head 0, heads 4-7 kv head 1: o ~ the constant (P quantisation aside)
    assert np.allclose(o[:, :, :4], 10, rtol=0.05) and np.allclose(o[:, :, 4:], 100, rtol=0.05)


def _ref_bwd(q, k, vq, s_v, o, dout, W):
    """float64 straight-through gradients with the forward's own O in D_i."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    c = 1.0 / math.sqrt(D)
    vh = vq.astype(np.float64) * np.float64(np.float32(s_v))
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(k.shape)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            Q, K, V = q[b, :, h].astype(np.float64), k[b, :, g].astype(np.float64), vh[b, :, g]
            dO, O = dout[b, :, h].astype(np.float64), o[b, :, h].astype(np.float64)
            S = Q @ K.T * c
            mask = np.tril(np.ones((T, T), bool))
            if W > 0:
                mask &= ~np.tril(np.ones((T, T), bool), -W)
            S = np.where(mask, S, -np.inf)
            A = np.exp(S - S.max(1, keepdims=True))
            A /= A.sum(1, keepdims=True)
            dA = dO @ V.T
            Dr = (dO * O).sum(1, keepdims=True)
            dS = A * (dA - Dr)
            dq[b, :, h] = dS @ K * c
            dk[b, :, g] += dS.T @ Q * c
            dv[b, :, g] += A.T @ dO
    return dq, dk, dv


def test_float64_backward_reference_against_finite_differences():
    # pins the reference formulas themselves: L = sum(dO * O(q, k, v)) for
    # unquantised softmax attention, with O recomputed in float64
    rng = np.random.default_rng(9)
    T, D, Hq, Hkv = 5, 4, 2, 1
    q = rng.standard_normal((1, T, Hq, D))
    k = rng.standard_normal((1, T, Hkv, D))
    v = rng.standard_normal((1, T, Hkv, D))
    dO = rng.standard_normal((1, T, Hq, D))

    def fwd(q, k, v):
        o = np.zeros((1, T, Hq, D))
        for h in range(Hq):
            S = q[0, :, h] @ k[0, :, 0].T / math.sqrt(D)
            S = np.where(np.tril(np.ones((T, T), bool)), S, -np.inf)
            A = np.exp(S - S.max(1, keepdims=True))
            A /= A.sum(1, keepdims=True)
            o[0, :, h] = A @ v[0, :, 0]
        return o

    o = fwd(q, k, v)
    eps = 1e-6
    # the analytic gradient of L, compared with central differences
    c = 1.0 / math.sqrt(D)
    gq, gk, gv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(k.shape)
    for h in range(Hq):
        Q, K, V = q[0, :, h], k[0, :, 0], v[0, :, 0]
        S = np.where(np.tril(np.ones((T, T), bool)), Q @ K.T * c, -np.inf)
        A = np.exp(S - S.max(1, keepdims=True))
        A /= A.sum(1, keepdims=True)
        dS = A * (dO[0, :, h] @ V.T - (dO[0, :, h] * o[0, :, h]).sum(1, keepdims=True))
        gq[0, :, h] = dS @ K * c
        gk[0, :, 0] += dS.T @ Q * c
        gv[0, :, 0] += A.T @ dO[0, :, h]
    for x, g, which in ((q, gq, 0), (k, gk, 1), (v, gv, 2)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = [[q, k, v], [q, k, v]]
            args[0][which], args[1][which] = xp, xm
            fd = ((dO * fwd(*args[0])).sum() - (dO * fwd(*args[1])).sum()) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-6, (which, idx, fd, g[idx])
    # and _ref_bwd implements the same formulas (V enters through vq * s_v)
    vq_like = v                                       # float "codes", scale 1
    dq2, dk2, dv2 = _ref_bwd(q, k, vq_like, 1.0, o, dO, 0)
    assert np.allclose(dq2, gq) and np.allclose(dk2, gk) and np.allclose(dv2, gv)


@pytest.mark.parametrize("W", [0, 7, 64, 90])
def test_backward_matches_float64_reference(orc, W):
    B, T, Hq, Hkv, D = 1, 140, 4, 2, 128
    q, k, vq = _case(10 + W, B, T, Hq, Hkv, D)
    s_v = 0.02
    o, m, l = orc.attn_fwd(q, k, vq, s_v, W)
    dout = (np.random.default_rng(W).standard_normal(o.shape) * 1e-3).astype(np.float32)
    dq, dk, dv = orc.attn_bwd(q, k, vq, s_v, o, dout, m, l, W)
    rq, rk, rv = _ref_bwd(q, k, vq, s_v, o, dout, W)
    for got, ref, what in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        scale = np.abs(ref).max()
        assert np.abs(got - ref).max() <= 2e-5 * scale, (what, np.abs(got - ref).max(), scale)


def test_sampled_rows_equal_full(orc):
    B, T, Hq, Hkv, D, W = 2, 90, 4, 2, 128, 30
    q, k, vq = _case(5, B, T, Hq, Hkv, D)
    o, m, l = orc.attn_fwd(q, k, vq, 0.03, W)
    rows = np.array([0, 5, 77, B * T * Hq - 1])
    o2, m2, l2 = orc.attn_fwd_rows(q, k, vq, 0.03, W, rows)
    assert np.array_equal(o2, o.reshape(-1, D)[rows])
    assert np.array_equal(m2, m.reshape(-1)[rows]) and np.array_equal(l2, l.reshape(-1)[rows])
    dout = (np.random.default_rng(1).standard_normal(o.shape) * 1e-3).astype(np.float32)
    dq, dk, dv = orc.attn_bwd(q, k, vq, 0.03, o, dout, m, l, W)
    krows = np.array([0, 3, 100, B * T * Hkv - 1])
    dq2, dk2, dv2 = orc.attn_bwd_rows(q, k, vq, 0.03, o, dout, m, l, W, rows, krows)
    assert np.array_equal(dq2, dq.reshape(-1, D)[rows])
    assert np.array_equal(dk2, dk.reshape(-1, D)[krows])
    assert np.array_equal(dv2, dv.reshape(-1, D)[krows])
