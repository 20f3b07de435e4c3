"""Pins the oracle's int8 forward and fp32 backward of the QAT linear layer.

Forward: brute-force exact integer dot products with Python ints, then the two
dequantising multiplies rounded exactly (int8 QAT linears: Open-1B review,
onedev.kr/papers/92, section "How to use").  Backward: for reductions of at
most 64 terms the canonical order is the textbook sequential dot product of the
rounded products; longer reductions are pinned by hand-built products whose
canonical sum is known (a wrong chunk size, order, index or transposed operand
gives another value) and by the error bound against the exact sum.
"""
import functools
import math
from fractions import Fraction

import numpy as np
import pytest

import exact_binary32 as E
from golden_io import f32_to_bits


def _q(rng, shape):
    return rng.integers(-127, 128, shape).astype(np.int8)


def _emu_fwd(xq, wq, s_x, s_w, m, n):
    acc = sum(int(a) * int(b) for a, b in zip(xq[m], wq[n]))
    return E.mul(E.mul(E.i2f(acc), E.f(s_x)), E.f(s_w))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (5, 7, 37), (8, 3, 130)])
def test_forward_brute_force(orc, M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    xq, wq = _q(rng, (M, K)), _q(rng, (N, K))
    s_x, s_w = float(np.float32(0.0371)), float(np.float32(0.00284))
    y = orc.linear_fwd(xq, wq, s_x, s_w)
    for m in range(M):
        for n in range(N):
            assert f32_to_bits(y[m, n]) == _emu_fwd(xq, wq, s_x, s_w, m, n).bits()


def test_forward_adversarial_magnitudes(orc):
    # all codes at +-127: |acc| = 16129 K crosses 2^24, where i2f must round
    for K in [1, 1040, 1041, 2048, 5632]:
        xq = np.full((2, K), 127, dtype=np.int8)
        wq = np.stack([np.full(K, 127, np.int8), np.full(K, -127, np.int8)])
        xq[1, ::2] = -127
        s_x, s_w = 1.0, float(np.float32(3.0))
        y = orc.linear_fwd(xq, wq, s_x, s_w)
        for m in range(2):
            for n in range(2):
                assert orc.int_dot(xq, wq, m, n) == int(xq[m].astype(np.int64) @ wq[n].astype(np.int64))
                assert f32_to_bits(y[m, n]) == _emu_fwd(xq, wq, s_x, s_w, m, n).bits()


def test_forward_sampled_matches_full(orc):
    rng = np.random.default_rng(9)
    xq, wq = _q(rng, (33, 70)), _q(rng, (17, 70))
    y = orc.linear_fwd(xq, wq, 0.5, 0.25)
    im, jn = rng.integers(0, 33, 50), rng.integers(0, 17, 50)
    assert np.array_equal(orc.linear_fwd_at(xq, wq, 0.5, 0.25, im, jn).view(np.uint32),
                          y[im, jn].view(np.uint32))


def _dequant(q, s):
    return E.mul(E.i2f(int(q)), E.f(s))


def _emu_seq_dot(us, vs):
    prods = [E.mul(u, v) for u, v in zip(us, vs)]
    return functools.reduce(E.add, prods[1:], prods[0])


@pytest.mark.parametrize("M,N,K", [(4, 1, 3), (6, 17, 5), (9, 64, 11), (64, 40, 3)])
def test_backward_short_reductions_are_textbook_dots(orc, M, N, K):
    # dX reduces over N, dW over M; both <= 64 here -> plain left-to-right dots
    rng = np.random.default_rng(M + N + K)
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    xq, wq = _q(rng, (M, K)), _q(rng, (N, K))
    s_x, s_w = float(np.float32(0.031)), float(np.float32(0.0027))
    dx = orc.linear_bwd_dx(dy, wq, s_w)
    dw = orc.linear_bwd_dw(dy, xq, s_x)
    for m in range(M):
        for k in range(K):
            ref = _emu_seq_dot([E.f(float(dy[m, n])) for n in range(N)],
                               [_dequant(wq[n, k], s_w) for n in range(N)])
            assert f32_to_bits(dx[m, k]) == ref.bits(), ("dx", m, k)
    for n in range(N):
        for k in range(K):
            ref = _emu_seq_dot([E.f(float(dy[m, n])) for m in range(M)],
                               [_dequant(xq[m, k], s_x) for m in range(M)])
            assert f32_to_bits(dw[n, k]) == ref.bits(), ("dw", n, k)


def test_backward_discriminating_products(orc):
    # products [2^24, 1, 1, ...] (130 terms): chunks 2^24 | 64 | 2 -> 2^24+66.
    # Only output (m=1, k=2) of dX / (n=1, k=2) of dW carries the pattern, so a
    # transposed operand or a wrong index lands elsewhere.
    L = 130
    M, N, K = 3, L, 4
    dy = np.zeros((M, N), dtype=np.float32)
    dy[1, :] = 1.0
    dy[1, 0] = 2.0 ** 24
    wq = np.zeros((N, K), dtype=np.int8)
    wq[:, 2] = 1
    dx = orc.linear_bwd_dx(dy, wq, 1.0)
    assert dx[1, 2] == 2.0 ** 24 + 66
    assert np.all(dx[[0, 2], :] == 0) and np.all(dx[1, [0, 1, 3]] == 0)

    M, N, K = L, 3, 4
    dy = np.zeros((M, N), dtype=np.float32)
    dy[:, 1] = 1.0
    dy[0, 1] = 2.0 ** 24
    xq = np.zeros((M, K), dtype=np.int8)
    xq[:, 2] = 1
    dw = orc.linear_bwd_dw(dy, xq, 1.0)
    assert dw[1, 2] == 2.0 ** 24 + 66
    assert np.count_nonzero(dw) == 1


def test_backward_dequant_scale_is_applied_per_operand(orc):
    # W^ = q (x) s_w: with s_w = 2^-3 and q = 3 every product is dy * 0.375
    M, N, K = 2, 70, 1
    dy = np.full((M, N), 1.0, dtype=np.float32)
    wq = np.full((N, K), 3, dtype=np.int8)
    dx = orc.linear_bwd_dx(dy, wq, 0.125)
    assert np.all(dx == np.float32(70 * 0.375))


@pytest.mark.parametrize("L", [200, 1000, 3000])
def test_backward_error_bound(orc, L):
    rng = np.random.default_rng(L)
    dy = (rng.standard_normal((2, L)) * 1e-3).astype(np.float32)
    wq = _q(rng, (L, 3))
    s_w = float(np.float32(0.0028))
    dx = orc.linear_bwd_dx(dy, wq, s_w)
    C = (L + 63) // 64
    d = 63 + math.ceil(math.log2(C))
    u = Fraction(1, 2 ** 24)
    gamma = (d + 1) * u / (1 - (d + 1) * u)  # +1 for the rounded product
    for m in range(2):
        for k in range(3):
            what = [Fraction(float(dy[m, n])) * Fraction(_dequant(wq[n, k], s_w).to_float())
                    for n in range(L)]
            err = abs(Fraction(float(dx[m, k])) - sum(what))
            assert err <= gamma * sum(abs(t) for t in what)


def test_backward_sampled_matches_full(orc):
    rng = np.random.default_rng(12)
    M, N, K = 150, 140, 9
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    xq, wq = _q(rng, (M, K)), _q(rng, (N, K))
    dx = orc.linear_bwd_dx(dy, wq, 0.003)
    dw = orc.linear_bwd_dw(dy, xq, 0.04)
    i, j = rng.integers(0, M, 40), rng.integers(0, K, 40)
    assert np.array_equal(orc.linear_bwd_dx_at(dy, wq, 0.003, i, j).view(np.uint32),
                          dx[i, j].view(np.uint32))
    i = rng.integers(0, N, 40)
    assert np.array_equal(orc.linear_bwd_dw_at(dy, xq, 0.04, i, j).view(np.uint32),
                          dw[i, j].view(np.uint32))


def test_backward_empty_reduction_is_positive_zero(orc):
    dy = np.zeros((3, 0), dtype=np.float32)
    wq = np.zeros((0, 4), dtype=np.int8)
    dx = orc.linear_bwd_dx(dy, wq, 1.0)
    assert dx.shape == (3, 4) and np.all(dx.view(np.uint32) == 0)
