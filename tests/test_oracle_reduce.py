"""Pins the oracle's micro-batch accumulation and TreeFold.

TreeFold (Open-1B review, onedev.kr/papers/92, section "Premises and limits":
the replica all-reduce is replayed by combining partials in the pairing order
of the cluster's recursive-doubling all-reduce) is pinned by hand-worked cases,
by an independent message-passing simulation of recursive doubling with the
non-power-of-two pre-step of Thakur, Rabenseifner and Gropp (IJHPCA 2005), by
the textbook pairwise tree for R = 2^k, and by layout independence.
"""
import numpy as np
import pytest

import exact_binary32 as E
from golden_io import f32_to_bits, treefold_cases


def _add(a, b):
    return E.add(E.f(float(a)), E.f(float(b))).to_float()


def test_treefold_golden(orc):
    for vals, exp in treefold_cases():
        assert f32_to_bits(orc.treefold_one(vals)) == exp, (vals, hex(exp))


def _simulate_recursive_doubling(vals):
    """Message-passing simulation: each rank holds a buffer; returns every
    rank's final buffer."""
    R = len(vals)
    buf = [float(v) for v in vals]
    p2 = 1
    while p2 * 2 <= R:
        p2 *= 2
    rem = R - p2
    # pre-step: even rank 2i sends to 2i+1 and drops out
    active = {}
    for rank in range(R):
        if rank < 2 * rem:
            if rank % 2 == 1:
                buf[rank] = _add(buf[rank - 1], buf[rank])   # lower rank first
                active[rank // 2] = rank
        else:
            active[rank - rem] = rank
    mask = 1
    while mask < p2:
        new = dict()
        for nr, rank in active.items():
            partner = active[nr ^ mask]
            lo, hi = (rank, partner) if nr < (nr ^ mask) else (partner, rank)
            new[rank] = _add(buf[lo], buf[hi])
        for rank, v in new.items():
            buf[rank] = v
        mask *= 2
    # post-step: odd ranks send the result back to the even rank that left
    for rank in range(0, 2 * rem, 2):
        buf[rank] = buf[rank + 1]
    return buf


@pytest.mark.parametrize("R", list(range(1, 17)) + [31, 32, 33, 64])
def test_treefold_matches_message_passing_simulation(orc, R):
    rng = np.random.default_rng(R)
    for _ in range(20):
        vals = (rng.standard_normal(R) * 10.0 ** rng.integers(-4, 5, R)).astype(np.float32)
        sim = _simulate_recursive_doubling(vals)
        ranks = orc.treefold_all_ranks(vals)
        assert len(set(f32_to_bits(v) for v in sim)) == 1          # every rank agrees
        assert [f32_to_bits(v) for v in ranks] == [f32_to_bits(v) for v in sim]
        assert f32_to_bits(orc.treefold_one(vals)) == f32_to_bits(sim[0])


@pytest.mark.parametrize("R", [1, 2, 4, 8, 16, 32, 64])
def test_power_of_two_is_adjacent_pair_tree(orc, R):
    rng = np.random.default_rng(100 + R)
    vals = (rng.standard_normal(R) * 10.0 ** rng.integers(-4, 5, R)).astype(np.float32)
    level = [float(v) for v in vals]
    while len(level) > 1:
        level = [_add(level[i], level[i + 1]) for i in range(0, len(level), 2)]
    assert f32_to_bits(orc.treefold_one(vals)) == f32_to_bits(level[0])


def test_treefold_r5_differs_from_stride_tree(orc):
    vals = np.array([2.0 ** 24, 1, 1, 1, -2.0 ** 24], dtype=np.float32)
    stride = _add(_add(_add(vals[0], vals[1]), _add(vals[2], vals[3])), vals[4])
    assert stride == 2.0
    assert orc.treefold_one(vals) == 1.0


def test_treefold_layout_independence(orc):
    rng = np.random.default_rng(77)
    R, n = 6, 5000
    block = (rng.standard_normal((R, n)) * 1e-3).astype(np.float32)
    ref = orc.treefold([block[r] for r in range(R)])
    separate = [block[r].copy() for r in range(R)]
    rev_block = np.ascontiguousarray(block[::-1])           # reversed memory order
    reversed_layout = [rev_block[R - 1 - r] for r in range(R)]
    strided = np.ascontiguousarray(block.T)                  # interleaved, copied out
    from_strided = [np.ascontiguousarray(strided[:, r]) for r in range(R)]
    for parts in (separate, reversed_layout, from_strided):
        assert np.array_equal(orc.treefold(parts).view(np.uint32), ref.view(np.uint32))


def test_treefold_pair_swap_invariance_and_order_sensitivity(orc):
    vals = np.array([1e8, 1.0, -1e8, 1.0, 3.0, 0.5], dtype=np.float32)
    base = orc.treefold_one(vals)
    swapped = vals[[1, 0, 3, 2, 5, 4]]                       # within first-level pairs
    assert f32_to_bits(orc.treefold_one(swapped)) == f32_to_bits(base)
    cross = vals[[0, 2, 1, 3, 4, 5]]                         # across pairs
    assert f32_to_bits(orc.treefold_one(cross)) != f32_to_bits(base)


def test_treefold_r1_is_a_copy(orc):
    x = np.array([1e-40, -0.0, 3.5], dtype=np.float32)      # bits kept verbatim
    assert np.array_equal(orc.treefold([x]).view(np.uint32), x.view(np.uint32))


def test_grad_accum_is_elementwise_add(orc):
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(3000) * 1e-3).astype(np.float32)
    g = (rng.standard_normal(3000) * 1e-3).astype(np.float32)
    a[:3], g[:3] = [-0.0, 1e-40, 2.0 ** 24], [-0.0, 1.0, 1.0]
    out = orc.grad_accum(a, g)
    for i in range(a.size):
        assert f32_to_bits(out[i]) == f32_to_bits(_add(a[i], g[i]))


def test_grad_accum_order_matters(orc):
    # ((1e8 + 1) + -1e8) = 0 but ((1e8 + -1e8) + 1) = 1: the fixed micro-batch
    # order is observable
    acc = np.array([1e8], np.float32)
    g1, g2 = np.array([1.0], np.float32), np.array([-1e8], np.float32)
    assert orc.grad_accum(orc.grad_accum(acc, g1), g2)[0] == 0.0
    assert orc.grad_accum(orc.grad_accum(acc, g2), g1)[0] == 1.0


# ----------------------------------------------------------------- level 2

def test_running_sum_is_the_textbook_left_fold(orc):
    rng = np.random.default_rng(17)
    for S in [1, 2, 3, 8, 13]:
        parts = [(rng.standard_normal(257) * 10.0 ** rng.integers(-3, 4, 257)).astype(np.float32)
                 for _ in range(S)]
        parts[0][:2] = [1e-40, -0.0]
        got = orc.running_sum(parts)
        for i in range(257):
            acc = float(parts[0][i])          # first partial taken as it is
            for s in range(1, S):
                acc = _add(acc, parts[s][i])
            assert f32_to_bits(got[i]) == f32_to_bits(acc), (S, i)


def test_running_sum_equals_streaming_accumulation(orc):
    # one resident partial: acc = P0, then acc (+)= P_s in shard order
    rng = np.random.default_rng(18)
    parts = [(rng.standard_normal(1000) * 1e-3).astype(np.float32) for _ in range(8)]
    acc = parts[0].copy()
    for p in parts[1:]:
        acc = orc.grad_accum(acc, p)
    assert np.array_equal(orc.running_sum(parts).view(np.uint32), acc.view(np.uint32))


def test_running_sum_order_is_observable(orc):
    parts = [np.array([2.0 ** 24], np.float32), np.array([1.0], np.float32),
             np.array([1.0], np.float32), np.array([2.0], np.float32)]
    # ((2^24 + 1) + 1) + 2 = 2^24 + 2, but (2^24 + 2) + (1 + 1) order differs from a tree
    assert orc.running_sum(parts)[0] == 2.0 ** 24 + 2
    assert orc.running_sum(parts[::-1])[0] == 2.0 ** 24 + 4
