"""GPU parity of the int8 P.V attention (repro_attn_fwd, through the C ABI)
against the oracle: o, the row maxima m and the row sums l bit for bit, on
ragged shapes, every mask kind and GQA grouping, and on sampled rows of the
full-size 4 x 4096-token, 16/4-head workload."""
import numpy as np
import pytest
import torch

import bitwise_reproducible_int8_gb300 as R
import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _exactness_checked():
    # the device's tensor-core exactness check runs first, so every cached
    # forward below takes the tensor-core P.V route (small caches cannot hold
    # the check's scratch and would otherwise take the CUDA-core route until a
    # larger call had run it)
    assert R.repro_selftest() == R.REPRO_OK

D = 128


def _case(seed, B, T, Hq, Hkv):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    vq = rng.integers(-127, 128, (B, T, Hkv, D)).astype(np.int8)
    s_v = np.float32(rng.uniform(0.005, 0.05))
    return q, k, vq, s_v


def gpu_attn_fwd(q, k, vq, s_v, W, cache=True, keep_cache=False):
    B, T, Hq, _ = q.shape
    o = torch.empty((B, T, Hq, D), device="cuda")
    m = torch.empty((B, T, Hq), device="cuda")
    l = torch.empty((B, T, Hq), device="cuda")
    ws = None
    if cache:
        ws = torch.empty(max(R.repro_attn_fwd_ws_bytes(B, T, Hq, W), 16), dtype=torch.uint8,
                         device="cuda")
    R.repro_attn_fwd(G.dev(q), G.dev(k), G.dev(vq), G.scalar(s_v), o, m, l, W, ws=ws)
    torch.cuda.synchronize()
    assert R.repro_device_check() == 0
    if keep_cache:
        return G.host(o), G.host(m), G.host(l), ws
    return G.host(o), G.host(m), G.host(l)


SHAPES = [(1, 1, 4, 2), (1, 5, 4, 2), (1, 63, 2, 2), (1, 64, 4, 1), (2, 65, 4, 2),
          (1, 130, 8, 2), (2, 200, 4, 4), (1, 257, 4, 2), (1, 600, 4, 2),
          (1, 130, 16, 2), (1, 70, 16, 1)]   # the last two: 8 and 16 query heads per kv head

# cached: the logit cache on, P.V on the tensor cores (the default); cached_dp4a:
# the cache on, P.V on CUDA cores (the launch-configuration hook's fwd_path 0);
# recomputed: no cache, P.V on CUDA cores.  T = 600 with W = 0 spans more than
# 512 keys, so the tensor-core route reads back two exact slices.
ROUTES = ["cached", "cached_dp4a", "recomputed"]


@pytest.fixture
def route(request):
    R.repro_set_launch_cfg(reset=True)
    if request.param == "cached_dp4a":
        R.repro_set_launch_cfg(fwd_path=0)
    yield request.param
    R.repro_set_launch_cfg(reset=True)


@pytest.mark.parametrize("route", ROUTES, indirect=True)
@pytest.mark.parametrize("W", [0, 1, 7, 64, 100])
@pytest.mark.parametrize("B,T,Hq,Hkv", SHAPES)
def test_attn_fwd_matches_oracle(orc, B, T, Hq, Hkv, W, route):
    q, k, vq, s_v = _case(B * 1000 + T * 10 + W, B, T, Hq, Hkv)
    o, m, l = gpu_attn_fwd(q, k, vq, s_v, W, route != "recomputed")
    ro, rm, rl = orc.attn_fwd(q, k, vq, s_v, W)
    G.assert_bits_equal(m, rm, f"m T={T} W={W}")
    G.assert_bits_equal(l, rl, f"l T={T} W={W}")
    G.assert_bits_equal(o, ro, f"o T={T} W={W}")


def test_attn_fwd_large_logits_and_zero_rows(orc):
    # logits far apart (many p flushed to 0, codes 0) and an all-zero query row
    q, k, vq, s_v = _case(7, 1, 150, 4, 2)
    q *= 8.0
    q[0, 10] = 0.0
    o, m, l = gpu_attn_fwd(q, k, vq, s_v, 0)
    ro, rm, rl = orc.attn_fwd(q, k, vq, s_v, 0)
    G.assert_bits_equal(m, rm, "m")
    G.assert_bits_equal(l, rl, "l")
    G.assert_bits_equal(o, ro, "o")


@pytest.mark.parametrize("W", [512, 0])
def test_attn_fwd_full_size_sampled(orc, W):
    # one micro-batch of the decoder: 4 sequences x 4096 tokens, 16 query and
    # 4 kv heads of 128; sliding window of 512 or full causal; both logit paths
    B, T, Hq, Hkv = 4, 4096, 16, 4
    q, k, vq, s_v = _case(100 + W, B, T, Hq, Hkv)
    o, m, l = gpu_attn_fwd(q, k, vq, s_v, W)
    o2, m2, l2 = gpu_attn_fwd(q, k, vq, s_v, W, cache=False)
    for x, y in ((o, o2), (m, m2), (l, l2)):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    rng = np.random.default_rng(W)
    nrow = B * T * Hq
    rows = np.unique(np.concatenate([rng.integers(0, nrow, 40), [0, 1, nrow - 1],
                                     [(3 * T + 4095) * Hq + 15, (2 * T + 511) * Hq + 3,
                                      (1 * T + 512) * Hq + 7]]))
    ro, rm, rl = orc.attn_fwd_rows(q, k, vq, s_v, W, rows)
    G.assert_bits_equal(o.reshape(-1, D)[rows], ro, "o rows")
    G.assert_bits_equal(m.reshape(-1)[rows], rm, "m rows")
    G.assert_bits_equal(l.reshape(-1)[rows], rl, "l rows")


def test_attn_fwd_repeatable():
    q, k, vq, s_v = _case(3, 2, 300, 8, 2)
    a = gpu_attn_fwd(q, k, vq, s_v, 100)
    b = gpu_attn_fwd(q, k, vq, s_v, 100)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=None):
    B, T, Hq, _ = q.shape
    Hkv = k.shape[2]
    dq = torch.empty((B, T, Hq, D), device="cuda")
    dk = torch.empty((B, T, Hkv, D), device="cuda")
    dv = torch.empty((B, T, Hkv, D), device="cuda")
    R.repro_attn_bwd(G.dev(q), G.dev(k), G.dev(vq), G.scalar(s_v), G.dev(o), G.dev(dout),
                     G.dev(m), G.dev(l), dq, dk, dv, W, fwd_ws=fwd_ws)
    torch.cuda.synchronize()
    assert R.repro_device_check() == 0
    return G.host(dq), G.host(dk), G.host(dv)


@pytest.mark.parametrize("logits", ["recomputed", "cached"])
@pytest.mark.parametrize("W", [0, 1, 7, 64, 100])
@pytest.mark.parametrize("B,T,Hq,Hkv", SHAPES)
def test_attn_bwd_matches_oracle(orc, B, T, Hq, Hkv, W, logits):
    q, k, vq, s_v = _case(B * 1000 + T * 10 + W + 7, B, T, Hq, Hkv)
    fwd_ws = None
    if logits == "cached":
        o, m, l, fwd_ws = gpu_attn_fwd(q, k, vq, s_v, W, keep_cache=True)
    else:
        o, m, l = orc.attn_fwd(q, k, vq, s_v, W)
    dout = (np.random.default_rng(T + W).standard_normal(o.shape) * 1e-3).astype(np.float32)
    dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=fwd_ws)
    rq, rk, rv = orc.attn_bwd(q, k, vq, s_v, o, dout, m, l, W)
    G.assert_bits_equal(dv, rv, f"dv T={T} W={W}")
    G.assert_bits_equal(dk, rk, f"dk T={T} W={W}")
    G.assert_bits_equal(dq, rq, f"dq T={T} W={W}")


@pytest.mark.parametrize("logits", ["recomputed", "cached"])
@pytest.mark.parametrize("W", [63, 65, 127, 128, 129, 192])
@pytest.mark.parametrize("B,T,Hq,Hkv", [(1, 300, 4, 2), (2, 257, 4, 1)])
def test_attn_bwd_windows_around_tile_multiples(orc, B, T, Hq, Hkv, W, logits):
    # a window edge just below, on and above a multiple of the 64-row tile
    # moves where each warp's fully valid middle range starts and ends
    q, k, vq, s_v = _case(B * 7 + T + W, B, T, Hq, Hkv)
    fwd_ws = None
    if logits == "cached":
        o, m, l, fwd_ws = gpu_attn_fwd(q, k, vq, s_v, W, keep_cache=True)
    else:
        o, m, l = orc.attn_fwd(q, k, vq, s_v, W)
    dout = (np.random.default_rng(W).standard_normal(o.shape) * 1e-3).astype(np.float32)
    dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=fwd_ws)
    rq, rk, rv = orc.attn_bwd(q, k, vq, s_v, o, dout, m, l, W)
    G.assert_bits_equal(dv, rv, f"dv T={T} W={W}")
    G.assert_bits_equal(dk, rk, f"dk T={T} W={W}")
    G.assert_bits_equal(dq, rq, f"dq T={T} W={W}")


@pytest.mark.parametrize("W", [0, 100])
def test_attn_bwd_fixed_point_magnitudes(orc, W):
    # key rows scaled by powers of two from 2^-40 to 2^12, so the dQ tile
    # partials T span the fixed-point conversion's ranges: |T 2^48| below 2^23
    # (rounded to the nearest integer, ties to even) and far above it (exact);
    # every dQ bit must still match the oracle's int64 sums
    B, T, Hq, Hkv = 1, 150, 2, 1
    q, k, vq, s_v = _case(171 + W, B, T, Hq, Hkv)
    q *= np.float32(2.0 ** -12)            # the logits stay moderate despite the scaling
    k *= np.exp2(np.arange(T) % 53 - 40).astype(np.float32)[None, :, None, None]
    o, m, l, fwd_ws = gpu_attn_fwd(q, k, vq, s_v, W, keep_cache=True)
    dout = np.random.default_rng(17).standard_normal(o.shape).astype(np.float32)
    rq, rk, rv = orc.attn_bwd(q, k, vq, s_v, o, dout, m, l, W)
    assert np.abs(rq).max() > 1.0 and np.abs(rq[rq != 0]).min() < 2.0 ** -30
    for fws in (fwd_ws, None):
        dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=fws)
        G.assert_bits_equal(dq, rq, "dq")
        G.assert_bits_equal(dk, rk, "dk")
        G.assert_bits_equal(dv, rv, "dv")


@pytest.mark.parametrize("cache", [True, False])
@pytest.mark.parametrize("W", [0, 100])
def test_attn_fwd_nan_keys(orc, W, cache):
    # a NaN in key rows 0 and 140 makes those keys' logits NaN for every query:
    # the row maximum passes over them (and is -inf for row 0, whose only key
    # is key 0); l and o are NaN exactly where a row sees one of those keys
    # and bit-identical to the oracle elsewhere
    B, T, Hq, Hkv = 1, 150, 2, 1
    q, k, vq, s_v = _case(404 + W, B, T, Hq, Hkv)
    k[0, 0, 0, 3] = np.nan
    k[0, 140, 0, 7] = np.nan
    o, m, l = gpu_attn_fwd(q, k, vq, s_v, W, cache=cache)
    ro, rm, rl = orc.attn_fwd(q, k, vq, s_v, W)
    assert np.isfinite(rm[0, 1:]).all() and np.all(rm[0, 0] == -np.inf)
    G.assert_bits_equal(m, rm, "m")
    for got, exp, what in ((l, rl, "l"), (o, ro, "o")):
        nan = np.isnan(exp)
        assert np.array_equal(np.isnan(got), nan), what
        G.assert_bits_equal(np.where(nan, 0, got).astype(np.float32),
                            np.where(nan, 0, exp).astype(np.float32), what)
    if W:
        assert not np.isnan(rl[0, 100:140]).any()   # rows that see neither key stay finite


@pytest.mark.parametrize("W", [0, 100])
def test_attn_bwd_fixed_point_saturation_and_nan(orc, W):
    # dQ partials beyond the fixed point's range: every third key row scaled
    # by 2^24 (q scaled down so the logits stay moderate), so tile partials
    # reach |T 2^48| >= 2^63 and saturate, and a row's saturated partials of
    # one sign wrap its int64 sum; one dO element is infinite, so that row's
    # dS and dQ partials are NaN and convert to 0.  dQ matches the oracle bit
    # for bit on both routes; dK and dV, which carry the NaNs, are NaN in the
    # same places and bit-identical elsewhere
    B, T, Hq, Hkv = 1, 200, 2, 1
    q, k, vq, s_v = _case(303 + W, B, T, Hq, Hkv)
    q *= np.float32(2.0 ** -24)
    k[:, ::3] *= np.float32(2.0 ** 24)
    o, m, l, fwd_ws = gpu_attn_fwd(q, k, vq, s_v, W, keep_cache=True)
    dout = np.random.default_rng(29).standard_normal(o.shape).astype(np.float32)
    dout[0, 137, 1, 5] = np.inf
    rq, rk, rv = orc.attn_bwd(q, k, vq, s_v, o, dout, m, l, W)
    assert np.all(rq[0, 137, 1] == 0) and np.isfinite(rq).all()
    with np.errstate(over="ignore", invalid="ignore"):
        big = np.abs(rq.astype(np.float64)) * 2.0 ** 48 / (1.0 / np.sqrt(128.0))
    assert (big > 2.0 ** 60).any()            # saturated or wrapped sums are present
    assert np.isnan(rk).any()
    for fws in (fwd_ws, None):
        dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=fws)
        G.assert_bits_equal(dq, rq, "dq")
        for got, exp, what in ((dk, rk, "dk"), (dv, rv, "dv")):
            nan = np.isnan(exp)
            assert np.array_equal(np.isnan(got), nan), what
            G.assert_bits_equal(np.where(nan, 0, got).astype(np.float32),
                                np.where(nan, 0, exp).astype(np.float32), what)


@pytest.mark.parametrize("W", [0, 100])
def test_attn_bwd_underflowing_probabilities(orc, W):
    # logits spread over hundreds: most p underflow to 0, so a and dS are
    # exact zeros and many backward terms are signed zeros, which the canonical
    # sums must keep with their signs
    B, T, Hq, Hkv = 1, 200, 4, 2
    q, k, vq, s_v = _case(91 + W, B, T, Hq, Hkv)
    q *= np.float32(40.0)
    o, m, l, fwd_ws = gpu_attn_fwd(q, k, vq, s_v, W, keep_cache=True)
    ro, rm, rl = orc.attn_fwd(q, k, vq, s_v, W)
    G.assert_bits_equal(o, ro, "o")
    dout = (np.random.default_rng(5).standard_normal(o.shape) * 1e-3).astype(np.float32)
    rq, rk, rv = orc.attn_bwd(q, k, vq, s_v, o, dout, m, l, W)
    for fws in (fwd_ws, None):
        dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=fws)
        G.assert_bits_equal(dv, rv, "dv")
        G.assert_bits_equal(dk, rk, "dk")
        G.assert_bits_equal(dq, rq, "dq")
    # the regime is real: many valid pairs sit far below their row maximum,
    # where e^(s - m) is an exact 0 in binary32 (checked in float64 here)
    g = np.arange(Hq) // (Hq // Hkv)
    s = np.einsum("bthd,bjhd->bhtj", q.astype(np.float64), k[:, :, g].astype(np.float64))
    s /= np.sqrt(128.0)
    t, j = np.arange(T)[:, None], np.arange(T)[None, :]
    valid = (j <= t) & ((W == 0) | (t - j < W))
    s = np.where(valid, s, -np.inf)
    below = (s - s.max(axis=-1, keepdims=True)) < -110.0
    assert below[..., valid].mean() > 0.3


@pytest.mark.parametrize("W", [0, 100])
def test_attn_bwd_row_sums_around_the_quotient_range(orc, W):
    # a = p (/) l is formed by correction when l is in [2^-30, 2^30) and by a
    # division otherwise (csrc/k_attn.cuh); a thread holds eight consecutive
    # rows, so l is changed per aligned group of eight rows: unchanged, scaled
    # out of the range both ways, at both ends of it (kept: 2^-30 and the
    # float below 2^30; divided: 2^30), and a group with a zero, a negative
    # and a NaN l.  Both backward routes match the oracle
    B, T, Hq, Hkv = 1, 200, 4, 2
    q, k, vq, s_v = _case(606 + W, B, T, Hq, Hkv)
    o, m, l, fwd_ws = gpu_attn_fwd(q, k, vq, s_v, W, keep_cache=True)
    l = l.copy()
    below_2_30 = np.nextafter(np.float32(2.0 ** 30), np.float32(0))
    for t in range(T):
        g = (t // 8) % 8
        if g == 1:
            l[0, t] *= np.float32(2.0 ** 40)
        elif g == 2:
            l[0, t] *= np.float32(2.0 ** -40)
        elif g == 3:
            l[0, t] = np.float32(2.0 ** -30)
        elif g == 4:
            l[0, t] = below_2_30
        elif g == 5:
            l[0, t] = np.float32(2.0 ** 30)
        elif g == 6 and t % 8 == 0:
            l[0, t] = 0.0
        elif g == 6 and t % 8 == 1:
            l[0, t] = -l[0, t]
        elif g == 6 and t % 8 == 2:
            l[0, t] = np.nan
    dout = (np.random.default_rng(61).standard_normal(o.shape) * 1e-3).astype(np.float32)
    rq, rk, rv = orc.attn_bwd(q, k, vq, s_v, o, dout, m, l, W)
    for fws in (fwd_ws, None):
        dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=fws)
        G.assert_bits_equal(dq, rq, "dq")
        for got, exp, what in ((dk, rk, "dk"), (dv, rv, "dv")):
            nan = np.isnan(exp)
            assert np.array_equal(np.isnan(got), nan), what
            G.assert_bits_equal(np.where(nan, 0, got).astype(np.float32),
                                np.where(nan, 0, exp).astype(np.float32), what)


@pytest.mark.parametrize("W", [512, 0])
def test_attn_bwd_full_size_sampled(orc, W):
    B, T, Hq, Hkv = 4, 4096, 16, 4
    q, k, vq, s_v = _case(200 + W, B, T, Hq, Hkv)
    o, m, l, fws = gpu_attn_fwd(q, k, vq, s_v, W, keep_cache=True)   # forward parity: above
    dout = (np.random.default_rng(W + 1).standard_normal(o.shape) * 1e-3).astype(np.float32)
    dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=fws)
    dq2, dk2, dv2 = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W)
    for x, y in ((dq, dq2), (dk, dk2), (dv, dv2)):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    rng = np.random.default_rng(W + 2)
    qrows = np.unique(np.concatenate([rng.integers(0, B * T * Hq, 24), [0, B * T * Hq - 1,
                                      (2 * T + 700) * Hq + 5]]))
    krows = np.unique(np.concatenate([rng.integers(0, B * T * Hkv, 24), [0, B * T * Hkv - 1,
                                      (1 * T + 4095) * Hkv + 2, (3 * T + 63) * Hkv + 1]]))
    rq, rk, rv = orc.attn_bwd_rows(q, k, vq, s_v, o, dout, m, l, W, qrows, krows)
    G.assert_bits_equal(dq.reshape(-1, D)[qrows], rq, "dq rows")
    G.assert_bits_equal(dk.reshape(-1, D)[krows], rk, "dk rows")
    G.assert_bits_equal(dv.reshape(-1, D)[krows], rv, "dv rows")


@pytest.mark.parametrize("W", [512, 0])
def test_attn_full_size_whole_tile_bands(orc, W):
    # every element of whole 64-row query tiles (o, m, l, dQ) and whole
    # 64-key tiles (dK, dV) at full size, on the bench's launch configuration
    # (cached forward, tensor-core P.V, cached backward): the first tile of a
    # sequence (truncated windows), the tile where the window first fills, and
    # the last tile, each in another sequence and head
    B, T, Hq, Hkv = 4, 4096, 16, 4
    q, k, vq, s_v = _case(300 + W, B, T, Hq, Hkv)
    o, m, l, fws = gpu_attn_fwd(q, k, vq, s_v, W, keep_cache=True)
    dout = (np.random.default_rng(W + 3).standard_normal(o.shape) * 1e-3).astype(np.float32)
    dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, W, fwd_ws=fws)
    i = np.arange(64)
    qrows = np.concatenate([(0 * T + i) * Hq + 0, (1 * T + 448 + i) * Hq + 7,
                            (3 * T + T - 64 + i) * Hq + 15])
    krows = np.concatenate([(0 * T + i) * Hkv + 0, (2 * T + 2048 + i) * Hkv + 3,
                            (3 * T + T - 64 + i) * Hkv + 1])
    ro, rm, rl = orc.attn_fwd_rows(q, k, vq, s_v, W, qrows)
    G.assert_bits_equal(o.reshape(-1, D)[qrows], ro, "o bands")
    G.assert_bits_equal(m.reshape(-1)[qrows], rm, "m bands")
    G.assert_bits_equal(l.reshape(-1)[qrows], rl, "l bands")
    rq, rk, rv = orc.attn_bwd_rows(q, k, vq, s_v, o, dout, m, l, W, qrows, krows)
    G.assert_bits_equal(dq.reshape(-1, D)[qrows], rq, "dq bands")
    G.assert_bits_equal(dk.reshape(-1, D)[krows], rk, "dk bands")
    G.assert_bits_equal(dv.reshape(-1, D)[krows], rv, "dv bands")


def test_attn_bwd_repeatable():
    q, k, vq, s_v = _case(4, 2, 300, 8, 2)
    o, m, l = gpu_attn_fwd(q, k, vq, s_v, 100)
    dout = (np.random.default_rng(0).standard_normal(o.shape) * 1e-3).astype(np.float32)
    a = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, 100)
    b = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, 100)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_attn_at_the_maximum_length(orc):
    # T = 131,072 is the longest sequence for which the exact int32 P.V sum
    # (at most 127 * 127 * T) fits; one head, full causal, sampled rows
    B, T, Hq, Hkv = 1, 131072, 1, 1
    q, k, vq, s_v = _case(131072, B, T, Hq, Hkv)
    vq[:] = 127                                  # the largest codes
    o, m, l = gpu_attn_fwd(q, k, vq, s_v, 0, cache=False)   # the cache would be 34 GB
    rows = np.array([0, 1, 4095, 65536, T - 2, T - 1])
    ro, rm, rl = orc.attn_fwd_rows(q, k, vq, s_v, 0, rows)
    G.assert_bits_equal(o.reshape(-1, D)[rows], ro, "o rows")
    G.assert_bits_equal(m.reshape(-1)[rows], rm, "m rows")
    G.assert_bits_equal(l.reshape(-1)[rows], rl, "l rows")
    dout = (np.random.default_rng(1).standard_normal(o.shape) * 1e-3).astype(np.float32)
    dq, dk, dv = gpu_attn_bwd(q, k, vq, s_v, o, dout, m, l, 0)
    krows = np.array([0, 1, T - 1])
    rq, rk, rv = orc.attn_bwd_rows(q, k, vq, s_v, o, dout, m, l, 0, rows, krows)
    G.assert_bits_equal(dq.reshape(-1, D)[rows], rq, "dq rows")
    G.assert_bits_equal(dk.reshape(-1, D)[krows], rk, "dk rows")
    G.assert_bits_equal(dv.reshape(-1, D)[krows], rv, "dv rows")


def test_attn_fwd_gate_falls_back_to_dp4a(orc):
    # with the forward's exactness check reported failed (test hook), the
    # cached forward computes P.V on CUDA cores: same bits, failure reported
    q, k, vq, s_v = _case(77, 1, 600, 4, 2)
    R.repro_set_launch_cfg(fwd_selftest=1)
    try:
        B, T, Hq, _ = q.shape
        o = torch.empty((B, T, Hq, D), device="cuda")
        m = torch.empty((B, T, Hq), device="cuda")
        l = torch.empty((B, T, Hq), device="cuda")
        ws = torch.empty(R.repro_attn_fwd_ws_bytes(B, T, Hq, 0), dtype=torch.uint8, device="cuda")
        R.repro_attn_fwd(G.dev(q), G.dev(k), G.dev(vq), G.scalar(s_v), o, m, l, 0, ws=ws)
        assert R.repro_device_check() == -9        # the failed check, reported once
        assert R.repro_device_check() == 0
    finally:
        R.repro_set_launch_cfg(reset=True)
    ro, rm, rl = orc.attn_fwd(q, k, vq, s_v, 0)
    G.assert_bits_equal(G.host(o), ro, "o")
    G.assert_bits_equal(G.host(l), rl, "l")
