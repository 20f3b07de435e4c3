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

D = 128


def _case(seed, B, T, Hq, Hkv):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    vq = rng.integers(-127, 128, (B, T, Hkv, D)).astype(np.int8)
    s_v = np.float32(rng.uniform(0.005, 0.05))
    return q, k, vq, s_v


def gpu_attn_fwd(q, k, vq, s_v, W):
    B, T, Hq, _ = q.shape
    o = torch.empty((B, T, Hq, D), device="cuda")
    m = torch.empty((B, T, Hq), device="cuda")
    l = torch.empty((B, T, Hq), device="cuda")
    R.repro_attn_fwd(G.dev(q), G.dev(k), G.dev(vq), G.scalar(s_v), o, m, l, W)
    torch.cuda.synchronize()
    assert R.repro_device_check() == 0
    return G.host(o), G.host(m), G.host(l)


SHAPES = [(1, 1, 4, 2), (1, 5, 4, 2), (1, 63, 2, 2), (1, 64, 4, 1), (2, 65, 4, 2),
          (1, 130, 8, 2), (2, 200, 4, 4), (1, 257, 4, 2)]


@pytest.mark.parametrize("W", [0, 1, 7, 64, 100])
@pytest.mark.parametrize("B,T,Hq,Hkv", SHAPES)
def test_attn_fwd_matches_oracle(orc, B, T, Hq, Hkv, W):
    q, k, vq, s_v = _case(B * 1000 + T * 10 + W, B, T, Hq, Hkv)
    o, m, l = gpu_attn_fwd(q, k, vq, s_v, W)
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
    # 4 kv heads of 128; sliding window of 512 or full causal
    B, T, Hq, Hkv = 4, 4096, 16, 4
    q, k, vq, s_v = _case(100 + W, B, T, Hq, Hkv)
    o, m, l = gpu_attn_fwd(q, k, vq, s_v, W)
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
