"""GPU tests of the debug mode (repro_set_debug): with REPRO_DEBUG_CHECK_FINITE
a NaN or an infinity in any float input of a call makes the next
repro_device_check return REPRO_ERR_NONFINITE; finite inputs report nothing,
the mode is off by default, and the results do not change with it."""
import numpy as np
import pytest
import torch

import bitwise_reproducible_int8_gb300 as R
import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.fixture
def debug_on():
    torch.cuda.synchronize()
    assert R.repro_device_check() == R.REPRO_OK
    R.repro_set_debug(R.REPRO_DEBUG_CHECK_FINITE)
    yield
    R.repro_set_debug(0)
    torch.cuda.synchronize()
    R.repro_device_check()


def _quant(x):
    q = torch.empty(x.numel(), dtype=torch.int8, device="cuda")
    R.repro_quant_i8(x, G.scalar(0.05), q)
    return q


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
@pytest.mark.parametrize("n,where", [(1 << 16, 12345), (1001, 1000), (3, 2)])
def test_nonfinite_input_reported(debug_on, bad, n, where):
    x = np.random.default_rng(n).standard_normal(n).astype(np.float32)
    x[where] = bad
    _quant(G.dev(x))
    assert R.repro_device_check() == R.REPRO_ERR_NONFINITE
    assert R.repro_device_check() == R.REPRO_OK            # the report clears the word


def test_finite_inputs_report_nothing_and_results_match(debug_on):
    x = np.random.default_rng(3).standard_normal(70_001).astype(np.float32)
    q_on = G.host(_quant(G.dev(x)))
    assert R.repro_device_check() == R.REPRO_OK
    R.repro_set_debug(0)
    q_off = G.host(_quant(G.dev(x)))
    assert np.array_equal(q_on, q_off)


def test_off_by_default():
    x = np.full(4096, np.nan, np.float32)
    _quant(G.dev(x))
    assert R.repro_device_check() == R.REPRO_OK


def test_scales_and_each_call_class(debug_on):
    rng = np.random.default_rng(5)
    # a NaN scale of the quantiser
    x = G.dev(rng.standard_normal(64).astype(np.float32))
    q = torch.empty(64, dtype=torch.int8, device="cuda")
    R.repro_quant_i8(x, G.scalar(float("nan")), q)
    assert R.repro_device_check() == R.REPRO_ERR_NONFINITE
    # the backward's dY
    M, N, K = 64, 32, 48
    dy = rng.standard_normal((M, N)).astype(np.float32)
    dy[5, 7] = np.inf
    wq = G.dev(rng.integers(-127, 128, (N, K)).astype(np.int8))
    dx = torch.empty((M, K), device="cuda")
    R.repro_linear_bwd(G.dev(dy), None, wq, None, G.scalar(0.01), dx=dx, dw=None)
    assert R.repro_device_check() == R.REPRO_ERR_NONFINITE
    # a TreeFold part
    parts = [G.dev(rng.standard_normal(1000).astype(np.float32)) for _ in range(3)]
    parts[2][999] = float("nan")
    out = torch.empty(1000, device="cuda")
    R.repro_treefold(parts, out)
    assert R.repro_device_check() == R.REPRO_ERR_NONFINITE
    # the attention forward's keys
    B, T, Hq, Hkv = 1, 70, 2, 1
    q = G.dev(rng.standard_normal((B, T, Hq, 128)).astype(np.float32))
    k = rng.standard_normal((B, T, Hkv, 128)).astype(np.float32)
    k[0, 33, 0, 100] = -np.inf
    vq = G.dev(rng.integers(-127, 128, (B, T, Hkv, 128)).astype(np.int8))
    o = torch.empty((B, T, Hq, 128), device="cuda")
    m = torch.empty((B, T, Hq), device="cuda")
    l = torch.empty((B, T, Hq), device="cuda")
    R.repro_attn_fwd(q, G.dev(k), vq, G.scalar(0.01), o, m, l, 0)
    assert R.repro_device_check() == R.REPRO_ERR_NONFINITE
    # and the same calls on finite inputs report nothing
    R.repro_treefold(parts[:2], out)
    assert R.repro_device_check() == R.REPRO_OK
