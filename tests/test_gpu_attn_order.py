"""GPU parity of the attention on the hand-worked order cases of
tests/golden/attn_order.txt: inputs on which another tile width, tile origin,
fold order or fixed-point placement gives other bits.  Every output of the
GPU forward / backward is compared bit for bit with the oracle, and the
case's own element with its hand-derived value."""
import numpy as np
import pytest
import torch

import bitwise_reproducible_int8_gb300 as R
import exact_binary32 as E
import gpu_helpers as G
from golden_io import attn_order_cases
from test_oracle_attn_order import _bits, _build, _c_bits, _canon_exact, exp_replay

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _exactness_checked():
    # the device's tensor-core exactness check runs first, so every cached
    # forward below takes the tensor-core P.V route (small caches cannot hold
    # the check's scratch and would otherwise take the CUDA-core route until a
    # larger call had run it)
    assert R.repro_selftest() == R.REPRO_OK


@pytest.mark.parametrize("case", list(attn_order_cases()), ids=lambda c: c["name"])
def test_gpu_attention_order_cases(orc, case):
    q, k, vq, dout, o = _build(case)
    T, W, Hq, Hkv = case["T"], case["W"], case["Hq"], case["Hkv"]
    row, col = case["row"], case["col"]
    expected = E.F32.from_bits(case["bits"])
    if case["times_c"]:
        expected = E.mul(expected, _c_bits())
    s_v = G.scalar(1.0)
    if case["kind"] in ("m", "l", "o"):
        ot = torch.empty((1, T, Hq, 128), device="cuda")
        mt = torch.empty((1, T, Hq), device="cuda")
        lt = torch.empty((1, T, Hq), device="cuda")
        R.repro_attn_fwd(G.dev(q), G.dev(k), G.dev(vq), s_v, ot, mt, lt, W)
        go, gm, gl = G.host(ot), G.host(mt), G.host(lt)
        ro, rm, rl = orc.attn_fwd(q, k, vq, 1.0, W)
        G.assert_bits_equal(go, ro, "o")
        G.assert_bits_equal(gm, rm, "m")
        G.assert_bits_equal(gl, rl, "l")
        got = {"m": gm.reshape(-1), "l": gl.reshape(-1), "o": go.reshape(-1, 128)[:, col]}[
            case["kind"]][row]
    else:
        m = np.zeros((1, T, Hq), np.float32)
        lsum = np.ones((1, T, Hq), np.float32)
        dq = torch.empty((1, T, Hq, 128), device="cuda")
        dk = torch.empty((1, T, Hkv, 128), device="cuda")
        dv = torch.empty((1, T, Hkv, 128), device="cuda")
        R.repro_attn_bwd(G.dev(q), G.dev(k), G.dev(vq), s_v, G.dev(o), G.dev(dout), G.dev(m),
                         G.dev(lsum), dq, dk, dv, W)
        gq, gk, gv = G.host(dq), G.host(dk), G.host(dv)
        rq, rk, rv = orc.attn_bwd(q, k, vq, 1.0, o, dout, m, lsum, W)
        G.assert_bits_equal(gq, rq, "dq")
        G.assert_bits_equal(gk, rk, "dk")
        G.assert_bits_equal(gv, rv, "dv")
        got = {"dq": gq, "dk": gk, "dv": gv}[case["kind"]].reshape(-1, 128)[row, col]
    assert R.repro_device_check() == 0
    assert _bits(got) == expected.bits(), (case["name"], hex(_bits(got)), hex(expected.bits()))


def test_gpu_row_sum_order_and_zero_maximum(orc):
    # as the oracle pins: key 0 at logit +0, keys 1..127 at RN(-192 c), so the
    # canonical row sum differs from a left fold; and all -0 logits give m = +0
    T = 128
    q = np.zeros((1, T, 2, 128), np.float32)
    k = np.zeros((1, T, 1, 128), np.float32)
    q[0, 127, 0, 0] = 1.0
    k[0, 1:, 0, 0] = -192.0
    k[0, :, 0, 1:] = -1.0          # head 1 (q = 0): every product -0, every logit -0
    vq = np.ones((1, T, 1, 128), np.int8)
    ot = torch.empty((1, T, 2, 128), device="cuda")
    mt = torch.empty((1, T, 2), device="cuda")
    lt = torch.empty((1, T, 2), device="cuda")
    R.repro_attn_fwd(G.dev(q), G.dev(k), G.dev(vq), G.scalar(1.0), ot, mt, lt, 0)
    go, gm, gl = G.host(ot), G.host(mt), G.host(lt)
    ro, rm, rl = orc.attn_fwd(q, k, vq, 1.0, 0)
    G.assert_bits_equal(gm, rm, "m")
    G.assert_bits_equal(gl, rl, "l")
    G.assert_bits_equal(go, ro, "o")
    s = E.mul(E.f(-192.0), _c_bits())
    p = E.F32.from_bits(exp_replay(s.to_float()))
    assert _bits(gl[0, 127, 0]) == _canon_exact([E.f(1.0)] + [p] * 127).bits()
    assert np.all(gm[0, :, 1].view(np.uint32) == 0)
