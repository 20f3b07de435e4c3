"""GPU parity of the optimiser step after TreeFold (global-norm clip + AdamW)
and of a two-step training loop on the tiny workload, against the oracle, bit
for bit."""
import numpy as np
import pytest

from bitwise_reproducible_int8_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import gpu_helpers as G  # noqa: E402
import bitwise_reproducible_int8_gb300 as R  # noqa: E402

HP = dict(lr=4.5e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0)


@pytest.fixture(autouse=True)
def _default_cfg():
    R.repro_set_launch_cfg(reset=True)
    yield
    R.repro_set_launch_cfg(reset=True)


def gpu_sumsq(g):
    out = torch.empty(1, device="cuda")
    R.repro_sumsq(G.dev(g), out)
    return G.host(out)[0]


@pytest.mark.parametrize("n", [1, 3, 64, 65, 1000, 300_001, 45_088_768])
def test_sumsq(orc, n):
    rng = np.random.default_rng(n % 1000)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[:min(n, 3)] = np.array([1e-40, -0.0, 3e-20], np.float32)[:min(n, 3)]
    G.assert_bits_equal(np.float32(gpu_sumsq(g)), np.float32(orc.sumsq(g)), f"sumsq n={n}")


@pytest.mark.parametrize("blk", [0, 3, 7, 10])
def test_sumsq_launch_invariance(orc, blk):
    rng = np.random.default_rng(5)
    g = (rng.standard_normal(200_003) * 1e-2).astype(np.float32)
    R.repro_set_launch_cfg(reduce_block_log2=blk)
    G.assert_bits_equal(np.float32(gpu_sumsq(g)), np.float32(orc.sumsq(g)), f"block 2^{blk}")


def _adamw_case(orc, n, t, hp, gscale, seed):
    rng = np.random.default_rng(seed)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3 * gscale).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-6 * gscale * gscale).astype(np.float32)
    g = (rng.standard_normal(n) * 0.03 * gscale).astype(np.float32)
    if n >= 4:
        p[:4] = [1e-40, -0.0, 0.0, 2.0 ** -10]
        g[:4] = [0.0, 1e-40, -1e-3, 5.0]
    s_ref = orc.sumsq(g)
    p_ref, m_ref, v_ref = orc.adamw_step(p, m, v, g, s_ref, t, **hp)
    tp, tm, tv, tg = G.dev(p), G.dev(m), G.dev(v), G.dev(g)
    ts = torch.empty(1, device="cuda")
    R.repro_sumsq(tg, ts)
    R.repro_adamw_step(tp, tm, tv, tg, ts, t, **hp)
    G.assert_bits_equal(G.host(ts), np.float32([s_ref]), "sumsq")
    G.assert_bits_equal(G.host(tp), p_ref, "p")
    G.assert_bits_equal(G.host(tm), m_ref, "m")
    G.assert_bits_equal(G.host(tv), v_ref, "v")


@pytest.mark.parametrize("t", [1, 2, 667, 100_000])
@pytest.mark.parametrize("gscale", [1e-4, 1.0, 30.0])
def test_adamw(orc, t, gscale):
    _adamw_case(orc, 10_003, t, HP, gscale, seed=t)


@pytest.mark.parametrize("hp", [dict(HP, lr=0.0), dict(HP, weight_decay=0.0),
                                dict(HP, max_norm=1e-3), dict(HP, beta1=0.0, beta2=0.0)])
def test_adamw_special_hparams(orc, hp):
    _adamw_case(orc, 4096, 3, hp, 1.0, seed=11)


def test_adamw_full_gradient_size(orc):
    # the block workload's flat gradient: 45,088,768 parameters
    _adamw_case(orc, 45_088_768, 1, HP, 1e-2, seed=99)


def test_two_training_steps_tiny(orc):
    """Re-pin and quantise W, forward, backward, accumulate two micro-batches,
    TreeFold over R = 4, clip + AdamW -- twice, the second step on the
    updated weights -- on the GPU and in the oracle."""
    wl = inputs.WORKLOADS["tiny"]
    W0 = inputs.weight(wl, 0)
    mbs = [(inputs.activation(wl, 0, j), inputs.upstream_grad(wl, 0, j)) for j in range(2)]
    noise = [inputs.replica_noise(wl, r, W0.size).reshape(W0.shape) for r in range(1, 4)]

    # oracle; the per-step state hash log covers (W, m, v) after each update
    W, m, v = W0.copy(), np.zeros_like(W0), np.zeros_like(W0)
    log = []
    for t in (1, 2):
        s_w = orc.wscale(W, 0)
        wq = orc.quant_i8(W, s_w)
        acc = None
        for X, dY in mbs:
            s_x = orc.wscale(X, 1)
            xq = orc.quant_i8(X, s_x)
            orc.linear_fwd(xq, wq, s_x, s_w)
            dw = orc.linear_bwd_dw(dY, xq, s_x)
            acc = dw if acc is None else orc.grad_accum(acc, dw)
        parts = [acc] + [orc.grad_accum(acc, nz) for nz in noise]
        g = orc.treefold(parts).reshape(W.shape)
        W, m, v = orc.adamw_step(W, m, v, g, orc.sumsq(g), t, **HP)
        log.append(orc.state_hash([W.tobytes(), m.tobytes(), v.tobytes()]))

    # GPU through the C ABI
    tW, tm, tv = G.dev(W0), torch.zeros(W0.shape, device="cuda"), torch.zeros(W0.shape, device="cuda")
    sw, sx, ss = (torch.empty(1, device="cuda") for _ in range(3))
    wq_t = torch.empty(W0.shape, dtype=torch.int8, device="cuda")
    xq_t = torch.empty(mbs[0][0].shape, dtype=torch.int8, device="cuda")
    y_t = torch.empty((wl.tokens, W0.shape[0]), device="cuda")
    gacc = torch.empty(W0.shape, device="cuda")
    tf = torch.empty(W0.shape, device="cuda")
    for t in (1, 2):
        R.repro_wscale(tW, 0, sw)
        R.repro_quant_i8(tW, sw, wq_t)
        for j, (X, dY) in enumerate(mbs):
            tX, tdY = G.dev(X), G.dev(dY)
            R.repro_wscale(tX, 1, sx)
            R.repro_quant_i8(tX, sx, xq_t)
            R.repro_linear_fwd(xq_t, wq_t, sx, sw, y_t)
            R.repro_linear_bwd(tdY, xq_t, None, sx, None, None, gacc, accumulate=j > 0)
        reps = [gacc]
        for nz in noise:
            r = gacc.clone()
            R.repro_grad_accum(r, G.dev(nz))
            reps.append(r)
        R.repro_treefold(reps, tf)
        R.repro_sumsq(tf, ss)
        R.repro_adamw_step(tW, tm, tv, tf, ss, t, **HP)
        digest = torch.zeros(32, dtype=torch.uint8, device="cuda")
        R.repro_state_hash([tW, tm, tv], digest)
        assert bytes(G.host(digest)) == log[t - 1], f"state hash after step {t}"
    assert log[0] != log[1]
    G.assert_bits_equal(G.host(tW), W, "W after two steps")
    G.assert_bits_equal(G.host(tm), m, "m after two steps")
    G.assert_bits_equal(G.host(tv), v, "v after two steps")
