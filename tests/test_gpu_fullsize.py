"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times: one step of the hot-path runner, then every output checked
against the oracle -- in full where the oracle is O(n) (scales, int8 codes)
and at sampled positions (corners of tiles and chunk boundaries plus seeded
random ones) for the forward, dX, the accumulated dW and TreeFold, which the
oracle evaluates one element at a time from the same host inputs."""
import numpy as np
import pytest

from bitwise_reproducible_int8_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import gpu_helpers as G  # noqa: E402
import bitwise_reproducible_int8_gb300 as R  # noqa: E402
from bitwise_reproducible_int8_gb300 import step as S  # noqa: E402

NSAMP = 512


def _samples(rng, rows, cols):
    fixed_r = [0, 1, 63, 64, 65, rows // 2, rows - 65, rows - 64, rows - 1]
    fixed_c = [0, 3, 63, 64, cols // 2, cols - 64, cols - 1]
    r = [x for x in fixed_r if 0 <= x < rows]
    c = [x for x in fixed_c if 0 <= x < cols]
    rr = np.array([a for a in r for _ in c] + list(rng.integers(0, rows, NSAMP)), np.int64)
    cc = np.array([b for _ in r for b in c] + list(rng.integers(0, cols, NSAMP)), np.int64)
    return rr, cc


@pytest.mark.parametrize("name", ["attn_out", "gate_up", "down_accum", "block", "block_audit"])
def test_fullsize_sampled(orc, name):
    R.repro_set_launch_cfg(reset=True)
    wl = inputs.WORKLOADS[name]
    host = S.generate_host_inputs(wl)
    hp = S.HotPathStep(wl, host)
    hp.use_optimizer = False      # the weights stay the inputs the oracle sees
    st = torch.cuda.current_stream()
    if wl.replicas > 1 or wl.shards > 1:
        hp.prepare(st)
    hp.run(st)
    torch.cuda.synchronize()
    assert R.repro_device_check() == 0

    rng = np.random.default_rng(7)
    offs, _ = S.grad_offsets(wl)
    J = wl.microbatches
    G_flat_idx, G_oracle = [], []
    for i, lin in enumerate(wl.linears):
        W = host.W[i]
        s_w = orc.wscale(W, 0)
        G.assert_bits_equal(G.host(hp.s_w[i:i + 1]), np.float32([s_w]), f"{name}/{lin.name} s_w")
        wq = orc.quant_i8(W, s_w)
        G.assert_bits_equal(G.host(hp.Wq[i]), wq, f"{name}/{lin.name} Wq")
        n_idx, k_idx = _samples(rng, lin.n_out, lin.k_in)
        g = None
        for j in range(J):
            X, dY = host.X[i][j], host.dY[i][j]
            s_x = orc.wscale(X, 1)
            xq = orc.quant_i8(X, s_x)
            dw = orc.linear_bwd_dw_at(dY, xq, s_x, n_idx, k_idx)
            g = dw if g is None else orc.grad_accum(g, dw)
        # the last micro-batch's forward-side buffers are still resident
        G.assert_bits_equal(G.host(hp.s_x[i:i + 1]), np.float32([s_x]), f"{name}/{lin.name} s_x")
        G.assert_bits_equal(G.host(hp.Xq[i]), xq, f"{name}/{lin.name} Xq")
        m_idx, c_idx = _samples(rng, wl.tokens, lin.n_out)
        G.assert_bits_equal(G.host(hp.Y[i])[m_idx, c_idx],
                            orc.linear_fwd_at(xq, wq, s_x, s_w, m_idx, c_idx),
                            f"{name}/{lin.name} Y")
        m_idx, k2 = _samples(rng, wl.tokens, lin.k_in)
        G.assert_bits_equal(G.host(hp.dX[i])[m_idx, k2],
                            orc.linear_bwd_dx_at(dY, wq, s_w, m_idx, k2),
                            f"{name}/{lin.name} dX")
        G.assert_bits_equal(G.host(hp.Gv[i])[n_idx, k_idx], g, f"{name}/{lin.name} dW accumulated")
        G_flat_idx.append(offs[i] + n_idx * lin.k_in + k_idx)
        G_oracle.append(g)

    idx = np.concatenate(G_flat_idx)
    g = np.concatenate(G_oracle)
    if wl.shards > 1:
        shards = [g] + [orc.grad_accum(g, host.shard_noise[s][idx]) for s in range(1, wl.shards)]
        g = orc.running_sum(shards)
        G.assert_bits_equal(G.host(hp.G2)[idx], g, f"{name} level-2 running sum")
    if wl.replicas > 1:
        parts = [g] + [orc.grad_accum(g, host.noise[r][idx]) for r in range(1, wl.replicas)]
        G.assert_bits_equal(G.host(hp.TF)[idx], orc.treefold(parts), f"{name} TreeFold")


def test_repeat_and_stream_determinism():
    # the same step twice, and on a side stream, gives identical bytes
    wl = inputs.WORKLOADS["attn_out"]
    hp = S.HotPathStep(wl)
    st = torch.cuda.current_stream()
    hp.run(st)
    torch.cuda.synchronize()
    ref = [G.host(t).copy() for t in (hp.Y[0], hp.dX[0], hp.G)]
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        hp.run(side)
    side.synchronize()
    for got, exp, what in zip([G.host(t) for t in (hp.Y[0], hp.dX[0], hp.G)], ref,
                              ["Y", "dX", "dW"]):
        G.assert_bits_equal(got, exp, f"repeat {what}")
