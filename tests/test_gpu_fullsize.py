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


def _band_rows(total, width):
    return np.concatenate([np.arange(width), np.arange(total - width, total)]).astype(np.int64)


@pytest.mark.parametrize("name", ["gate_up", "down_accum"])
def test_fullsize_whole_tile_bands(orc, name):
    # every element of whole tile bands at the full sizes: the first and last
    # 128-row bands of Y and dX (every column: the forward's and dX kernel's
    # first and last tile rows), and the first and last 64-column bands of
    # the accumulated dW (every row: the dW kernel's first and last tile
    # columns, across every reduction segment)
    R.repro_set_launch_cfg(reset=True)
    wl = inputs.WORKLOADS[name]
    host = S.generate_host_inputs(wl)
    hp = S.HotPathStep(wl, host)
    hp.run(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert R.repro_device_check() == 0
    lin, J, M = wl.linears[0], wl.microbatches, wl.tokens
    W = host.W[0]
    s_w = orc.wscale(W, 0)
    wq = orc.quant_i8(W, s_w)
    rows = _band_rows(M, 128)
    cols = _band_rows(lin.k_in, 64)
    # dW bands: every row n, columns in the two bands, accumulated over J
    n_all = np.repeat(np.arange(lin.n_out, dtype=np.int64), cols.size)
    k_all = np.tile(cols, lin.n_out)
    g = None
    for j in range(J):
        X, dY = host.X[0][j], host.dY[0][j]
        s_x = orc.wscale(X, 1)
        xq = orc.quant_i8(X, s_x)
        dw = orc.linear_bwd_dw_at(dY, xq, s_x, n_all, k_all)
        g = dw if g is None else orc.grad_accum(g, dw)
    G.assert_bits_equal(G.host(hp.Gv[0])[:, cols].ravel(), g, f"{name} dW column bands")
    # Y and dX bands of the last micro-batch (still resident)
    m_y = np.repeat(rows, lin.n_out)
    c_y = np.tile(np.arange(lin.n_out, dtype=np.int64), rows.size)
    G.assert_bits_equal(G.host(hp.Y[0])[rows].ravel(),
                        orc.linear_fwd_at(xq, wq, s_x, s_w, m_y, c_y), f"{name} Y row bands")
    m_x = np.repeat(rows, lin.k_in)
    c_x = np.tile(np.arange(lin.k_in, dtype=np.int64), rows.size)
    G.assert_bits_equal(G.host(hp.dX[0])[rows].ravel(),
                        orc.linear_bwd_dx_at(dY, wq, s_w, m_x, c_x), f"{name} dX row bands")


def test_block_steps_repeat_bit_for_bit():
    # the benchmark's own set-up (dW on its second stream, fused accumulation,
    # TreeFold over six replicas): two steps give the same TreeFold bytes
    R.repro_set_launch_cfg(reset=True)
    wl = inputs.WORKLOADS["block"]
    hp = S.HotPathStep(wl)
    assert hp.s_dw is not None
    st = torch.cuda.Stream()
    hp.prepare(st)
    hp.run(st)
    st.synchronize()
    first = G.host(hp.TF).copy()
    hp.run(st)
    st.synchronize()
    assert R.repro_device_check() == 0
    G.assert_bits_equal(G.host(hp.TF), first, "block TreeFold, second step")
