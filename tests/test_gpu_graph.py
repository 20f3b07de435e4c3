"""CUDA-graph capture.  Every call of the library only enqueues on the caller's
stream, allocates nothing and never synchronises, so a whole step (scales,
quantisation, forward, backward with fused accumulation, level-2 running sum,
TreeFold) and the attention forward + backward capture into one CUDA graph.
Replays must write the same bits as the eager calls, every time, into outputs
that were wiped before each replay."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import gpu_helpers as G  # noqa: E402
import bitwise_reproducible_int8_gb300 as R  # noqa: E402
from bitwise_reproducible_int8_gb300 import inputs  # noqa: E402
from bitwise_reproducible_int8_gb300 import step as S  # noqa: E402


def _bits(t):
    a = t.detach().cpu().numpy()
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint8).copy()


def _wipe(ts):
    for t in ts:
        if t.dtype == torch.float32:
            t.fill_(float("nan"))
        else:
            t.fill_(0x55)
    torch.cuda.synchronize()   # the fills run on the default stream, the replays on their own


# the tiny workload (64 tokens, TreeFold over 4) and a mid-size one with two
# micro-batches (accumulation in the dW epilogue), two shards and a dW
# reduction of 64 chunks
MID = inputs.Workload("graph_mid", 4096, (inputs.Linear("a", 512, 256), inputs.Linear("b", 256, 768)),
                      2, 3, 40, 50, "graph capture case", 2)


@pytest.mark.parametrize("wl,dw_stream", [(inputs.WORKLOADS["tiny"], False), (MID, False),
                                          (MID, True)], ids=["tiny", "mid", "mid-two-streams"])
def test_step_graph_replays_match_eager(wl, dw_stream):
    st = torch.cuda.Stream()
    hp = S.HotPathStep(wl, dw_stream=dw_stream)
    with torch.cuda.stream(st):
        if wl.replicas > 1 or wl.shards > 1:
            hp.prepare(st)
        hp.run(st)
    st.synchronize()
    outs = [hp.result(), hp.G] + hp.Y + hp.dX + hp.Wq + hp.Xq + [hp.s_w, hp.s_x]
    eager = [_bits(t) for t in outs]
    g = hp.capture(st)
    for _ in range(2):
        _wipe(outs)
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        for i, (t, e) in enumerate(zip(outs, eager)):
            assert np.array_equal(_bits(t), e), f"output {i} differs after a graph replay"
    assert R.repro_device_check(st) == R.REPRO_OK


def test_step_with_optimizer_refuses_capture():
    wl = inputs.Workload("opt", 64, (inputs.Linear("o", 128, 256),), 1, 2, 0, 0, "", 1, True)
    hp = S.HotPathStep(wl)
    with pytest.raises(RuntimeError):
        hp.capture(torch.cuda.Stream())


@pytest.mark.parametrize("W", [0, 64])
def test_attention_graph_replays_match_eager(W):
    aw = inputs.ATTN_WORKLOADS["attn_tiny"]
    q, k, v, do = (G.dev(a) for a in inputs.attn_inputs(aw))
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    s_v = torch.zeros(1, dtype=torch.float32, device="cuda")
    vq = torch.empty(v.shape, dtype=torch.int8, device="cuda")
    o = torch.empty_like(q)
    m = torch.empty((B, T, Hq), device="cuda")
    l = torch.empty((B, T, Hq), device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    ws_s = torch.empty(max(R.repro_wscale_ws_bytes(v.numel()), 16), dtype=torch.uint8,
                       device="cuda")
    ws_f = torch.empty(max(R.repro_attn_fwd_ws_bytes(B, T, Hq, W), 16), dtype=torch.uint8,
                       device="cuda")
    ws_b = torch.empty(max(R.repro_attn_bwd_ws_bytes(B, T, Hq, W), 16), dtype=torch.uint8,
                       device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()

    def run():
        R.repro_wscale(v, R.REPRO_SCALE_ACT_AMAX, s_v, ws=ws_s, stream=st)
        R.repro_quant_i8(v, s_v, vq, stream=st)
        R.repro_attn_fwd(q, k, vq, s_v, o, m, l, W, ws=ws_f, stream=st)
        R.repro_attn_bwd(q, k, vq, s_v, o, do, m, l, dq, dk, dv, W, ws=ws_b, fwd_ws=ws_f,
                         stream=st)

    with torch.cuda.stream(st):
        run()
    st.synchronize()
    outs = [s_v, vq, o, m, l, dq, dk, dv]
    eager = [_bits(t) for t in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        run()
    for _ in range(2):
        _wipe(outs)
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        for i, (t, e) in enumerate(zip(outs, eager)):
            assert np.array_equal(_bits(t), e), f"attention output {i} differs after a replay"
    assert R.repro_device_check(st) == R.REPRO_OK


def test_overlapped_input_refill_keeps_bits():
    # the end-to-end pattern: each step's inputs are copied from pinned host
    # memory on a copy stream, each buffer refilled as soon as the previous step
    # has last read it (run()'s done events); every step's result must be the
    # device-resident step's, bit for bit
    wl = MID
    st, cp = torch.cuda.Stream(), torch.cuda.Stream()
    hp = S.HotPathStep(wl, dw_stream=True)   # inputs read on both streams
    with torch.cuda.stream(st):
        hp.prepare(st)
        hp.run(st)
    st.synchronize()
    expect = _bits(hp.result())
    L, J = len(wl.linears), wl.microbatches
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    hX = [[pin(hp.host.X[i][j]) for j in range(J)] for i in range(L)]
    hdY = [[pin(hp.host.dY[i][j]) for j in range(J)] for i in range(L)]
    hW = [pin(hp.host.W[i]) for i in range(L)]
    out = torch.empty(hp.result().shape, dtype=torch.float32, pin_memory=True)
    for t in hp.X[0] + hp.X[1] + hp.dY[0] + hp.dY[1] + hp.W:
        t.fill_(float("nan"))   # every input must come from the copies
    torch.cuda.synchronize()
    prev = None
    for _ in range(3):
        done = [None] * (J + 1)
        evs = []
        with torch.cuda.stream(cp):
            if prev is None:
                cp.wait_stream(st)
            else:
                for ev in prev[J]:
                    cp.wait_event(ev)
            for i in range(L):
                hp.W[i].copy_(hW[i], non_blocking=True)
            for j in range(J):
                if prev is not None:
                    for ev in prev[j]:
                        cp.wait_event(ev)
                for i in range(L):
                    hp.X[i][j].copy_(hX[i][j], non_blocking=True)
                    hp.dY[i][j].copy_(hdY[i][j], non_blocking=True)
                e = torch.cuda.Event()
                e.record(cp)
                evs.append(e)
        hp.run(st, wait_events=evs, done_events=done)
        prev = done
        with torch.cuda.stream(st):
            out.copy_(hp.result(), non_blocking=True)
        st.synchronize()
        assert np.array_equal(out.numpy().view(np.uint32), expect)
    assert R.repro_device_check(st) == R.REPRO_OK


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "unfused"])
def test_dw_stream_matches_one_stream(fused):
    # dW on its own stream (concurrent with the forward and dX) and dW after dX
    # on the one stream give the same bits
    outs = []
    for dw_stream in (True, False):
        hp = S.HotPathStep(MID, fused_accum=fused, dw_stream=dw_stream)
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            hp.prepare(st)
            hp.run(st)
            hp.run(st)
        st.synchronize()
        outs.append([_bits(t) for t in [hp.result(), hp.G] + hp.dX + hp.Y])
        assert R.repro_device_check(st) == R.REPRO_OK
    for i, (a, b) in enumerate(zip(*outs)):
        assert np.array_equal(a, b), f"output {i} differs between one and two streams"
